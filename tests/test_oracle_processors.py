"""Pins of the oracle's logits processors and stop tokens (banned tokens,
repetition penalty, stop on the committed prefix)."""
import numpy as np

import oracle
import workloads
from conftest import hand_workload, load_golden


def _rows(spec):
    return np.array([[float(x) for x in r.split()] for r in " ".join(spec).split("|")], np.float32)


def _greedy(rows, drafts, **proc):
    G = len(drafts)
    w = hand_workload(rows, None, drafts, entry="logits", u=np.zeros(G), E=np.ones((1, rows.shape[1])),
                      temperature=[0.0])
    w.update(proc)
    return oracle.verify(w, with_diag=False)


def _lists(ids):
    ids = np.asarray(ids, np.int32)
    return np.array([len(ids)], np.int64), ids


def test_greedy_golden_cases():
    g = load_golden("processors_examples.txt")
    for c in ("g1", "g2", "g3", "g5"):
        rows = _rows(g[f"{c}_rows"])
        drafts = [int(x) for x in g[f"{c}_drafts"]]
        proc = {"repetition_penalty": np.array([float(g[f"{c}_theta"][0])], np.float32)}
        proc["penalty_cu"], proc["penalty_ids"] = _lists([int(x) for x in g[f"{c}_context"]])
        if f"{c}_banned" in g:
            proc["banned_cu"], proc["banned_ids"] = _lists([int(x) for x in g[f"{c}_banned"]])
        o = _greedy(rows, drafts, **proc)
        expect = [int(x) for x in g[f"{c}_expect"]]
        n = o["num_accepted"][0] + 1
        assert list(o["out_tokens"][0, :n]) == expect, c
        assert o["status"] == 0


def test_golden_g1_commit_length():
    g = load_golden("processors_examples.txt")
    rows = _rows(g["g1_rows"])
    proc = {"repetition_penalty": np.array([2.0], np.float32)}
    proc["penalty_cu"], proc["penalty_ids"] = _lists([0, 2])
    o = _greedy(rows, [1, 1], **proc)
    assert o["num_accepted"][0] == 1 and list(o["out_tokens"][0]) == [1, 0, -1]


def test_penalty_without_context_list():
    """g1's rows with theta 2 and no context list: position 0 is unprocessed
    ([2.0 1.5 -1.0] -> argmax 0 != y0 = 1)... so take y0 = 0: accepted, then
    position 1 penalises y0: [1.0 1.5 -1.0] -> argmax 1."""
    g = load_golden("processors_examples.txt")
    rows = _rows(g["g1_rows"])
    o = _greedy(rows, [0, 0], repetition_penalty=np.array([2.0], np.float32))
    assert o["num_accepted"][0] == 1 and list(o["out_tokens"][0, :2]) == [0, 1]


def test_stop_token_truncates_commit_and_rollback():
    g = load_golden("processors_examples.txt")
    drafts = [int(x) for x in g["g4_drafts"]]
    am = [int(x) for x in g["g4_argmax"]]
    V = 10
    rows = np.zeros((len(am), V), np.float32)
    rows[np.arange(len(am)), am] = 3.0
    w = hand_workload(rows, None, drafts, entry="logits", u=np.zeros(3), E=np.ones((1, V)), temperature=[0.0],
                      ncomp=[100], slots=np.arange(4, dtype=np.int64))
    o = oracle.verify(w, with_diag=False)
    assert o["num_accepted"][0] == 3 and o["num_computed_tokens"][0] == 100
    w["stop_cu"], w["stop_ids"] = _lists([int(x) for x in g["g4_stop"]])
    o = oracle.verify(w, with_diag=False)
    A = int(g["g4_A"][0])
    assert o["num_accepted"][0] == A
    assert list(o["out_tokens"][0]) == [int(x) for x in g["g4_expect"]] + [-1] * (3 - A)
    assert o["num_computed_tokens"][0] == 100 - (3 - A)  # rollback of the verify tokens after the stop
    assert list(o["slot_mapping"]) == [0, 1, -1, -1]
    w["stop_ids"] = np.array([7], np.int32)  # the bonus itself: nothing changes
    assert oracle.verify(w, with_diag=False)["num_accepted"][0] == 3
    w["stop_ids"] = np.array([4], np.int32)  # the first token: A = 0
    assert oracle.verify(w, with_diag=False)["num_accepted"][0] == 0


def test_identical_processing_of_target_and_draft():
    """y = 0 penalised on both sides: p' = q', so any u < 1 accepts; a draft
    side left unprocessed would give p'(0)/q(0) = 0.667 and reject u = 0.9."""
    t = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 0.0]], np.float32)
    d = np.array([[1.0, 0.0, 0.0]], np.float32)
    w = hand_workload(t, d, [0], entry="logits", u=[0.9], E=np.ones((1, 3)), temperature=[1.0])
    w["repetition_penalty"] = np.array([4.0], np.float32)
    w["penalty_cu"], w["penalty_ids"] = _lists([0])
    o = oracle.verify(w, with_diag=False)
    assert o["num_accepted"][0] == 1
    np.testing.assert_allclose(o["dbg_py"][0], o["dbg_qy"][0], rtol=0, atol=0)


def test_theta_one_and_empty_lists_change_nothing():
    w = workloads.make("fused", N=6, V=3000, seed=12)
    base = oracle.verify(w, with_diag=False)
    w2 = dict(w)
    w2["repetition_penalty"] = np.ones(6, np.float32)
    w2["penalty_cu"] = np.arange(1, 7, dtype=np.int64) * 50
    w2["penalty_ids"] = np.random.default_rng(0).integers(0, 3000, size=300).astype(np.int32)
    w2["banned_cu"] = np.zeros(6, np.int64)
    w2["banned_ids"] = np.zeros(0, np.int32)
    o = oracle.verify(w2, with_diag=False)
    for k in ("out_tokens", "num_accepted"):
        np.testing.assert_array_equal(o[k], base[k])


def test_bf16_rounding_of_penalised_logits():
    """bf16 row [1.0, 0.333984375]: token 0 penalised by theta 3 gives
    fp32 0.3333333, rounded to bf16 0.333984375 -- a tie, lowest index wins
    (without the rounding token 1 would win)."""
    vals = np.array([[1.0, 0.333984375, -8.0], [0.0, 0.0, 0.0]], np.float32)
    bits = workloads._to_bf16_bits(vals)
    assert workloads.bf16_bits_to_f32(bits)[0, 1] == np.float32(0.333984375)
    w = hand_workload(bits, None, [0], entry="logits", dtype="bf16", u=[0.0], E=np.ones((1, 3)),
                      temperature=[0.0])
    w["repetition_penalty"] = np.array([3.0], np.float32)
    w["penalty_cu"], w["penalty_ids"] = _lists([0])
    o = oracle.verify(w, with_diag=False)
    assert o["out_tokens"][0, 0] == 0


def test_bad_lists_and_theta():
    t = np.zeros((2, 4), np.float32)
    w = hand_workload(t, None, [0], entry="logits", u=[0.0], E=np.ones((1, 4)), temperature=[0.0])
    w["stop_cu"], w["stop_ids"] = np.array([3], np.int64), np.array([1], np.int32)  # runs past the end
    o = oracle.verify(w, with_diag=False)
    assert o["status"] == oracle.BAD_LIST and o["num_accepted"][0] == 0
    w = hand_workload(t, None, [0], entry="logits", u=[0.0], E=np.ones((1, 4)), temperature=[0.0])
    w["repetition_penalty"] = np.array([0.0], np.float32)
    w["penalty_cu"], w["penalty_ids"] = _lists([1])
    assert oracle.verify(w, with_diag=False)["status"] == oracle.BAD_PARAM


# ----------------------------------------------------------------------------
# the order: temperature, top-k, top-p on the raw row, then the processors
# ----------------------------------------------------------------------------
def _case_lists(g, c):
    kw = {}
    if f"{c}_banned" in g:
        kw["banned_cu"], kw["banned_ids"] = _lists([int(x) for x in g[f"{c}_banned"]])
    if f"{c}_theta" in g:
        kw["repetition_penalty"] = np.array([float(g[f"{c}_theta"][0])], np.float32)
        kw["penalty_cu"], kw["penalty_ids"] = _lists([int(x) for x in g[f"{c}_context"]])
    return kw


def test_order_golden_sampler_rows():
    """The draft-side sampler's transformed rows on the hand-worked cases t1-t5
    (each separates the pages' order from processors-first)."""
    g = load_golden("processors_order_examples.txt")
    for c in ("t1", "t2", "t3", "t4", "t5"):
        row = np.array([[float(x) for x in g[f"{c}_row"]]], np.float32)
        V = row.shape[1]
        s = oracle.sample_rows(row, temperature=[float(g[f"{c}_temp"][0])], top_k=[int(g[f"{c}_topk"][0])],
                               top_p=[float(g[f"{c}_topp"][0])], exponentials=np.ones((1, V)), **_case_lists(g, c))
        if f"{c}_status" in g:
            assert s["status"] == int(g[f"{c}_status"][0]) and s["tokens"][0] == -1, c
            continue
        assert s["status"] == 0, c
        expect = np.array([float(x) for x in g[f"{c}_expect"]], np.float32)
        np.testing.assert_allclose(s["probs"][0], expect, rtol=0, atol=1e-7, err_msg=c)


def test_order_golden_verifier_rows():
    """The same cases through the verifier: the target and draft rows of one
    position are the case's row, and the draft id walks over the vocabulary,
    so dbg_py/dbg_qy read the whole transformed row back."""
    g = load_golden("processors_order_examples.txt")
    for c in ("t1", "t2", "t3", "t4", "t5"):
        row = np.array([float(x) for x in g[f"{c}_row"]], np.float32)
        V = row.shape[0]
        for y in range(V):
            t = np.stack([row, np.zeros(V, np.float32)])
            w = hand_workload(t, row[None, :], [y], entry="logits", u=[0.5], E=np.ones((1, V)),
                              temperature=[float(g[f"{c}_temp"][0])], top_k=[int(g[f"{c}_topk"][0])],
                              top_p=[float(g[f"{c}_topp"][0])])
            w.update(_case_lists(g, c))
            o = oracle.verify(w, with_diag=False)
            if f"{c}_status" in g:
                assert o["status"] == int(g[f"{c}_status"][0]) and o["num_accepted"][0] == 0, c
                assert list(o["out_tokens"][0]) == [-1, -1], c
                continue
            exp_y = float(g[f"{c}_expect"][y])
            assert abs(o["dbg_py"][0] - exp_y) <= 1e-7 and abs(o["dbg_qy"][0] - exp_y) <= 1e-7, (c, y)


def test_order_golden_commit():
    """v1: the commit itself differs between the two orders."""
    g = load_golden("processors_order_examples.txt")
    t = _rows(g["v1_target"])
    d = _rows(g["v1_draft"])
    w = hand_workload(t, d, [int(x) for x in g["v1_drafts"]], entry="logits", u=[float(g["v1_u"][0])],
                      E=np.ones((1, t.shape[1])), temperature=[1.0], top_k=[int(g["v1_topk"][0])], top_p=[1.0])
    w["banned_cu"], w["banned_ids"] = _lists([int(x) for x in g["v1_banned"]])
    o = oracle.verify(w, with_diag=False)
    assert o["status"] == 0
    assert o["num_accepted"][0] == int(g["v1_A"][0])
    assert list(o["out_tokens"][0]) == [int(x) for x in g["v1_expect"]]
    assert o["dbg_py"][0] == float(g["v1_py"][0]) and o["dbg_qy"][0] == float(g["v1_qy"][0])


def test_order_golden_sampler_token():
    g = load_golden("processors_order_examples.txt")
    row = np.array([[float(x) for x in g["s1_row"]]], np.float32)
    for E in (np.ones((1, 4)), np.array([[1.0, 5.0, 0.01, 1.0]])):
        s = oracle.sample_rows(row, temperature=[1.0], top_k=[2], exponentials=E, banned_cu=[1],
                               banned_ids=np.array([0], np.int32))
        assert s["tokens"][0] == int(g["s1_token"][0]) and s["status"] == 0
        np.testing.assert_array_equal(s["probs"][0], np.array([float(x) for x in g["s1_expect"]], np.float32))


def test_transform_row_without_processors_matches_plain_transform():
    """The processed-row entry with no processed row is the plain transform,
    and a processed row equal to the raw row changes nothing."""
    rng = np.random.default_rng(4)
    for _ in range(20):
        l = (rng.standard_normal(300) * 2).astype(np.float32)
        k, tp, T = int(rng.integers(0, 60)), float(rng.uniform(0.2, 1.0)), float(rng.uniform(0.3, 2))
        a, ea, ra = oracle.logits_to_probs(l, T, k, tp)
        b, eb, rb = oracle.transform_row(l, None, T, k, tp)
        c, ec, rc = oracle.transform_row(l, l.copy(), T, k, tp)
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(a, c)
        assert ra == rb == rc == 0 and ea == eb == ec


def test_planted_mistakes_are_caught(oracle_mod, tmp_path):
    import ctypes  # noqa: F401
    import subprocess
    src = oracle_mod._SRC.read_text()
    tests = (test_greedy_golden_cases, test_golden_g1_commit_length, test_penalty_without_context_list,
             test_stop_token_truncates_commit_and_rollback,
             test_identical_processing_of_target_and_draft, test_bf16_rounding_of_penalised_logits,
             test_order_golden_sampler_rows, test_order_golden_verifier_rows, test_order_golden_commit,
             test_order_golden_sampler_token)
    mutants = {
        "drafts not in the set": ("for (int k = 0; k < nextra; ++k) {", "for (int k = 0; k < nextra - 1; ++k) {"),
        "penalty overrides ban": ("      if (x >= 0 && x < V && !mark[x]) mark[x] = 2;\n    }\n    for (int k = 0; k < nextra",
                                  "      if (x >= 0 && x < V) mark[x] = 2;\n    }\n    for (int k = 0; k < nextra"),
        "drafts only with a context list": ("a->penalty_ids, pb, pe, a->draft_ids + s, j);",
                                            "a->penalty_ids, pb, pe, a->draft_ids + s, a->penalty_cu ? j : 0);"),
        "no bf16 rounding": ("row[x] = dtype == ORC_BF16 ? round_to_bf16(v) : v;", "row[x] = v;"),
        "penalty branches swapped": ("float v = row[x] > 0.0f ? row[x] / *theta : row[x] * *theta;",
                                     "float v = row[x] > 0.0f ? row[x] * *theta : row[x] / *theta;"),
        "penalty always divides": ("float v = row[x] > 0.0f ? row[x] / *theta : row[x] * *theta;",
                                   "float v = row[x] / *theta;"),
        "stop off by one": ("        A = m;\n        break;", "        A = m > 0 ? m - 1 : 0;\n        break;"),
        "draft side unprocessed": ("  if (has_processors(a)) {\n    memcpy(proc",
                                   "  if (has_processors(a) && is_target) {\n    memcpy(proc"),
        "verifier: processors before the cuts": ("int rc = oracle_transform_row(tmp, lp, a->vocab_size",
                                                 "int rc = oracle_transform_row(lp ? lp : tmp, lp, a->vocab_size"),
        "sampler: processors before the cuts": (
            "oracle_transform_row(l, (banned_cu || repetition_penalty) ? lp : NULL,",
            "oracle_transform_row((banned_cu || repetition_penalty) ? lp : l, (banned_cu || repetition_penalty) ? lp : NULL,"),
        "processed values ignored": ("const float *v = lp ? lp : l;", "const float *v = l;"),
        "all-banned kept set not flagged": ("if (m2 == -INFINITY) return ORC_BAD_VALUES;", "if (m2 == -INFINITY) m2 = 0;"),
    }
    for name, (old, new) in mutants.items():
        assert src.count(old) == 1, name
        msrc = tmp_path / f"p_{abs(hash(name))}.c"
        msrc.write_text(src.replace(old, new, 1))
        so = tmp_path / f"p_{abs(hash(name))}.so"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so),
                        str(msrc), "-lm"], check=True)
        saved, orig_build = oracle_mod._LIB, oracle_mod.build
        try:
            oracle_mod._LIB = None
            oracle_mod.build = lambda force=False, _so=so: _so
            caught = False
            for t in tests:
                try:
                    t()
                except AssertionError:
                    caught = True
                    break
        finally:
            oracle_mod.build, oracle_mod._LIB = orig_build, saved
        assert caught, name


def test_sampler_applies_the_same_processors():
    """The draft-side sampler's probability row under processors equals the
    verifier's q row at the same position (identical transforms on q), and a
    banned argmax is never drafted greedily."""
    rng = np.random.default_rng(3)
    V = 40
    d = rng.standard_normal((1, V)).astype(np.float32) * 2
    t = rng.standard_normal((2, V)).astype(np.float32) * 2
    ctx = np.array([int(np.argmax(d[0])), 7, 7, 3], np.int32)
    ban = np.array([11, 12], np.int32)
    s = oracle.sample_rows(d, temperature=[0.9], top_k=[10], top_p=[0.95], exponentials=np.ones((1, V)),
                           repetition_penalty=[1.7], penalty_cu=[len(ctx)], penalty_ids=ctx, banned_cu=[2],
                           banned_ids=ban)
    assert s["status"] == 0
    y = int(s["tokens"][0])
    w = hand_workload(t, d, [y], entry="logits", u=[0.999999], E=np.ones((1, V)), temperature=[0.9],
                      top_k=[10], top_p=[0.95])
    w["repetition_penalty"] = np.array([1.7], np.float32)
    w["penalty_cu"], w["penalty_ids"] = np.array([len(ctx)], np.int64), ctx
    w["banned_cu"], w["banned_ids"] = np.array([2], np.int64), ban
    o = oracle.verify(w)
    assert o["dbg_qy"][0] == s["probs"][0, y]
    assert np.all(s["probs"][0, ban] == 0)
    g = oracle.sample_rows(d, temperature=[0.0], banned_cu=[1], banned_ids=np.array([int(np.argmax(d[0]))],
                                                                                     np.int32))
    assert g["tokens"][0] != int(np.argmax(d[0]))
    bad = oracle.sample_rows(d, temperature=[0.9], banned_cu=[5], banned_ids=ban)
    assert bad["status"] == oracle.BAD_LIST and bad["tokens"][0] == -1
