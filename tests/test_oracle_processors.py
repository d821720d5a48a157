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


def test_planted_mistakes_are_caught(oracle_mod, tmp_path):
    import ctypes  # noqa: F401
    import subprocess
    src = oracle_mod._SRC.read_text()
    tests = (test_greedy_golden_cases, test_golden_g1_commit_length, test_penalty_without_context_list,
             test_stop_token_truncates_commit_and_rollback,
             test_identical_processing_of_target_and_draft, test_bf16_rounding_of_penalised_logits)
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
        "draft side unprocessed": ("load_row(base, a->dtype, row, stride, a->vocab_size, tmp);\n  process_row(a, i, s, j, tmp);",
                                   "load_row(base, a->dtype, row, stride, a->vocab_size, tmp);\n"
                                   "  if (is_target) process_row(a, i, s, j, tmp);"),
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
