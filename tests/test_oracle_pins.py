"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test names the passage it checks.  Nothing here compares the oracle with
itself: the expected values are the pages' worked examples (tests/golden),
hand-derived consequences of the pages' formulas, exact counts over a grid of
uniforms, published known-answer vectors, or a library routine for a special
case.
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

from conftest import hand_workload, load_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

U_GRID = ((np.arange(1000) + 0.5) / 1000).astype(np.float32)  # 1000 uniforms, one per 1/1000 bin


def _idx(vocab, names):
    return [vocab.index(n) for n in names]


# ----------------------------------------------------------------------------
# Philox4x32-10: known-answer vectors published with Random123 for the
# generator of Salmon et al., "Parallel random numbers: as easy as 1, 2, 3"
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("ctr,key,expect", [
    ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
    ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
    ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
])
def test_philox_known_answers(oracle_mod, ctr, key, expect):
    assert list(oracle_mod.philox4x32_10(ctr, key)) == expect


def test_production_draws_have_the_stated_laws(oracle_mod):
    """u ~ U[0,1) on the 2^-24 grid, E ~ Exp(1); Kolmogorov-Smirnov on 200000 draws
    over four seeds (many requests, positions and vocabulary entries)."""
    u = np.array([oracle_mod.uniform(s, 3, r, j) for s in range(4) for r in range(5000) for j in range(10)])
    E = np.array([oracle_mod.exponential(s, 3, r, x) for s in range(4) for r in range(500) for x in range(100)],
                 dtype=np.float64)
    assert u.min() >= 0 and u.max() < 1
    assert np.all(np.floor(u * 2 ** 24) == u * 2 ** 24)
    assert scipy.stats.kstest(u, "uniform").pvalue > 0.01
    assert E.min() > 0
    assert scipy.stats.kstest(E, "expon").pvalue > 0.01
    # u and E streams of one request differ, requests differ, offsets differ
    assert oracle_mod.uniform(1, 0, 0, 0) != oracle_mod.uniform(1, 0, 1, 0)
    assert oracle_mod.uniform(1, 0, 0, 0) != oracle_mod.uniform(1, 1, 0, 0)


# ----------------------------------------------------------------------------
# Page 2, section 05 / 07: the two-token worked example
# ----------------------------------------------------------------------------
def _two_token(u, E=(1.0, 1.0)):
    g = load_golden("two_token_worked_example.txt")
    V = g["vocab"]
    q = [float(x) for x in g["draft_probs"]]
    p0 = [float(x) for x in g["target_probs_row0"]]
    p1 = [float(x) for x in g["target_probs_row1"]]
    return g, hand_workload([p0, p1], [q], _idx(V, g["draft"]), u=[u], E=[E])


def test_worked_example_rejects_and_commits_A(oracle_mod):
    g, w = _two_token(float(g_u := load_golden("two_token_worked_example.txt")["uniform"][0]))
    V = g["vocab"]
    rng = np.random.default_rng(5)
    for E in [(1.0, 1.0), (0.01, 5.0), (5.0, 0.01)] + [tuple(rng.exponential(size=2)) for _ in range(20)]:
        w["exponentials"] = np.asarray([E], np.float32)
        r = oracle_mod.verify(w)
        assert r["out_tokens"].tolist() == [[V.index(g["expected_output"][0]), -1]]
        assert r["num_accepted"].tolist() == [0]
        assert r["status"] == 0


def test_worked_example_acceptance_probability_and_marginal(oracle_mod):
    """alpha(B) = 0.5; the first committed token has marginal (0.6, 0.4)."""
    g = load_golden("two_token_worked_example.txt")
    V = g["vocab"]
    q = np.array([float(x) for x in g["draft_probs"]])
    p0 = [float(x) for x in g["target_probs_row0"]]
    p1 = [float(x) for x in g["target_probs_row1"]]
    counts = np.zeros(2)
    for y in (0, 1):
        n = len(U_GRID)
        w = hand_workload([p0, p1] * n, [[q[0], q[1]]] * n, [y] * n, [1] * n,
                          u=U_GRID, E=np.ones((n, 2)))
        w["target"] = np.tile(np.array([p0, p1], np.float32), (n, 1))
        r = oracle_mod.verify(w)
        first = r["out_tokens"][:, 0]
        if y == V.index("B"):
            acc = (r["num_accepted"] == 1).mean()
            assert acc == pytest.approx(float(g["acceptance_probability"][0]), abs=0)
        counts += q[y] * np.bincount(first, minlength=2) / n
    assert counts == pytest.approx([float(x) for x in g["marginal"]], abs=1e-12)


def test_worked_example_accept_then_bonus(oracle_mod):
    """u=0.3 < 0.5 accepts B; the bonus comes from the last target row (0.3, 0.7)."""
    _, w = _two_token(0.3, (1.0, 1.0))
    r = oracle_mod.verify(w)
    assert r["out_tokens"].tolist() == [[1, 1]] and r["num_accepted"].tolist() == [1]
    w["exponentials"] = np.asarray([[0.1, 1.0]], np.float32)  # 0.3/0.1 = 3 > 0.7/1
    assert oracle_mod.verify(w)["out_tokens"].tolist() == [[1, 0]]


# ----------------------------------------------------------------------------
# Page 2, section 18 exercises (answers from section 04's formulas)
# ----------------------------------------------------------------------------
def test_exercise_acceptance_rate_and_residual(oracle_mod):
    g = load_golden("exercise_three_token.txt")
    q = [float(x) for x in g["draft_probs"]]
    p = [float(x) for x in g["target_probs"]]
    y = g["vocab"].index(g["draft"][0])
    n = len(U_GRID)
    w = hand_workload(np.tile(np.array([p, p], np.float32), (n, 1)), [q] * n, [y] * n, [1] * n,
                      u=U_GRID, E=np.ones((n, 3)))
    r = oracle_mod.verify(w)
    assert (r["num_accepted"] == 1).mean() == pytest.approx(float(g["acceptance_probability"][0]), abs=0)
    # residual distribution: force rejection (u=0.999) and draw many replacements
    m = 60000
    rng = np.random.default_rng(11)
    w = hand_workload(np.tile(np.array([p, p], np.float32), (m, 1)), [q] * m, [y] * m, [1] * m,
                      u=np.full(m, 0.999), E=rng.exponential(size=(m, 3)))
    r = oracle_mod.verify(w)
    assert np.all(r["num_accepted"] == 0)
    cnt = np.bincount(r["out_tokens"][:, 0], minlength=3)
    res = np.array([float(x) for x in g["residual_normalised"]])
    assert cnt[0] == 0  # (p - q)+ is 0 at A: never drawn back
    assert scipy.stats.chisquare(cnt[1:], m * res[1:]).pvalue > 0.01


def test_exercise_gamma4_reject_at_third(oracle_mod):
    """gamma=4, third candidate rejected: 3 tokens committed, KV rollback 2."""
    g = load_golden("exercise_three_token.txt")
    V = 3
    one = lambda k: [1.0 if x == k else 0.0 for x in range(V)]
    # rows 0,1 accept (p=q one-hot on the draft), row 2 rejects (p(y)=0), row 3 unused
    p = [one(0), one(1), one(2), one(0), one(1)]
    q = [one(0), one(1), one(0), one(0)]
    ids = [0, 1, 0, 0]
    w = hand_workload(p, q, ids, u=[0.5] * 4, E=[[1, 1, 1]], ncomp=[100], slots=[10, 11, 12, 13, 14])
    r = oracle_mod.verify(w)
    A = int(g["reject_at_candidate"][0]) - 1
    assert r["num_accepted"].tolist() == [A]
    assert (r["out_tokens"][0] >= 0).sum() == int(g["committed"][0])
    assert r["out_tokens"][0].tolist() == [0, 1, 2, -1, -1]
    assert 100 - r["num_computed_tokens"][0] == int(g["rollback"][0])
    assert r["slot_mapping"].tolist() == [10, 11, 12, -1, -1]


# ----------------------------------------------------------------------------
# Page 3, section 3.2: block-granular rollback
# ----------------------------------------------------------------------------
def test_kv_rollback_example(oracle_mod):
    g = load_golden("kv_rollback_example.txt")
    bs = int(g["block_size"][0])
    n0 = int(g["num_computed_tokens_before"][0])
    K = int(g["draft"][0])
    A = int(g["accepted"][0])
    V = 4
    one = lambda k: [1.0 if x == k else 0.0 for x in range(V)]
    ids = [1] * K
    q = [one(1)] * K
    p = [one(1)] * A + [one(2)] * (K + 1 - A)  # accept A drafts, reject the next
    block_table = np.arange(1000, 1000 + 64 + 1) * 7  # arbitrary physical block ids
    pos = np.arange(n0 - K - 1, n0)
    slots = block_table[pos // bs] * bs + pos % bs
    w = hand_workload(p, q, ids, u=[0.5] * K, E=[[1] * V], ncomp=[n0], slots=slots)
    r = oracle_mod.verify(w)
    n1 = int(r["num_computed_tokens"][0])
    assert r["num_accepted"][0] == A
    assert n1 == int(g["num_computed_tokens_after"][0])
    assert (n1 // bs, n1 % bs) == (int(g["block"][0]), int(g["offset"][0]))
    # slots of positions >= n1 are invalidated, the others kept
    kept = r["slot_mapping"] >= 0
    assert kept.tolist() == (pos < n1).tolist()
    assert np.array_equal(r["slot_mapping"][kept], slots[kept])


# ----------------------------------------------------------------------------
# Page 2, section 03 / page 1 "Greedy kernel": greedy verification
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("entry", ["probs", "logits_f32", "logits_bf16"])
def test_greedy_example(oracle_mod, entry):
    g = load_golden("greedy_example.txt")
    vocab = g["vocab"]
    V = len(vocab)
    draft = _idx(vocab, g["draft"])
    am = _idx(vocab, g["target_argmax"])
    rng = np.random.default_rng(3)
    rows = []
    for k in am:
        r = rng.uniform(0.0, 0.1, size=V)
        r[k] = 0.5
        rows.append(r / r.sum())
    rows = np.array(rows, np.float32)
    kw = dict(temperature=[0.0])
    if entry == "probs":
        target = rows
        w = hand_workload(target, None, draft, **kw)
    else:
        lg = np.log(rows.astype(np.float64))
        if entry == "logits_bf16":
            bits = (lg.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            w = hand_workload(bits, None, draft, entry="logits", dtype="bf16", **kw)
        else:
            w = hand_workload(lg.astype(np.float32), None, draft, entry="logits", **kw)
    w["uniforms"] = np.zeros(len(draft), np.float32)
    w["exponentials"] = np.ones((1, V), np.float32)
    r = oracle_mod.verify(w)
    assert r["out_tokens"][0].tolist() == _idx(vocab, g["expected_commit"]) + [-1, -1]
    assert r["num_accepted"].tolist() == [2]
    # all four match: gamma + 1 tokens, the last one the argmax of the 5th row
    w["draft_ids"] = np.array(am[:4], np.int32)
    r = oracle_mod.verify(w)
    assert (r["out_tokens"][0] >= 0).sum() == int(g["all_match_commit_count"][0])
    assert r["out_tokens"][0].tolist() == am


def test_greedy_lowest_index_tie(oracle_mod):
    p = [[0.1, 0.4, 0.4, 0.1], [0.25, 0.25, 0.25, 0.25]]
    w = hand_workload(p, None, [2], temperature=[0.0], u=[0], E=[[1] * 4])
    r = oracle_mod.verify(w)
    assert r["out_tokens"].tolist() == [[1, -1]]  # index 1 wins the 0.4 tie; y=2 mismatches
    w["draft_ids"] = np.array([1], np.int32)
    r = oracle_mod.verify(w)
    assert r["out_tokens"].tolist() == [[1, 0]]  # bonus: 4-way tie -> index 0


# ----------------------------------------------------------------------------
# Acceptance-test edge cases (page 2 sections 04/06; page 1 "Random kernel")
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("u,qy,py,accept", [
    (0.5, 0.5, 0.25, False),      # u*q == p exactly: strict '<' rejects
    (0.0, 0.9, 1e-30, True),      # u = 0 accepts whenever p(y) > 0
    (0.0, 0.9, 0.0, False),       # ... and rejects when p(y) = 0
    (0.7, 0.0, 0.3, True),        # q(y) = 0 < p(y): always accepted, no clamp needed
    (0.7, 0.0, 0.0, False),       # p = q = 0 at y: rejected
    (1 - 2 ** -24, 0.3, 0.3, True),  # p == q accepts for every u < 1
    (0.999, 0.8, 0.79, False),
])
def test_acceptance_edges(oracle_mod, u, qy, py, accept):
    V = 3
    p0 = np.array([py, 0.5 * (1 - py), 0.5 * (1 - py)], np.float32)
    q0 = np.array([qy, 0.5 * (1 - qy), 0.5 * (1 - qy)], np.float32)
    w = hand_workload([p0, [0.2, 0.3, 0.5]], [q0], [0], u=[u], E=[[1, 1, 1]])
    r = oracle_mod.verify(w)
    assert bool(r["num_accepted"][0] == 1) == accept


def test_equal_p_q_always_accepts(oracle_mod):
    rng = np.random.default_rng(0)
    V, n = 16, 1000
    rows = rng.dirichlet(np.ones(V), size=n).astype(np.float32)
    ids = np.array([rng.choice(V, p=r / r.sum()) for r in rows.astype(np.float64)], np.int32)
    target = np.empty((2 * n, V), np.float32)
    target[0::2] = rows
    target[1::2] = rows
    w = hand_workload(target, rows, ids, [1] * n, u=rng.random(n), E=rng.exponential(size=(n, V)))
    assert np.all(oracle_mod.verify(w)["num_accepted"] == 1)


def test_one_hot_target(oracle_mod):
    """p = e_k: accept iff y == k, and the replacement is k."""
    V = 5
    k = 3
    pk = [1.0 if x == k else 0.0 for x in range(V)]
    q = [0.2] * 5
    for y in range(V):
        w = hand_workload([pk, pk], [q], [y], u=[0.999], E=[[0.5, 2, 0.1, 3, 1]])
        r = oracle_mod.verify(w)
        assert r["num_accepted"][0] == (1 if y == k else 0)
        assert r["out_tokens"][0].tolist() == ([k, k] if y == k else [k, -1])


def test_race_ties_take_lowest_index(oracle_mod):
    # residual (0, 0.2, 0.2, 0.2) and E chosen so two keys tie exactly
    p = [0.1, 0.3, 0.3, 0.3]
    q = [0.7, 0.1, 0.1, 0.1]
    w = hand_workload([p, p], [q], [0], u=[0.99], E=[[1.0, 2.0, 0.5, 0.5]])
    assert oracle_mod.verify(w)["out_tokens"].tolist() == [[2, -1]]
    # +inf keys (tiny E) tie too: the lowest index still wins
    w["exponentials"] = np.array([[1.0, 1e-45, 1.0, 1e-45]], np.float32)
    assert oracle_mod.verify(w)["out_tokens"].tolist() == [[1, -1]]


def test_all_zero_residual_falls_back_to_p(oracle_mod):
    # p <= q everywhere (fp rounding corner), y rejected because u*q >= p
    q = np.array([0.25, 0.25, 0.25, 0.25], np.float32)
    p = (q * np.float32(0.999)).astype(np.float32)
    w = hand_workload([p, p], [q], [1], u=[0.9995], E=[[3.0, 1.0, 0.5, 2.0]])
    r = oracle_mod.verify(w)
    assert r["num_accepted"][0] == 0
    assert r["out_tokens"][0, 0] == 2  # argmax p/E = argmax 1/E -> index 2
    assert r["diag"][0, oracle_mod.DIAG_FALLBACK] == 1
    assert r["status"] == 0


def test_empty_distribution_status(oracle_mod):
    w = hand_workload([[0.0, 0.0, 0.0]], None, [], u=[], E=[[1, 1, 1]], temperature=[1.0])
    w["draft"] = np.zeros((0, 3), np.float32)
    r = oracle_mod.verify(w)
    assert r["out_tokens"].tolist() == [[0]]
    assert r["status"] == oracle_mod.EMPTY_DISTRIBUTION


def test_gamma_zero_request_gets_bonus(oracle_mod):
    p = [[0.1, 0.9, 0.0], [0.5, 0.5, 0.0], [0.0, 0.0, 1.0]]
    q = [[0.1, 0.9, 0.0]]
    w = hand_workload(p, q, [1], [0, 1], u=[0.5], E=[[1, 1, 1], [1, 1, 1]], ncomp=[7, 9], slots=[1, 2, 3])
    r = oracle_mod.verify(w)
    # request 0: gamma 0 -> bonus argmax(p/E) of its only row (index 1)
    # request 1: target rows 1..2; draft 1 accepted (p=0.5, u*q = 0.45), bonus from row 2 -> 2
    assert r["out_tokens"].tolist() == [[1, -1], [1, 2]]
    assert r["num_accepted"].tolist() == [0, 1]
    assert r["num_computed_tokens"].tolist() == [7, 9]
    assert r["slot_mapping"].tolist() == [1, 2, 3]


def test_ragged_row_indexing(oracle_mod):
    """Request i's target rows start at s_i + i (s_i = exclusive prefix sum of
    gamma), its draft rows at s_i (page 1, "SpecDecodeMetadata")."""
    V = 8
    one = lambda k: [1.0 if x == k else 0.0 for x in range(V)]
    gam = [2, 0, 3]
    # request 0: drafts (3, 4): accept 3, reject 4 -> replacement 6
    # request 1: no drafts: bonus 5
    # request 2: drafts (1, 2, 7): all accepted, bonus 0
    tgt = [one(3), one(6), one(1),  # req 0 rows (third unused)
           one(5),                  # req 1 row
           one(1), one(2), one(7), one(0)]  # req 2 rows
    drf = [one(3), one(4), one(1), one(2), one(7)]
    ids = [3, 4, 1, 2, 7]
    w = hand_workload(tgt, drf, ids, gam, u=[0.5] * 5, E=np.ones((3, V)),
                      ncomp=[50, 60, 70], slots=list(range(100, 108)))
    r = oracle_mod.verify(w)
    assert r["out_tokens"].tolist() == [[3, 6, -1, -1], [5, -1, -1, -1], [1, 2, 7, 0]]
    assert r["num_accepted"].tolist() == [1, 0, 3]
    assert r["num_computed_tokens"].tolist() == [49, 60, 70]
    assert r["slot_mapping"].tolist() == [100, 101, -1, 103, 104, 105, 106, 107]


def test_batch_has_no_cross_talk(oracle_mod):
    """Page 2 section 14: one all-accept and one first-position reject in a batch
    give the same results as when run alone."""
    import workloads
    w = workloads.make("tiny", seed=9)
    full = oracle_mod.verify(w)
    for i in range(w["N"]):
        sub = dict(w)
        G = w["gamma"]
        sub.update(N=1, T=G, draft_ids=w["draft_ids"][i * G:(i + 1) * G],
                   target=w["target"][i * (G + 1):(i + 1) * (G + 1)], draft=w["draft"][i * G:(i + 1) * G],
                   temperature=w["temperature"][i:i + 1], uniforms=w["uniforms"][i * G:(i + 1) * G],
                   exponentials=w["exponentials"][i:i + 1], num_computed_tokens=w["num_computed_tokens"][i:i + 1],
                   slot_mapping=w["slot_mapping"][i * (G + 1):(i + 1) * (G + 1)])
        one = oracle_mod.verify(sub)
        assert one["out_tokens"][0].tolist() == full["out_tokens"][i].tolist()
        assert one["num_computed_tokens"][0] == full["num_computed_tokens"][i]


# ----------------------------------------------------------------------------
# invariants on seeded workloads (page 2 sections 09 and 13)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("name,kw", [("tiny", {}), ("random", dict(N=16, V=4099)),
                                     ("ragged", dict(N=24, V=3001)), ("fused", dict(N=8, V=2048))])
def test_invariants(oracle_mod, name, kw):
    import workloads
    w = workloads.make(name, **kw)
    r = oracle_mod.verify(w)
    gam = workloads.gammas_of(w)
    A = r["num_accepted"]
    out = r["out_tokens"]
    assert r["status"] == 0
    s = 0
    for i in range(w["N"]):
        g = int(gam[i])
        committed = (out[i] >= 0).sum()
        assert 1 <= committed == A[i] + 1 <= g + 1  # S = A + 1
        assert np.all(out[i, :A[i] + 1] >= 0) and np.all(out[i, A[i] + 1:] == -1)
        assert out[i, :A[i]].tolist() == w["draft_ids"][s:s + A[i]].tolist()
        dec = w["num_computed_tokens"][i] - r["num_computed_tokens"][i]
        nslots = (r["slot_mapping"][s + i:s + i + g + 1] == -1).sum()
        assert dec == nslots == g - A[i]
        if A[i] < g and r["diag"][i, oracle_mod.DIAG_PATH] == 0 and r["diag"][i, oracle_mod.DIAG_FALLBACK] == 0:
            assert out[i, A[i]] != w["draft_ids"][s + A[i]]  # replacement != rejected draft
        s += g


# ----------------------------------------------------------------------------
# data errors: the request emits nothing and a status bit is raised
# ----------------------------------------------------------------------------
def test_status_bits_and_invalid_requests(oracle_mod):
    p = [[0.5, 0.5], [0.5, 0.5], [0.5, 0.5], [0.5, 0.5]]
    q = [[0.5, 0.5], [0.5, 0.5]]
    base = dict(u=[0.1, 0.1], E=[[1, 1], [1, 1]], ncomp=[10, 10], slots=[1, 2, 3, 4])
    # draft id out of range at an examined position
    r = oracle_mod.verify(hand_workload(p, q, [0, 5], [1, 1], **base))
    assert r["status"] == oracle_mod.BAD_DRAFT_ID
    assert r["out_tokens"].tolist() == [[0, 0], [-1, -1]] or r["out_tokens"][1].tolist() == [-1, -1]
    assert r["num_accepted"][1] == 0 and r["num_computed_tokens"][1] == 10
    # bad cu (decreasing)
    w = hand_workload(p, q, [0, 1], [1, 1], **base)
    w["cu_num_draft_tokens"] = np.array([2, 1], np.int32)
    r = oracle_mod.verify(w)
    assert r["status"] & oracle_mod.BAD_CU and r["out_tokens"][1].tolist() == [-1, -1]
    # negative temperature
    r = oracle_mod.verify(hand_workload(p, q, [0, 1], [1, 1], temperature=[1.0, -1.0], **base))
    assert r["status"] == oracle_mod.BAD_PARAM and r["out_tokens"][1].tolist() == [-1, -1]
    # bad exponential where a key is needed: key 0, status raised, output defined
    w = hand_workload([[0.9, 0.1], [0.5, 0.5]], [[0.1, 0.9]], [1], u=[0.99], E=[[-1.0, 1.0]])
    r = oracle_mod.verify(w)
    assert r["status"] & oracle_mod.BAD_EXPONENTIAL
    # draft rows missing for a random request
    w = hand_workload(p[:2], None, [0], u=[0.1], E=[[1, 1]])
    r = oracle_mod.verify(w)
    assert r["status"] == oracle_mod.MISSING_DRAFT and r["out_tokens"].tolist() == [[-1, -1]]
    # a bad id after the first rejection is never examined
    pr = [[1.0, 0.0], [0.5, 0.5], [0.5, 0.5]]
    r = oracle_mod.verify(hand_workload(pr, [[0.0, 1.0], [0.5, 0.5]], [1, 9], u=[0.5, 0.5], E=[[1, 1]]))
    assert r["status"] == 0 and r["out_tokens"].tolist() == [[0, -1, -1]]


def test_subnormal_temperature_is_a_bad_parameter(oracle_mod):
    """Reading: a temperature in (0, FLT_MIN) is invalid (its reciprocal leaves
    the fp32 range); FLT_MIN itself is valid and behaves as a sharp softmax."""
    p = [[0.5, 0.5], [0.5, 0.5]]
    q = [[0.25, 0.75]]
    for t, bad in ((1e-40, True), (float(np.float32(1.1754944e-38) / 2), True), (1.1754944e-38, False)):
        r = oracle_mod.verify(hand_workload(p, q, [1], u=[0.9], E=[[1.0, 2.0]], temperature=[t]))
        assert (r["status"] == oracle_mod.BAD_PARAM) == bad, t
        if bad:
            assert r["out_tokens"].tolist() == [[-1, -1]] and r["num_accepted"][0] == 0
    l = np.array([[1.0, 0.5, -2.0]], np.float32)
    s = oracle_mod.sample_rows(l, temperature=[1e-40], exponentials=np.ones((1, 3)))
    assert s["status"] == oracle_mod.BAD_PARAM and s["tokens"][0] == -1
    s = oracle_mod.sample_rows(l, temperature=[1.1754944e-38], exponentials=np.ones((1, 3)))
    assert s["status"] == 0 and s["tokens"][0] == 0
    np.testing.assert_array_equal(s["probs"][0], np.array([1.0, 0.0, 0.0], np.float32))


# ----------------------------------------------------------------------------
# logits -> probabilities (page 1 "Rejection sampling": temperature, top-k,
# top-p applied identically; page 2 sections 06 and 14)
# ----------------------------------------------------------------------------
def test_plain_softmax_special_case(oracle_mod):
    rng = np.random.default_rng(1)
    l = (rng.standard_normal(5000) * 3).astype(np.float32)
    for T in (1.0, 0.7, 2.5):
        pr, edge, rc = oracle_mod.logits_to_probs(l, T)
        ref = scipy.special.softmax(l.astype(np.float64) / np.float64(np.float32(T)))
        assert rc == 0 and edge == 0
        # the oracle rounds its double result once: within half an fp32 ulp of the library value
        assert np.all(np.abs(pr.astype(np.float64) - ref) <= ref * 2.0 ** -24 * (1 + 1e-9))


def test_top_k_keeps_ties(oracle_mod):
    l = np.array([1.0, 5.0, 3.0, 3.0, 3.0, -2.0, 4.0], np.float32)
    pr, _, _ = oracle_mod.logits_to_probs(l, 1.0, top_k=3)
    keep = pr > 0
    assert keep.tolist() == [False, True, True, True, True, False, True]  # 5, 4 and all three 3s
    ref = scipy.special.softmax(l[keep].astype(np.float64))
    assert np.allclose(pr[keep], ref, atol=1e-7)
    pr1, _, _ = oracle_mod.logits_to_probs(l, 0.5, top_k=1)
    assert pr1.tolist() == [0, 1, 0, 0, 0, 0, 0]
    assert np.array_equal(oracle_mod.logits_to_probs(l, 1.0, top_k=0)[0] > 0, np.ones(7, bool))
    assert np.array_equal(oracle_mod.logits_to_probs(l, 1.0, top_k=7)[0] > 0, np.ones(7, bool))


def test_top_p_cut(oracle_mod):
    probs = np.array([0.05, 0.5, 0.15, 0.3])
    l = np.log(probs).astype(np.float32)
    pr, edge, _ = oracle_mod.logits_to_probs(l, 1.0, top_p=0.7)
    # descending 0.5, 0.3 (cum 0.8 >= 0.7): keep two, renormalise to 0.625 / 0.375
    assert pr == pytest.approx([0, 0.625, 0, 0.375], abs=1e-6)
    assert edge == 0
    pr, _, _ = oracle_mod.logits_to_probs(l, 1.0, top_p=0.45)
    assert pr == pytest.approx([0, 1, 0, 0], abs=1e-7)
    # ties at the cut are kept
    l2 = np.log(np.array([0.4, 0.2, 0.2, 0.2])).astype(np.float32)
    pr, _, _ = oracle_mod.logits_to_probs(l2, 1.0, top_p=0.5)
    assert (pr > 0).tolist() == [True, True, True, True]
    # top-k then top-p compose: top-2 of (0.5, 0.3) renormalised gives (0.625, 0.375); top_p 0.6 keeps one
    pr, _, _ = oracle_mod.logits_to_probs(l, 1.0, top_k=2, top_p=0.6)
    assert pr == pytest.approx([0, 1, 0, 0], abs=1e-7)
    pr, _, _ = oracle_mod.logits_to_probs(l, 1.0, top_k=2, top_p=0.7)
    assert pr == pytest.approx([0, 0.625, 0, 0.375], abs=1e-6)


def test_logits_edge_values(oracle_mod):
    l = np.array([0.0, -np.inf, 1.0, -np.inf], np.float32)
    pr, _, rc = oracle_mod.logits_to_probs(l, 1.0)
    assert rc == 0 and pr[1] == 0 and pr[3] == 0
    assert pr[0] + pr[2] == pytest.approx(1.0, abs=1e-7)
    assert oracle_mod.logits_to_probs(np.array([np.nan, 0], np.float32), 1.0)[2] == oracle_mod.BAD_VALUES
    assert oracle_mod.logits_to_probs(np.array([np.inf, 0], np.float32), 1.0)[2] == oracle_mod.BAD_VALUES
    assert oracle_mod.logits_to_probs(np.array([-np.inf, -np.inf], np.float32), 1.0)[2] == oracle_mod.BAD_VALUES


def test_logits_entry_matches_probs_entry_on_softmax_rows(oracle_mod):
    """At T=1 without top-k/top-p the logits entry is the probability entry on
    softmax rows (library softmax, rounded to fp32); decisions may differ only
    where a diagnostic margin is below the rounding of that softmax."""
    import workloads
    w = workloads.make("random", N=24, V=3000)
    lw = dict(w)
    rng = np.random.default_rng(4)
    tl = (rng.standard_normal(w["target"].shape) * 2).astype(np.float32)
    dl = (tl[np.repeat(np.arange(w["N"]) * (w["gamma"] + 1), w["gamma"]) + np.tile(np.arange(w["gamma"]), w["N"])]
          + rng.standard_normal(w["draft"].shape).astype(np.float32) * 0.5).astype(np.float32)
    lw.update(entry="logits", dtype="f32", target=tl, draft=dl)
    pw = dict(w)
    pw.update(target=scipy.special.softmax(tl.astype(np.float64), axis=-1).astype(np.float32),
              draft=scipy.special.softmax(dl.astype(np.float64), axis=-1).astype(np.float32))
    rl = oracle_mod.verify(lw)
    rp = oracle_mod.verify(pw)
    same = (rl["out_tokens"] == rp["out_tokens"]).all(axis=1)
    close = (rl["diag"][:, 0] < 1e-6) | (rl["diag"][:, 1] < 1e-6)
    assert np.all(same | close)
    assert same.mean() > 0.9


# ----------------------------------------------------------------------------
# Page 1, "About synthetic / block verification": preset acceptance rates
# ----------------------------------------------------------------------------
def test_synthetic_acceptance_lengths_follow_the_rates(oracle_mod):
    """With u on a uniform grid, the fraction of requests accepting at least k
    drafts is exactly prod_{j<k} rate_j, whatever p and q are."""
    import workloads
    n, G, V = 1000, 3, 50
    w = workloads.make("random", N=n, gamma=G, V=V, seed=3)
    rates = np.array([0.9, 0.6, 0.5], np.float32)
    # per-position u grids, shuffled independently so positions are uncorrelated
    rng = np.random.default_rng(0)
    u = np.stack([rng.permutation(U_GRID) for _ in range(G)], axis=1).reshape(-1)
    w["uniforms"] = u
    r = oracle_mod.verify(w, synthetic_rates=rates)
    A = r["num_accepted"]
    assert (A >= 1).mean() == pytest.approx(0.9, abs=0)
    # later positions: conditional rates hold on the exact grid counts
    assert ((A >= 2).sum()) == int(((u.reshape(n, G)[:, 0] < 0.9) & (u.reshape(n, G)[:, 1] < 0.6)).sum())
    acc = r["out_tokens"]
    for i in range(n):  # accepted tokens are the drafts; the next one is a residual draw (not the draft)
        assert acc[i, :A[i]].tolist() == w["draft_ids"][i * G:i * G + A[i]].tolist()
    assert np.all(np.isnan(r["dbg_py"]))  # the synthetic test uses no p(y), q(y): none are reported


def test_synthetic_rates_must_be_non_increasing(oracle_mod):
    import workloads
    w = workloads.make("tiny")
    r = oracle_mod.verify(w, synthetic_rates=np.array([0.5, 0.7, 0.2, 0.1], np.float32))
    assert r["status"] == oracle_mod.BAD_PARAM and np.all(r["out_tokens"] == -1)
    r = oracle_mod.verify(w, synthetic_rates=np.array([1.0, 1.0, 1.0, 1.0], np.float32))
    assert np.all(r["num_accepted"] == 4)  # u < 1 always: every draft kept, bonus drawn


def test_threaded_oracle_is_the_oracle(oracle_mod):
    """The threaded helpers that the full-size GPU tests use give exactly the
    single-threaded oracle's results (every output, ragged batch, production
    draws; sampler rows with their streams)."""
    import workloads
    w = workloads.make("ragged", N=40, V=3000, test_mode=False)
    a = oracle_mod.verify(w, production=True, seed=3, offset=2)
    b = oracle_mod.verify_parallel(w, production=True, seed=3, offset=2, threads=7)
    assert a["status"] == b["status"]
    for k in ("out_tokens", "num_accepted", "num_computed_tokens", "slot_mapping", "dbg_py", "dbg_qy", "diag"):
        np.testing.assert_array_equal(np.nan_to_num(a[k], nan=-9), np.nan_to_num(b[k], nan=-9), err_msg=k)
    rows = w["draft"][:30]
    kw = dict(temperature=np.full(30, 0.9, np.float32), top_k=np.full(30, 20), seed=4, offset=1, rng_row_base=3)
    x = oracle_mod.sample_rows(rows, **kw)
    y = oracle_mod.sample_rows_parallel(rows, threads=4, **kw)
    np.testing.assert_array_equal(x["tokens"], y["tokens"])
    np.testing.assert_array_equal(x["probs"], y["probs"])
    np.testing.assert_array_equal(x["diag"], y["diag"])
