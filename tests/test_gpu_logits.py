"""Parity of the CUDA logits entry with the CPU oracle (GPU required).

Greedy rows compare raw logits, so their outputs are exact.  Random rows go
through temperature, top-k, softmax and top-p on both sides; the oracle does it
in double and rounds to fp32, the kernel in fp32.  The contract: p(y) and q(y)
agree within 1e-6 absolute; committed tokens, num_accepted and the KV rollback
agree exactly except where the oracle reports a decision within tolerance of
flipping.  The exemptions are narrow and each one frees only what it can
change:
  * an acceptance test that a perturbation of p and q inside both 1e-6
    absolute and 1e-5 relative could flip (|u*q - p| below both bounds): the
    acceptance count, the tokens and the rollback of that request are free,
    and p(y), q(y) are still compared on the positions both sides examined;
  * a race whose two leading keys such a perturbation could swap: only the
    drawn token (the last committed one) is free; the acceptance count, the
    accepted tokens, the rollback and every p(y), q(y) must match;
  * a top-p cut whose value-group sum lies within 1e-6 of top_p (the kept set
    itself may differ): the request's outputs are free.
Exempted requests are counted, printed, and never more than 5% of a batch.
"""
import numpy as np
import pytest
import scipy.stats

import oracle
import workloads
from conftest import hand_workload

pytestmark = pytest.mark.gpu
TOL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from speculative_decoding_token_rejection_gb300 import _build
    _build.build()
    oracle.build()


def H():
    import gpu_harness
    return gpu_harness


def exempt_classes(o, production=False):
    """Per request: (acceptance within the band, race within the band, top-p
    edge), from the oracle's diagnostics."""
    d = o["diag"]
    accept = d[:, oracle.DIAG_ACCEPT_MARGIN] < 1
    race = d[:, oracle.DIAG_RACE_FLIP] < 1
    if production:  # production E can differ by an ulp of log: relative key gaps below 1e-6 too
        race |= d[:, oracle.DIAG_RACE_RELGAP] < TOL
    edge = d[:, oracle.DIAG_TOPP_EDGE] > 0
    return accept, race, edge


def exempt_mask(o, production=False):
    accept, race, edge = exempt_classes(o, production)
    return accept | race | edge


def compare_logits(g, o, w, production=False, max_exempt_frac=0.05):
    assert max_exempt_frac <= 0.05
    accept, race, edge = exempt_classes(o, production)
    free = accept | edge  # the acceptance count itself may differ
    ex = free | race
    gam = workloads.gammas_of(w)
    A_g, A_o = g["num_accepted"], o["num_accepted"]
    np.testing.assert_array_equal(A_g[~free], A_o[~free])
    np.testing.assert_array_equal(g["out_tokens"][~ex], o["out_tokens"][~ex])
    assert g["status"] == o["status"]
    s = 0
    for i in range(w["N"]):
        gi = int(gam[i])
        if not free[i]:
            if race[i]:  # only the drawn token may differ
                a = int(A_o[i])
                np.testing.assert_array_equal(g["out_tokens"][i, :a], o["out_tokens"][i, :a])
                np.testing.assert_array_equal(g["out_tokens"][i, a + 1:], o["out_tokens"][i, a + 1:])
            if o["num_computed_tokens"] is not None:
                assert g["num_computed_tokens"][i] == o["num_computed_tokens"][i]
            if o["slot_mapping"] is not None:
                np.testing.assert_array_equal(g["slot_mapping"][s + i:s + i + gi + 1],
                                              o["slot_mapping"][s + i:s + i + gi + 1])
        if not edge[i]:
            for key in ("dbg_py", "dbg_qy"):
                og, gg = o[key][s:s + gi], g[key][s:s + gi]
                if not free[i]:  # the same positions were examined
                    np.testing.assert_array_equal(np.isnan(og), np.isnan(gg))
                m = ~np.isnan(og) & ~np.isnan(gg)  # positions both sides examined
                assert np.all(np.abs(gg[m] - og[m]) <= TOL), (i, key, gg[m], og[m])
        s += gi
    if ex.any():
        print(f"exempt: {int(accept.sum())} acceptance, {int(race.sum())} race, {int(edge.sum())} top-p edge "
              f"of {w['N']} requests")
    assert ex.mean() <= max_exempt_frac, f"{ex.sum()} of {w['N']} requests exempted"
    return int(ex.sum())


# ----------------------------------------------------------------------------
# greedy: exact
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("kw", [{}, dict(N=7, V=3001), dict(N=20, gamma=9, V=5000)])
def test_greedy_workload_exact(kw):
    w = workloads.make("greedy", **kw)
    H().assert_same(H().run_gpu(w), oracle.verify(w, with_diag=False), check_dbg=False)


def test_greedy_fp32_logits_exact():
    w = workloads.make("greedy", N=16, V=4096)
    w = dict(w, dtype="f32", target=workloads.bf16_bits_to_f32(w["target"]) * np.float32(1.001))
    H().assert_same(H().run_gpu(w), oracle.verify(w, with_diag=False), check_dbg=False)


def test_greedy_matching_drafts_get_bonus():
    w = workloads.make("greedy", N=10, V=2000, seed=5)
    G = w["gamma"]
    t32 = workloads.bf16_bits_to_f32(w["target"])
    for i in range(0, 10, 2):  # even requests: drafts equal the target argmax -> gamma+1 tokens
        w["draft_ids"][i * G:(i + 1) * G] = t32[i * (G + 1):i * (G + 1) + G].argmax(axis=1)
    o = oracle.verify(w, with_diag=False)
    H().assert_same(H().run_gpu(w), o, check_dbg=False)
    assert (o["num_accepted"][::2] == G).all()


# ----------------------------------------------------------------------------
# random rows: within the stated tolerance
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("name,kw", [
    ("ragged", {}),                          # N=256, V=128256, half greedy, T=1 dense rows
    ("ragged", dict(N=40, V=3001)),          # unaligned rows (scalar path)
    ("fused", dict(N=24, V=8192)),           # top-k 50 + top-p 0.9, T=0.8
    ("fused", dict(N=16, gamma=3, V=20000)),
])
def test_random_logits_test_mode(name, kw):
    w = workloads.make(name, **kw)
    o = oracle.verify(w)
    g = H().run_gpu(w)
    compare_logits(g, o, w)


def test_fused_full_size_test_mode():
    """N=512, gamma=7, V=151936 bf16 logits in test mode (explicit u and E):
    every request against the oracle (threaded over the host's cores)."""
    w = workloads.make("fused")
    g = H().run_gpu(w)
    o = oracle.verify_parallel(w)
    compare_logits(g, o, w)
    assert g["status"] == 0
    A = g["num_accepted"]
    assert np.all((A >= 0) & (A <= w["gamma"]))
    assert np.all((g["out_tokens"] >= 0).sum(axis=1) == A + 1)


def test_fp32_logits_fused():
    w = workloads.make("fused", N=12, V=6000)
    w = dict(w, dtype="f32", target=workloads.bf16_bits_to_f32(w["target"]),
             draft=workloads.bf16_bits_to_f32(w["draft"]))
    compare_logits(H().run_gpu(w), oracle.verify(w), w)


@pytest.mark.parametrize("cluster,V", [(1, 40000), (2, 40000), (1, 20480), (1, 20488)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_in_place_chunks_beyond_register_groups(cluster, V, dtype):
    """Rows read in place whose chunk is larger than the 20480 bf16 elements
    whose group maxima stay in registers take the group-walk scan instead;
    20480 itself is the last chunk on the register path."""
    w = workloads.make("fused", N=12, V=V, seed=16)
    if dtype == "fp32":
        w = dict(w, dtype="f32", target=workloads.bf16_bits_to_f32(w["target"]),
                 draft=workloads.bf16_bits_to_f32(w["draft"]))
    o = oracle.verify(w)
    g = H().run_gpu(w, cluster_ctas=cluster)
    compare_logits(g, o, w)


@pytest.mark.parametrize("top_k,top_p,temp,N", [
    (1, 1.0, 1.0, 10), (5, 1.0, 0.5, 10), (0, 0.5, 1.0, 10), (7, 0.3, 0.9, 10), (4095, 0.95, 1.3, 10),
    (20, 1e-4, 1.0, 10),
    # a flattened row (T = 2) with a wide nucleus
    (0, 0.8, 2.0, 40)])
def test_sampling_parameter_grid(top_k, top_p, temp, N):
    w = workloads.make("fused", N=N, V=4096, seed=31)
    w["top_k"] = np.full(N, top_k, np.int32)
    w["top_p"] = np.full(N, top_p, np.float32)
    w["temperature"] = np.full(N, temp, np.float32)
    compare_logits(H().run_gpu(w), oracle.verify(w), w)


def test_top_k_ties_at_threshold():
    """Sixteen requests whose rows hold a ten-way tie at the top-k threshold
    (top_k 4 keeps the maximum and all ten tied keys), drafts among the tied
    ids; the oracle exempts none of them."""
    V, N, G = 64, 16, 5
    rng = np.random.default_rng(2)
    t, d, ids = [], [], []
    for _ in range(N):
        rows = rng.standard_normal((G + 1, V)).astype(np.float32)
        rows[:, 5:15] = 2.0  # ten-way tie
        rows[:, 3] = 3.0
        t.append(rows)
        d.append(rows[:G] + np.float32(0.01))
        ids += list(rng.choice([5, 9, 3, 14, 0, 20], size=G))
    w = hand_workload(np.concatenate(t), np.concatenate(d), ids, entry="logits", u=rng.random(N * G),
                      E=rng.exponential(size=(N, V)), top_k=[4] * N, top_p=[1.0] * N, temperature=[1.0] * N)
    o = oracle.verify(w)
    assert compare_logits(H().run_gpu(w), o, w) == 0
    assert len(set(o["num_accepted"].tolist())) > 2


def test_logits_status_cases():
    V = 16
    good = np.zeros((2, V), np.float32)
    good[:, 3] = 1.0
    cases = []
    bad = good.copy()
    bad[0, 7] = np.nan
    cases.append((bad, oracle.BAD_VALUES))
    bad = good.copy()
    bad[0, 2] = np.inf
    cases.append((bad, oracle.BAD_VALUES))
    bad = good.copy()
    bad[0, :] = -np.inf
    cases.append((bad, oracle.BAD_VALUES))
    ninf = good.copy()
    ninf[0, 8:] = -np.inf
    cases.append((ninf, 0))
    for tgt, code in cases:
        w = hand_workload(tgt, good[:1], [3], entry="logits", u=[0.5], E=[np.ones(V)], temperature=[1.0])
        o = oracle.verify(w)
        g = H().run_gpu(w)
        assert o["status"] == code
        H().assert_same(g, o, check_dbg=False)
    w = hand_workload(good, good[:1], [3], entry="logits", u=[0.5], E=[np.ones(V)], temperature=[1.0],
                      top_p=[0.0])
    o = oracle.verify(w)
    assert o["status"] == oracle.BAD_PARAM
    H().assert_same(H().run_gpu(w), o, check_dbg=False)
    # NaN on the greedy path; a NaN in an unread row is never seen
    w = hand_workload(np.array([[0, 1, np.nan, 0], [0, 0, 0, 0]], np.float32), None, [1], entry="logits",
                      temperature=[0.0], u=[0], E=[[1] * 4])
    H().assert_same(H().run_gpu(w), oracle.verify(w, with_diag=False), check_dbg=False)
    w = hand_workload(np.array([[0, 1, 0, 0], [0, np.nan, 0, 0]], np.float32), None, [2], entry="logits",
                      temperature=[0.0], u=[0], E=[[1] * 4])
    o = oracle.verify(w, with_diag=False)
    assert o["status"] == 0
    H().assert_same(H().run_gpu(w), o, check_dbg=False)


# ----------------------------------------------------------------------------
# production mode
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("name,kw", [("ragged", dict(N=48, V=9000)), ("fused", dict(N=24, V=12000))])
def test_production_logits_matches_oracle_philox(name, kw):
    w = workloads.make(name, test_mode=False, **kw)
    o = oracle.verify(w, production=True, seed=8, offset=2)
    g = H().run_gpu(w, production=True, seed=8, offset=2)
    compare_logits(g, o, w, production=True)


def test_production_logits_chi_square():
    """V=6 logits with T=0.7, top-k 4, top-p 0.9: the first committed token
    follows the transformed target row (10^6 trials)."""
    n, V, G = 1_000_000, 6, 2
    rng = np.random.default_rng(3)
    tl = rng.standard_normal((G + 1, V)).astype(np.float32)
    dl = (tl[:G] + rng.standard_normal((G, V)).astype(np.float32) * 0.8).astype(np.float32)
    kw = dict(temp=0.7, k=4, p=0.9)
    p0, _, _ = oracle.logits_to_probs(tl[0], kw["temp"], kw["k"], kw["p"])
    q = [oracle.logits_to_probs(dl[j], kw["temp"], kw["k"], kw["p"])[0] for j in range(G)]
    ids = np.stack([rng.choice(V, size=n, p=q[j].astype(np.float64) / q[j].astype(np.float64).sum())
                    for j in range(G)], axis=1).reshape(-1)
    w = hand_workload(np.tile(tl, (n, 1)), np.tile(dl, (n, 1)), ids, entry="logits",
                      temperature=np.full(n, kw["temp"]), top_k=np.full(n, kw["k"]), top_p=np.full(n, kw["p"]))
    g = H().run_gpu(w, production=True, seed=19, offset=4)
    assert g["status"] == 0
    first = np.bincount(g["out_tokens"][:, 0], minlength=V)
    expect = p0.astype(np.float64)
    assert np.all(first[expect == 0] == 0)
    nz = expect > 0
    assert scipy.stats.chisquare(first[nz], n * expect[nz] / expect[nz].sum()).pvalue > 0.01


@pytest.mark.parametrize("rates", [[0.9, 0.8, 0.5, 0.5, 0.3, 0.3, 0.1], [1.0] * 7, [0.3, 0.4, 0, 0, 0, 0, 0]])
def test_synthetic_acceptance_logits(rates):
    w = workloads.make("fused", N=24, V=8192, seed=5)
    o = oracle.verify(w, synthetic_rates=np.array(rates, np.float32))
    g = H().run_gpu(w, synthetic_rates=rates)
    compare_logits(g, o, w)
    if rates[1] > rates[0]:
        assert o["status"] == oracle.BAD_PARAM


@pytest.mark.parametrize("shape", ["normal", "ties", "spiky", "monotone"])
@pytest.mark.parametrize("top_k", [1, 8, 9, 100, 255, 256, 257])
def test_top_k_threshold_bound_cases(shape, top_k):
    """Rows chosen so the threshold sits at every kind of place relative to a
    CTA's largest keys: heavy ties, a few spikes over a flat floor, and a
    monotone row whose top k all lie in one CTA's chunk; k on both sides of
    32 x warps (where the per-CTA threshold bound switches off)."""
    N, V = 24, 40000
    w = workloads.make("fused", N=N, V=V, seed=41)
    rng = np.random.default_rng(top_k * 7 + len(shape))
    G = w["gamma"]
    rows = N * (G + 1) + N * G
    if shape == "normal":
        l = rng.standard_normal((rows, V)).astype(np.float32) * 2.5
    elif shape == "ties":
        l = rng.integers(0, 6, size=(rows, V)).astype(np.float32)
    elif shape == "spiky":
        l = np.full((rows, V), -5.0, np.float32)
        l[:, rng.integers(0, V, size=3)] = 10.0
        l += rng.integers(0, 2, size=(rows, V)).astype(np.float32) * 0.5
    else:
        l = np.tile(-np.arange(V, dtype=np.float32) * 0.01, (rows, 1))
        l += rng.standard_normal((rows, V)).astype(np.float32) * 0.02
    bits = workloads._to_bf16_bits(l)
    w["target"] = bits[:N * (G + 1)]
    w["draft"] = bits[N * (G + 1):]
    w["top_k"] = np.full(N, top_k, np.int32)
    w["top_p"] = np.full(N, 0.95 if top_k > 8 else 1.0, np.float32)
    compare_logits(H().run_gpu(w), oracle.verify(w), w)


@pytest.mark.parametrize("name,kw,production", [("fused", dict(N=40, V=151936), False),
                                                ("fused", dict(N=24, V=12000), True),
                                                ("ragged", dict(N=48, V=9000), False)])
def test_draft_rows_in_place_and_resident_agree(name, kw, production):
    """The two forms of the logits kernel -- row chunks read in place
    (default) or copied into shared memory -- against the oracle and against
    each other (identical except inside the tolerance band)."""
    import speculative_decoding_token_rejection_gb300 as sv
    w = workloads.make(name, test_mode=not production, **kw)
    o = oracle.verify(w, production=production, seed=6, offset=1)
    g_in_place = H().run_gpu(w, production=production, seed=6, offset=1)
    g_res = H().run_gpu(w, production=production, seed=6, offset=1, flags=sv.SV_FLAG_RESIDENT_ROWS)
    compare_logits(g_in_place, o, w, production=production, max_exempt_frac=0.05)
    compare_logits(g_res, o, w, production=production, max_exempt_frac=0.05)
    np.testing.assert_array_equal(g_in_place["num_accepted"], g_res["num_accepted"])


@pytest.mark.parametrize("cluster", [1, 2, 4, 16])
@pytest.mark.parametrize("resident", [False, True])
def test_explicit_cluster_sizes(cluster, resident):
    """Every cluster size in both forms; V=12008 leaves a ragged last chunk
    (16-byte aligned rows, chunks of 12008 / C rounded up to 8 elements)."""
    import speculative_decoding_token_rejection_gb300 as sv
    w = workloads.make("fused", N=20, V=12008, seed=15)
    o = oracle.verify(w)
    g = H().run_gpu(w, cluster_ctas=cluster, flags=sv.SV_FLAG_RESIDENT_ROWS if resident else 0)
    compare_logits(g, o, w)


@pytest.mark.parametrize("top_k,top_p,temp,N", [
    (2000, 1.0, 0.8, 12),      # top-k threshold several windows below the maximum
    (2000, 0.9, 0.8, 12),      # ... with a cut inside its window or above it (the multi-pass selection)
    (600, 0.3, 1.0, 12),
    (0, 0.9, 0.8, 24),         # top-p alone, cut below the first window
    (0, 0.95, 0.8, 12),        # a wider nucleus: more windows
    (0, 0.98, 0.6, 12),
    (5000, 0.97, 1.2, 12)])
def test_thresholds_below_the_first_window(top_k, top_p, temp, N):
    """Rows whose threshold or cut lies below the first 128-key window, on a
    vocabulary large enough for several windows."""
    w = workloads.make("fused", N=N, V=40000, seed=37)
    w["top_k"] = np.full(N, top_k, np.int32)
    w["top_p"] = np.full(N, top_p, np.float32)
    w["temperature"] = np.full(N, temp, np.float32)
    o = oracle.verify(w)
    g = H().run_gpu(w)
    compare_logits(g, o, w)
    _valid_outputs(g, w)


def _valid_outputs(g, w):
    A = g["num_accepted"]
    assert np.all((A >= 0) & (A <= w["gamma"]))
    for i in range(w["N"]):
        assert np.all((g["out_tokens"][i, :A[i] + 1] >= 0) & (g["out_tokens"][i, :A[i] + 1] < w["V"]))
        assert np.all(g["out_tokens"][i, A[i] + 1:] == -1)


def test_flat_rows_cut_near_one_are_valid():
    """A nucleus of 0.9999 on flat rows (T = 2.5): every key near the cut
    carries less than 1e-6 of mass, so every cut lies inside the tolerance band
    and the kept set may legitimately differ from the oracle's.  Not a parity
    case: the outputs must be valid (counts in range, committed tokens in the
    vocabulary, -1 after them, accepted tokens equal to the drafts)."""
    w = workloads.make("fused", N=12, V=40000, seed=37)
    w["top_k"] = np.zeros(12, np.int32)
    w["top_p"] = np.full(12, 0.9999, np.float32)
    w["temperature"] = np.full(12, 2.5, np.float32)
    g = H().run_gpu(w)
    assert g["status"] == 0
    _valid_outputs(g, w)
    G = w["gamma"]
    for i in range(12):
        a = int(g["num_accepted"][i])
        assert list(g["out_tokens"][i, :a]) == list(w["draft_ids"][i * G:i * G + a])
