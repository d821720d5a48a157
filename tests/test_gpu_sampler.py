"""Parity of the CUDA draft-side sampler with the oracle (GPU required).

Every transformed probability row must agree with the oracle's within 1e-6
absolute (a full-row check of the logits transform shared with the verifier's
logits entry); sampled tokens must agree except where the oracle reports a
race a perturbation inside 1e-6 absolute and 1e-5 relative could flip, or a
top-p edge.  Greedy rows are exact.  Production draws pass a chi-square test.
"""
import numpy as np
import pytest
import scipy.stats

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from speculative_decoding_token_rejection_gb300 import _build
    _build.build()
    oracle.build()


def run_sampler(rows_np, temp, k, p, E=None, seed=0, offset=0, base=0, bf16=False, cluster=0, flags=0, test_flags=0,
                hints=0):
    import torch
    import gpu_harness
    import speculative_decoding_token_rejection_gb300 as sv
    dev = torch.device("cuda:0")
    if bf16:
        logits = torch.from_numpy(rows_np.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        logits = torch.from_numpy(np.ascontiguousarray(rows_np, np.float32)).to(dev)
    R, V = rows_np.shape
    tokens = torch.full((R,), -7, dtype=torch.int32, device=dev)
    probs = torch.zeros((R, V), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t = lambda a, dt: None if a is None else torch.as_tensor(np.asarray(a), dtype=dt).to(dev)
    sv.spec_verify_sample(gpu_harness.verifier(cluster, flags).handle, logits=logits, tokens=tokens, probs=probs,
                          temperature=t(temp, torch.float32), top_k=t(k, torch.int32), top_p=t(p, torch.float32),
                          exponentials=t(E, torch.float32), seed=seed, offset=offset, rng_row_base=base,
                          status=status, test_flags=test_flags, hints=hints)
    torch.cuda.synchronize()
    return tokens.cpu().numpy(), probs.cpu().numpy(), int(status.item())


def check(rows, temp, k, p, E=None, production=False, bf16=False, budget=0.05, seed=0, offset=0, base=0, cluster=0,
          flags=0, hints=0):
    assert budget <= 0.05
    o = oracle.sample_rows(rows, temperature=temp, top_k=k, top_p=p, exponentials=E, seed=seed, offset=offset,
                           rng_row_base=base)
    tok, pr, st = run_sampler(rows, temp, k, p, E, bf16=bf16, seed=seed, offset=offset, base=base, cluster=cluster,
                              flags=flags, hints=hints)
    assert st == o["status"]
    temp = np.asarray(temp)
    rnd = temp > 0
    np.testing.assert_array_equal(tok[~rnd], o["tokens"][~rnd])  # greedy: exact
    assert np.max(np.abs(pr[rnd] - o["probs"][rnd])) <= 1e-6
    ex = (o["diag"][:, 0] < 1) | (o["diag"][:, 1] > 0)
    keep = ~ex
    np.testing.assert_array_equal(tok[keep], o["tokens"][keep])
    assert ex.mean() <= budget, ex.sum()
    return tok


def fused_rows(R=64, V=151936):
    w = workloads.make("fused", N=max(1, R // 7), V=V, test_mode=False)
    return w["draft"][:R]


@pytest.mark.parametrize("cluster", [0, 4, 8, 16])
@pytest.mark.parametrize("resident", [False, True])
def test_sampler_forms_and_cluster_sizes(cluster, resident):
    """Rows read in place (default) or copied into shared memory, at the
    automatic cluster size and explicit ones: 4 CTAs give chunks of 37984
    keys (beyond the register-held group maxima), 8 and 16 stay within."""
    import speculative_decoding_token_rejection_gb300 as sv
    rows = fused_rows(24, 151936)
    R, V = rows.shape
    E = np.random.default_rng(2).standard_exponential((R, V), dtype=np.float32)
    temp = np.where(np.arange(R) % 6 == 5, 0.0, 0.8).astype(np.float32)
    check(rows, temp, np.full(R, 50), np.full(R, 0.9, np.float32), E, bf16=True, cluster=cluster,
          flags=sv.SV_FLAG_RESIDENT_ROWS if resident else 0)


@pytest.mark.parametrize("V", [151936, 5000, 4097])
def test_sampler_fused_rows_test_mode(V):
    rows = fused_rows(64, V)
    R = rows.shape[0]
    rng = np.random.default_rng(1)
    E = rng.standard_exponential((R, V), dtype=np.float32)
    check(rows, np.full(R, 0.8, np.float32), np.full(R, 50), np.full(R, 0.9, np.float32), E, bf16=True)


@pytest.mark.parametrize("k,p,temp", [(0, 1.0, 1.0), (0, 0.95, 0.7), (200, 1.0, 1.3), (1, 1.0, 1.0)])
def test_sampler_parameter_grid_fp32(k, p, temp):
    rng = np.random.default_rng(2)
    R, V = 48, 6000
    rows = (rng.standard_normal((R, V)) * 2.0).astype(np.float32)
    E = rng.standard_exponential((R, V), dtype=np.float32)
    check(rows, np.full(R, temp, np.float32), np.full(R, k), np.full(R, p, np.float32), E, budget=0.05)


def test_sampler_greedy_rows_and_status():
    rng = np.random.default_rng(3)
    rows = (rng.standard_normal((6, 300)) * 2).astype(np.float32)
    rows[4, 17] = np.nan
    temp = np.array([0, 1, 0, 0.5, 1, -2], np.float32)
    E = rng.standard_exponential((6, 300), dtype=np.float32)
    tok = check(rows, temp, np.zeros(6), np.ones(6, np.float32), E)
    assert tok[4] == -1 and tok[5] == -1


def test_sampler_production_matches_oracle_philox():
    rows = fused_rows(48, 20000)
    R = rows.shape[0]
    check(rows, np.full(R, 0.8, np.float32), np.full(R, 50), np.full(R, 0.9, np.float32), None, bf16=True,
          seed=5, offset=2, base=9)


def test_sampler_production_chi_square():
    rng = np.random.default_rng(4)
    V, R = 7, 1_000_000
    l = (rng.standard_normal(V) * 1.5).astype(np.float32)
    probs, _, _ = oracle.logits_to_probs(l, 0.7, 4, 0.9)
    tok, _, st = run_sampler(np.tile(l, (R, 1)), np.full(R, 0.7, np.float32), np.full(R, 4),
                             np.full(R, 0.9, np.float32), None, seed=21, offset=3)
    assert st == 0
    cnt = np.bincount(tok, minlength=V)
    e = probs.astype(np.float64)
    assert np.all(cnt[e == 0] == 0)
    nz = e > 0
    assert scipy.stats.chisquare(cnt[nz], R * e[nz] / e[nz].sum()).pvalue > 0.01


def _proc_lists(R, V, rng):
    ctx = [rng.integers(-2, V + 2, size=int(rng.integers(0, 60))) for _ in range(R)]
    ban = [rng.integers(0, V, size=int(rng.integers(0, 8))) for _ in range(R)]
    out = {"repetition_penalty": rng.uniform(0.6, 2.0, size=R).astype(np.float32)}
    for name, lists in (("penalty", ctx), ("banned", ban)):
        out[f"{name}_cu"] = np.cumsum([len(x) for x in lists]).astype(np.int64)
        out[f"{name}_ids"] = np.concatenate(lists).astype(np.int32)
    return out


@pytest.mark.parametrize("form", ["in_place", "resident", "one_cta"])
@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("temp", [0.0, 0.8])
def test_sampler_with_processors(bf16, temp, form):
    """Banned tokens and the repetition penalty per row, against the oracle,
    with the rows read in place or copied into shared memory by a cluster per
    row, or by one CTA per row: tokens exact (outside the tolerance band of
    the race) and the written q rows within 1e-6."""
    import torch
    import speculative_decoding_token_rejection_gb300 as sv
    rng = np.random.default_rng(int(bf16) + 2)
    R, V = 24, 20000
    rows = rng.standard_normal((R, V)).astype(np.float32) * 2.5
    if bf16:
        rows = workloads._to_bf16_bits(rows)
    lists = _proc_lists(R, V, rng)
    # the argmax of a few rows is banned outright
    E = rng.exponential(size=(R, V)).astype(np.float32)
    kw = dict(temperature=np.full(R, temp, np.float32), top_k=np.full(R, 50, np.int32),
              top_p=np.full(R, 0.9, np.float32))
    o = oracle.sample_rows(rows, exponentials=E, **kw, repetition_penalty=lists["repetition_penalty"],
                           penalty_cu=lists["penalty_cu"], penalty_ids=lists["penalty_ids"],
                           banned_cu=lists["banned_cu"], banned_ids=lists["banned_ids"])
    dev = torch.device("cuda:0")
    t = (torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16) if bf16 else torch.from_numpy(rows)).to(dev)
    tok = torch.full((R,), -7, dtype=torch.int32, device=dev)
    probs = torch.zeros((R, V), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flags = {"in_place": 0, "resident": sv.SV_FLAG_RESIDENT_ROWS, "one_cta": sv.SV_FLAG_ONE_CTA_PER_REQUEST}[form]
    h = sv.spec_verify_create(R, 1, V, device=0, flags=flags)
    try:
        T = lambda x, dt: torch.as_tensor(x).to(dev)
        sv.spec_verify_sample(h, logits=t, tokens=tok, probs=probs, exponentials=torch.from_numpy(E).to(dev),
                              temperature=T(kw["temperature"], None), top_k=T(kw["top_k"], None),
                              top_p=T(kw["top_p"], None), status=st,
                              repetition_penalty=T(lists["repetition_penalty"], None),
                              penalty_cu=T(lists["penalty_cu"], None), penalty_token_ids=T(lists["penalty_ids"], None),
                              banned_cu=T(lists["banned_cu"], None), banned_token_ids=T(lists["banned_ids"], None))
        torch.cuda.synchronize()
    finally:
        sv.spec_verify_destroy(h)
    assert int(st.item()) == o["status"]
    g = tok.cpu().numpy()
    exempt = (o["diag"][:, 0] < 1) | (o["diag"][:, 1] > 0)
    np.testing.assert_array_equal(g[~exempt], o["tokens"][~exempt])
    assert exempt.mean() <= 0.05
    if temp > 0:
        d = np.abs(probs.cpu().numpy() - o["probs"])
        assert d.max() <= 1e-6


# ----------------------------------------------------------------------------
# one CTA per row (SV_FLAG_ONE_CTA_PER_REQUEST, or the small-top-k hint on a
# batch of at least two rows per SM): the same contract
# ----------------------------------------------------------------------------
def _one_cta():
    import speculative_decoding_token_rejection_gb300 as sv
    return sv.SV_FLAG_ONE_CTA_PER_REQUEST


@pytest.mark.parametrize("V", [151936, 5000, 4097, 13])
def test_sampler_one_cta_per_row_fused_rows(V):
    rows = fused_rows(64, V)
    R = rows.shape[0]
    E = np.random.default_rng(6).standard_exponential((R, V), dtype=np.float32)
    temp = np.where(np.arange(R) % 9 == 4, 0.0, 0.8).astype(np.float32)
    check(rows, temp, np.full(R, min(50, V - 1)), np.full(R, 0.9, np.float32), E, bf16=True, flags=_one_cta())


@pytest.mark.parametrize("k,p,temp", [(0, 1.0, 1.0), (0, 0.95, 0.7), (200, 1.0, 1.3), (1, 1.0, 1.0), (256, 0.9, 0.8),
                                      (257, 0.9, 0.8)])
def test_sampler_one_cta_per_row_grid_fp32(k, p, temp):
    rng = np.random.default_rng(7)
    R, V = 48, 6000
    rows = (rng.standard_normal((R, V)) * 2.0).astype(np.float32)
    E = rng.standard_exponential((R, V), dtype=np.float32)
    check(rows, np.full(R, temp, np.float32), np.full(R, k), np.full(R, p, np.float32), E, flags=_one_cta())


def test_sampler_one_cta_per_row_greedy_and_status():
    rng = np.random.default_rng(8)
    rows = (rng.standard_normal((6, 300)) * 2).astype(np.float32)
    rows[4, 17] = np.nan
    temp = np.array([0, 1, 0, 0.5, 1, -2], np.float32)
    E = rng.standard_exponential((6, 300), dtype=np.float32)
    tok = check(rows, temp, np.full(6, 3), np.ones(6, np.float32), E, flags=_one_cta())
    assert tok[4] == -1 and tok[5] == -1


def test_sampler_one_cta_per_row_production():
    rows = fused_rows(48, 20000)
    R = rows.shape[0]
    check(rows, np.full(R, 0.8, np.float32), np.full(R, 50), np.full(R, 0.9, np.float32), None, bf16=True,
          seed=5, offset=2, base=9, flags=_one_cta())


def test_sampler_one_cta_per_row_chi_square():
    """Production draws of the per-row form follow the transformed row."""
    rng = np.random.default_rng(9)
    V, R = 7, 1_000_000
    l = (rng.standard_normal(V) * 1.5).astype(np.float32)
    probs, _, _ = oracle.logits_to_probs(l, 0.7, 4, 0.9)
    tok, _, st = run_sampler(np.tile(l, (R, 1)), np.full(R, 0.7, np.float32), np.full(R, 4),
                             np.full(R, 0.9, np.float32), None, seed=22, offset=3, flags=_one_cta())
    assert st == 0
    cnt = np.bincount(tok, minlength=V)
    e = probs.astype(np.float64)
    assert np.all(cnt[e == 0] == 0)
    nz = e > 0
    assert scipy.stats.chisquare(cnt[nz], R * e[nz] / e[nz].sum()).pvalue > 0.01


def test_sampler_forms_agree_bitwise_with_hint():
    """512 fused rows (the bench's draft step): the hinted call takes one CTA
    per row; tokens and probability rows equal the cluster form's bit for bit."""
    import speculative_decoding_token_rejection_gb300 as sv
    w = workloads.make("fused", seed=3, test_mode=False)
    rows = w["draft"][::7][:512]
    R = rows.shape[0]
    args = (rows, np.full(R, 0.8, np.float32), np.full(R, 50), np.full(R, 0.9, np.float32), None)
    t0, p0, s0 = run_sampler(*args, bf16=True, seed=4, offset=1)
    t1, p1, s1 = run_sampler(*args, bf16=True, seed=4, offset=1, hints=sv.SV_HINT_SMALL_TOP_K)
    assert s0 == s1 == 0
    np.testing.assert_array_equal(t0, t1)
    np.testing.assert_array_equal(p0, p1)
