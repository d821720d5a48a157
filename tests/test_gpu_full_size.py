"""Parity at the full sizes and in the launch configurations that bench.py
times (GPU required): N=512 requests, gamma=7, V=151936, production Philox
draws at the bench's seeds, automatic cluster sizes.  The GPU runs every
request and the oracle checks every request (the logits batches and the
sampler rows through the threaded oracle over the host's cores).
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def H():
    import gpu_harness
    return gpu_harness


def compare(g, o, w, **kw):
    from test_gpu_logits import compare_logits
    return compare_logits(g, o, w, **kw)


_CACHE = {}


def fused_probs():
    if "probs" not in _CACHE:
        _CACHE["probs"] = workloads.make("fused_probs", seed=3, test_mode=False)
    return _CACHE["probs"]


def fused_logits():
    if "logits" not in _CACHE:
        _CACHE["logits"] = workloads.make("fused", seed=3, test_mode=False)
    return _CACHE["logits"]


@pytest.mark.parametrize("offset", [0, 7])
def test_probability_entry_bench_batch(offset):
    """The headline batch (fp32 probability rows) at the bench's seed: every
    request against the oracle."""
    w = fused_probs()
    o = oracle.verify(w, production=True, seed=20240601, offset=offset)
    g = H().run_gpu(w, production=True, seed=20240601, offset=offset)
    compare(g, o, w, production=True, max_exempt_frac=0.01)


def test_synthetic_acceptance_bench_batch():
    """The headline batch with the bench's preset rates: every request."""
    rates = np.array([0.8, 0.7, 0.6, 0.5, 0.4, 0.3, 0.2], np.float32)
    w = fused_probs()
    o = oracle.verify(w, production=True, seed=20240605, offset=3, synthetic_rates=rates)
    g = H().run_gpu(w, production=True, seed=20240605, offset=3, synthetic_rates=rates)
    compare(g, o, w, production=True, max_exempt_frac=0.01)


@pytest.mark.parametrize("form", ["cluster", "stream"])
def test_logits_entry_bench_batch(form):
    """The fused logits batch (bf16, T=0.8, top-k 50, top-p 0.9) in both
    forms: clusters (rows read in place, 8 CTAs per request; no hint) and,
    with the small-top-k hint the bench passes, one CTA per request: every
    one of the 512 requests against the oracle."""
    import speculative_decoding_token_rejection_gb300 as sv
    w = fused_logits()
    hints = sv.SV_HINT_SMALL_TOP_K if form == "stream" else 0
    g = H().run_gpu(w, production=True, seed=20240602, offset=5, hints=hints)
    o = oracle.verify_parallel(w, production=True, seed=20240602, offset=5)
    n_ex = compare(g, o, w, production=True)
    print(f"logits batch: {n_ex} of {w['N']} requests exempted")
    A = g["num_accepted"]
    assert np.all((A >= 0) & (A <= w["gamma"]))


@pytest.mark.parametrize("form", ["cluster", "stream"])
def test_logits_processors_bench_batch(form):
    """The fused logits batch with the bench's processors (repetition
    penalty 1.2 over 512 context ids, 16 banned and 2 stop ids per request),
    in both forms (the small-top-k hint the bench passes selects one CTA per
    request): every one of the 512 requests against the oracle."""
    import bench
    import speculative_decoding_token_rejection_gb300 as sv
    w = dict(fused_logits())
    w.update(bench.processor_lists(w["N"], w["V"], seed=11))
    hints = sv.SV_HINT_SMALL_TOP_K if form == "stream" else 0
    g = H().run_gpu(w, production=True, seed=20240604, offset=2, hints=hints)
    o = oracle.verify_parallel(w, production=True, seed=20240604, offset=2)
    n_ex = compare(g, o, w, production=True)
    print(f"processors batch: {n_ex} of {w['N']} requests exempted")
    assert g["status"] == 0


@pytest.mark.parametrize("position", [0, 6])
def test_draft_sampler_bench_rows(position):
    """One draft step of the fused batch as the bench samples it (512 bf16
    rows of V=151936, 4 CTAs per row, rows read in place, q rows written):
    every row's token and transformed row against the oracle."""
    import speculative_decoding_token_rejection_gb300 as sv
    w = fused_logits()
    N, G, V = w["N"], w["gamma"], w["V"]
    rows = np.ascontiguousarray(w["draft"].reshape(N, G, V)[:, position, :])
    dev = torch.device("cuda:0")
    t = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).to(dev)
    temp = np.asarray(w["temperature"], np.float32)
    kw = dict(temperature=temp, top_k=np.full(N, 50, np.int32), top_p=np.full(N, 0.9, np.float32))
    tok = torch.full((N,), -7, dtype=torch.int32, device=dev)
    probs = torch.zeros((N, V), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    h = sv.spec_verify_create(N, 1, V, device=0)
    try:
        T = lambda x: torch.as_tensor(x).to(dev)
        sv.spec_verify_sample(h, logits=t, tokens=tok, probs=probs, temperature=T(kw["temperature"]),
                              top_k=T(kw["top_k"]), top_p=T(kw["top_p"]), seed=20240603, offset=position,
                              rng_row_base=0, status=st)
        torch.cuda.synchronize()
    finally:
        sv.spec_verify_destroy(h)
    assert int(st.item()) == 0
    o = oracle.sample_rows_parallel(rows, temperature=temp, top_k=kw["top_k"], top_p=kw["top_p"], seed=20240603,
                                    offset=position, rng_row_base=0)
    g = tok.cpu().numpy()
    exempt = (o["diag"][:, 0] < 1) | (o["diag"][:, 1] > 0)
    print(f"sampler rows: {int(exempt.sum())} of {N} exempted")
    np.testing.assert_array_equal(g[~exempt], o["tokens"][~exempt])
    assert exempt.mean() <= 0.05
    pg = probs.cpu().numpy()
    keep = o["diag"][:, 1] == 0  # rows whose kept set is not at a top-p edge
    assert np.max(np.abs(pg[keep] - o["probs"][keep])) <= 1e-6
    assert np.all((g >= 0) & (g < V))
