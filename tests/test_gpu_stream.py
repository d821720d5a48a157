"""Parity of the one-CTA-per-request ("stream") form of the logits entry with
the CPU oracle (GPU required), under the handle flag
SV_FLAG_ONE_CTA_PER_REQUEST.  The same contract and exemption rules as the
cluster form (test_gpu_logits.compare_logits): the form changes how a row's
floor, top-k threshold, top-p cut and race are found (block maxima, then
candidates), never what they are.  The cases cover the candidate path (top-k
1 .. 256, ties at the floor, signed zeros, rows shorter than a block step or
with a ragged tail) and every way out of it (top-k off or above 256, fp32 rows
beyond the block maxima's room, candidates overflowing their room), each of
which takes the exact multi-pass statistics.
"""
import numpy as np
import pytest

import oracle
import workloads
from conftest import hand_workload

pytestmark = pytest.mark.gpu


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


def run(w, **kw):
    import speculative_decoding_token_rejection_gb300 as sv
    return H().run_gpu(w, flags=sv.SV_FLAG_ONE_CTA_PER_REQUEST, **kw)


def compare(g, o, w, **kw):
    from test_gpu_logits import compare_logits
    return compare_logits(g, o, w, **kw)


def with_params(w, **over):
    w = dict(w)
    N = w["N"]
    for k, v in over.items():
        w[k] = np.full(N, v, np.int32 if k == "top_k" else np.float32)
    return w


@pytest.mark.parametrize("name,kw,over", [
    ("fused", dict(N=24, V=8192), {}),
    ("fused", dict(N=16, V=151936), {}),
    ("fused", dict(N=12, V=20007), {}),         # a ragged tail (fewer than a 16-byte group)
    ("ragged", dict(N=40, V=9000), {}),          # greedy and random requests, ragged gamma
    ("fused", dict(N=20, V=12000), dict(top_k=1)),
    ("fused", dict(N=20, V=12000), dict(top_k=256)),
    ("fused", dict(N=20, V=12000), dict(top_k=257)),  # above the candidate path: exact statistics
    ("fused", dict(N=20, V=12000), dict(top_k=0)),    # top-k off: exact statistics
    ("fused", dict(N=20, V=12000), dict(top_k=8, top_p=1.0)),
    ("fused", dict(N=6, V=100), {}),             # fewer groups than one step
    ("fused", dict(N=6, V=13), dict(top_k=3)),   # a single group and a tail
    ("fused", dict(N=6, V=2053), dict(top_k=200)),
    ("fused", dict(N=8, V=151936), dict(top_k=256)),
    ("fused", dict(N=8, V=151936), dict(top_k=256, top_p=1.0)),
])
def test_stream_test_mode(name, kw, over):
    w = with_params(workloads.make(name, **kw), **over)
    n_ex = compare(run(w), oracle.verify(w), w)
    print(f"{name} {kw} {over}: {n_ex} exempted")


@pytest.mark.parametrize("V", [6000, 140000])
def test_stream_fp32_logits(V):
    """fp32 rows: 16-bit block keys from the high key bits; rows beyond the
    block maxima's room (131072 fp32 logits) take the exact statistics."""
    w = workloads.make("fused", N=12 if V < 10000 else 3, V=V)
    w = dict(w, dtype="f32", target=workloads.bf16_bits_to_f32(w["target"]),
             draft=workloads.bf16_bits_to_f32(w["draft"]))
    compare(run(w), oracle.verify(w), w)


@pytest.mark.parametrize("shape", ["ties", "spiky", "monotone", "signed_zeros"])
@pytest.mark.parametrize("top_k", [1, 9, 100, 256])
def test_stream_floor_cases(shape, top_k):
    """Rows that put the block floor at awkward places: heavy ties at the
    floor, a few spikes over a flat floor, a monotone row whose top k sit in
    a few blocks, and rows of +0.0 / -0.0 (the NaN-propagating maximum may
    return either zero; the floor's block test allows for it)."""
    N, V = 24, 40000  # (24 requests: one race exemption stays within the 5% budget)
    w = workloads.make("fused", N=N, V=V, seed=43)
    rng = np.random.default_rng(top_k * 11 + len(shape))
    G = w["gamma"]
    rows = N * (G + 1) + N * G
    if shape == "ties":
        l = rng.integers(0, 6, size=(rows, V)).astype(np.float32)
    elif shape == "spiky":
        l = np.full((rows, V), -5.0, np.float32)
        l[:, rng.integers(0, V, size=3)] = 10.0
        l += rng.integers(0, 2, size=(rows, V)).astype(np.float32) * 0.5
    elif shape == "monotone":
        l = np.tile(-np.arange(V, dtype=np.float32) * 0.01, (rows, 1))
        l += rng.standard_normal((rows, V)).astype(np.float32) * 0.02
    else:
        l = rng.choice(np.array([-0.0, 0.0, -1.0, -2.0], np.float32), size=(rows, V))
        l[:, rng.integers(0, V, size=top_k // 2)] = 0.5
    bits = workloads._to_bf16_bits(l)
    w["target"] = bits[:N * (G + 1)]
    w["draft"] = bits[N * (G + 1):]
    w = with_params(w, top_k=top_k, top_p=0.95 if top_k > 8 else 1.0)
    compare(run(w), oracle.verify(w), w)


@pytest.mark.parametrize("name,kw", [("fused", dict(N=24, V=12000)), ("ragged", dict(N=48, V=9000))])
def test_stream_production_philox(name, kw):
    w = workloads.make(name, test_mode=False, **kw)
    g = run(w, production=True, seed=20240611, offset=2)
    o = oracle.verify(w, production=True, seed=20240611, offset=2)
    compare(g, o, w, production=True)


def test_stream_synthetic_acceptance():
    rates = [0.9, 0.8, 0.5, 0.5, 0.3, 0.3, 0.1]
    w = workloads.make("fused", N=16, V=12000)
    o = oracle.verify(w, synthetic_rates=np.array(rates, np.float32))
    compare(run(w, synthetic_rates=rates), o, w)


def test_stream_status_cases():
    """Invalid values and parameters are reported as in the cluster form."""
    V = 16
    good = np.zeros((2, V), np.float32)
    good[:, 3] = 1.0
    cases = []
    for col, val in ((7, np.nan), (2, np.inf)):
        bad = good.copy()
        bad[0, col] = val
        cases.append((bad, oracle.BAD_VALUES))
    bad = good.copy()
    bad[0, :] = -np.inf
    cases.append((bad, oracle.BAD_VALUES))
    ninf = good.copy()
    ninf[0, 8:] = -np.inf
    cases.append((ninf, 0))
    for tgt, code in cases:
        for top_k in (None, [2]):
            w = hand_workload(tgt, good[:1], [3], entry="logits", u=[0.5], E=[np.ones(V)], temperature=[1.0],
                              top_k=top_k)
            o = oracle.verify(w)
            assert o["status"] == code
            H().assert_same(run(w), o, check_dbg=False)
    w = hand_workload(good, good[:1], [3], entry="logits", u=[0.5], E=[np.ones(V)], temperature=[1.0],
                      top_p=[0.0])
    o = oracle.verify(w)
    assert o["status"] == oracle.BAD_PARAM
    H().assert_same(run(w), o, check_dbg=False)


def test_stream_processors_bench_lists():
    """The bench's processors (repetition penalty over 512 context ids, 16
    banned and 2 stop ids per request) in the one-CTA form."""
    import bench
    w = dict(workloads.make("fused", N=16, V=12000))
    w.update(bench.processor_lists(w["N"], w["V"], seed=5))
    compare(run(w), oracle.verify(w), w)


@pytest.fixture
def one_cta_everywhere():
    import gpu_harness
    import speculative_decoding_token_rejection_gb300 as sv
    gpu_harness.EXTRA_FLAGS = sv.SV_FLAG_ONE_CTA_PER_REQUEST
    yield
    gpu_harness.EXTRA_FLAGS = 0


@pytest.mark.parametrize("name,kw", [
    ("test_random_logits_with_processors", dict(dtype="bf16", theta=1.3)),
    ("test_random_logits_with_processors", dict(dtype="f32", theta=0.7)),
    ("test_greedy_with_processors_exact", {}),
    ("test_ragged_production_with_processors", {}),
    ("test_processors_statistics_paths", dict(top_k=50, top_p=0.9, temp=0.8, V=151936, cluster=0)),
    ("test_processors_statistics_paths", dict(top_k=0, top_p=0.9, temp=0.8, V=151936, cluster=0)),
    ("test_processors_statistics_paths", dict(top_k=2000, top_p=1.0, temp=0.8, V=30000, cluster=0)),
    ("test_processed_keys_win_races_and_windows", dict(top_k=50, top_p=0.9)),
    ("test_synthetic_mode_with_processors", {}),
    ("test_list_and_theta_errors", {}),
    ("test_everything_banned_is_bad_values", {}),
    ("test_order_golden_cases", dict(resident=False)),
    ("test_banned_maximum_far_above_the_rest", dict(resident=False)),
    ("test_penalty_raising_past_the_fp32_range", {}),
    ("test_banned_nucleus_is_bad_values", {}),
])
def test_stream_processor_cases(name, kw, one_cta_everywhere):
    """The processor cases of test_gpu_processors.py, rerun with every call in
    the one-CTA form: the kept set from the raw candidates, the processed kept
    candidates summed afresh (or, off the candidate path, the exact statistics'
    correction), the draft token's marks, the race over processed weights, and
    greedy rows' argmax over the processed row."""
    import test_gpu_processors
    getattr(test_gpu_processors, name)(**kw)


def test_stream_and_cluster_forms_agree_bitwise():
    """Both forms compute the same fixed-point masses, cuts, normalisers and
    race keys, so their outputs are identical, p(y) and q(y) included."""
    w = workloads.make("fused", N=64, V=151936, seed=9, test_mode=False)
    a = H().run_gpu(w, production=True, seed=20240612, offset=1)
    b = run(w, production=True, seed=20240612, offset=1)
    for k in ("out_tokens", "num_accepted", "num_computed_tokens", "slot_mapping"):
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_array_equal(a["dbg_py"], b["dbg_py"])
    np.testing.assert_array_equal(a["dbg_qy"], b["dbg_qy"])
    assert a["status"] == b["status"] == 0


@pytest.mark.parametrize("V", [262144, 262152])
def test_stream_block_capacity_edge(V):
    """bf16 rows of exactly the block maxima's room (32 steps, 4096 blocks per
    row) take the candidate path; 8 logits more leave it for the exact
    statistics."""
    w = workloads.make("fused", N=4, V=V, seed=47)
    compare(run(w), oracle.verify(w), w)


def test_stream_processors_at_the_capacity_edge():
    """Processors with row bitmaps of a 262144-logit vocabulary (64 KB per
    CTA)."""
    import bench
    w = dict(workloads.make("fused", N=4, V=262144, seed=48))
    w.update(bench.processor_lists(w["N"], w["V"], seed=6))
    compare(run(w), oracle.verify(w), w)
