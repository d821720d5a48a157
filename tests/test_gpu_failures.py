"""Failure detection on the GPU without faulting it (GPU required).

The bulk row copies into shared memory complete on an mbarrier whose waits
poll a bounded number of times; a give-up raises SV_DATA_COPY_TIMEOUT and the
request emits nothing.  A test cannot make a copy hang without faulting a GPU,
so the call flag SV_TEST_EXPIRE_COPY_WAIT makes the first wait give up at
once while the second, ordinary wait still lets every copy land: the CTA
then carries on exactly as after a real give-up.  Also here: invalid
temperatures (negative, infinite, subnormal) on every entry."""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def H():
    import gpu_harness
    return gpu_harness


@pytest.mark.parametrize("procs", [False, True])
def test_expired_copy_wait_reports_and_emits_nothing(procs):
    import speculative_decoding_token_rejection_gb300 as sv
    w = workloads.make("ragged", N=24, V=9000, seed=4)  # half greedy, half random
    if procs:
        from test_gpu_processors import add_lists
        add_lists(w, np.random.default_rng(3), theta=1.4, n_ctx=50, n_ban=4)
    o = oracle.verify(w)
    flags = sv.SV_FLAG_RESIDENT_ROWS
    g = H().run_gpu(w, flags=flags, test_flags=sv.SV_TEST_EXPIRE_COPY_WAIT)
    assert g["status"] & sv.DATA_STATUS_BITS["COPY_TIMEOUT"]
    greedy = np.asarray(w["temperature"]) == 0
    copied = ~greedy | procs  # greedy rows are copied only to be processed
    gam = workloads.gammas_of(w)
    s = 0
    for i in range(w["N"]):
        if copied[i]:
            assert np.all(g["out_tokens"][i] == -1) and g["num_accepted"][i] == 0, i
            assert g["num_computed_tokens"][i] == w["num_computed_tokens"][i]  # KV bookkeeping untouched
            np.testing.assert_array_equal(g["slot_mapping"][s + i:s + i + gam[i] + 1],
                                          w["slot_mapping"][s + i:s + i + gam[i] + 1])
        else:  # streamed rows, no copy: the ordinary result
            np.testing.assert_array_equal(g["out_tokens"][i], o["out_tokens"][i])
        s += int(gam[i])
    # the next call on the same handle, without the flag, is the ordinary one
    from test_gpu_logits import compare_logits
    compare_logits(H().run_gpu(w, flags=flags), o, w)


def test_expired_copy_wait_in_the_sampler():
    import speculative_decoding_token_rejection_gb300 as sv
    from test_gpu_sampler import run_sampler
    rng = np.random.default_rng(5)
    R, V = 12, 5000
    rows = workloads._to_bf16_bits((rng.standard_normal((R, V)) * 2.5).astype(np.float32))
    E = rng.standard_exponential((R, V), dtype=np.float32)
    temp = np.full(R, 0.8, np.float32)
    tok, _, st = run_sampler(rows, temp, np.full(R, 50), np.full(R, 0.9, np.float32), E, bf16=True,
                             flags=sv.SV_FLAG_RESIDENT_ROWS, test_flags=sv.SV_TEST_EXPIRE_COPY_WAIT)
    assert st == sv.DATA_STATUS_BITS["COPY_TIMEOUT"] and np.all(tok == -1)
    o = oracle.sample_rows(rows, temperature=temp, top_k=np.full(R, 50), top_p=np.full(R, 0.9, np.float32),
                           exponentials=E)
    tok, _, st = run_sampler(rows, temp, np.full(R, 50), np.full(R, 0.9, np.float32), E, bf16=True,
                             flags=sv.SV_FLAG_RESIDENT_ROWS)
    assert st == 0
    ex = (o["diag"][:, 0] < 1) | (o["diag"][:, 1] > 0)
    np.testing.assert_array_equal(tok[~ex], o["tokens"][~ex])


@pytest.mark.parametrize("name", ["random", "fused"])
def test_invalid_temperatures(name):
    """Negative, infinite, NaN and subnormal temperatures are bad parameters
    (the request emits nothing) on both entries; FLT_MIN itself is valid."""
    w = workloads.make(name, N=6, V=2000, seed=8)
    temps = np.array([-1.0, np.inf, np.nan, 1e-40, 1.1754944e-38, 0.9], np.float32)
    w["temperature"] = temps
    o = oracle.verify(w)
    g = H().run_gpu(w)
    assert o["status"] & oracle.BAD_PARAM and g["status"] == o["status"]
    assert np.all(g["out_tokens"][:4] == -1) and np.all(g["num_accepted"][:4] == 0)
    np.testing.assert_array_equal(g["num_accepted"], o["num_accepted"])
    np.testing.assert_array_equal(g["out_tokens"], o["out_tokens"])


def test_invalid_temperatures_in_the_sampler():
    from test_gpu_sampler import run_sampler
    rng = np.random.default_rng(6)
    rows = (rng.standard_normal((5, 700)) * 2).astype(np.float32)
    temp = np.array([1e-40, -0.5, np.inf, 1.1754944e-38, 0.7], np.float32)
    E = rng.standard_exponential((5, 700), dtype=np.float32)
    o = oracle.sample_rows(rows, temperature=temp, exponentials=E)
    tok, _, st = run_sampler(rows, temp, None, None, E)
    assert st == o["status"] == oracle.BAD_PARAM
    np.testing.assert_array_equal(tok, o["tokens"])
