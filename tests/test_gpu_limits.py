"""The largest sizes a handle accepts: max_spec_len = SV_MAX_SPEC_LEN (256)
with every draft accepted, and the largest vocabulary the test handle is
created for (2^18), on both entries and the sampler."""
import numpy as np
import pytest

import oracle
import workloads
from conftest import hand_workload

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def H():
    import gpu_harness
    return gpu_harness


def _all_accepted(entry, N, G, V, seed):
    """Draft rows equal to the target rows: p(y) = q(y) > 0, so u q < p for
    every u < 1 and all G drafts are accepted; the bonus is raced over the
    last row."""
    rng = np.random.default_rng(seed)
    rows = rng.standard_normal((N * (G + 1), V)).astype(np.float32) * 2
    drafts = np.concatenate([rows[i * (G + 1):i * (G + 1) + G] for i in range(N)])
    if entry == "probs":
        e = np.exp(rows - rows.max(axis=1, keepdims=True))
        rows = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
        drafts = np.concatenate([rows[i * (G + 1):i * (G + 1) + G] for i in range(N)])
    ids = np.array([int(np.argmax(d)) for d in drafts], np.int32)
    dtype = "bf16" if entry == "logits" else "f32"
    if dtype == "bf16":
        rows, drafts = workloads._to_bf16_bits(rows), workloads._to_bf16_bits(drafts)
    return hand_workload(rows, drafts, ids, entry=entry, dtype=dtype, u=rng.random(N * G) * 0.999,
                         E=rng.exponential(size=(N, V)), temperature=np.ones(N, np.float32))


@pytest.mark.parametrize("entry", ["probs", "logits"])
def test_longest_speculation_all_accepted(entry):
    import speculative_decoding_token_rejection_gb300 as sv
    G = sv.SV_MAX_SPEC_LEN
    w = _all_accepted(entry, 3, G, 2048, seed=4)
    o = oracle.verify(w)
    assert np.all(o["num_accepted"] == G)
    g = H().run_gpu(w)
    if entry == "probs":
        H().assert_same(g, o)
    else:
        from test_gpu_logits import compare_logits
        assert compare_logits(g, o, w) == 0
        np.testing.assert_array_equal(g["num_accepted"], o["num_accepted"])
        np.testing.assert_array_equal(g["out_tokens"][:, :G], o["out_tokens"][:, :G])


@pytest.mark.parametrize("name,entry", [("fused", "logits"), ("random", "probs")])
def test_largest_vocabulary(name, entry):
    V = 1 << 18
    w = workloads.make(name, N=6, gamma=3, V=V, seed=23)
    assert w["entry"] == entry
    o = oracle.verify(w)
    g = H().run_gpu(w)
    if entry == "probs":
        H().assert_same(g, o)
    else:
        from test_gpu_logits import compare_logits
        assert compare_logits(g, o, w) == 0


def test_sampler_largest_vocabulary():
    from test_gpu_sampler import check
    rng = np.random.default_rng(9)
    V = 1 << 18
    rows = workloads._to_bf16_bits(rng.standard_normal((6, V)).astype(np.float32) * 2.5)
    E = rng.exponential(size=(6, V)).astype(np.float32)
    check(rows, np.full(6, 0.8, np.float32), np.full(6, 50, np.int32), np.full(6, 0.9, np.float32), E=E,
          bf16=True)
