"""Logits processors (banned tokens, repetition penalty) and stop tokens on
the GPU against the oracle, through the C ABI."""
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


def compare(g, o, w, **kw):
    from test_gpu_logits import compare_logits
    return compare_logits(g, o, w, **kw)


def add_lists(w, rng, *, theta=1.3, n_ctx=200, n_ban=12, stop_from_drafts=True, ban_drafts=True):
    """Per-request context, banned and stop lists with repeats, ids outside
    [0, V), drafts among the banned ids (forced rejections) and drafts among
    the stop ids (truncated commits)."""
    N, V, G = w["N"], w["V"], w["gamma"]
    gam = workloads.gammas_of(w)
    starts = np.concatenate([[0], np.cumsum(gam)[:-1]])
    ctx, ban, stop = [], [], []
    for i in range(N):
        c = rng.integers(-3, V + 3, size=int(rng.integers(0, n_ctx)))
        if len(c) > 4:
            c[1] = c[0]  # a repeat
        ctx.append(c)
        b = rng.integers(0, V, size=int(rng.integers(0, n_ban)))
        if ban_drafts and gam[i] > 2 and i % 5 == 0:
            b = np.append(b, w["draft_ids"][starts[i] + 2])
        ban.append(b)
        st = rng.integers(0, V, size=int(rng.integers(0, 3)))
        if stop_from_drafts and gam[i] > 1 and i % 3 == 0:
            st = np.append(st, w["draft_ids"][starts[i] + 1])
        stop.append(st)
    for name, lists in (("penalty", ctx), ("banned", ban), ("stop", stop)):
        w[f"{name}_cu"] = np.cumsum([len(x) for x in lists]).astype(np.int64)
        w[f"{name}_ids"] = (np.concatenate(lists) if sum(len(x) for x in lists) else np.zeros(0)).astype(np.int32)
    w["repetition_penalty"] = np.full(N, theta, np.float32)
    return w


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("theta", [1.3, 0.7])
def test_random_logits_with_processors(dtype, theta):
    w = workloads.make("fused", N=30, V=12000, seed=21)
    if dtype == "f32":
        w = dict(w, dtype="f32", target=workloads.bf16_bits_to_f32(w["target"]),
                 draft=workloads.bf16_bits_to_f32(w["draft"]))
    add_lists(w, np.random.default_rng(4), theta=theta)
    o = oracle.verify(w)
    compare(H().run_gpu(w), o, w, max_exempt_frac=0.1)
    assert (o["num_accepted"] < workloads.gammas_of(w)).any()


def test_greedy_with_processors_exact():
    w = workloads.make("greedy", N=24, V=32000, seed=8)
    # make drafts match the unprocessed argmax so processors decide the outcomes
    rng = np.random.default_rng(5)
    add_lists(w, rng, theta=3.0, n_ctx=50, n_ban=4)
    o = oracle.verify(w, with_diag=False)
    H().assert_same(H().run_gpu(w), o, check_dbg=False)


def test_ragged_production_with_processors():
    w = workloads.make("ragged", N=40, V=9000, test_mode=False)
    add_lists(w, np.random.default_rng(6), theta=1.8)
    o = oracle.verify(w, production=True, seed=3, offset=5)
    g = H().run_gpu(w, production=True, seed=3, offset=5)
    compare(g, o, w, production=True, max_exempt_frac=0.1)


@pytest.mark.parametrize("top_k,top_p,temp,V,cluster", [
    (50, 0.9, 0.8, 151936, 0),     # the fused setting at its vocabulary: 8 CTAs, register-held group maxima
    (0, 0.9, 0.8, 151936, 0),      # top-p alone: cuts in windows below the first
    (0, 1.0, 0.8, 151936, 0),      # temperature alone: dense sums and race
    (2000, 1.0, 0.8, 30000, 0),    # a deep top-k threshold
    (50, 0.9, 0.8, 40000, 1),      # one CTA per request over a 40000-key chunk
])
def test_processors_statistics_paths(top_k, top_p, temp, V, cluster):
    """Every statistics path with processors (rows copied into shared memory
    and rewritten there) against the oracle: the fused setting at its
    vocabulary, cuts in windows below the first, dense rows, a deep top-k
    threshold, and one CTA per request over a 40000-key chunk."""
    w = workloads.make("fused", N=16, V=V, seed=23)
    w["top_k"] = np.full(16, top_k, np.int32)
    w["top_p"] = np.full(16, top_p, np.float32)
    w["temperature"] = np.full(16, temp, np.float32)
    add_lists(w, np.random.default_rng(9), theta=1.5, n_ctx=400, n_ban=20)
    o = oracle.verify(w)
    compare(H().run_gpu(w, cluster_ctas=cluster), o, w, max_exempt_frac=0.5)


@pytest.mark.parametrize("top_k,top_p", [(50, 0.9), (0, 0.9)])
def test_processed_keys_win_races_and_windows(top_k, top_p):
    """Processors that move keys into the kept set and onto the race's top
    (theta < 1 raises every penalised logit), so processed keys decide group
    maxima, window counts and race winners; against the oracle."""
    w = workloads.make("fused", N=24, V=20000, seed=29)
    w["top_k"] = np.full(24, top_k, np.int32)
    w["top_p"] = np.full(24, top_p, np.float32)
    add_lists(w, np.random.default_rng(10), theta=0.5, n_ctx=2000, n_ban=40)
    o = oracle.verify(w)
    compare(H().run_gpu(w), o, w, max_exempt_frac=0.3)


def test_synthetic_mode_with_processors():
    w = workloads.make("fused", N=20, V=8192, seed=9)
    add_lists(w, np.random.default_rng(7))
    rates = np.array([0.9, 0.8, 0.8, 0.5, 0.4, 0.2, 0.1], np.float32)
    o = oracle.verify(w, synthetic_rates=rates)
    compare(H().run_gpu(w, synthetic_rates=rates), o, w, max_exempt_frac=0.1)


def test_stop_tokens_probability_entry_exact():
    w = workloads.make("random", N=32, V=6000, seed=2)
    rng = np.random.default_rng(8)
    gam = workloads.gammas_of(w)
    starts = np.concatenate([[0], np.cumsum(gam)[:-1]])
    stop = [np.array([w["draft_ids"][starts[i] + i % gam[i]]]) if i % 2 else np.zeros(0, np.int64)
            for i in range(w["N"])]
    w["stop_cu"] = np.cumsum([len(x) for x in stop]).astype(np.int64)
    w["stop_ids"] = np.concatenate(stop).astype(np.int32)
    o = oracle.verify(w)
    H().assert_same(H().run_gpu(w), o)
    base = oracle.verify({k: v for k, v in w.items() if not k.startswith("stop")})
    assert (o["num_accepted"] < base["num_accepted"]).any()  # some commits were cut
    assert rng is not None


def test_list_and_theta_errors():
    V = 16
    t = np.zeros((3, V), np.float32)
    t[:, 3] = 2.0
    d = t[:2].copy()
    for key, val, code in [("stop_cu", np.array([5], np.int64), oracle.BAD_LIST),
                           ("banned_cu", np.array([-1], np.int64), oracle.BAD_LIST),
                           ("repetition_penalty", np.array([-1.0], np.float32), oracle.BAD_PARAM),
                           ("repetition_penalty", np.array([np.inf], np.float32), oracle.BAD_PARAM)]:
        w = hand_workload(t, d, [3, 3], entry="logits", u=[0.5, 0.5], E=np.ones((1, V)), temperature=[1.0])
        w[key] = val
        if key.endswith("_cu"):
            w[key.replace("_cu", "_ids")] = np.array([3, 4], np.int32)
        o = oracle.verify(w)
        assert o["status"] == code
        H().assert_same(H().run_gpu(w), o, check_dbg=False)


def test_everything_banned_is_bad_values():
    V = 32
    rng = np.random.default_rng(1)
    t = rng.standard_normal((3, V)).astype(np.float32)
    w = hand_workload(t, t[:2] + 0.1, [1, 2], entry="logits", u=[0.2, 0.3], E=np.ones((1, V)), temperature=[1.0])
    w["banned_cu"] = np.array([V], np.int64)
    w["banned_ids"] = np.arange(V, dtype=np.int32)
    o = oracle.verify(w)
    assert o["status"] == oracle.BAD_VALUES
    H().assert_same(H().run_gpu(w), o, check_dbg=False)
