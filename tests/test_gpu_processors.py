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
    compare(H().run_gpu(w), o, w)
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
    compare(g, o, w, production=True)


@pytest.mark.parametrize("top_k,top_p,temp,V,cluster", [
    (50, 0.9, 0.8, 151936, 0),     # the fused setting at its vocabulary: 8 CTAs, register-held group maxima
    (0, 0.9, 0.8, 151936, 0),      # top-p alone: cuts in windows below the first
    (0, 1.0, 0.8, 151936, 0),      # temperature alone: dense sums and race
    (2000, 1.0, 0.8, 30000, 0),    # a deep top-k threshold
    (50, 0.9, 0.8, 40000, 1),      # one CTA per request over a 40000-key chunk
])
def test_processors_statistics_paths(top_k, top_p, temp, V, cluster):
    """Every statistics path with processors against the oracle: the fused
    setting at its vocabulary, cuts in windows below the first, dense rows, a
    deep top-k threshold, and one CTA per request over a 40000-key chunk."""
    N = 32
    w = workloads.make("fused", N=N, V=V, seed=23)
    w["top_k"] = np.full(N, top_k, np.int32)
    w["top_p"] = np.full(N, top_p, np.float32)
    w["temperature"] = np.full(N, temp, np.float32)
    add_lists(w, np.random.default_rng(9), theta=1.5, n_ctx=400, n_ban=20)
    o = oracle.verify(w)
    compare(H().run_gpu(w, cluster_ctas=cluster), o, w)


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
    compare(H().run_gpu(w), o, w)


def test_synthetic_mode_with_processors():
    w = workloads.make("fused", N=20, V=8192, seed=9)
    add_lists(w, np.random.default_rng(7))
    rates = np.array([0.9, 0.8, 0.8, 0.5, 0.4, 0.2, 0.1], np.float32)
    o = oracle.verify(w, synthetic_rates=rates)
    compare(H().run_gpu(w, synthetic_rates=rates), o, w)


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


# ----------------------------------------------------------------------------
# the order: temperature, top-k, top-p on the raw rows, then the processors
# ----------------------------------------------------------------------------
def _golden_lists(g, c):
    kw = {}
    if f"{c}_banned" in g:
        ids = np.array([int(x) for x in g[f"{c}_banned"]], np.int32)
        kw["banned_cu"], kw["banned_ids"] = np.array([len(ids)], np.int64), ids
    if f"{c}_theta" in g:
        ids = np.array([int(x) for x in g[f"{c}_context"]], np.int32)
        kw["repetition_penalty"] = np.array([float(g[f"{c}_theta"][0])], np.float32)
        kw["penalty_cu"], kw["penalty_ids"] = np.array([len(ids)], np.int64), ids
    return kw


@pytest.mark.parametrize("resident", [False, True])
def test_order_golden_cases(resident):
    """The hand-worked cases that separate the pages' order from
    processors-first, through the GPU: every transformed probability of each
    case row (the draft id walks over the vocabulary), and the commit that
    differs between the two orders, exactly as the oracle and the fixture."""
    import speculative_decoding_token_rejection_gb300 as sv
    from conftest import load_golden
    g = load_golden("processors_order_examples.txt")
    flags = sv.SV_FLAG_RESIDENT_ROWS if resident else 0
    for c in ("t1", "t2", "t3", "t4", "t5"):
        row = np.array([float(x) for x in g[f"{c}_row"]], np.float32)
        V = row.shape[0]
        N = V  # one request per draft id
        t = np.concatenate([np.stack([row, np.zeros(V, np.float32)]) for _ in range(N)])
        d = np.tile(row, (N, 1))
        E = np.tile(np.arange(1, V + 1, dtype=np.float32), (N, 1))  # distinct keys: no race ties
        w = hand_workload(t, d, list(range(V)), entry="logits", u=[0.5] * N, E=E,
                          temperature=[float(g[f"{c}_temp"][0])] * N, top_k=[int(g[f"{c}_topk"][0])] * N,
                          top_p=[float(g[f"{c}_topp"][0])] * N)
        for k, v in _golden_lists(g, c).items():
            if k.endswith("_cu"):
                v = v[0] * np.arange(1, N + 1, dtype=np.int64)
            elif k.endswith("_ids"):
                v = np.tile(v, N)
            else:
                v = np.full(N, v[0], np.float32)
            w[k] = v
        o = oracle.verify(w)
        r = H().run_gpu(w, flags=flags)
        if f"{c}_status" in g:
            assert o["status"] == r["status"] == int(g[f"{c}_status"][0]), c
            assert np.all(r["out_tokens"] == -1) and np.all(r["num_accepted"] == 0), c
            continue
        compare(r, o, w)
        expect = np.array([float(x) for x in g[f"{c}_expect"]], np.float32)
        assert np.all(np.abs(r["dbg_py"] - expect) <= 1e-6) and np.all(np.abs(r["dbg_qy"] - expect) <= 1e-6), c
    tg = np.array([[float(x) for x in r.split()] for r in " ".join(g["v1_target"]).split("|")], np.float32)
    dr = np.array([[float(x) for x in g["v1_draft"]]], np.float32)
    w = hand_workload(tg, dr, [int(x) for x in g["v1_drafts"]], entry="logits", u=[float(g["v1_u"][0])],
                      E=np.ones((1, tg.shape[1])), temperature=[1.0], top_k=[int(g["v1_topk"][0])], top_p=[1.0])
    w.update(_golden_lists(g, "v1"))
    r = H().run_gpu(w, flags=flags)
    assert r["status"] == 0 and r["num_accepted"][0] == int(g["v1_A"][0])
    assert list(r["out_tokens"][0]) == [int(x) for x in g["v1_expect"]]
    assert r["dbg_py"][0] == float(g["v1_py"][0]) and r["dbg_qy"][0] == float(g["v1_qy"][0])


def _spiked(N, V, seed, top, gap_rest):
    """bf16 logits rows N(0, 1) whose maximum is `top` at index 7 (every row),
    with the rest `gap_rest` lower on average."""
    rng = np.random.default_rng(seed)
    G = 3
    rows = (rng.standard_normal((N * (G + 1) + N * G, V)) + (top - gap_rest)).astype(np.float32)
    rows[:, 7] = top
    bits = workloads._to_bf16_bits(rows)
    w = hand_workload(bits[:N * (G + 1)], bits[N * (G + 1):], rng.integers(0, V, size=N * G), entry="logits",
                      dtype="bf16", u=rng.random(N * G), E=rng.exponential(size=(N, V)),
                      temperature=np.full(N, 0.8, np.float32), top_k=np.full(N, 50, np.int32),
                      top_p=np.full(N, 0.9, np.float32))
    w["draft_ids"][::G] = 7  # position 0 drafts the spiked id
    return w


@pytest.mark.parametrize("resident", [False, True])
def test_banned_maximum_far_above_the_rest(resident):
    """The row maximum is banned and every other kept key lies ~40 nats below
    it: the corrected normaliser cancels to nothing relative to the raw
    maximum, so the kernel recomputes the kept set's statistics against its
    largest unbanned value (the oracle renormalises in double)."""
    import speculative_decoding_token_rejection_gb300 as sv
    w = _spiked(24, 3000, 5, top=40.0, gap_rest=40.0 * 0.8 + 3)
    w["top_p"] = np.ones(24, np.float32)  # top-k 50 alone: the kept set is the maximum and 49 keys far below
    w["banned_cu"] = np.arange(1, 25, dtype=np.int64)
    w["banned_ids"] = np.full(24, 7, np.int32)
    o = oracle.verify(w)
    assert o["status"] == 0 and np.all(o["dbg_py"][::3] == 0)  # y = 7 is banned at position 0
    compare(H().run_gpu(w, flags=sv.SV_FLAG_RESIDENT_ROWS if resident else 0), o, w)


def test_penalty_raising_past_the_fp32_range():
    """theta 1e-3 raises the maximum (l / theta, l > 0) so far that its weight
    relative to the raw maximum overflows fp32: the kernel recomputes the
    statistics against the processed maximum.  theta 2e-38 overflows the
    processed logit itself to +inf: no distribution, the bad-values status."""
    for theta, status in ((1e-3, 0), (2e-38, oracle.BAD_VALUES)):
        w = _spiked(16, 3000, 6, top=10.0, gap_rest=4.0)
        w["repetition_penalty"] = np.full(16, theta, np.float32)
        w["penalty_cu"] = np.arange(1, 17, dtype=np.int64)
        w["penalty_ids"] = np.full(16, 7, np.int32)
        o = oracle.verify(w)
        assert o["status"] == status
        r = H().run_gpu(w)
        if status:
            H().assert_same(r, o, check_dbg=False)
        else:
            compare(r, o, w)


def test_banned_nucleus_is_bad_values():
    """top_p small enough that each row's nucleus is its maximum alone, and
    the maximum banned: no distribution is left (oracle: bad values)."""
    w = _spiked(16, 3000, 7, top=12.0, gap_rest=10.0)
    w["top_k"] = np.zeros(16, np.int32)
    w["top_p"] = np.full(16, 0.5, np.float32)
    w["banned_cu"] = np.arange(1, 17, dtype=np.int64)
    w["banned_ids"] = np.full(16, 7, np.int32)
    o = oracle.verify(w)
    assert o["status"] == oracle.BAD_VALUES and np.all(o["num_accepted"] == 0)
    H().assert_same(H().run_gpu(w), o, check_dbg=False)


@pytest.mark.parametrize("resident", [False, True])
def test_processors_in_both_forms(resident):
    """The fused setting with the bench's kind of lists, rows read in place
    (the default) or copied into shared memory: both against the oracle."""
    import speculative_decoding_token_rejection_gb300 as sv
    w = workloads.make("fused", N=32, V=30000, seed=41)
    add_lists(w, np.random.default_rng(12), theta=1.2, n_ctx=512, n_ban=16)
    o = oracle.verify(w)
    compare(H().run_gpu(w, flags=sv.SV_FLAG_RESIDENT_ROWS if resident else 0), o, w)
