"""Parity of the CUDA probability entry with the CPU oracle (GPU required).

Test mode (u and E given as tensors): every output -- committed tokens,
num_accepted, num_computed_tokens, slot_mapping, the gathered p(y)/q(y) and the
status word -- must be bit-exact.  Production mode (Philox inside the kernel)
is compared with the oracle's own Philox draws: the acceptance counts are exact
(u is exact on both sides); a token may differ only where the oracle reports
two race keys within a relative 1e-6 of each other (E = -ln U is evaluated by
different log routines), and such requests are counted.  The production
sampler must also pass the chi-square test of the closed-form outcome law.
"""
import numpy as np
import pytest
import scipy.stats

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


# ----------------------------------------------------------------------------
# hand-built edge cases: identical outputs and status bits
# ----------------------------------------------------------------------------
def _one(k, V):
    return [1.0 if x == k else 0.0 for x in range(V)]


def edge_cases():
    c = {}
    c["worked_example_reject"] = hand_workload([[0.6, 0.4], [0.3, 0.7]], [[0.2, 0.8]], [1], u=[0.7], E=[[1, 1]])
    c["worked_example_accept"] = hand_workload([[0.6, 0.4], [0.3, 0.7]], [[0.2, 0.8]], [1], u=[0.3], E=[[0.1, 1]])
    c["tie_reject"] = hand_workload([[0.25, 0.75], [0.5, 0.5]], [[0.5, 0.5]], [0], u=[0.5], E=[[1, 1]])
    c["race_tie"] = hand_workload([[0.1, 0.3, 0.3, 0.3]] * 2, [[0.7, 0.1, 0.1, 0.1]], [0], u=[0.99],
                                  E=[[1.0, 2.0, 0.5, 0.5]])
    c["race_inf_tie"] = hand_workload([[0.1, 0.3, 0.3, 0.3]] * 2, [[0.7, 0.1, 0.1, 0.1]], [0], u=[0.99],
                                      E=[[1.0, 1e-45, 1.0, 1e-45]])
    q = np.array([0.25] * 4, np.float32)
    p = (q * np.float32(0.999)).astype(np.float32)
    c["fallback"] = hand_workload([p, p], [q], [1], u=[0.9995], E=[[3.0, 1.0, 0.5, 2.0]])
    c["empty"] = hand_workload([[0.0, 0.0, 0.0]], np.zeros((0, 3)), [], u=[], E=[[1, 1, 1]])
    c["gamma0_and_ragged"] = hand_workload([_one(3, 8), _one(6, 8), _one(1, 8), _one(5, 8), _one(1, 8),
                                            _one(2, 8), _one(7, 8), _one(0, 8)],
                                           [_one(3, 8), _one(4, 8), _one(1, 8), _one(2, 8), _one(7, 8)],
                                           [3, 4, 1, 2, 7], [2, 0, 3], u=[0.5] * 5, E=np.ones((3, 8)),
                                           ncomp=[50, 0, 70], slots=list(range(100, 108)))
    pp = [[0.5, 0.5]] * 4
    base = dict(u=[0.1, 0.1], E=[[1, 1], [1, 1]], ncomp=[10, 10], slots=[1, 2, 3, 4])
    c["bad_draft_id"] = hand_workload(pp, [[0.5, 0.5]] * 2, [0, 5], [1, 1], **base)
    w = hand_workload(pp, [[0.5, 0.5]] * 2, [0, 1], [1, 1], **base)
    w["cu_num_draft_tokens"] = np.array([2, 1], np.int32)
    c["bad_cu"] = w
    c["bad_temperature"] = hand_workload(pp, [[0.5, 0.5]] * 2, [0, 1], [1, 1], temperature=[1.0, float("nan")],
                                         **base)
    c["bad_exponential"] = hand_workload([[0.9, 0.1], [0.5, 0.5]], [[0.1, 0.9]], [1], u=[0.99], E=[[-1.0, 1.0]])
    c["missing_draft"] = hand_workload([[0.5, 0.5]] * 2, None, [0], u=[0.1], E=[[1, 1]])
    c["bad_id_after_reject"] = hand_workload([[1.0, 0.0], [0.5, 0.5], [0.5, 0.5]], [[0.0, 1.0], [0.5, 0.5]],
                                             [1, 9], u=[0.5, 0.5], E=[[1, 1]])
    rows = np.full((5, 5), 0.05, np.float32)
    for j, k in enumerate([0, 1, 4, 0, 3]):
        rows[j, k] = 0.8
    c["greedy_example"] = hand_workload(rows, None, [0, 1, 2, 3], temperature=[0.0], u=[0] * 4, E=[[1] * 5])
    c["greedy_all_match"] = hand_workload(rows, None, [0, 1, 4, 0], temperature=[0.0], u=[0] * 4, E=[[1] * 5])
    c["greedy_ties"] = hand_workload([[0.1, 0.4, 0.4, 0.1], [0.25] * 4], None, [1], temperature=[0.0], u=[0],
                                     E=[[1] * 4])
    c["greedy_nan"] = hand_workload([[0.1, np.nan, 0.4, 0.1], [0.25] * 4], None, [1], temperature=[0.0], u=[0],
                                    E=[[1] * 4])
    c["greedy_neg_zero"] = hand_workload([[-0.0, 0.0, -1.0], [0.0, -0.0, -2.0]], None, [1], temperature=[0.0],
                                         u=[0], E=[[1] * 3])
    # mixed batch: an all-accept request next to a first-position reject (page 2, section 14)
    c["cross_talk"] = hand_workload([_one(1, 4), _one(2, 4), _one(3, 4), _one(0, 4), _one(1, 4), _one(2, 4)],
                                    [_one(1, 4), _one(2, 4), _one(2, 4), _one(2, 4)], [1, 2, 2, 2], [2, 2],
                                    u=[0.5] * 4, E=np.ones((2, 4)), ncomp=[20, 30], slots=list(range(6)))
    return c


@pytest.mark.parametrize("name", sorted(edge_cases()))
@pytest.mark.parametrize("cluster", [1, 4])
def test_edge_cases(name, cluster):
    w = edge_cases()[name]
    o = oracle.verify(w, with_diag=False)
    g = H().run_gpu(w, cluster_ctas=cluster)
    H().assert_same(g, o)


# ----------------------------------------------------------------------------
# seeded workloads, test mode: bit-exact
# ----------------------------------------------------------------------------
CASES = [
    ("tiny", {}),
    ("random", {}),                       # N=64, gamma=4, V=128256
    ("random", dict(N=9, V=4099)),        # rows not 16-byte aligned: scalar path
    ("random", dict(N=17, V=4100)),       # aligned rows, ragged last chunk
    ("random", dict(N=5, gamma=0, V=5000)),
    ("random", dict(N=3, gamma=31, V=3000)),
    ("fused_probs", dict(N=32, V=8192)),  # sparse rows (top-50 support)
]


@pytest.mark.parametrize("name,kw", CASES)
def test_seeded_test_mode(name, kw):
    w = workloads.make(name, **kw)
    o = oracle.verify(w, with_diag=False)
    g = H().run_gpu(w)
    H().assert_same(g, o)
    assert g["status"] == 0


@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
def test_cluster_sizes_agree(cluster):
    w = workloads.make("random", N=12, V=20000, seed=21)
    o = oracle.verify(w, with_diag=False)
    H().assert_same(H().run_gpu(w, cluster_ctas=cluster), o)


def test_mixed_greedy_and_random():
    w = workloads.make("random", N=40, V=6000, seed=8)
    w["temperature"] = np.where(np.arange(40) % 3 == 0, 0.0, 1.0).astype(np.float32)
    # make some greedy requests match: set their drafts to the target argmax
    G = w["gamma"]
    for i in range(0, 40, 6):
        for j in range(G):
            w["draft_ids"][i * G + j] = int(np.argmax(w["target"][i * (G + 1) + j]))
    o = oracle.verify(w, with_diag=False)
    H().assert_same(H().run_gpu(w), o)
    assert (o["num_accepted"][::6] == G).all()


def test_ragged_probs():
    w = workloads.make("random", N=50, V=7000, seed=13)
    rng = np.random.default_rng(1)
    gam = rng.integers(0, w["gamma"] + 1, size=50)
    # keep a prefix of each request's drafts to build a ragged batch
    G = w["gamma"]
    keep_d = np.concatenate([np.arange(i * G, i * G + g) for i, g in enumerate(gam)])
    keep_t = np.concatenate([np.arange(i * (G + 1), i * (G + 1) + g + 1) for i, g in enumerate(gam)])
    w.update(draft_ids=w["draft_ids"][keep_d], draft=w["draft"][keep_d], target=w["target"][keep_t],
             uniforms=w["uniforms"][keep_d], cu_num_draft_tokens=np.cumsum(gam).astype(np.int32),
             T=int(gam.sum()), slot_mapping=w["slot_mapping"][keep_t])
    o = oracle.verify(w, with_diag=False)
    H().assert_same(H().run_gpu(w), o)


def test_full_size_headline_batch_test_mode():
    """N=512, gamma=7, V=151936 fp32 probability rows: every request checked."""
    w = _headline()
    o = oracle.verify(w, with_diag=False)
    H().assert_same(H().run_gpu(w), o)


_HEAD = {}


def _headline():
    if "w" not in _HEAD:
        _HEAD["w"] = workloads.make("fused_probs")
    return _HEAD["w"]


# ----------------------------------------------------------------------------
# production mode (in-kernel Philox)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("name,kw,seed,offset", [
    ("random", {}, 1234, 0),
    ("random", dict(N=9, V=4099), 5, 77),
    ("fused_probs", dict(N=64, V=16384), 99, 3),
])
def test_production_matches_oracle_philox(name, kw, seed, offset):
    w = workloads.make(name, test_mode=False, **kw)
    o = oracle.verify(w, production=True, seed=seed, offset=offset, rng_request_base=7)
    g = H().run_gpu(w, production=True, seed=seed, offset=offset, rng_request_base=7)
    near = o["diag"][:, oracle.DIAG_RACE_RELGAP] < 1e-6
    H().assert_same(g, o, exempt=near)
    assert near.sum() <= max(1, w["N"] // 100)


def test_production_full_size_headline():
    w = dict(_headline())
    w["uniforms"] = w["exponentials"] = None
    o = oracle.verify(w, production=True, seed=42, offset=9)
    g = H().run_gpu(w, production=True, seed=42, offset=9)
    near = o["diag"][:, oracle.DIAG_RACE_RELGAP] < 1e-6
    H().assert_same(g, o, exempt=near)
    assert near.sum() <= 5


def test_production_is_deterministic_and_offset_sensitive():
    w = workloads.make("random", N=32, V=9000, test_mode=False)
    a = H().run_gpu(w, production=True, seed=3, offset=1)
    b = H().run_gpu(w, production=True, seed=3, offset=1)
    c = H().run_gpu(w, production=True, seed=3, offset=2)
    np.testing.assert_array_equal(a["out_tokens"], b["out_tokens"])
    assert not np.array_equal(a["out_tokens"], c["out_tokens"])


def _closed_form_case():
    import test_oracle_stats as st
    return st


@pytest.mark.parametrize("seed", [11, 12])
def test_production_chi_square_closed_form(seed):
    """10^6 requests at V=3, gamma=2 with drafts y_j ~ q_j: the GPU's outcome
    frequencies match the exact closed form (page 2, section 04) at p > 0.01."""
    st = _closed_form_case()
    n = 1_000_000
    rng = np.random.default_rng(seed)
    w = st._sample_workload(n, rng)
    w["uniforms"] = w["exponentials"] = None
    g = H().run_gpu(w, production=True, seed=seed, offset=0)
    assert g["status"] == 0
    assert st._chi2_outcomes(g["out_tokens"], g["num_accepted"], n) > 0.01
    first = np.bincount(g["out_tokens"][:, 0], minlength=st.V)
    assert scipy.stats.chisquare(first, n * np.array(st.P_ROWS[0]) / 16).pvalue > 0.01


def test_production_chi_square_v8_first_token():
    """V=8, gamma=3: the first committed token follows p_0 (10^6 trials)."""
    n = 1_000_000
    V, G = 8, 3
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.ones(V), size=G + 1).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, size=G).astype(np.float32)
    ids = np.stack([rng.choice(V, size=n, p=q[j].astype(np.float64) / q[j].astype(np.float64).sum())
                    for j in range(G)], axis=1).reshape(-1)
    w = hand_workload(np.tile(p, (n, 1)), np.tile(q, (n, 1)), ids)
    g = H().run_gpu(w, production=True, seed=77, offset=1)
    first = np.bincount(g["out_tokens"][:, 0], minlength=V)
    expect = p[0].astype(np.float64) / p[0].astype(np.float64).sum()
    assert scipy.stats.chisquare(first, n * expect).pvalue > 0.01


@pytest.mark.parametrize("production", [False, True])
def test_pinned_host_rows_zero_copy(production):
    """Probability rows left in pinned host memory (the path the end-to-end
    figure measures: the kernel reads them over the host link) against the
    oracle, bit for bit, in test mode (E in host memory too) and with
    production draws."""
    import torch
    import speculative_decoding_token_rejection_gb300 as sv
    w = workloads.make("fused_probs", N=48, V=16384)
    dev = torch.device("cuda:0")
    ref = oracle.verify(w, production=production, seed=12, offset=3)
    t = workloads.as_torch(w, dev)
    hp = torch.from_numpy(w["target"]).pin_memory()
    hq = torch.from_numpy(w["draft"]).pin_memory()
    hE = torch.from_numpy(w["exponentials"]).pin_memory()
    N, G, T = w["N"], w["gamma"], w["T"]
    out = torch.full((N, G + 1), -7, dtype=torch.int32, device=dev)
    nacc = torch.full((N,), -7, dtype=torch.int32, device=dev)
    ncomp = t["num_computed_tokens"].clone()
    slots = t["slot_mapping"].clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dpy = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    dqy = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    sv.spec_verify_run(H().verifier().handle, entry="probs", draft_ids=t["draft_ids"], target=hp, draft=hq,
                       temperature=t["temperature"], uniforms=None if production else t["uniforms"],
                       exponentials=None if production else hE, seed=12, offset=3, out_tokens=out,
                       num_accepted=nacc, num_computed_tokens=ncomp, slot_mapping=slots, dbg_py=dpy, dbg_qy=dqy,
                       status=status, device=dev, host_rows=True)
    torch.cuda.synchronize()
    g = dict(out_tokens=out.cpu().numpy(), num_accepted=nacc.cpu().numpy(), num_computed_tokens=ncomp.cpu().numpy(),
             slot_mapping=slots.cpu().numpy(), dbg_py=dpy.cpu().numpy(), dbg_qy=dqy.cpu().numpy(),
             status=int(status.item()))
    near = ref["diag"][:, oracle.DIAG_RACE_RELGAP] < 1e-6 if production else None  # an ulp of log in E
    H().assert_same(g, ref, exempt=near)
    assert near is None or near.sum() <= 1


@pytest.mark.parametrize("rates", [[0.9, 0.7, 0.7, 0.2], [1.0, 1.0, 1.0, 1.0], [0.0, 0.0, 0.0, 0.0],
                                   [0.5, 0.6, 0.1, 0.0]])
@pytest.mark.parametrize("production", [False, True])
def test_synthetic_acceptance_probs(rates, production):
    """Synthetic mode (preset non-increasing rates): bit-exact with the oracle,
    including the bad-rates status for the increasing set."""
    w = workloads.make("random", N=40, V=6000, seed=17, test_mode=not production)
    o = oracle.verify(w, production=production, seed=3, offset=1, synthetic_rates=np.array(rates, np.float32))
    g = H().run_gpu(w, production=production, seed=3, offset=1, synthetic_rates=rates)
    H().assert_same(g, o)
