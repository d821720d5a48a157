"""The CUDA n-gram proposer against the oracle (through the C ABI)."""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _sv():
    import speculative_decoding_token_rejection_gb300 as sv
    return sv


_HANDLES = {}


def handle(R, k):
    key = (R, k)
    if key not in _HANDLES:
        _HANDLES[key] = _sv().spec_verify_create(max(R, 1), max(k, 0), 1, device=0)
    return _HANDLES[key]


def run_gpu(tokens, cu, *, min_n, max_n, k, mml, misalign=0):
    dev = torch.device("cuda:0")
    R = len(cu)
    # misalign: the token buffer starts `misalign` int32 past a 16-byte boundary (plain loads, no bulk copies)
    t = torch.as_tensor(np.concatenate([np.zeros(misalign, np.int32), np.asarray(tokens, np.int32)])).to(dev)
    t = t[misalign:]
    c = torch.as_tensor(np.asarray(cu, np.int64)).to(dev)
    out = torch.full((R, k), -7, dtype=torch.int32, device=dev)
    num = torch.full((R,), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _sv().spec_verify_ngram_propose(handle(R, k), token_ids=t, cu_num_tokens=c, draft_token_ids=out,
                                    num_draft_tokens=num, min_ngram=min_n, max_ngram=max_n, max_model_len=mml,
                                    status=st)
    torch.cuda.synchronize()
    return dict(draft_token_ids=out.cpu().numpy(), num_draft_tokens=num.cpu().numpy(), status=int(st.item()))


def check(tokens, cu, misalign=0, **kw):
    g = run_gpu(tokens, cu, misalign=misalign, **kw)
    o = oracle.ngram_propose(tokens, cu, min_ngram=kw["min_n"], max_ngram=kw["max_n"], k=kw["k"],
                             max_model_len=kw["mml"])
    np.testing.assert_array_equal(g["num_draft_tokens"], o["num_draft_tokens"])
    np.testing.assert_array_equal(g["draft_token_ids"], o["draft_token_ids"])
    assert g["status"] == o["status"]
    return g


@pytest.mark.parametrize("alphabet", [2, 3, 5, 1000])
def test_small_random_batches(alphabet):
    rng = np.random.default_rng(alphabet)
    for rep in range(6):
        lens = rng.integers(0, 300, size=37)
        lens[::9] = rng.integers(0, 4, size=lens[::9].shape)  # very short histories too
        tokens = rng.integers(0, alphabet, size=int(lens.sum())).astype(np.int32)
        min_n = int(rng.integers(1, 4))
        max_n = int(rng.integers(min_n, 9))
        k = int(rng.integers(0, 9))
        g = check(tokens, np.cumsum(lens), min_n=min_n, max_n=max_n, k=k, mml=int(rng.integers(150, 400)))
        if alphabet <= 3 and k > 0:
            assert (g["num_draft_tokens"] > 0).any()


def test_repetitive_histories_moderate():
    tokens, cu = workloads.make_histories(48, min_len=300, max_len=5000, vocab=50, p_copy=0.6, seed=3)
    for (min_n, max_n, k) in [(5, 5, 7), (2, 5, 4), (1, 64, 8), (3, 12, 0)]:
        check(tokens, cu, min_n=min_n, max_n=max_n, k=k, mml=1 << 20)


def test_max_model_len_and_edges():
    rng = np.random.default_rng(8)
    hist = [np.array([1, 2, 3, 4, 1, 2, 3]), np.array([3, 3, 3, 3, 3]), np.zeros(0, np.int64), np.array([9]),
            rng.integers(0, 2, size=200)]
    tokens = np.concatenate(hist).astype(np.int32)
    cu = np.cumsum([len(h) for h in hist])
    for mml in (1, 5, 7, 8, 10, 1000):
        for (min_n, max_n) in [(1, 1), (1, 3), (3, 3), (2, 64)]:
            check(tokens, cu, min_n=min_n, max_n=max_n, k=6, mml=mml)


def test_bad_ranges_report_status():
    tokens = np.arange(40, dtype=np.int32) % 4
    cu = np.array([10, 8, 30, 41], np.int64)  # request 1 ends before it starts; request 3 runs past the end
    g = check(tokens, cu, min_n=1, max_n=3, k=3, mml=100)
    assert g["status"] == oracle.BAD_CU
    assert g["num_draft_tokens"][1] == 0 and g["num_draft_tokens"][3] == 0


def test_full_batch_sampled():
    """The default batch (512 requests, 1024..16384 tokens) in one launch; the
    oracle checks a seeded sample of requests one by one."""
    tokens, cu = workloads.make_histories()
    k, min_n, max_n = 7, 5, 5
    g = run_gpu(tokens, cu, min_n=min_n, max_n=max_n, k=k, mml=1 << 20)
    assert g["status"] == 0
    starts = np.concatenate([[0], cu[:-1]])
    for q in np.random.default_rng(0).choice(len(cu), size=24, replace=False):
        h = tokens[starts[q]:cu[q]]
        o = oracle.ngram_propose(h, [len(h)], min_ngram=min_n, max_ngram=max_n, k=k, max_model_len=1 << 20)
        assert g["num_draft_tokens"][q] == o["num_draft_tokens"][0]
        np.testing.assert_array_equal(g["draft_token_ids"][q], o["draft_token_ids"][0])
    assert (g["num_draft_tokens"] > 0).mean() > 0.25  # half the segments repeat: many tails were seen before


@pytest.mark.parametrize("misalign", [0, 1, 3])
def test_histories_across_chunks(misalign):
    """Histories longer than one shared-memory chunk (12284 tokens), with
    matches on both sides of every chunk boundary (a three-token alphabet),
    through bulk copies (aligned buffer) and plain loads (misaligned)."""
    rng = np.random.default_rng(17 + misalign)
    lens = np.array([12283, 12284, 12285, 12290, 24570, 30001, 5, 4097])
    tokens = rng.integers(0, 3, size=int(lens.sum())).astype(np.int32)
    cu = np.cumsum(lens)
    for (min_n, max_n, k) in [(8, 8, 5), (1, 20, 7), (3, 5, 3)]:
        check(tokens, cu, misalign=misalign, min_n=min_n, max_n=max_n, k=k, mml=1 << 20)


@pytest.mark.parametrize("misalign", [1, 2])
def test_repetitive_histories_misaligned_buffer(misalign):
    tokens, cu = workloads.make_histories(24, min_len=300, max_len=20000, vocab=50, p_copy=0.6, seed=5)
    check(tokens, cu, misalign=misalign, min_n=5, max_n=5, k=7, mml=1 << 20)
