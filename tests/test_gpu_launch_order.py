"""Launch order (GPU required).  By default every kernel is launched with
programmatic stream serialization, so it may be scheduled while the previous
kernel in the stream is still running; its first instruction waits for that
grid.  These tests run calls back to back, with no synchronisation between
them, where each call reads what the kernel just before it wrote -- the KV
bookkeeping (num_computed_tokens, slot_mapping) updated in place by the
previous verification, rows or histories written by a torch kernel -- and
compare with the oracle applied the same number of times, in the default
mode and under SV_FLAG_SERIAL_LAUNCH (plain stream order), and through a
CUDA graph of the same calls."""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CHAIN = 6  # calls back to back on the same bookkeeping buffers


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from speculative_decoding_token_rejection_gb300 import _build
    _build.build()
    oracle.build()


def _sv():
    import speculative_decoding_token_rejection_gb300 as sv
    return sv


_HANDLES = {}


def handle(flags):
    if flags not in _HANDLES:
        _HANDLES[flags] = _sv().Verifier(256, 8, 1 << 15, device=0, flags=flags)
    return _HANDLES[flags].handle


def chained_oracle(w, n):
    """The oracle applied n times, each time to the bookkeeping the previous
    application left; returns the last result."""
    nc, sl = w["num_computed_tokens"], w["slot_mapping"]
    for _ in range(n):
        o = oracle.verify(w, num_computed_tokens=nc, slot_mapping=sl)
        nc, sl = o["num_computed_tokens"], o["slot_mapping"]
    return o


def enqueue_verify(h, t, w, ncomp, slots, out, nacc, status):
    _sv().spec_verify_run(
        h, entry=w["entry"], draft_ids=t["draft_ids"], target=t["target"], draft=t["draft"],
        cu_num_draft_tokens=t["cu_num_draft_tokens"], temperature=t["temperature"], top_k=t.get("top_k"),
        top_p=t.get("top_p"), uniforms=t["uniforms"], exponentials=t["exponentials"], out_tokens=out,
        num_accepted=nacc, num_computed_tokens=ncomp, slot_mapping=slots, status=status)


def flags_of(mode):
    sv = _sv()
    return {"default": 0, "serial": sv.SV_FLAG_SERIAL_LAUNCH,
            "one_cta": sv.SV_FLAG_ONE_CTA_PER_REQUEST,
            "one_cta_serial": sv.SV_FLAG_ONE_CTA_PER_REQUEST | sv.SV_FLAG_SERIAL_LAUNCH}[mode]


CASES = [("random", dict(N=48, gamma=5, V=3000)),   # probability entry
         ("fused", dict(N=40, gamma=6, V=9000))]   # logits entry (bf16)


@pytest.mark.parametrize("name,kw", CASES)
@pytest.mark.parametrize("mode", ["default", "serial", "one_cta", "one_cta_serial"])
def test_verify_chain_reads_previous_bookkeeping(name, kw, mode):
    """CHAIN verifications back to back, each reading num_computed_tokens and
    slot_mapping as the previous kernel left them; the target rows are
    written by a torch kernel just before the first call."""
    w = workloads.make(name, **kw)
    dev = torch.device("cuda:0")
    t = workloads.as_torch(w, dev)
    src = t["target"].clone()
    t["target"].zero_()
    N, G = w["N"], w["gamma"]
    ncomp = t["num_computed_tokens"].clone()
    slots = t["slot_mapping"].clone()
    outs = [torch.full((N, G + 1), -7, dtype=torch.int32, device=dev) for _ in range(CHAIN)]
    naccs = [torch.full((N,), -7, dtype=torch.int32, device=dev) for _ in range(CHAIN)]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    h = handle(flags_of(mode))
    torch.cuda.synchronize()
    torch.mul(src, 1, out=t["target"])  # rows written by a kernel right before the first call
    for k in range(CHAIN):
        enqueue_verify(h, t, w, ncomp, slots, outs[k], naccs[k], status)
    torch.cuda.synchronize()
    o = chained_oracle(w, CHAIN)
    np.testing.assert_array_equal(ncomp.cpu().numpy(), o["num_computed_tokens"])
    np.testing.assert_array_equal(slots.cpu().numpy(), o["slot_mapping"])
    assert int(status.item()) == o["status"]
    if w["entry"] == "probs":  # test mode is bit-exact for the probability entry
        for k in range(CHAIN):
            np.testing.assert_array_equal(naccs[k].cpu().numpy(), o["num_accepted"])
            np.testing.assert_array_equal(outs[k].cpu().numpy(), o["out_tokens"])
    else:  # every call of the chain gives the same result, with the oracle's acceptance counts
        np.testing.assert_array_equal(naccs[0].cpu().numpy(), o["num_accepted"])
        for k in range(1, CHAIN):
            np.testing.assert_array_equal(naccs[k].cpu().numpy(), naccs[0].cpu().numpy())
            np.testing.assert_array_equal(outs[k].cpu().numpy(), outs[0].cpu().numpy())


@pytest.mark.parametrize("mode", ["default", "serial"])
def test_verify_chain_in_cuda_graph(mode):
    """Three chained verifications captured in a CUDA graph and the graph
    replayed twice: the bookkeeping sees all six calls in order."""
    w = workloads.make("random", N=32, gamma=4, V=2048)
    dev = torch.device("cuda:0")
    t = workloads.as_torch(w, dev)
    N, G = w["N"], w["gamma"]
    ncomp = t["num_computed_tokens"].clone()
    slots = t["slot_mapping"].clone()
    out = torch.full((N, G + 1), -7, dtype=torch.int32, device=dev)
    nacc = torch.full((N,), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    h = handle(flags_of(mode))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for _ in range(3):
                enqueue_verify(h, t, w, ncomp, slots, out, nacc, status)
    torch.cuda.synchronize()
    ncomp.copy_(t["num_computed_tokens"])  # (capture launched nothing; restore anyway)
    slots.copy_(t["slot_mapping"])
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    o = chained_oracle(w, 6)
    np.testing.assert_array_equal(ncomp.cpu().numpy(), o["num_computed_tokens"])
    np.testing.assert_array_equal(slots.cpu().numpy(), o["slot_mapping"])
    np.testing.assert_array_equal(nacc.cpu().numpy(), o["num_accepted"])
    np.testing.assert_array_equal(out.cpu().numpy(), o["out_tokens"])


@pytest.mark.parametrize("mode", ["default", "serial"])
def test_ngram_reads_histories_written_just_before(mode):
    """Histories written by a torch kernel right before each of several
    back-to-back proposer calls (each call sees its own batch)."""
    sv = _sv()
    dev = torch.device("cuda:0")
    flags = flags_of(mode)
    h = sv.spec_verify_create(64, 5, 1, device=0, flags=flags)
    try:
        batches = [workloads.make_histories(R=64, min_len=16, max_len=1500, vocab=40, seed=70 + b) for b in range(4)]
        n = max(len(tk) for tk, _ in batches)
        buf = torch.zeros(n, dtype=torch.int32, device=dev)
        srcs = [torch.as_tensor(np.pad(tk, (0, n - len(tk)))).to(dev) for tk, _ in batches]
        cus = [torch.as_tensor(cu).to(dev) for _, cu in batches]
        outs = [torch.full((64, 5), -7, dtype=torch.int32, device=dev) for _ in batches]
        nums = [torch.full((64,), -7, dtype=torch.int32, device=dev) for _ in batches]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        for b in range(len(batches)):
            torch.add(srcs[b], 0, out=buf)  # this call's histories, written by a kernel
            sv.spec_verify_ngram_propose(h, token_ids=buf, cu_num_tokens=cus[b], draft_token_ids=outs[b],
                                         num_draft_tokens=nums[b], min_ngram=2, max_ngram=4, max_model_len=1 << 20,
                                         status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for b, (tk, cu) in enumerate(batches):
            o = oracle.ngram_propose(tk, cu, min_ngram=2, max_ngram=4, k=5, max_model_len=1 << 20)
            np.testing.assert_array_equal(nums[b].cpu().numpy(), o["num_draft_tokens"])
            np.testing.assert_array_equal(outs[b].cpu().numpy(), o["draft_token_ids"])
    finally:
        sv.spec_verify_destroy(h)


@pytest.mark.parametrize("mode", ["default", "serial", "one_cta"])
def test_sampler_then_verify_same_stream(mode):
    """The draft-side sampler writes its tokens and q rows; the verification
    enqueued right after reads them as draft ids and draft rows (the pipeline
    order of a speculative step).  The result equals the oracle run on the
    sampler's outputs as they ended up."""
    sv = _sv()
    w = workloads.make("fused", N=24, gamma=1, V=5000)
    dev = torch.device("cuda:0")
    t = workloads.as_torch(w, dev)
    N, V = w["N"], w["V"]
    flags = flags_of(mode)
    h = handle(flags)
    tok = torch.full((N,), -7, dtype=torch.int32, device=dev)
    q = torch.full((N, V), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    hints = sv.SV_HINT_SMALL_TOP_K if mode == "one_cta" else 0
    draft_rows = t["draft"]  # [T=N, V] bf16 logits, one draft position per request
    torch.cuda.synchronize()
    sv.spec_verify_sample(h, logits=draft_rows, tokens=tok, probs=q, temperature=t["temperature"],
                          top_k=t.get("top_k"), top_p=t.get("top_p"), exponentials=t["exponentials"],
                          status=status, hints=hints)
    out = torch.full((N, 2), -7, dtype=torch.int32, device=dev)
    nacc = torch.full((N,), -7, dtype=torch.int32, device=dev)
    # the probability entry with the sampler's q rows as both draft and target rows (p = q, the
    # bonus row a copy too); the copies and the verification are enqueued without a pause
    target = torch.repeat_interleave(q, 2, dim=0)
    sv.spec_verify_run(h, entry="probs", draft_ids=tok, target=target, draft=q, cu_num_draft_tokens=None,
                       temperature=torch.ones(N, device=dev), uniforms=t["uniforms"],
                       exponentials=t["exponentials"], out_tokens=out, num_accepted=nacc, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # p = q, so every sampled token is accepted (u * q(y) < q(y) for u < 1 and q(y) > 0)
    np.testing.assert_array_equal(nacc.cpu().numpy(), np.ones(N, np.int32))
    np.testing.assert_array_equal(out.cpu().numpy()[:, 0], tok.cpu().numpy())
    assert (tok.cpu().numpy() >= 0).all()
