"""World-size-2 sharding of a verification batch, on the CPU with gloo.

Each rank takes its contiguous request range (speculative_decoding_token_
rejection_gb300.shard), verifies it with the oracle in production mode keyed by
its first global request index, and rank 0 gathers the shards: the result
equals the unsharded batch exactly.  The same host logic drives the per-GPU
shards of bench.py under torchrun.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_token_rejection_gb300.shard import shard_bounds, shard_workload


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _with_lists(w):
    """Processor and stop lists on a workload (deterministic, per request)."""
    rng = np.random.default_rng(11)
    N, V = w["N"], w["V"]
    for name, n in (("penalty", 30), ("banned", 5), ("stop", 2)):
        lens = rng.integers(0, n, size=N)
        w[f"{name}_cu"] = np.cumsum(lens).astype(np.int64)
        w[f"{name}_ids"] = rng.integers(0, V, size=int(lens.sum())).astype(np.int32)
    if w["entry"] != "logits":
        for name in ("penalty", "banned"):
            w.pop(f"{name}_cu")
            w.pop(f"{name}_ids")
    else:
        w["repetition_penalty"] = rng.uniform(0.8, 1.6, size=N).astype(np.float32)
    return w


def _worker(rank, world, port, name, kw, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lists = kw.pop("lists", False)
        w = workloads.make(name, test_mode=False, **kw)
        if lists:
            w = _with_lists(w)
        sh = shard_workload(w, rank, world)
        r = oracle.verify(sh, production=True, seed=5, offset=3, rng_request_base=sh["rng_request_base"],
                          with_diag=False)
        part = {k: r[k] for k in ("out_tokens", "num_accepted", "num_computed_tokens", "slot_mapping")}
        part["status"] = r["status"]
        gathered = [None] * world
        dist.all_gather_object(gathered, part)
        if rank == 0:
            full = oracle.verify(w, production=True, seed=5, offset=3, with_diag=False)
            ok = all(np.array_equal(np.concatenate([g[k] for g in gathered]), full[k])
                     for k in ("out_tokens", "num_accepted", "num_computed_tokens", "slot_mapping"))
            ok = ok and all(g["status"] == 0 for g in gathered)
            q.put(ok)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,kw", [("random", dict(N=9, V=3000)), ("ragged", dict(N=13, V=2000)),
                                     ("fused", dict(N=6, V=4096)), ("fused", dict(N=7, V=4096, lists=True)),
                                     ("random", dict(N=9, V=3000, lists=True))])
def test_two_rank_shards_equal_unsharded(name, kw):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, name, kw, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    assert q.get(timeout=10) is True


def test_shard_bounds_cover_the_batch():
    for n in (0, 1, 7, 512):
        for world in (1, 2, 3, 8):
            spans = [shard_bounds(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1


def _ngram_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    import workloads
    from speculative_decoding_token_rejection_gb300.shard import shard_histories
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        tokens, cu = workloads.make_histories(11, min_len=20, max_len=300, vocab=7, seed=4)
        t, c, _ = shard_histories(tokens, cu, rank, world)
        r = oracle.ngram_propose(t, c, min_ngram=2, max_ngram=4, k=5, max_model_len=1000)
        gathered = [None] * world
        dist.all_gather_object(gathered, r)
        if rank == 0:
            full = oracle.ngram_propose(tokens, cu, min_ngram=2, max_ngram=4, k=5, max_model_len=1000)
            ok = all(np.array_equal(np.concatenate([g[k] for g in gathered]), full[k])
                     for k in ("draft_token_ids", "num_draft_tokens"))
            q.put(ok and (full["num_draft_tokens"] > 0).any())
    finally:
        dist.destroy_process_group()


def test_two_rank_ngram_shards_equal_unsharded():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ngram_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok
