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


def _worker(rank, world, port, name, kw, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.make(name, test_mode=False, **kw)
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
                                     ("fused", dict(N=6, V=4096))])
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
