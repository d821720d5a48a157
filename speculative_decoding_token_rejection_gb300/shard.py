"""Request-range sharding of a verification batch across ranks.

Requests are independent ("vLLM source walk-through (10)", section "Greedy
kernel": one program per request), so a batch splits into contiguous request
ranges with no exchange step.  A shard keeps its requests' rows, re-bases
``cu_num_draft_tokens`` and carries ``rng_request_base`` = its first global
request index, so production-mode draws -- keyed by the global request index
-- are the same whichever way the batch is split.

Works on dicts of numpy arrays or torch tensors with the keys used by
``workloads.make`` (host bookkeeping only; no verifier arithmetic).
"""
from __future__ import annotations


def shard_bounds(num_reqs: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced request range [r0, r1) of ``rank``."""
    if not (0 <= rank < world):
        raise ValueError("rank out of range")
    base, extra = divmod(num_reqs, world)
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def _starts(w: dict):
    """Exclusive prefix sums s_i of the draft counts (length N+1)."""
    N, G = int(w["N"]), int(w["gamma"])
    cu = w.get("cu_num_draft_tokens")
    if cu is None:
        return [i * G for i in range(N + 1)]
    vals = [int(v) for v in (cu.tolist() if hasattr(cu, "tolist") else cu)]
    return [0] + vals


def shard_workload(w: dict, rank: int, world: int) -> dict:
    """The sub-batch of ``rank``: rows, ids, parameters and bookkeeping of its
    requests, ``cu`` re-based, plus ``rng_request_base``."""
    r0, r1 = shard_bounds(int(w["N"]), rank, world)
    s = _starts(w)
    d0, d1 = s[r0], s[r1]          # draft rows / tokens
    t0, t1 = d0 + r0, d1 + r1      # target rows / verify tokens
    out = dict(w)
    out.update(N=r1 - r0, T=d1 - d0, rng_request_base=r0, shard=(r0, r1))
    out["draft_ids"] = w["draft_ids"][d0:d1]
    out["target"] = w["target"][t0:t1]
    if w.get("draft") is not None:
        out["draft"] = w["draft"][d0:d1]
    cu = w.get("cu_num_draft_tokens")
    if cu is not None:
        out["cu_num_draft_tokens"] = cu[r0:r1] - d0
    for k in ("temperature", "top_k", "top_p", "num_computed_tokens"):
        if w.get(k) is not None:
            out[k] = w[k][r0:r1]
    if w.get("uniforms") is not None:
        out["uniforms"] = w["uniforms"][d0:d1]
    if w.get("exponentials") is not None:
        out["exponentials"] = w["exponentials"][r0:r1]
    if w.get("slot_mapping") is not None:
        out["slot_mapping"] = w["slot_mapping"][t0:t1]
    return out
