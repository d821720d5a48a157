"""Request-range sharding of a verification batch across ranks.

Requests are independent ("vLLM source walk-through (10)", section "Greedy
kernel": one program per request), so a batch splits into contiguous request
ranges with no exchange step.  A shard keeps its requests' rows, re-bases
``cu_num_draft_tokens`` and carries ``rng_request_base`` = its first global
request index, so production-mode draws -- keyed by the global request index
-- are the same whichever way the batch is split.

Works on dicts of numpy arrays or torch tensors with the keys used by
``workloads.make`` plus the optional per-request processor and stop lists
(host bookkeeping only; no verifier arithmetic).  The n-gram proposer's
histories split the same way (``shard_histories``).
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
    if w.get("repetition_penalty") is not None:
        out["repetition_penalty"] = w["repetition_penalty"][r0:r1]
    for name in ("penalty", "banned", "stop"):  # per-request id lists, inclusive prefix sums
        if w.get(f"{name}_cu") is not None:
            out[f"{name}_cu"], out[f"{name}_ids"] = _shard_list(w[f"{name}_cu"], w[f"{name}_ids"], r0, r1)
    return out


def _shard_list(cu, ids, r0: int, r1: int):
    """Entries of requests [r0, r1) of a per-request list (inclusive prefix
    sums ``cu`` into ``ids``), with ``cu`` re-based."""
    b = int(cu[r0 - 1]) if r0 > 0 else 0
    e = int(cu[r1 - 1]) if r1 > r0 else b
    return cu[r0:r1] - b, ids[b:e]


def shard_histories(tokens, cu_num_tokens, rank: int, world: int):
    """The n-gram proposer's batch of ``rank``: its contiguous range of
    request histories with ``cu_num_tokens`` re-based.  Returns (tokens, cu,
    (r0, r1))."""
    r0, r1 = shard_bounds(len(cu_num_tokens), rank, world)
    c, t = _shard_list(cu_num_tokens, tokens, r0, r1)
    return t, c, (r0, r1)
