"""Seeded synthetic workloads for the batched speculative-decoding verifier.

This module only *makes inputs*: draft/target logits or probability rows, draft
ids, uniforms ``u`` and exponentials ``E`` for test mode, the ragged
``cu_num_draft_tokens`` layout and the KV bookkeeping (``num_computed_tokens``,
``slot_mapping``).  It holds none of the verifier's arithmetic: no acceptance
test, no residual, no race and no rollback.  To *make* the fused workload's
draft ids and probability rows it samples from the stated distribution
(temperature 0.8, top-k 50, top-p 0.9) with a float32 recipe of its own
(``_nucleus_rows``: library topk and softmax, a numpy cumulative sum); the
verifier's transform itself lives in the oracle and the kernels.  Both the
CPU oracle and the CUDA path are fed from it with byte-identical arrays.

Shapes follow the tutorial page "Speculative Decoding: propose, verify, accept",
section 02: draft ids ``[N, gamma]``, draft rows ``[N, gamma, V]`` and target rows
``[N, gamma+1, V]``.  Requests are stored flattened and request-major, the
layout of vLLM's ``SpecDecodeMetadata`` (vLLM source walk-through part 10,
section "SpecDecodeMetadata"): draft row ``s_i + j`` and target row ``s_i + i + j``
with ``s_i`` the exclusive prefix sum of the per-request draft counts.

Recipes (one per named workload; sizes can be shrunk for parity tests):

* ``tiny``    N=4, gamma=4, V=1000; fp32 probability rows.  Target logits
  ~N(0, 2^2), draft logits = target + N(0, 0.5^2); both turned into probability
  rows with a plain float32 softmax (input synthesis); draft ids drawn from the
  draft rows by inverse CDF; u ~ U[0,1), E ~ Exp(1).
* ``greedy``  N=64, gamma=5, V=32000; bf16 logits, target ~N(0, 3^2), draft =
  target + N(0, 1); temperature 0; draft ids = argmax of the draft logits
  (greedy drafting); the draft logits themselves are not passed.
* ``random``  N=64, gamma=4, V=128256; as ``tiny`` with sigma 2 / 0.5.
* ``fused``   N=512, gamma=7, V=151936; bf16 logits, target ~N(0, 2.5^2), draft
  = target + N(0, 0.7^2); temperature 0.8, top-k 50, top-p 0.9 per request.
  Draft ids are drawn from the transformed draft rows (``_nucleus_rows``), as
  the draft-side sampler would draw them, so every draft lies in q's support.
* ``fused_probs``  the same batch materialised as fp32 probability rows for the
  probability entry: every target and draft row through ``_nucleus_rows``
  (its 50 largest logits, a float32 softmax at T=0.8, cut to the shortest
  descending prefix reaching 0.9 with ties at the cut kept, renormalised; zero
  elsewhere), and the same draft ids.
* ``ragged``  N=256, gamma_i ~ U{0..8} (ragged via ``cu_num_draft_tokens``),
  V=128256; bf16 logits, target ~N(0, 2^2), per-request draft noise sigma in
  {0.1, 1.0, 3.0}; a seeded half of the requests is greedy (T=0), the rest T=1
  without top-k/top-p; num_computed_tokens_i ~ U[gamma_i+1, 4096]; a random
  block table with block_size 16 gives int64 slot_mapping entries for the
  gamma_i+1 verify tokens at positions ncomp_i-gamma_i-1 .. ncomp_i-1.

N-gram proposer histories (``make_histories``; "vLLM source walk-through
(10)", section "NgramProposer": useful on repetitive text such as code,
formatted output and chat templates): each request's history starts with 32
fresh tokens; then, segment after segment (lengths U{8..64}), with probability
``p_copy`` an earlier stretch of the same history is repeated, else fresh tokens
are drawn uniformly from ``vocab`` ids.  Lengths are U{min_len..max_len}; the
``ngram`` batch is R=512, lengths 1024..16384, vocab 151936, p_copy 0.5.
"""
from __future__ import annotations

import numpy as np

BLOCK_SIZE = 16
MAX_CONTEXT = 4096

# name -> (N, gamma, V, entry, default seed)
WORKLOADS = {
    "tiny": dict(N=4, gamma=4, V=1000, entry="probs", seed=0),
    "greedy": dict(N=64, gamma=5, V=32000, entry="logits", seed=1),
    "random": dict(N=64, gamma=4, V=128256, entry="probs", seed=2),
    "fused": dict(N=512, gamma=7, V=151936, entry="logits", seed=3),
    "fused_probs": dict(N=512, gamma=7, V=151936, entry="probs", seed=3),
    "ragged": dict(N=256, gamma=8, V=128256, entry="logits", seed=4),
}


# ----------------------------------------------------------------------------
# small helpers (input synthesis only)
# ----------------------------------------------------------------------------
def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 -> bfloat16 (round-to-nearest-even) and return the raw
    uint16 bit patterns.  Inputs here are finite normals, so no NaN handling."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _softmax_rows_f32(x: np.ndarray) -> np.ndarray:
    """Plain float32 softmax over the last axis, used only to *make* probability
    rows for the probability entry."""
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m, dtype=np.float32)
    return (e / e.sum(axis=-1, keepdims=True, dtype=np.float32)).astype(np.float32)


def _inverse_cdf(rng: np.random.Generator, w: np.ndarray) -> np.ndarray:
    """Draw one index per row of non-negative weights ``w`` (rows of any scale)."""
    c = np.cumsum(w.astype(np.float64), axis=-1)
    t = rng.random(w.shape[0]) * c[:, -1]
    idx = (c < t[:, None]).sum(axis=-1)
    return np.minimum(idx, w.shape[-1] - 1).astype(np.int32)


def _exponentials(rng: np.random.Generator, shape) -> np.ndarray:
    e = rng.standard_exponential(shape, dtype=np.float32)
    e[e <= 0] = np.float32(1e-30)  # Exp(1) draws of exactly 0 are measure-zero; keep E > 0
    return e


def _kv_bookkeeping(rng, gammas: np.ndarray):
    """num_computed_tokens and int64 slot_mapping for the verify-token layout."""
    N = gammas.shape[0]
    ncomp = np.array([rng.integers(g + 1, MAX_CONTEXT + 1) for g in gammas], dtype=np.int32)
    blocks_per_req = MAX_CONTEXT // BLOCK_SIZE
    pool = rng.permutation(N * blocks_per_req).astype(np.int64).reshape(N, blocks_per_req)
    slots = []
    for i, g in enumerate(gammas):
        pos = np.arange(ncomp[i] - g - 1, ncomp[i], dtype=np.int64)
        slots.append(pool[i, pos // BLOCK_SIZE] * BLOCK_SIZE + pos % BLOCK_SIZE)
    return ncomp, np.concatenate(slots).astype(np.int64), pool


def _layout(gammas: np.ndarray):
    cu = np.cumsum(gammas).astype(np.int32)
    T = int(cu[-1]) if len(cu) else 0
    return cu, T


# ----------------------------------------------------------------------------
# public entry point
# ----------------------------------------------------------------------------
def make(name: str, seed: int | None = None, *, N: int | None = None, gamma: int | None = None,
         V: int | None = None, test_mode: bool = True) -> dict:
    """Build one workload.  Returns a dict of numpy arrays plus metadata.

    Keys: ``entry`` ('probs'|'logits'), ``dtype`` ('f32'|'bf16'), ``N``, ``gamma``
    (max_spec_len), ``V``, ``T`` (total draft tokens), ``draft_ids`` [T] int32,
    ``cu_num_draft_tokens`` [N] int32 or None (uniform gamma), ``target``
    [T+N, V] (float32 rows or uint16 bf16 bits), ``draft`` [T, V] or None,
    ``temperature`` [N] f32 or None, ``top_k`` [N] int32 or None, ``top_p`` [N]
    f32 or None, ``uniforms`` [T] f32 / ``exponentials`` [N, V] f32 (test mode,
    else None), ``num_computed_tokens`` [N] int32 and ``slot_mapping`` [T+N]
    int64 (or None).
    """
    spec = dict(WORKLOADS[name])
    N = spec["N"] if N is None else N
    G = spec["gamma"] if gamma is None else gamma
    V = spec["V"] if V is None else V
    seed = spec["seed"] if seed is None else seed
    rng = np.random.default_rng(seed)
    fn = {"tiny": _dense_probs, "random": _dense_probs, "greedy": _greedy, "fused": _fused,
          "fused_probs": _fused, "ragged": _ragged}[name]
    out = fn(name, rng, N, G, V)
    out.update(name=name, N=N, gamma=G, V=V, seed=seed)
    if test_mode:
        out["uniforms"] = rng.random(out["T"], dtype=np.float32)
        out["exponentials"] = _exponentials(rng, (N, V))
    else:
        out["uniforms"] = None
        out["exponentials"] = None
    return out


def _dense_probs(name, rng, N, G, V):
    sig_t, sig_d = 2.0, 0.5
    gammas = np.full(N, G, dtype=np.int64)
    T = N * G
    tl = rng.standard_normal((N, G + 1, V), dtype=np.float32) * np.float32(sig_t)
    dl = tl[:, :G] + rng.standard_normal((N, G, V), dtype=np.float32) * np.float32(sig_d)
    p = _softmax_rows_f32(tl).reshape(T + N, V)
    q = _softmax_rows_f32(dl).reshape(T, V)
    ids = _inverse_cdf(rng, q) if T else np.zeros(0, np.int32)
    ncomp, slots, _ = _kv_bookkeeping(rng, gammas)
    return dict(entry="probs", dtype="f32", T=T, draft_ids=ids, cu_num_draft_tokens=None,
                target=p, draft=q, temperature=np.ones(N, np.float32), top_k=None, top_p=None,
                num_computed_tokens=ncomp, slot_mapping=slots)


def _greedy(name, rng, N, G, V):
    gammas = np.full(N, G, dtype=np.int64)
    T = N * G
    tl = rng.standard_normal((N, G + 1, V), dtype=np.float32) * np.float32(3.0)
    t_bits = _to_bf16_bits(tl).reshape(T + N, V)
    dl = bf16_bits_to_f32(t_bits.reshape(N, G + 1, V)[:, :G]) + rng.standard_normal((N, G, V), dtype=np.float32)
    d_bits = _to_bf16_bits(dl).reshape(T, V)
    ids = bf16_bits_to_f32(d_bits).argmax(axis=-1).astype(np.int32)  # greedy drafting
    ncomp, slots, _ = _kv_bookkeeping(rng, gammas)
    return dict(entry="logits", dtype="bf16", T=T, draft_ids=ids, cu_num_draft_tokens=None,
                target=t_bits, draft=None, temperature=np.zeros(N, np.float32), top_k=None,
                top_p=None, num_computed_tokens=ncomp, slot_mapping=slots)


def _nucleus_rows(rows_f32: np.ndarray, temp: float, k: int, top_p: float):
    """Input synthesis for the fused workload.  For each row: the indices of its
    largest values -- the k largest and every value tied with the k-th -- and
    their weights: a float32 softmax of value/temp over that set, cut to the
    shortest descending prefix whose float64 cumulative sum reaches ``top_p``
    (every entry equal to the last kept value kept too), renormalised in
    float64 and rounded to float32; 0 for the entries the cut drops.  Returns
    (indices [rows, m], weights [rows, m]) with m >= k."""
    import torch
    x = torch.from_numpy(np.ascontiguousarray(rows_f32))
    m = min(x.shape[-1], 4 * k)
    while True:  # widen until no row's tie at the k-th value runs past the m taken
        vals, idx = torch.topk(x, m, dim=-1, largest=True, sorted=True)
        if m == x.shape[-1] or bool((vals[:, -1] < vals[:, k - 1]).all()):
            break
        m = min(x.shape[-1], 2 * m)
    in_k = vals >= vals[:, k - 1:k]
    z = torch.where(in_k, vals / temp, torch.tensor(float("-inf")))
    w = torch.softmax(z, dim=-1, dtype=torch.float32).numpy().astype(np.float64)
    v = vals.numpy()
    first = (np.cumsum(w, axis=-1) < top_p).sum(axis=-1)  # first entry reaching top_p
    first = np.minimum(first, in_k.numpy().sum(axis=-1) - 1)
    keep = v >= v[np.arange(v.shape[0]), first][:, None]
    w = np.where(keep, w, 0.0)
    w /= w.sum(axis=-1, keepdims=True)
    return idx.numpy().astype(np.int64), w.astype(np.float32)


def _fused(name, rng, N, G, V):
    """Chunks of requests are generated in parallel threads, each from its own
    child stream of the workload seed, so the result does not depend on the
    thread count."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    temp, k, top_p = 0.8, 50, 0.9
    gammas = np.full(N, G, dtype=np.int64)
    T = N * G
    kk = min(k, V)
    t_bits = np.empty((N, G + 1, V), dtype=np.uint16)
    d_bits = np.empty((N, G, V), dtype=np.uint16)
    ids = np.zeros((N, G), dtype=np.int32)
    probs = name == "fused_probs"
    if probs:
        p = np.zeros((N, G + 1, V), dtype=np.float32)
        q = np.zeros((N, G, V), dtype=np.float32)
    step = 16
    chunk_seeds = rng.integers(0, 2 ** 63 - 1, size=(N + step - 1) // step)

    def work(c):
        r0, r1 = c * step, min(N, (c + 1) * step)
        crng = np.random.default_rng(int(chunk_seeds[c]))
        tl = crng.standard_normal((r1 - r0, G + 1, V), dtype=np.float32) * np.float32(2.5)
        t_bits[r0:r1] = _to_bf16_bits(tl)
        dl = bf16_bits_to_f32(t_bits[r0:r1, :G]) + \
            crng.standard_normal((r1 - r0, G, V), dtype=np.float32) * np.float32(0.7)
        d_bits[r0:r1] = _to_bf16_bits(dl)
        if G:
            d32 = bf16_bits_to_f32(d_bits[r0:r1]).reshape(-1, V)
            d_idx, d_w = _nucleus_rows(d32, temp, kk, top_p)
            pick = _inverse_cdf(crng, d_w)
            ids[r0:r1] = d_idx[np.arange(d_idx.shape[0]), pick].reshape(r1 - r0, G)
            if probs:
                np.put_along_axis(q[r0:r1].reshape(-1, V), d_idx, d_w, axis=-1)
        if probs:
            t_idx, t_w = _nucleus_rows(bf16_bits_to_f32(t_bits[r0:r1]).reshape(-1, V), temp, kk, top_p)
            np.put_along_axis(p[r0:r1].reshape(-1, V), t_idx, t_w, axis=-1)

    nchunks = len(chunk_seeds)
    with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1, 16)) as ex:
        list(ex.map(work, range(nchunks)))
    ncomp, slots, _ = _kv_bookkeeping(rng, gammas)
    out = dict(T=T, draft_ids=ids.reshape(-1), cu_num_draft_tokens=None,
               temperature=np.full(N, temp, np.float32), top_k=np.full(N, k, np.int32),
               top_p=np.full(N, top_p, np.float32), num_computed_tokens=ncomp, slot_mapping=slots)
    if not probs:
        out.update(entry="logits", dtype="bf16", target=t_bits.reshape(T + N, V), draft=d_bits.reshape(T, V))
        return out
    # fused_probs: sparse fp32 probability rows of the same distributions
    out.update(entry="probs", dtype="f32", target=p.reshape(T + N, V), draft=q.reshape(T, V), top_k=None,
               top_p=None)
    return out


def _ragged(name, rng, N, G, V):
    gammas = rng.integers(0, G + 1, size=N).astype(np.int64)
    cu, T = _layout(gammas)
    sig_choices = np.array([0.1, 1.0, 3.0], dtype=np.float32)
    sig = sig_choices[rng.integers(0, 3, size=N)]
    greedy = np.zeros(N, dtype=bool)
    greedy[rng.permutation(N)[: N // 2]] = True
    temperature = np.where(greedy, 0.0, 1.0).astype(np.float32)
    t_bits = np.empty((T + N, V), dtype=np.uint16)
    d_bits = np.empty((T, V), dtype=np.uint16)
    ids = np.empty(T, dtype=np.int32)
    s = 0
    for i in range(N):
        g = int(gammas[i])
        tl = rng.standard_normal((g + 1, V), dtype=np.float32) * np.float32(2.0)
        t_bits[s + i: s + i + g + 1] = _to_bf16_bits(tl)
        if g:
            dl = bf16_bits_to_f32(t_bits[s + i: s + i + g]) + \
                rng.standard_normal((g, V), dtype=np.float32) * sig[i]
            d_bits[s: s + g] = _to_bf16_bits(dl)
            d32 = bf16_bits_to_f32(d_bits[s: s + g])
            if greedy[i]:
                ids[s: s + g] = d32.argmax(axis=-1)
            else:
                ids[s: s + g] = _inverse_cdf(rng, _softmax_rows_f32(d32))
        s += g
    ncomp, slots, _ = _kv_bookkeeping(rng, gammas)
    return dict(entry="logits", dtype="bf16", T=T, draft_ids=ids, cu_num_draft_tokens=cu,
                target=t_bits, draft=d_bits, temperature=temperature, top_k=None, top_p=None,
                num_computed_tokens=ncomp, slot_mapping=slots, sigma=sig)


def gammas_of(w: dict) -> np.ndarray:
    """Per-request draft counts of a workload (from its layout, not its values)."""
    if w["cu_num_draft_tokens"] is None:
        return np.full(w["N"], w["gamma"], dtype=np.int64)
    cu = w["cu_num_draft_tokens"].astype(np.int64)
    return np.diff(np.concatenate([[0], cu]))


def as_torch(w: dict, device="cpu", pin: bool = False) -> dict:
    """Convert the array fields of a workload to torch tensors (bf16 bits are
    viewed as torch.bfloat16).  Pure marshalling."""
    import torch
    out = {}
    for k, v in w.items():
        if isinstance(v, np.ndarray):
            if v.dtype == np.uint16:
                t = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16)
            else:
                t = torch.from_numpy(v)
            if pin and device == "cpu":
                t = t.pin_memory()
            elif device != "cpu":
                t = t.to(device, non_blocking=False)
            out[k] = t
        else:
            out[k] = v
    return out


NGRAM = dict(R=512, min_len=1024, max_len=16384, vocab=151936, p_copy=0.5, seed=9)


def make_histories(R: int = NGRAM["R"], *, min_len: int = NGRAM["min_len"], max_len: int = NGRAM["max_len"],
                   vocab: int = NGRAM["vocab"], p_copy: float = NGRAM["p_copy"], seed: int = NGRAM["seed"]):
    """Token histories for the n-gram proposer: returns (tokens int32 [total],
    cu_num_tokens int64 [R] inclusive prefix sums).  Pure input synthesis."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(min_len, max_len + 1, size=R)
    hist = []
    for L in lens:
        h = np.empty(int(L), np.int32)
        n0 = min(32, int(L))
        h[:n0] = rng.integers(0, vocab, size=n0)
        pos = n0
        while pos < L:
            seg = min(int(rng.integers(8, 65)), int(L) - pos)
            if pos >= 16 and rng.random() < p_copy:
                src = int(rng.integers(0, pos - 8))
                for c in range(seg):  # element by element: a repeat may run into itself
                    h[pos + c] = h[src + c]
            else:
                h[pos:pos + seg] = rng.integers(0, vocab, size=seg)
            pos += seg
        hist.append(h)
    tokens = np.concatenate(hist) if hist else np.zeros(0, np.int32)
    cu = np.cumsum(lens).astype(np.int64)
    return tokens, cu
