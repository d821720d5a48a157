"""TEST INFRASTRUCTURE -- the CPU oracle of the batched speculative-decoding verifier.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it: the arithmetic lives in ``sv_oracle.c`` (plain C, one
request and one row at a time, see that file's header for the pages it
follows); this module only compiles it with gcc and marshals numpy arrays
through ctypes.

Diagnostics (``diag`` columns): DIAG_ACCEPT_MARGIN and DIAG_RACE_FLIP are
"flip indices" -- the perturbation of p and q needed to change that decision,
in units of the tolerance (1e-6 absolute and 1e-5 relative); below 1 means a
perturbation inside both bounds could flip it.  DIAG_RACE_RELGAP is the
relative gap between the winning race key and the runner-up.

Status bits mirror the library's documented meaning: 1 bad cu range, 2 draft id
outside [0, V), 4 bad exponential draw, 8 empty distribution, 16 NaN/inf
values, 32 bad sampling parameter, 64 draft rows missing, 256 bad processor or
stop list range.

Logits processors and stop tokens come with the workload dict (optional keys):
``repetition_penalty`` [N], ``penalty_cu``/``penalty_ids`` (each request's
context tokens), ``banned_cu``/``banned_ids`` and ``stop_cu``/``stop_ids``
(inclusive prefix sums into the id arrays, like ``cu_num_draft_tokens``).
"""
from __future__ import annotations

import ctypes
import os
import pathlib
import subprocess
import tempfile

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SRC = _HERE / "sv_oracle.c"
_LIB_PATH = _HERE / "_build" / "liboracle_sv.so"
_LIB = None

NDIAG = 6
DIAG_ACCEPT_MARGIN, DIAG_RACE_FLIP, DIAG_RACE_RELGAP, DIAG_TOPP_EDGE, DIAG_FALLBACK, DIAG_PATH = range(6)

BAD_CU, BAD_DRAFT_ID, BAD_EXPONENTIAL, EMPTY_DISTRIBUTION, BAD_VALUES, BAD_PARAM, MISSING_DRAFT = (
    1, 2, 4, 8, 16, 32, 64)
BAD_LIST = 256

_P = ctypes.c_void_p


class _Args(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32), ("max_spec_len", ctypes.c_int32), ("vocab_size", ctypes.c_int32),
        ("entry", ctypes.c_int32), ("dtype", ctypes.c_int32), ("pad0", ctypes.c_int32),
        ("num_draft_tokens_total", ctypes.c_int64),
        ("draft_ids", _P), ("cu_num_draft_tokens", _P),
        ("target", _P), ("target_row_stride", ctypes.c_int64),
        ("draft", _P), ("draft_row_stride", ctypes.c_int64),
        ("temperature", _P), ("top_k", _P), ("top_p", _P),
        ("uniforms", _P), ("exponentials", _P), ("exponentials_row_stride", ctypes.c_int64),
        ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
        ("rng_request_base", ctypes.c_uint32), ("pad1", ctypes.c_uint32),
        ("out_tokens", _P), ("num_accepted", _P), ("num_computed_tokens", _P), ("slot_mapping", _P),
        ("dbg_py", _P), ("dbg_qy", _P), ("status", _P), ("diag", _P), ("synthetic_rates", _P),
        ("repetition_penalty", _P), ("penalty_cu", _P), ("penalty_ids", _P), ("penalty_total", ctypes.c_int64),
        ("banned_cu", _P), ("banned_ids", _P), ("banned_total", ctypes.c_int64),
        ("stop_cu", _P), ("stop_ids", _P), ("stop_total", ctypes.c_int64),
    ]


def build(force: bool = False) -> pathlib.Path:
    """Compile sv_oracle.c with gcc (no FMA contraction, no fast-math)."""
    if not force and _LIB_PATH.exists() and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB_PATH
    _LIB_PATH.parent.mkdir(parents=True, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_LIB_PATH.parent)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-o", tmp, str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(str(build()))
        lib.oracle_verify.argtypes = [ctypes.POINTER(_Args)]
        lib.oracle_verify_range.argtypes = [ctypes.POINTER(_Args), ctypes.c_int, ctypes.c_int]
        lib.oracle_philox4x32_10.argtypes = [_P, _P, _P]
        lib.oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        lib.oracle_uniform.restype = ctypes.c_float
        lib.oracle_exponential.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        lib.oracle_exponential.restype = ctypes.c_float
        lib.oracle_logits_to_probs.argtypes = [_P, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_float,
                                               _P, _P]
        lib.oracle_transform_row.argtypes = [_P, _P, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_float,
                                             _P, _P]
        lib.oracle_sample_rows.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_int64,
                                           _P, _P, _P, _P, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_uint32, _P, _P, _P, _P,
                                           _P, _P, _P, ctypes.c_int64, _P, _P, ctypes.c_int64]
        lib.oracle_ngram_propose.argtypes = [ctypes.c_int32, _P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.c_int64, _P, _P]
        assert lib.oracle_sizeof_args() == ctypes.sizeof(_Args), "oracle_args layout mismatch"
        _LIB = lib
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------------------
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, offset: int, req: int, j: int) -> float:
    return float(_lib().oracle_uniform(seed, offset, req, j))


def exponential(seed: int, offset: int, req: int, x: int) -> np.float32:
    return np.float32(_lib().oracle_exponential(seed, offset, req, x))


def logits_to_probs(logits, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """Temperature, top-k, softmax, top-p and renormalisation of one logits row.
    Returns (fp32 probabilities, top-p edge flag, status code)."""
    l = _c(logits, np.float32)
    out = np.zeros_like(l)
    edge = np.zeros(1, dtype=np.int32)
    rc = _lib().oracle_logits_to_probs(_ptr(l), l.shape[0], temperature, int(top_k), top_p, _ptr(out), _ptr(edge))
    return out, int(edge[0]), int(rc)


def transform_row(logits, processed, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """The transform in the pages' order: temperature, top-k and top-p placed
    on the raw row ``logits``, then the processed values ``processed`` (the same
    row after banned ids and repetition penalty, or None) on the kept entries,
    renormalised.  Returns (fp32 probabilities, top-p edge flag, status code)."""
    l = _c(logits, np.float32)
    lp = _c(processed, np.float32)
    out = np.zeros_like(l)
    edge = np.zeros(1, dtype=np.int32)
    rc = _lib().oracle_transform_row(_ptr(l), _ptr(lp), l.shape[0], temperature, int(top_k), top_p, _ptr(out),
                                     _ptr(edge))
    return out, int(edge[0]), int(rc)


def verify(w: dict, *, production: bool = False, seed: int = 0, offset: int = 0, rng_request_base: int = 0,
           with_diag: bool = True, req_range=None, num_computed_tokens=None, slot_mapping=None,
           synthetic_rates=None) -> dict:
    """Run the oracle on a workload dict (see ``workloads.make``).

    Test mode uses ``w['uniforms']`` / ``w['exponentials']``; ``production=True``
    draws them from Philox4x32-10 with (seed, offset).  Returns a dict with
    out_tokens [N, gamma+1], num_accepted [N], num_computed_tokens [N],
    slot_mapping [T+N] (updated copies), dbg_py/dbg_qy [T] (NaN where not
    examined), status (int) and diag [N, NDIAG].
    """
    lib = _lib()
    N, G, V, T = int(w["N"]), int(w["gamma"]), int(w["V"]), int(w["T"])
    is_logits = w["entry"] == "logits"
    bf16 = w["dtype"] == "bf16"
    tdt = np.uint16 if bf16 else np.float32
    ids = _c(w["draft_ids"], np.int32)
    cu = _c(w["cu_num_draft_tokens"], np.int32)
    tgt = _c(w["target"], tdt)
    drf = _c(w["draft"], tdt)
    temp = _c(w["temperature"], np.float32)
    topk = _c(w.get("top_k"), np.int32)
    topp = _c(w.get("top_p"), np.float32)
    u = None if production else _c(w["uniforms"], np.float32)
    E = None if production else _c(w["exponentials"], np.float32)
    if not production and (u is None or E is None):
        raise ValueError("test mode needs uniforms and exponentials")
    nc_in = w.get("num_computed_tokens") if num_computed_tokens is None else num_computed_tokens
    sm_in = w.get("slot_mapping") if slot_mapping is None else slot_mapping
    out = np.full((N, G + 1), -7, dtype=np.int32)  # every entry is written
    nacc = np.full(N, -7, dtype=np.int32)
    ncomp = None if nc_in is None else np.array(nc_in, dtype=np.int32, copy=True)
    slots = None if sm_in is None else np.array(sm_in, dtype=np.int64, copy=True)
    dpy = np.full(max(T, 1), np.nan, dtype=np.float32)
    dqy = np.full(max(T, 1), np.nan, dtype=np.float32)
    status = np.zeros(1, dtype=np.int32)
    diag = np.zeros((N, NDIAG), dtype=np.float64) if with_diag else None
    a = _Args()
    a.num_reqs, a.max_spec_len, a.vocab_size = N, G, V
    a.entry = 1 if is_logits else 0
    a.dtype = 1 if bf16 else 0
    a.num_draft_tokens_total = T
    a.draft_ids, a.cu_num_draft_tokens = _ptr(ids), _ptr(cu)
    a.target, a.target_row_stride = _ptr(tgt), V
    a.draft, a.draft_row_stride = _ptr(drf), V
    a.temperature, a.top_k, a.top_p = _ptr(temp), _ptr(topk), _ptr(topp)
    a.uniforms, a.exponentials, a.exponentials_row_stride = _ptr(u), _ptr(E), V
    a.seed, a.offset, a.rng_request_base = seed, offset, rng_request_base
    a.out_tokens, a.num_accepted = _ptr(out), _ptr(nacc)
    a.num_computed_tokens, a.slot_mapping = _ptr(ncomp), _ptr(slots)
    a.dbg_py, a.dbg_qy, a.status, a.diag = _ptr(dpy), _ptr(dqy), _ptr(status), _ptr(diag)
    rates = _c(synthetic_rates, np.float32)
    a.synthetic_rates = _ptr(rates)
    keep = []
    theta = _c(w.get("repetition_penalty"), np.float32)
    keep.append(theta)
    a.repetition_penalty = _ptr(theta)
    for name in ("penalty", "banned", "stop"):
        cu_l = _c(w.get(f"{name}_cu"), np.int64)
        ids_l = _c(w.get(f"{name}_ids"), np.int32)
        keep += [cu_l, ids_l]
        setattr(a, f"{name}_cu", _ptr(cu_l))
        setattr(a, f"{name}_ids", _ptr(ids_l))
        setattr(a, f"{name}_total", 0 if ids_l is None else int(ids_l.shape[0]))
    if req_range is None:
        rc = lib.oracle_verify(ctypes.byref(a))
    else:
        rc = lib.oracle_verify_range(ctypes.byref(a), int(req_range[0]), int(req_range[1]))
    if rc != 0:
        raise RuntimeError(f"oracle_verify failed with {rc}")
    return dict(out_tokens=out, num_accepted=nacc, num_computed_tokens=ncomp, slot_mapping=slots,
                dbg_py=dpy[:T], dbg_qy=dqy[:T], status=int(status[0]), diag=diag)


def _threads(threads):
    return max(1, threads if threads else (os.cpu_count() or 1))


def verify_parallel(w: dict, *, threads: int = 0, **kw) -> dict:
    """``verify`` over every request of ``w``, the requests split into
    contiguous ranges run on host threads (ctypes releases the GIL during each
    call; the C oracle keeps no global state), then merged.  Each range is the
    oracle as it stands; the result is the one ``verify`` gives."""
    from concurrent.futures import ThreadPoolExecutor
    N = int(w["N"])
    cuts = np.linspace(0, N, min(_threads(threads), max(N, 1)) + 1).astype(int)
    ranges = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    if len(ranges) <= 1:
        return verify(w, **kw)
    with ThreadPoolExecutor(len(ranges)) as ex:
        parts = list(ex.map(lambda r: verify(w, req_range=r, **kw), ranges))
    if w.get("cu_num_draft_tokens") is not None:
        cu = np.asarray(w["cu_num_draft_tokens"], np.int64)
    else:
        cu = (np.arange(1, N + 1) * int(w["gamma"])).astype(np.int64)
    start = lambda i: int(cu[i - 1]) if i > 0 else 0
    out = {k: (None if v is None else np.array(v, copy=True)) for k, v in parts[0].items() if k != "status"}
    status = 0
    for (a, b), r in zip(ranges, parts):
        status |= r["status"]
        for k in ("out_tokens", "num_accepted", "num_computed_tokens", "diag"):
            if out.get(k) is not None:
                out[k][a:b] = r[k][a:b]
        for k in ("dbg_py", "dbg_qy"):
            out[k][start(a):start(b)] = r[k][start(a):start(b)]
        if out.get("slot_mapping") is not None:  # verify-token layout: request i at s_i + i .. s_i + i + gamma_i
            out["slot_mapping"][start(a) + a:start(b) + b] = r["slot_mapping"][start(a) + a:start(b) + b]
    out["status"] = status
    return out


def sample_rows(logits, *, temperature=None, top_k=None, top_p=None, exponentials=None, seed=0, offset=0,
                rng_row_base=0, with_probs=True, repetition_penalty=None, penalty_cu=None, penalty_ids=None,
                banned_cu=None, banned_ids=None):
    """Draft-side sampler: one token per logits row (fp32 array [R, V] or bf16
    bits uint16 [R, V]).  Test mode when ``exponentials`` is given.  Optional
    logits processors per row (lists as in ``verify``).  Returns dict(tokens
    [R], probs [R, V] or None, status, diag [R, 2] = race flip index, top-p
    edge flag)."""
    lib = _lib()
    bf16 = logits.dtype == np.uint16
    l = _c(logits, np.uint16 if bf16 else np.float32)
    R, V = l.shape
    temp = _c(temperature, np.float32)
    tk = _c(top_k, np.int32)
    tp = _c(top_p, np.float32)
    E = _c(exponentials, np.float32)
    tokens = np.full(R, -7, np.int32)
    probs = np.zeros((R, V), np.float32) if with_probs else None
    status = np.zeros(1, np.int32)
    diag = np.zeros((R, 2), np.float64)
    theta = _c(repetition_penalty, np.float32)
    pcu, pids = _c(penalty_cu, np.int64), _c(penalty_ids, np.int32)
    bcu, bids = _c(banned_cu, np.int64), _c(banned_ids, np.int32)
    rc = lib.oracle_sample_rows(R, V, 1 if bf16 else 0, _ptr(l), V, _ptr(temp), _ptr(tk), _ptr(tp), _ptr(E), V,
                                seed, offset, rng_row_base, _ptr(tokens), _ptr(probs), _ptr(status), _ptr(diag),
                                _ptr(theta), _ptr(pcu), _ptr(pids), 0 if pids is None else int(pids.shape[0]),
                                _ptr(bcu), _ptr(bids), 0 if bids is None else int(bids.shape[0]))
    if rc != 0:
        raise RuntimeError(f"oracle_sample_rows failed with {rc}")
    return dict(tokens=tokens, probs=probs, status=int(status[0]), diag=diag)


def sample_rows_parallel(logits, *, threads: int = 0, **kw):
    """``sample_rows`` with the rows split into contiguous ranges run on host
    threads, then concatenated (per-row arguments are sliced; production
    draws keep their stream by offsetting ``rng_row_base``)."""
    from concurrent.futures import ThreadPoolExecutor
    R = logits.shape[0]
    cuts = np.linspace(0, R, min(_threads(threads), max(R, 1)) + 1).astype(int)
    ranges = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    per_row = ("temperature", "top_k", "top_p", "exponentials", "repetition_penalty")
    if any(kw.get(k) is not None for k in ("penalty_cu", "banned_cu")):
        raise ValueError("sample_rows_parallel takes no processor lists")

    def run(r):
        a, b = r
        sub = {k: (None if v is None else np.asarray(v)[a:b]) if k in per_row else v for k, v in kw.items()}
        sub["rng_row_base"] = int(kw.get("rng_row_base", 0)) + a
        return sample_rows(logits[a:b], **sub)

    with ThreadPoolExecutor(max(1, len(ranges))) as ex:
        parts = list(ex.map(run, ranges))
    probs = None if parts[0]["probs"] is None else np.concatenate([p["probs"] for p in parts])
    status = 0
    for p in parts:
        status |= p["status"]
    return dict(tokens=np.concatenate([p["tokens"] for p in parts]), probs=probs, status=status,
                diag=np.concatenate([p["diag"] for p in parts]))


def ngram_propose(tokens, cu_num_tokens, *, min_ngram: int, max_ngram: int, k: int, max_model_len: int):
    """N-gram proposals for a ragged batch of token histories (request q owns
    tokens[cu[q-1]:cu[q]]).  Returns dict(draft_token_ids [R, k] with -1
    padding, num_draft_tokens [R], status)."""
    t = _c(np.asarray(tokens), np.int32)
    cu = _c(np.asarray(cu_num_tokens), np.int64)
    R = int(cu.shape[0])
    out = np.full((R, max(k, 0)), -1, np.int32)
    num = np.zeros(R, np.int32)
    st = _lib().oracle_ngram_propose(R, _ptr(t), _ptr(cu), int(t.shape[0]), int(min_ngram), int(max_ngram), int(k),
                                     int(max_model_len), _ptr(out), _ptr(num))
    return dict(draft_token_ids=out, num_draft_tokens=num, status=int(st))
