"""Python binding of the GB300 speculative-decoding verifier (rejection sampler).

A thin ctypes layer over ``libspec_verify.so`` (declared in
``include/spec_verify.h``): it checks tensor devices, dtypes and strides,
passes raw device pointers and the current CUDA stream, and returns.  Every
step of the verification runs in the library's CUDA kernels; there is no
Python or CPU fallback -- if the library is missing the import of this module
still works but every call raises ``NativeLibraryMissing``.

Functions keep the C names: ``spec_verify_create``, ``spec_verify_run``,
``spec_verify_destroy``, ``spec_verify_check_args``,
``spec_verify_status_string``; ``Verifier`` bundles them with output
allocation for convenience.
"""
from __future__ import annotations

import ctypes
import pathlib
from dataclasses import dataclass
from typing import Optional

_PKG = pathlib.Path(__file__).resolve().parent
LIB_PATH = _PKG / "libspec_verify.so"

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_CAPACITY = range(5)
SV_ENTRY_PROBS, SV_ENTRY_LOGITS = 0, 1
SV_F32, SV_BF16 = 0, 1
SV_MAX_SPEC_LEN = 256
DATA_STATUS_BITS = {
    "BAD_CU": 1, "BAD_DRAFT_ID": 2, "BAD_EXPONENTIAL": 4, "EMPTY_DISTRIBUTION": 8,
    "BAD_VALUES": 16, "BAD_PARAM": 32, "MISSING_DRAFT": 64, "COPY_TIMEOUT": 128,
}

_P = ctypes.c_void_p


SV_FLAG_RESIDENT_ROWS = 1
SV_FLAG_ONE_CTA_PER_REQUEST = 2
SV_FLAG_SERIAL_LAUNCH = 4
SV_HINT_SMALL_TOP_K = 1
SV_SMALL_TOP_K_MAX = 256
SV_TEST_EXPIRE_COPY_WAIT = 1


class SpecVerifyConfig(ctypes.Structure):
    _fields_ = [("max_num_reqs", ctypes.c_int32), ("max_spec_len", ctypes.c_int32),
                ("vocab_size", ctypes.c_int32), ("device", ctypes.c_int32),
                ("cluster_ctas", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class SpecVerifyArgs(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32), ("max_spec_len", ctypes.c_int32), ("vocab_size", ctypes.c_int32),
        ("entry", ctypes.c_int32), ("dtype", ctypes.c_int32), ("hints", ctypes.c_uint32),
        ("num_draft_tokens_total", ctypes.c_int64),
        ("draft_ids", _P), ("cu_num_draft_tokens", _P),
        ("target", _P), ("target_row_stride", ctypes.c_int64),
        ("draft", _P), ("draft_row_stride", ctypes.c_int64),
        ("temperature", _P), ("top_k", _P), ("top_p", _P),
        ("uniforms", _P), ("exponentials", _P), ("exponentials_row_stride", ctypes.c_int64),
        ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
        ("rng_request_base", ctypes.c_uint32), ("test_flags", ctypes.c_uint32),
        ("out_tokens", _P), ("num_accepted", _P), ("num_computed_tokens", _P), ("slot_mapping", _P),
        ("dbg_py", _P), ("dbg_qy", _P), ("status", _P), ("synthetic_acceptance_rates", _P),
        ("repetition_penalty", _P), ("penalty_cu", _P), ("penalty_token_ids", _P), ("penalty_total", ctypes.c_int64),
        ("banned_cu", _P), ("banned_token_ids", _P), ("banned_total", ctypes.c_int64),
        ("stop_cu", _P), ("stop_token_ids", _P), ("stop_total", ctypes.c_int64),
    ]


class SpecVerifySampleArgs(ctypes.Structure):
    _fields_ = [
        ("num_rows", ctypes.c_int32), ("vocab_size", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("hints", ctypes.c_uint32),
        ("logits", _P), ("row_stride", ctypes.c_int64),
        ("temperature", _P), ("top_k", _P), ("top_p", _P),
        ("exponentials", _P), ("exponentials_row_stride", ctypes.c_int64),
        ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
        ("rng_row_base", ctypes.c_uint32), ("test_flags", ctypes.c_uint32),
        ("tokens", _P), ("probs", _P), ("probs_row_stride", ctypes.c_int64), ("status", _P),
        ("repetition_penalty", _P), ("penalty_cu", _P), ("penalty_token_ids", _P), ("penalty_total", ctypes.c_int64),
        ("banned_cu", _P), ("banned_token_ids", _P), ("banned_total", ctypes.c_int64),
    ]


class SpecVerifyNgramArgs(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32), ("min_ngram", ctypes.c_int32), ("max_ngram", ctypes.c_int32),
        ("num_spec_tokens", ctypes.c_int32), ("max_model_len", ctypes.c_int64),
        ("num_tokens_total", ctypes.c_int64), ("token_ids", _P), ("cu_num_tokens", _P),
        ("draft_token_ids", _P), ("num_draft_tokens", _P), ("status", _P),
    ]


class NativeLibraryMissing(RuntimeError):
    pass


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{spec_verify_status_string(code)}: {msg}")
        self.code = code


_LIB = None
EXPORTED = ("spec_verify_create", "spec_verify_run", "spec_verify_destroy", "spec_verify_check_args",
            "spec_verify_status_string", "spec_verify_last_error", "spec_verify_abi_version",
            "spec_verify_sizeof_config", "spec_verify_sizeof_args", "spec_verify_sample",
            "spec_verify_check_sample_args", "spec_verify_sizeof_sample_args", "spec_verify_ngram_propose",
            "spec_verify_check_ngram_args", "spec_verify_sizeof_ngram_args")


def load_library(path: Optional[str] = None):
    """Load libspec_verify.so (once) and bind its prototypes."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = pathlib.Path(path) if path else LIB_PATH
    if not p.exists():
        raise NativeLibraryMissing(f"{p} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(str(p))
    lib.spec_verify_create.argtypes = [ctypes.POINTER(SpecVerifyConfig), ctypes.POINTER(ctypes.c_void_p)]
    lib.spec_verify_create.restype = ctypes.c_int
    lib.spec_verify_run.argtypes = [ctypes.c_void_p, ctypes.POINTER(SpecVerifyArgs), ctypes.c_void_p]
    lib.spec_verify_run.restype = ctypes.c_int
    lib.spec_verify_destroy.argtypes = [ctypes.c_void_p]
    lib.spec_verify_destroy.restype = ctypes.c_int
    lib.spec_verify_check_args.argtypes = [ctypes.POINTER(SpecVerifyConfig), ctypes.POINTER(SpecVerifyArgs)]
    lib.spec_verify_check_args.restype = ctypes.c_int
    lib.spec_verify_status_string.argtypes = [ctypes.c_int]
    lib.spec_verify_status_string.restype = ctypes.c_char_p
    lib.spec_verify_last_error.argtypes = []
    lib.spec_verify_last_error.restype = ctypes.c_char_p
    lib.spec_verify_abi_version.restype = ctypes.c_uint32
    lib.spec_verify_sizeof_config.restype = ctypes.c_size_t
    lib.spec_verify_sizeof_args.restype = ctypes.c_size_t
    lib.spec_verify_sample.argtypes = [ctypes.c_void_p, ctypes.POINTER(SpecVerifySampleArgs), ctypes.c_void_p]
    lib.spec_verify_sample.restype = ctypes.c_int
    lib.spec_verify_check_sample_args.argtypes = [ctypes.POINTER(SpecVerifyConfig),
                                                  ctypes.POINTER(SpecVerifySampleArgs)]
    lib.spec_verify_check_sample_args.restype = ctypes.c_int
    lib.spec_verify_sizeof_sample_args.restype = ctypes.c_size_t
    lib.spec_verify_ngram_propose.argtypes = [ctypes.c_void_p, ctypes.POINTER(SpecVerifyNgramArgs), ctypes.c_void_p]
    lib.spec_verify_ngram_propose.restype = ctypes.c_int
    lib.spec_verify_check_ngram_args.argtypes = [ctypes.POINTER(SpecVerifyConfig), ctypes.POINTER(SpecVerifyNgramArgs)]
    lib.spec_verify_check_ngram_args.restype = ctypes.c_int
    lib.spec_verify_sizeof_ngram_args.restype = ctypes.c_size_t
    if lib.spec_verify_sizeof_config() != ctypes.sizeof(SpecVerifyConfig) or \
            lib.spec_verify_sizeof_args() != ctypes.sizeof(SpecVerifyArgs) or \
            lib.spec_verify_sizeof_sample_args() != ctypes.sizeof(SpecVerifySampleArgs) or \
            lib.spec_verify_sizeof_ngram_args() != ctypes.sizeof(SpecVerifyNgramArgs):
        raise RuntimeError("spec_verify struct layout differs from the binding")
    if path is None:
        _LIB = lib
    return lib


def spec_verify_status_string(code: int) -> str:
    return load_library().spec_verify_status_string(int(code)).decode()


def _check(code: int):
    if code != SV_OK:
        raise SpecVerifyError(code, load_library().spec_verify_last_error().decode())


def make_config(max_num_reqs: int, max_spec_len: int, vocab_size: int, device: int = 0,
                cluster_ctas: int = 0, flags: int = 0) -> SpecVerifyConfig:
    return SpecVerifyConfig(int(max_num_reqs), int(max_spec_len), int(vocab_size), int(device),
                            int(cluster_ctas), int(flags))


def spec_verify_create(max_num_reqs: int, max_spec_len: int, vocab_size: int, device: int = 0,
                       cluster_ctas: int = 0, flags: int = 0) -> int:
    cfg = make_config(max_num_reqs, max_spec_len, vocab_size, device, cluster_ctas, flags)
    h = ctypes.c_void_p()
    _check(load_library().spec_verify_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def spec_verify_destroy(handle: int) -> None:
    _check(load_library().spec_verify_destroy(ctypes.c_void_p(handle)))


# ----------------------------------------------------------------------------
# argument marshalling
# ----------------------------------------------------------------------------
def _ptr(t, dtype, name, device, numel=None, ndim=None, contiguous=True):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _rows(t, name, device, V, nrows, dtypes, host_ok=False):
    """A [rows, >=V] tensor whose rows are unit-stride; returns (ptr, row_stride).
    With host_ok, a pinned host tensor is accepted too: its address is valid on
    the device (unified addressing) and the kernel reads the rows it needs
    directly from host memory."""
    if t is None:
        return None, 0
    if t.dim() != 2 or t.shape[1] != V or t.shape[0] != nrows:
        raise ValueError(f"{name} must have shape [{nrows}, {V}], got {tuple(t.shape)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} dtype {t.dtype} not in {dtypes}")
    if nrows == 0:
        return None, V  # nothing to read; torch gives empty dims arbitrary strides
    if (V > 1 and t.stride(1) != 1) or (nrows > 1 and t.stride(0) < V):
        raise ValueError(f"{name} rows must be unit-stride and non-overlapping")
    if t.device != device and not (host_ok and t.device.type == "cpu" and t.is_pinned()):
        raise ValueError(f"{name} is on {t.device}, expected {device}" +
                         (" or pinned host memory" if host_ok else ""))
    return t.data_ptr(), (t.stride(0) if nrows > 1 else V)


def build_args(*, entry: str, draft_ids, target, out_tokens, num_accepted, draft=None, cu_num_draft_tokens=None,
               temperature=None, top_k=None, top_p=None, uniforms=None, exponentials=None, seed: int = 0,
               offset: int = 0, rng_request_base: int = 0, num_computed_tokens=None, slot_mapping=None,
               dbg_py=None, dbg_qy=None, status=None, device=None,
               host_rows: bool = False, synthetic_acceptance_rates=None, repetition_penalty=None,
               penalty_cu=None, penalty_token_ids=None, banned_cu=None, banned_token_ids=None, stop_cu=None,
               stop_token_ids=None, test_flags: int = 0, hints: int = 0) -> SpecVerifyArgs:
    """Validate tensors and fill a SpecVerifyArgs (no device work).

    Logits processors (logits entry) and stop tokens (both entries) come as
    per-request lists: ``*_cu`` int64 [N] inclusive prefix sums into the
    int32 ``*_token_ids``; ``repetition_penalty`` float32 [N].

    ``host_rows=True`` (probability entry only) lets ``target``/``draft``/
    ``exponentials`` live in pinned host memory: the kernel then pulls only
    the rows a call needs over the host link instead of the caller copying
    every row first.  ``device`` must then be given (the GPU running the call)."""
    import torch
    if entry not in ("probs", "logits"):
        raise ValueError("entry must be 'probs' or 'logits'")
    if host_rows and entry != "probs":
        raise ValueError("host_rows is supported by the probability entry only")
    if device is None:
        if host_rows:
            raise ValueError("host_rows needs an explicit device")
        device = target.device
    device = torch.device(device)
    N = out_tokens.shape[0]
    G = out_tokens.shape[1] - 1
    V = target.shape[-1]
    T = draft_ids.numel()
    if target.dtype == torch.bfloat16:
        dt = SV_BF16
    elif target.dtype == torch.float32:
        dt = SV_F32
    else:
        raise TypeError("target must be float32 or bfloat16")
    dts = (target.dtype,)
    a = SpecVerifyArgs()
    a.num_reqs, a.max_spec_len, a.vocab_size = N, G, V
    a.entry = SV_ENTRY_PROBS if entry == "probs" else SV_ENTRY_LOGITS
    a.dtype = dt
    a.num_draft_tokens_total = T
    a.draft_ids = _ptr(draft_ids, torch.int32, "draft_ids", device)
    a.cu_num_draft_tokens = _ptr(cu_num_draft_tokens, torch.int32, "cu_num_draft_tokens", device, numel=N)
    a.target, a.target_row_stride = _rows(target, "target", device, V, T + N, dts, host_rows)
    a.draft, a.draft_row_stride = _rows(draft, "draft", device, V, T, dts, host_rows)
    a.temperature = _ptr(temperature, torch.float32, "temperature", device, numel=N)
    a.top_k = _ptr(top_k, torch.int32, "top_k", device, numel=N)
    a.top_p = _ptr(top_p, torch.float32, "top_p", device, numel=N)
    a.uniforms = _ptr(uniforms, torch.float32, "uniforms", device, numel=T)
    if exponentials is not None:
        a.exponentials, a.exponentials_row_stride = _rows(exponentials, "exponentials", device, V, N,
                                                          (torch.float32,), host_rows)
    a.seed, a.offset, a.rng_request_base = int(seed), int(offset), int(rng_request_base)
    a.test_flags = int(test_flags)
    a.hints = int(hints)
    a.out_tokens = _ptr(out_tokens, torch.int32, "out_tokens", device, ndim=2)
    a.num_accepted = _ptr(num_accepted, torch.int32, "num_accepted", device, numel=N)
    a.num_computed_tokens = _ptr(num_computed_tokens, torch.int32, "num_computed_tokens", device, numel=N)
    a.slot_mapping = _ptr(slot_mapping, torch.int64, "slot_mapping", device, numel=T + N)
    a.dbg_py = _ptr(dbg_py, torch.float32, "dbg_py", device, numel=T)
    a.dbg_qy = _ptr(dbg_qy, torch.float32, "dbg_qy", device, numel=T)
    a.status = _ptr(status, torch.int32, "status", device, numel=1)
    a.synthetic_acceptance_rates = _ptr(synthetic_acceptance_rates, torch.float32, "synthetic_acceptance_rates",
                                        device, numel=G)
    a.repetition_penalty = _ptr(repetition_penalty, torch.float32, "repetition_penalty", device, numel=N)
    for name, cu_l, ids_l in (("penalty", penalty_cu, penalty_token_ids), ("banned", banned_cu, banned_token_ids),
                              ("stop", stop_cu, stop_token_ids)):
        setattr(a, f"{name}_cu", _ptr(cu_l, torch.int64, f"{name}_cu", device, numel=N))
        has_ids = ids_l is not None and ids_l.numel() > 0
        setattr(a, f"{name}_token_ids", _ptr(ids_l, torch.int32, f"{name}_token_ids", device, ndim=1)
                if has_ids else None)
        setattr(a, f"{name}_total", int(ids_l.numel()) if ids_l is not None else 0)
    return a


def spec_verify_run(handle: int, stream=None, **kw) -> None:
    """Enqueue one verification on ``stream`` (default: torch's current stream).
    Keyword arguments are those of ``build_args``."""
    import torch
    a = build_args(**kw)
    if stream is None:
        stream = torch.cuda.current_stream(kw.get("device") or kw["target"].device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(load_library().spec_verify_run(ctypes.c_void_p(handle), ctypes.byref(a), ctypes.c_void_p(s)))


def build_sample_args(*, logits, tokens, probs=None, temperature=None, top_k=None, top_p=None, exponentials=None,
                      seed: int = 0, offset: int = 0, rng_row_base: int = 0, status=None, repetition_penalty=None,
                      penalty_cu=None, penalty_token_ids=None, banned_cu=None,
                      banned_token_ids=None, test_flags: int = 0, hints: int = 0) -> SpecVerifySampleArgs:
    """Validate tensors and fill a SpecVerifySampleArgs (no device work).
    Logits processors per row as in ``build_args``."""
    import torch
    device = logits.device
    R, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = SV_BF16
    elif logits.dtype == torch.float32:
        dt = SV_F32
    else:
        raise TypeError("logits must be float32 or bfloat16")
    a = SpecVerifySampleArgs()
    a.num_rows, a.vocab_size, a.dtype = R, V, dt
    a.logits, a.row_stride = _rows(logits, "logits", device, V, R, (logits.dtype,))
    a.temperature = _ptr(temperature, torch.float32, "temperature", device, numel=R)
    a.top_k = _ptr(top_k, torch.int32, "top_k", device, numel=R)
    a.top_p = _ptr(top_p, torch.float32, "top_p", device, numel=R)
    if exponentials is not None:
        a.exponentials, a.exponentials_row_stride = _rows(exponentials, "exponentials", device, V, R,
                                                          (torch.float32,))
    a.seed, a.offset, a.rng_row_base = int(seed), int(offset), int(rng_row_base)
    a.test_flags = int(test_flags)
    a.hints = int(hints)
    a.tokens = _ptr(tokens, torch.int32, "tokens", device, numel=R)
    if probs is not None:
        a.probs, a.probs_row_stride = _rows(probs, "probs", device, V, R, (torch.float32,))
    a.status = _ptr(status, torch.int32, "status", device, numel=1)
    a.repetition_penalty = _ptr(repetition_penalty, torch.float32, "repetition_penalty", device, numel=R)
    for name, cu_l, ids_l in (("penalty", penalty_cu, penalty_token_ids), ("banned", banned_cu, banned_token_ids)):
        setattr(a, f"{name}_cu", _ptr(cu_l, torch.int64, f"{name}_cu", device, numel=R))
        has_ids = ids_l is not None and ids_l.numel() > 0
        setattr(a, f"{name}_token_ids", _ptr(ids_l, torch.int32, f"{name}_token_ids", device, ndim=1)
                if has_ids else None)
        setattr(a, f"{name}_total", int(ids_l.numel()) if ids_l is not None else 0)
    return a


def spec_verify_sample(handle: int, stream=None, **kw) -> None:
    """Enqueue the draft-side sampler on ``stream`` (default: torch's current
    stream).  Keyword arguments are those of ``build_sample_args``."""
    import torch
    a = build_sample_args(**kw)
    if stream is None:
        stream = torch.cuda.current_stream(kw["logits"].device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(load_library().spec_verify_sample(ctypes.c_void_p(handle), ctypes.byref(a), ctypes.c_void_p(s)))


def spec_verify_check_sample_args(config: SpecVerifyConfig, args: SpecVerifySampleArgs) -> int:
    """Host-only validation of sampler arguments; returns the sv_status code."""
    return int(load_library().spec_verify_check_sample_args(ctypes.byref(config), ctypes.byref(args)))


def build_ngram_args(*, token_ids, cu_num_tokens, draft_token_ids, num_draft_tokens, min_ngram: int, max_ngram: int,
                     max_model_len: int, status=None) -> SpecVerifyNgramArgs:
    """Validate tensors and fill a SpecVerifyNgramArgs (no device work).  The
    number of proposed tokens k is draft_token_ids.shape[1]."""
    import torch
    device = cu_num_tokens.device
    R = int(cu_num_tokens.numel())
    if draft_token_ids.dim() != 2 or draft_token_ids.shape[0] != R:
        raise ValueError(f"draft_token_ids must have shape [{R}, k], got {tuple(draft_token_ids.shape)}")
    a = SpecVerifyNgramArgs()
    a.num_reqs, a.min_ngram, a.max_ngram = R, int(min_ngram), int(max_ngram)
    a.num_spec_tokens = int(draft_token_ids.shape[1])
    a.max_model_len = int(max_model_len)
    a.num_tokens_total = int(token_ids.numel())
    a.token_ids = _ptr(token_ids, torch.int32, "token_ids", device, ndim=1) if token_ids.numel() else None
    a.cu_num_tokens = _ptr(cu_num_tokens, torch.int64, "cu_num_tokens", device, ndim=1) if R else None
    a.draft_token_ids = _ptr(draft_token_ids, torch.int32, "draft_token_ids", device) if draft_token_ids.numel() else None
    a.num_draft_tokens = _ptr(num_draft_tokens, torch.int32, "num_draft_tokens", device, numel=R) if R else None
    a.status = _ptr(status, torch.int32, "status", device, numel=1)
    return a


def spec_verify_ngram_propose(handle: int, stream=None, **kw) -> None:
    """Enqueue the batched n-gram proposer on ``stream`` (default: torch's
    current stream).  Keyword arguments are those of ``build_ngram_args``."""
    import torch
    a = build_ngram_args(**kw)
    if stream is None:
        stream = torch.cuda.current_stream(kw["cu_num_tokens"].device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(load_library().spec_verify_ngram_propose(ctypes.c_void_p(handle), ctypes.byref(a), ctypes.c_void_p(s)))


def spec_verify_check_ngram_args(config: SpecVerifyConfig, args: SpecVerifyNgramArgs) -> int:
    """Host-only validation of n-gram proposer arguments; returns the sv_status code."""
    return int(load_library().spec_verify_check_ngram_args(ctypes.byref(config), ctypes.byref(args)))


def spec_verify_check_args(config: SpecVerifyConfig, args: SpecVerifyArgs) -> int:
    """Host-only validation; returns the sv_status code."""
    return int(load_library().spec_verify_check_args(ctypes.byref(config), ctypes.byref(args)))


@dataclass
class VerifyResult:
    out_tokens: "object"
    num_accepted: "object"
    status: "object"


class Verifier:
    """A handle plus output allocation.  ``verify`` returns device tensors."""

    def __init__(self, max_num_reqs: int, max_spec_len: int, vocab_size: int, device: int = 0,
                 cluster_ctas: int = 0, flags: int = 0):
        self.device = device
        self.handle = spec_verify_create(max_num_reqs, max_spec_len, vocab_size, device, cluster_ctas, flags)

    def close(self):
        if self.handle:
            spec_verify_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def verify(self, *, entry: str, draft_ids, target, max_spec_len: int, num_reqs: int, stream=None,
               out_tokens=None, num_accepted=None, status=None, **kw) -> VerifyResult:
        import torch
        dev = target.device
        if out_tokens is None:
            out_tokens = torch.empty((num_reqs, max_spec_len + 1), dtype=torch.int32, device=dev)
        if num_accepted is None:
            num_accepted = torch.empty((num_reqs,), dtype=torch.int32, device=dev)
        if status is None:
            status = torch.zeros((1,), dtype=torch.int32, device=dev)
        spec_verify_run(self.handle, stream=stream, entry=entry, draft_ids=draft_ids, target=target,
                        out_tokens=out_tokens, num_accepted=num_accepted, status=status, **kw)
        return VerifyResult(out_tokens, num_accepted, status)
