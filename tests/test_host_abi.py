"""Host-side checks of the C ABI: the library builds, loads without a GPU,
exports every function include/spec_verify.h declares, its structs match the
binding, and spec_verify_check_args rejects bad calls before any launch."""
import ctypes
import re

import pytest

from conftest import ROOT

import speculative_decoding_token_rejection_gb300 as sv


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_token_rejection_gb300 import _build
    _build.build()
    return sv.load_library()


def declared_functions():
    text = (ROOT / "include" / "spec_verify.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify_\w+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(sv.EXPORTED) == set(names)


def test_abi_description(lib):
    assert lib.spec_verify_abi_version() == 8
    assert lib.spec_verify_sizeof_args() == ctypes.sizeof(sv.SpecVerifyArgs)
    assert lib.spec_verify_sizeof_config() == ctypes.sizeof(sv.SpecVerifyConfig)


def test_status_strings(lib):
    assert [sv.spec_verify_status_string(c) for c in range(5)] == [
        "SV_OK", "SV_ERR_INVALID_ARG", "SV_ERR_UNSUPPORTED", "SV_ERR_CUDA", "SV_ERR_CAPACITY"]


FAKE = 0x10000  # never dereferenced: check_args only looks at pointer presence


def good_args(N=4, G=3, V=1000):
    a = sv.SpecVerifyArgs()
    a.num_reqs, a.max_spec_len, a.vocab_size = N, G, V
    a.entry, a.dtype = sv.SV_ENTRY_PROBS, sv.SV_F32
    a.num_draft_tokens_total = N * G
    a.draft_ids = FAKE
    a.target, a.target_row_stride = FAKE, V
    a.draft, a.draft_row_stride = FAKE, V
    a.out_tokens = FAKE
    a.num_accepted = FAKE
    return a


def cfg(**kw):
    c = dict(max_num_reqs=8, max_spec_len=4, vocab_size=2000)
    c.update(kw)
    return sv.make_config(**c)


@pytest.mark.parametrize("mutate,code", [
    (lambda a: None, sv.SV_OK),
    (lambda a: setattr(a, "num_reqs", 9), sv.SV_ERR_CAPACITY),
    (lambda a: setattr(a, "num_reqs", -1), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "max_spec_len", 5), sv.SV_ERR_CAPACITY),
    (lambda a: setattr(a, "vocab_size", 2001), sv.SV_ERR_CAPACITY),
    (lambda a: setattr(a, "vocab_size", 0), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "entry", 7), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "dtype", sv.SV_BF16), sv.SV_ERR_UNSUPPORTED),  # probs entry is fp32 only
    (lambda a: (setattr(a, "entry", sv.SV_ENTRY_LOGITS), setattr(a, "dtype", sv.SV_BF16)), sv.SV_OK),
    (lambda a: setattr(a, "entry", sv.SV_ENTRY_LOGITS), sv.SV_OK),  # fp32 logits
    (lambda a: setattr(a, "hints", 2), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "hints", 1), sv.SV_OK),
    (lambda a: setattr(a, "num_draft_tokens_total", 11), sv.SV_ERR_INVALID_ARG),  # != N*G without cu
    (lambda a: setattr(a, "draft_ids", None), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "target", None), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "target_row_stride", 999), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "draft_row_stride", 10), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "uniforms", FAKE), sv.SV_ERR_INVALID_ARG),  # without exponentials
    (lambda a: (setattr(a, "uniforms", FAKE), setattr(a, "exponentials", FAKE),
                setattr(a, "exponentials_row_stride", 1000)), sv.SV_OK),
    (lambda a: (setattr(a, "uniforms", FAKE), setattr(a, "exponentials", FAKE),
                setattr(a, "exponentials_row_stride", 10)), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "exponentials", FAKE), sv.SV_ERR_INVALID_ARG),  # test mode, T > 0, no uniforms
    (lambda a: (setattr(a, "exponentials", FAKE), setattr(a, "exponentials_row_stride", 1000),
                setattr(a, "num_reqs", 2), setattr(a, "max_spec_len", 0),
                setattr(a, "num_draft_tokens_total", 0)), sv.SV_OK),  # T = 0: uniforms may be absent
    (lambda a: setattr(a, "out_tokens", None), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "num_accepted", None), sv.SV_ERR_INVALID_ARG),
    (lambda a: (setattr(a, "cu_num_draft_tokens", FAKE), setattr(a, "num_draft_tokens_total", 5)), sv.SV_OK),
    (lambda a: (setattr(a, "cu_num_draft_tokens", FAKE), setattr(a, "num_draft_tokens_total", 13)),
     sv.SV_ERR_INVALID_ARG),  # T > N*G
    (lambda a: (setattr(a, "num_reqs", 0), setattr(a, "num_draft_tokens_total", 0),
                setattr(a, "target", None)), sv.SV_OK),  # empty batch: no pointers needed
    # processors belong to the logits entry; stop tokens to both
    (lambda a: setattr(a, "repetition_penalty", FAKE), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "banned_cu", FAKE), sv.SV_ERR_INVALID_ARG),
    (lambda a: (setattr(a, "entry", sv.SV_ENTRY_LOGITS), setattr(a, "repetition_penalty", FAKE),
                setattr(a, "penalty_cu", FAKE), setattr(a, "penalty_token_ids", FAKE),
                setattr(a, "penalty_total", 3)), sv.SV_OK),
    (lambda a: (setattr(a, "entry", sv.SV_ENTRY_LOGITS), setattr(a, "banned_cu", FAKE),
                setattr(a, "banned_total", 3)), sv.SV_ERR_INVALID_ARG),  # ids missing
    (lambda a: (setattr(a, "entry", sv.SV_ENTRY_LOGITS), setattr(a, "banned_cu", FAKE),
                setattr(a, "banned_total", 0)), sv.SV_OK),  # empty lists need no ids
    (lambda a: (setattr(a, "stop_cu", FAKE), setattr(a, "stop_token_ids", FAKE), setattr(a, "stop_total", 2)),
     sv.SV_OK),
    (lambda a: (setattr(a, "stop_cu", FAKE), setattr(a, "stop_token_ids", FAKE), setattr(a, "stop_total", -1)),
     sv.SV_ERR_INVALID_ARG),
])
def test_check_args(lib, mutate, code):
    a = good_args()
    mutate(a)
    assert sv.spec_verify_check_args(cfg(), a) == code


@pytest.mark.parametrize("kw,code", [
    (dict(max_num_reqs=0), sv.SV_ERR_INVALID_ARG),
    (dict(max_spec_len=257), sv.SV_ERR_INVALID_ARG),
    (dict(vocab_size=0), sv.SV_ERR_INVALID_ARG),
    (dict(cluster_ctas=3), sv.SV_ERR_INVALID_ARG),
    (dict(cluster_ctas=16), sv.SV_OK),
    (dict(flags=sv.SV_FLAG_RESIDENT_ROWS), sv.SV_OK),
    (dict(flags=sv.SV_FLAG_ONE_CTA_PER_REQUEST), sv.SV_OK),
    (dict(flags=sv.SV_FLAG_SERIAL_LAUNCH), sv.SV_OK),
    (dict(flags=sv.SV_FLAG_SERIAL_LAUNCH | sv.SV_FLAG_ONE_CTA_PER_REQUEST), sv.SV_OK),
    (dict(flags=8), sv.SV_ERR_INVALID_ARG),
])
def test_check_config(lib, kw, code):
    assert sv.spec_verify_check_args(cfg(**kw), good_args()) == code


def test_null_pointers_rejected(lib):
    assert lib.spec_verify_check_args(None, None) == sv.SV_ERR_INVALID_ARG
    c = cfg()
    assert lib.spec_verify_check_args(ctypes.byref(c), None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_run(None, None, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_destroy(None) == sv.SV_OK
    h = ctypes.c_void_p()
    assert lib.spec_verify_create(None, ctypes.byref(h)) == sv.SV_ERR_INVALID_ARG


def test_create_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(sv.SpecVerifyError) as ei:
        sv.spec_verify_create(4, 4, 1000)
    assert ei.value.code == sv.SV_ERR_CUDA


def test_gpu_test_workloads_pass_host_marshalling(lib):
    """Every workload the GPU tests send goes through the binding's tensor
    checks and the library's host validation without error (CPU tensors: the
    pointers are only checked for presence)."""
    import torch
    import workloads
    import test_gpu_probs as tg
    cases = list(tg.edge_cases().values())
    cases += [workloads.make(n, **kw) for n, kw in tg.CASES if n != "fused_probs" or kw]
    cases += [workloads.make("greedy", N=7, V=3001), workloads.make("ragged", N=40, V=3001),
              workloads.make("fused", N=24, V=8192)]
    cfg_ = sv.make_config(1 << 20, sv.SV_MAX_SPEC_LEN, 1 << 18)
    for w in cases:
        t = workloads.as_torch(w, "cpu")
        N, G, T = w["N"], w["gamma"], w["T"]
        for production in (False, True):
            a = sv.build_args(
                entry=w["entry"], draft_ids=t["draft_ids"], target=t["target"], draft=t["draft"],
                cu_num_draft_tokens=t["cu_num_draft_tokens"], temperature=t["temperature"],
                top_k=t.get("top_k"), top_p=t.get("top_p"),
                uniforms=None if production else t["uniforms"],
                exponentials=None if production else t["exponentials"],
                out_tokens=torch.empty((N, G + 1), dtype=torch.int32), num_accepted=torch.empty(N, dtype=torch.int32),
                num_computed_tokens=t.get("num_computed_tokens"), slot_mapping=t.get("slot_mapping"),
                dbg_py=torch.empty(T), dbg_qy=torch.empty(T), status=torch.zeros(1, dtype=torch.int32))
            assert sv.spec_verify_check_args(cfg_, a) == sv.SV_OK, (w.get("name"), production,
                                                                   lib.spec_verify_last_error())


def _sample_args(R=4, V=1000):
    a = sv.SpecVerifySampleArgs()
    a.num_rows, a.vocab_size, a.dtype = R, V, sv.SV_BF16
    a.logits, a.row_stride = FAKE, V
    a.tokens = FAKE
    return a


@pytest.mark.parametrize("mutate,code", [
    (lambda a: None, sv.SV_OK),
    (lambda a: setattr(a, "num_rows", 9), sv.SV_ERR_CAPACITY),
    (lambda a: setattr(a, "num_rows", -1), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "vocab_size", 2001), sv.SV_ERR_CAPACITY),
    (lambda a: setattr(a, "dtype", 5), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "logits", None), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "row_stride", 999), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "tokens", None), sv.SV_ERR_INVALID_ARG),
    (lambda a: (setattr(a, "probs", FAKE), setattr(a, "probs_row_stride", 10)), sv.SV_ERR_INVALID_ARG),
    (lambda a: (setattr(a, "exponentials", FAKE), setattr(a, "exponentials_row_stride", 1000)), sv.SV_OK),
    (lambda a: setattr(a, "test_flags", 3), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "test_flags", 1), sv.SV_OK),
    (lambda a: setattr(a, "hints", 2), sv.SV_ERR_INVALID_ARG),
    (lambda a: setattr(a, "hints", sv.SV_HINT_SMALL_TOP_K), sv.SV_OK),
    (lambda a: (setattr(a, "num_rows", 0), setattr(a, "logits", None)), sv.SV_OK),
])
def test_check_sample_args(lib, mutate, code):
    a = _sample_args()
    mutate(a)
    assert sv.spec_verify_check_sample_args(cfg(), a) == code


def _ngram_args(sv, **kw):
    a = sv.SpecVerifyNgramArgs()
    a.num_reqs, a.min_ngram, a.max_ngram, a.num_spec_tokens = 4, 2, 5, 3
    a.max_model_len, a.num_tokens_total = 100, 50
    a.token_ids, a.cu_num_tokens, a.draft_token_ids, a.num_draft_tokens = 0x1000, 0x2000, 0x3000, 0x4000
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("mutate,code", [
    ({}, 0), (dict(num_reqs=0, token_ids=None, cu_num_tokens=None), 0), (dict(num_reqs=-1), 1),
    (dict(num_reqs=1 << 20), 4), (dict(num_spec_tokens=-1), 1), (dict(num_spec_tokens=9), 4),
    (dict(min_ngram=0), 1), (dict(max_ngram=1), 1), (dict(min_ngram=3, max_ngram=65), 2),
    (dict(max_model_len=0), 1), (dict(num_tokens_total=-1), 1), (dict(cu_num_tokens=None), 1),
    (dict(token_ids=None), 1), (dict(token_ids=None, num_tokens_total=0), 0), (dict(num_draft_tokens=None), 1),
    (dict(draft_token_ids=None), 1), (dict(draft_token_ids=None, num_spec_tokens=0), 0)])
def test_check_ngram_args(lib, mutate, code):
    import speculative_decoding_token_rejection_gb300 as sv
    cfg = sv.make_config(64, 8, 1000)
    assert sv.spec_verify_check_ngram_args(cfg, _ngram_args(sv, **mutate)) == code
