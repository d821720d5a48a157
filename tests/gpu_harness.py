"""Helpers shared by the GPU tests: run a workload through the C ABI (via the
Python binding) and through the oracle, and compare."""
import numpy as np
import torch

import speculative_decoding_token_rejection_gb300 as sv
import workloads

_VERIFIERS = {}


def verifier(cluster_ctas=0, flags=0):
    key = (cluster_ctas, flags)
    if key not in _VERIFIERS:
        _VERIFIERS[key] = sv.Verifier(1 << 20, sv.SV_MAX_SPEC_LEN, 1 << 19, device=0, cluster_ctas=cluster_ctas,
                                      flags=flags)
    return _VERIFIERS[key]


def processor_args(w, dev):
    """Logits processors and stop tokens of a workload dict (optional keys, the
    names the oracle reads) as binding keyword arguments."""
    out = {}
    if w.get("repetition_penalty") is not None:
        out["repetition_penalty"] = torch.as_tensor(np.asarray(w["repetition_penalty"], np.float32)).to(dev)
    for name, kw in (("penalty", "penalty"), ("banned", "banned"), ("stop", "stop")):
        if w.get(f"{name}_cu") is not None:
            out[f"{kw}_cu"] = torch.as_tensor(np.asarray(w[f"{name}_cu"], np.int64)).to(dev)
            out[f"{kw}_token_ids"] = torch.as_tensor(np.asarray(w[f"{name}_ids"], np.int32)).to(dev)
    return out


# handle flags OR-ed into every run_gpu call (a test module sets it to rerun
# other modules' cases in another form of the kernels)
EXTRA_FLAGS = 0


def run_gpu(w, *, production=False, seed=0, offset=0, rng_request_base=0, cluster_ctas=0, stream=None,
            synthetic_rates=None, flags=0, test_flags=0, hints=0):
    """Run the CUDA path on workload ``w``; returns numpy results like oracle.verify."""
    flags |= EXTRA_FLAGS
    dev = torch.device("cuda:0")
    t = workloads.as_torch(w, dev)
    N, G, T = w["N"], w["gamma"], w["T"]
    out = torch.full((N, G + 1), -7, dtype=torch.int32, device=dev)
    nacc = torch.full((N,), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dpy = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    dqy = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    ncomp = t.get("num_computed_tokens")
    slots = t.get("slot_mapping")
    ncomp = None if ncomp is None else ncomp.clone()
    slots = None if slots is None else slots.clone()
    sv.spec_verify_run(
        verifier(cluster_ctas, flags).handle, stream=stream, entry=w["entry"], draft_ids=t["draft_ids"],
        target=t["target"], draft=t["draft"], cu_num_draft_tokens=t["cu_num_draft_tokens"],
        temperature=t["temperature"], top_k=t.get("top_k"), top_p=t.get("top_p"),
        uniforms=None if production else t["uniforms"], exponentials=None if production else t["exponentials"],
        seed=seed, offset=offset, rng_request_base=rng_request_base, out_tokens=out, num_accepted=nacc,
        num_computed_tokens=ncomp, slot_mapping=slots, dbg_py=dpy, dbg_qy=dqy, status=status,
        synthetic_acceptance_rates=None if synthetic_rates is None else
        torch.as_tensor(np.asarray(synthetic_rates, np.float32)).to(dev), test_flags=test_flags, hints=hints,
        **processor_args(w, dev))
    torch.cuda.synchronize()
    cpu = lambda x: None if x is None else x.cpu().numpy()
    return dict(out_tokens=cpu(out), num_accepted=cpu(nacc), num_computed_tokens=cpu(ncomp),
                slot_mapping=cpu(slots), dbg_py=cpu(dpy), dbg_qy=cpu(dqy), status=int(status.item()))


def assert_same(g, o, *, check_dbg=True, exempt=None):
    """Bit-exact comparison of every output; ``exempt`` masks requests whose
    token may legitimately differ (their acceptance count must still match)."""
    N = o["out_tokens"].shape[0]
    keep = np.ones(N, bool) if exempt is None else ~exempt
    np.testing.assert_array_equal(g["num_accepted"], o["num_accepted"])
    np.testing.assert_array_equal(g["out_tokens"][keep], o["out_tokens"][keep])
    if o["num_computed_tokens"] is not None:
        np.testing.assert_array_equal(g["num_computed_tokens"], o["num_computed_tokens"])
    if o["slot_mapping"] is not None:
        np.testing.assert_array_equal(g["slot_mapping"], o["slot_mapping"])
    assert g["status"] == o["status"], (g["status"], o["status"])
    if check_dbg:
        np.testing.assert_array_equal(np.isnan(g["dbg_py"]), np.isnan(o["dbg_py"]))
        m = ~np.isnan(o["dbg_py"])
        np.testing.assert_array_equal(g["dbg_py"][m].view(np.uint32), o["dbg_py"][m].view(np.uint32))
        np.testing.assert_array_equal(g["dbg_qy"][m].view(np.uint32), o["dbg_qy"][m].view(np.uint32))
