#!/usr/bin/env python
"""Benchmark of the batched speculative-decoding verifier on one GB300.

Workload (one "step" = one verification call over the whole batch): N=512
requests, gamma=7 drafts each, V=151936, fp32 probability rows with the
fused workload's sparse support (50 largest logits at T=0.8), production-mode
randomness (Philox inside the kernel; the offset advances every step).  Inputs
are synthetic (workloads.py) and resident in HBM before timing.  The rows one
step touches (~0.6 GB) exceed the 126 MB L2 several times over, so no flush is
inserted.

Prints one JSON line: verified draft tokens/s for the whole job, the roofline
of the verifier kernel against the measured HBM copy bandwidth, the logits
entry on the same batch shape (and two other sampling settings on its rows),
the n-gram proposer on its own batch, the other next-step calls (synthetic
acceptance, the logits entry with processors, the draft-side sampler with and
without q rows), end-to-end figures through the C ABI with inputs in pinned
host memory (zero-copy rows, and full copies), the CPU oracle on all host
cores and on one as a reported baseline, and the SM clocks sampled during the
timed region.  --impl reference times the CPU oracle itself on the same
batch (all host cores).

  python bench.py [--steps K] [--warmup W] [--impl ours|reference] [--gpus N]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import pathlib
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "verified draft tokens/s at N=512,gamma=7,V=151936; achieved HBM GB/s vs ~8 TB/s"
UNIT = "verified draft tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "fused_probs"
KERNEL_SOURCES = ["sv_probs.cu", "sv_device.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cluster", type=int, default=0, help="CTAs per request (0 = automatic)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--requests", type=int, default=0, help="override the batch size (profiling runs only)")
    ap.add_argument("--logits-steps", type=int, default=300)
    ap.add_argument("--no-logits", action="store_true")
    ap.add_argument("--logits-variant-steps", type=int, default=30)
    ap.add_argument("--ngram-steps", type=int, default=200)
    ap.add_argument("--logits-form", choices=["auto", "cluster", "stream"], default="auto",
                    help="logits entry: library choice with the small-top-k hint, clusters only, or one CTA per request")
    ap.add_argument("--logits-resident", action="store_true",
                    help="keep both row chunks of the logits entry in shared memory (comparison runs)")
    ap.add_argument("--no-ngram", action="store_true")
    ap.add_argument("--sampler-steps", type=int, default=100)
    ap.add_argument("--processor-steps", type=int, default=100)
    ap.add_argument("--synthetic-steps", type=int, default=1000)
    ap.add_argument("--no-next", action="store_true",
                    help="skip the draft-side sampler, processors and synthetic-acceptance objects")
    ap.add_argument("--serial-launch", action="store_true",
                    help="create every handle with SV_FLAG_SERIAL_LAUNCH (plain stream order; comparison runs)")
    args = ap.parse_args()
    global LAUNCH_FLAGS
    if args.serial_launch:
        LAUNCH_FLAGS = 4  # SV_FLAG_SERIAL_LAUNCH (checked against the binding in main)
    return args


# flags OR-ed into every handle the bench creates (SV_FLAG_SERIAL_LAUNCH under --serial-launch)
LAUNCH_FLAGS = 0


def measured_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback (6.8 TB/s earlier GB300 copy measurement)"


LOGITS_KERNEL_SOURCES = ["sv_logits.cuh", "sv_logits.cu", "sv_logits_bf16.cu", "sv_logits_f32.cu", "sv_sample_bf16.cu",
                         "sv_sample_f32.cu", "sv_device.cuh"]  # (the processor units instantiate the same templates)
STREAM_KERNEL_SOURCES = ["sv_stream.cuh", "sv_stream_bf16.cu", "sv_logits.cuh", "sv_device.cuh"]
NGRAM_KERNEL_SOURCES = ["sv_ngram.cu", "sv_device.cuh"]


def kernel_source_hash(sources=None) -> str:
    """Hash of the kernel sources with comments and whitespace removed, so an
    edit to the documentation does not retire the stored ncu counters (the
    sources hold no string literal with a comment marker)."""
    h = hashlib.sha256()
    for n in (sources or KERNEL_SOURCES):
        text = (ROOT / "speculative_decoding_token_rejection_gb300" / "csrc" / n).read_text()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def stored_traffic(name="verify_probs_fused_probs", sources=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = ROOT / "profiles" / f"{name}.traffic.json"
    if not p.exists():
        return None, None
    d = json.loads(p.read_text())
    if d.get("kernel_source_sha") != kernel_source_hash(sources):
        return None, d.get("kernel_source_sha")
    return d.get("dram_bytes_per_launch"), d.get("kernel_source_sha")


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.dev = device_index

    def start(self):
        import torch
        sel = str(self.dev)
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:
            inside = [s for _, s in self.samples]
            window = "whole run (timed region shorter than the 200 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for s in inside for k in range(4) if len(s) > 5 + k and "Active" in s[5 + k]
                          and "Not" not in s[5 + k]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((num(s[3]) or 0.0) for s in inside)}


# ----------------------------------------------------------------------------
def algorithmic_bytes(nacc, gammas, V, G):
    """Minimal bytes one call must move per request (probability entry,
    production mode): draft ids, the gathered p(y)/q(y) at examined positions,
    one streamed row pair (rejection) or one row (bonus), the temperature, the
    output row and num_accepted, num_computed_tokens read+write and the slot
    entries set to -1."""
    import numpy as np
    A = nacc.astype(np.int64)
    g = gammas.astype(np.int64)
    gathered = np.minimum(A + 1, g)
    row = np.where(A < g, 8 * V, 4 * V)
    per = 4 * g + 8 * gathered + row + 4 + 4 * (G + 1) + 4 + 8 + 8 * (g - A)
    return int(per.sum())


def logits_algorithmic_bytes(nacc, gammas, temps, V, G, elem=2):
    """Minimal bytes of one logits-entry call: the logits rows a sequential
    verifier must read -- target rows 0..A, and for random requests draft rows
    0..min(A, gamma-1) -- plus ids, parameters, outputs and KV bookkeeping."""
    import numpy as np
    A = nacc.astype(np.int64)
    g = gammas.astype(np.int64)
    rows = np.where(temps == 0, A + 1, (A + 1) + np.minimum(A + 1, g))
    per = rows * V * elem + 4 * g + 12 + 4 * (G + 1) + 4 + 8 + 8 * (g - A)
    return int(per.sum())


def time_logits_entry(args, sv, lib, dev, world, rank, dist, stream, top_k=50, top_p=0.9, steps=None, w=None):
    """The logits entry on the same batch shape: bf16 target/draft logits with
    T=0.8, top-k 50, top-p 0.9 per request (production Philox); other
    sampling settings on the same rows with ``top_k`` / ``top_p``."""
    import numpy as np
    import torch
    import workloads
    if w is None:
        w = workloads.make("fused", seed=3 + 1000 * rank, test_mode=False, N=args.requests or None)
    N, G, V, T = w["N"], w["gamma"], w["V"], w["T"]
    w = dict(w, top_k=np.full(N, top_k, np.int32), top_p=np.full(N, top_p, np.float32))
    gam = workloads.gammas_of(w)
    t = workloads.as_torch(w, dev)
    flags = (sv.SV_FLAG_RESIDENT_ROWS if args.logits_resident else 0) | LAUNCH_FLAGS
    if args.logits_form == "stream":
        flags |= sv.SV_FLAG_ONE_CTA_PER_REQUEST
    ver = sv.Verifier(N, G, V, device=dev.index, cluster_ctas=args.cluster, flags=flags)
    # the caller knows its sampling parameters: top-k 50 is a small top-k
    hints = sv.SV_HINT_SMALL_TOP_K if (0 < top_k <= sv.SV_SMALL_TOP_K_MAX and args.logits_form != "cluster") else 0
    K = max(3, min(args.steps, steps or args.logits_steps))
    W = args.warmup
    nacc = torch.empty((K + W, N), dtype=torch.int32, device=dev)
    out = torch.empty((N, G + 1), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    a = sv.build_args(entry="logits", draft_ids=t["draft_ids"], target=t["target"], draft=t["draft"],
                      temperature=t["temperature"], top_k=t["top_k"], top_p=t["top_p"], out_tokens=out,
                      num_accepted=nacc[0], num_computed_tokens=t["num_computed_tokens"].clone(),
                      slot_mapping=t["slot_mapping"].clone(), status=status, seed=20240602,
                      rng_request_base=rank * N, hints=hints)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    h = ctypes.c_void_p(ver.handle)

    def step(k):
        a.offset = k
        a.num_accepted = nacc.data_ptr() + 4 * N * k
        if lib.spec_verify_run(h, ctypes.byref(a), sptr) != 0:
            raise RuntimeError(lib.spec_verify_last_error().decode())

    for k in range(W):
        step(k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for k in range(K):
        step(W + k)
    ev[1].record(stream)
    torch.cuda.synchronize()
    total_ms = ev[0].elapsed_time(ev[1])
    if dist:
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    na = nacc[W:].cpu().numpy()
    alg = float(np.mean([logits_algorithmic_bytes(na[k], gam, w["temperature"], V, G) for k in range(K)]))
    ms = total_ms / K
    peak, src = measured_peak()
    full = (2 * T + N) * V * 2
    # the form the library takes (include/spec_verify.h: the flag, or the hint on a batch of at least two
    # requests per SM; never with resident rows)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream_form = not args.logits_resident and (args.logits_form == "stream" or (hints and N >= 2 * sms))
    sources = STREAM_KERNEL_SOURCES if stream_form else LOGITS_KERNEL_SOURCES
    traffic, traffic_sha = stored_traffic("verify_logits_fused_stream" if stream_form else "verify_logits_fused",
                                          sources)
    if traffic is not None and (N != 512 or top_k != 50 or top_p != 0.9):
        traffic = None  # the stored counters are scaled to a 512-request launch of this setting
    ver.close()
    return {"value": world * T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": K,
            "config": {"workload": f"fused: N={N} gamma={G} V={V} bf16 logits, T=0.8, top-k {top_k if top_k > 0 else 'off'}, "
                                   f"top-p {top_p if top_p < 1 else 'off'}, production Philox", "entry": "logits",
                       "rows": "shared memory" if args.logits_resident else "read in place (L2 prefetch)",
                       "hints": "small top-k" if hints else "none",
                       "form": "one CTA per request" if stream_form else "clusters"},
            "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": alg / (ms / 1e3) / 1e9 / peak, "traffic": traffic, "peak_source": src,
                         "algorithmic_bytes_per_launch": alg, "full_tensor_bytes": full,
                         "full_tensor_equiv_gbs": full / (ms / 1e3) / 1e9,
                         "full_tensor_equiv_of_peak": full / (ms / 1e3) / 1e9 / peak,
                         "kernel_source_sha": kernel_source_hash(sources),
                         "traffic_source_sha": traffic_sha},
            "acceptance": {"mean_accepted": float(na.mean()),
                           "A_hist": np.bincount(na.reshape(-1), minlength=G + 1).tolist()},
            "gpu_launches": K, "_w": w}


def _timed_launches(step, K, W, stream, dev, dist):
    """W untimed launches, then K launches between CUDA events on ``stream``;
    the mean milliseconds per launch (max over ranks)."""
    import torch
    for k in range(W):
        step(k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(K):
        step(W + k)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    if dist:
        tt = torch.tensor([ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    return ms


def time_sampler(args, sv, dev, world, rank, dist, stream, w, write_q):
    """The draft-side sampler on one draft step of the fused batch: one bf16
    row of V=151936 per request (N=512 rows), T=0.8, top-k 50, top-p 0.9,
    production Philox.  Launch k samples draft position k mod gamma, so
    consecutive launches read different rows (155.6 MB per launch, above the
    L2 size).  With ``write_q`` the transformed fp32 row of every request is
    written out too, in the probability entry's q layout."""
    import numpy as np
    import torch
    N, G, V = w["N"], w["gamma"], w["V"]
    draft = torch.from_numpy(w["draft"].view(np.int16)).view(torch.bfloat16).to(dev).view(N, G, V)
    temp = torch.from_numpy(np.asarray(w["temperature"], np.float32)).to(dev)
    top_k = torch.full((N,), 50, dtype=torch.int32, device=dev)
    top_p = torch.full((N,), 0.9, dtype=torch.float32, device=dev)
    tokens = torch.empty((N,), dtype=torch.int32, device=dev)
    probs = torch.empty((N, V), dtype=torch.float32, device=dev) if write_q else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    h = sv.spec_verify_create(N, 1, V, device=dev.index, cluster_ctas=args.cluster, flags=LAUNCH_FLAGS)
    lib = sv.load_library()
    sptr = ctypes.c_void_p(stream.cuda_stream)
    # the caller knows its sampling parameters: top-k 50 is a small top-k (one CTA per row on a large batch)
    hints = sv.SV_HINT_SMALL_TOP_K if args.logits_form != "cluster" else 0
    flags_f = sv.SV_FLAG_ONE_CTA_PER_REQUEST if args.logits_form == "stream" else 0
    if flags_f:
        sv.spec_verify_destroy(h)
        h = sv.spec_verify_create(N, 1, V, device=dev.index, cluster_ctas=args.cluster, flags=flags_f | LAUNCH_FLAGS)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream_form = bool(flags_f) or (bool(hints) and N >= 2 * sms)
    built = [sv.build_sample_args(logits=draft[:, j, :], tokens=tokens, probs=probs, temperature=temp,
                                  top_k=top_k, top_p=top_p, seed=20240603, rng_row_base=rank * N, status=status,
                                  hints=hints)
             for j in range(G)]

    def step(k):
        a = built[k % G]
        a.offset = k
        if lib.spec_verify_sample(ctypes.c_void_p(h), ctypes.byref(a), sptr) != 0:
            raise RuntimeError(lib.spec_verify_last_error().decode())

    K = max(3, min(args.steps, args.sampler_steps))
    ms = _timed_launches(step, K, args.warmup, stream, dev, dist)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    sv.spec_verify_destroy(h)
    alg = N * V * 2 + N * (4 + 4 + 4 + 4) + (N * V * 4 if write_q else 0)
    peak, src = measured_peak()
    sources = STREAM_KERNEL_SOURCES if stream_form else LOGITS_KERNEL_SOURCES
    traffic, traffic_sha = (None, None) if write_q else stored_traffic(
        "draft_sampler_fused_rows_per_row" if stream_form else "draft_sampler_fused_rows", sources)
    if traffic is not None and N != 512:
        traffic = None  # the stored counters are scaled to a 512-row launch
    return {"value": world * N / (ms / 1e3), "unit": "sampled tokens/s", "ms_per_step": ms, "steps": K,
            "config": {"workload": f"draft step of the fused batch: {N} bf16 rows of V={V}, T=0.8, top-k 50, "
                                   "top-p 0.9, production Philox" + (", fp32 q rows written" if write_q else ""),
                       "form": "one CTA per row" if stream_form else "clusters",
                       "l2": f"no flush: launch k reads draft position k mod {G} ({N * V * 2 / 1e6:.1f} MB per "
                             f"launch; {N * G * V * 2 / 1e6:.0f} MB over {G} launches, > 126 MB L2)"},
            "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": alg / (ms / 1e3) / 1e9 / peak, "traffic": traffic, "peak_source": src,
                         "algorithmic_bytes_per_launch": alg,
                         "kernel_source_sha": kernel_source_hash(sources),
                         "traffic_source_sha": traffic_sha},
            "gpu_launches": K}


def processor_lists(N, V, seed, context=512, banned=16, stop=2):
    """Per-request logits processors of a serving batch: a repetition penalty
    of 1.2 over the last ``context`` tokens of each request's context, ``banned``
    banned ids and ``stop`` stop ids (uniform over the vocabulary), as
    inclusive int64 prefix sums and int32 ids."""
    import numpy as np
    rng = np.random.default_rng(seed)
    out = {"repetition_penalty": np.full(N, 1.2, np.float32)}
    for name, n in (("penalty", context), ("banned", banned), ("stop", stop)):
        out[f"{name}_cu"] = np.arange(1, N + 1, dtype=np.int64) * n
        out[f"{name}_ids"] = rng.integers(0, V, size=N * n).astype(np.int32)
    return out


def time_processors(args, sv, lib, dev, world, rank, dist, stream, w):
    """The logits entry on the fused batch with logits processors and stop
    tokens: repetition penalty 1.2 over a 512-token context per request (the
    request's drafts join it as they are committed), 16 banned ids and 2 stop
    ids per request.  The kept sets are placed on the raw rows (read in place
    unless --logits-resident) and the processors then act on the kept entries;
    with the small-top-k hint the call takes one CTA per request."""
    import numpy as np
    import torch
    import workloads
    N, G, V, T = w["N"], w["gamma"], w["V"], w["T"]
    w = dict(w, top_k=np.full(N, 50, np.int32), top_p=np.full(N, 0.9, np.float32))
    gam = workloads.gammas_of(w)
    t = workloads.as_torch(w, dev)
    pl = {k: torch.from_numpy(v).to(dev) for k, v in processor_lists(N, V, seed=11 + 1000 * rank).items()}
    flags = (sv.SV_FLAG_RESIDENT_ROWS if args.logits_resident else 0) | LAUNCH_FLAGS
    if args.logits_form == "stream":
        flags |= sv.SV_FLAG_ONE_CTA_PER_REQUEST
    ver = sv.Verifier(N, G, V, device=dev.index, cluster_ctas=args.cluster, flags=flags)
    # top-k 50 is a small top-k: with the hint a batch of two requests per SM takes one CTA per request
    hints = sv.SV_HINT_SMALL_TOP_K if args.logits_form != "cluster" else 0
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream_form = not args.logits_resident and (args.logits_form == "stream" or (hints and N >= 2 * sms))
    K = max(3, min(args.steps, args.processor_steps))
    nacc = torch.empty((K + args.warmup, N), dtype=torch.int32, device=dev)
    out = torch.empty((N, G + 1), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    a = sv.build_args(entry="logits", draft_ids=t["draft_ids"], target=t["target"], draft=t["draft"],
                      temperature=t["temperature"], top_k=t["top_k"], top_p=t["top_p"], out_tokens=out,
                      num_accepted=nacc[0], status=status, seed=20240604, rng_request_base=rank * N,
                      repetition_penalty=pl["repetition_penalty"], penalty_cu=pl["penalty_cu"],
                      penalty_token_ids=pl["penalty_ids"], banned_cu=pl["banned_cu"],
                      banned_token_ids=pl["banned_ids"], stop_cu=pl["stop_cu"], stop_token_ids=pl["stop_ids"],
                      hints=hints)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    h = ctypes.c_void_p(ver.handle)

    def step(k):
        a.offset = k
        a.num_accepted = nacc.data_ptr() + 4 * N * k
        if lib.spec_verify_run(h, ctypes.byref(a), sptr) != 0:
            raise RuntimeError(lib.spec_verify_last_error().decode())

    ms = _timed_launches(step, K, args.warmup, stream, dev, dist)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    na = nacc[args.warmup:].cpu().numpy()
    lists = sum(int(v.numel()) * v.element_size() for v in pl.values())
    alg = float(np.mean([logits_algorithmic_bytes(na[k], gam, w["temperature"], V, G) for k in range(K)])) + lists
    peak, src = measured_peak()
    ver.close()
    return {"value": world * T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": K,
            "config": {"workload": f"fused: N={N} gamma={G} V={V} bf16 logits, T=0.8, top-k 50, top-p 0.9, "
                                   "repetition penalty 1.2 over 512 context ids, 16 banned ids, 2 stop ids per "
                                   "request, production Philox", "entry": "logits",
                       "rows": "shared memory" if args.logits_resident else "read in place (L2 prefetch)",
                       "form": "one CTA per request" if stream_form else "clusters"},
            "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": alg / (ms / 1e3) / 1e9 / peak, "traffic": None, "peak_source": src,
                         "algorithmic_bytes_per_launch": alg},
            "acceptance": {"mean_accepted": float(na.mean())}, "gpu_launches": K}


SYNTHETIC_RATES = [0.8, 0.7, 0.6, 0.5, 0.4, 0.3, 0.2]
NGRAM_BATCHES = 12  # history batches the n-gram launches rotate over (together above the L2 size)


def time_synthetic(args, sv, lib, dev, world, rank, dist, stream, t, gammas, N, G, V, T):
    """The probability entry on the headline batch in synthetic acceptance
    mode: position j is accepted with the preset rate r_j (non-increasing), so
    no p(y), q(y) are gathered; the race still streams the row pair of the
    stopping position (or the bonus row)."""
    import numpy as np
    import torch
    rates = torch.tensor(SYNTHETIC_RATES[:G] + [0.0] * max(0, G - len(SYNTHETIC_RATES)), dtype=torch.float32,
                         device=dev)
    ver = sv.Verifier(N, G, V, device=dev.index, cluster_ctas=args.cluster, flags=LAUNCH_FLAGS)
    K = max(3, min(args.steps, args.synthetic_steps))
    nacc = torch.empty((K + args.warmup, N), dtype=torch.int32, device=dev)
    out = torch.empty((N, G + 1), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    a = sv.build_args(entry="probs", draft_ids=t["draft_ids"], target=t["target"], draft=t["draft"],
                      temperature=t["temperature"], out_tokens=out, num_accepted=nacc[0], status=status,
                      seed=20240605, rng_request_base=rank * N, synthetic_acceptance_rates=rates)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    h = ctypes.c_void_p(ver.handle)

    def step(k):
        a.offset = k
        a.num_accepted = nacc.data_ptr() + 4 * N * k
        if lib.spec_verify_run(h, ctypes.byref(a), sptr) != 0:
            raise RuntimeError(lib.spec_verify_last_error().decode())

    ms = _timed_launches(step, K, args.warmup, stream, dev, dist)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    na = nacc[args.warmup:].cpu().numpy().astype(np.int64)
    g = gammas.astype(np.int64)
    # the probability entry's bytes without the gathers: ids, the raced row(s), outputs
    alg = float(np.mean([int((4 * g + np.where(na[k] < g, 8 * V, 4 * V) + 4 + 4 * (G + 1) + 4).sum())
                         for k in range(K)])) + 4 * G
    peak, src = measured_peak()
    ver.close()
    return {"value": world * T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": K,
            "config": {"workload": f"fused_probs: N={N} gamma={G} V={V} fp32 rows, synthetic rates "
                                   f"{SYNTHETIC_RATES[:G]}, production Philox", "entry": "probs"},
            "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": alg / (ms / 1e3) / 1e9 / peak, "traffic": None, "peak_source": src,
                         "algorithmic_bytes_per_launch": alg},
            "acceptance": {"mean_accepted": float(na.mean()),
                           "A_hist": np.bincount(na.reshape(-1), minlength=G + 1).tolist()},
            "gpu_launches": K}


def time_ngram(args, sv, dev, world, rank, dist, stream):
    """The batched n-gram proposer on its default batch shape (512 repetitive
    histories of 1024..16384 tokens, min/max n-gram 5, k = 7).  One batch of
    histories (~18.5 MB) fits in L2, so the launches rotate over NGRAM_BATCHES
    different batches (~148 MB together, above the L2 size): launch k reads
    batch k mod NGRAM_BATCHES, which the previous launches have evicted, and
    the launches run back to back between two CUDA events, as a serving step
    issues them (the per-launch figure is the whole run's time over the
    launches)."""
    import numpy as np
    import torch
    import workloads
    batches = []
    for b in range(NGRAM_BATCHES):
        tokens, cu = workloads.make_histories(seed=workloads.NGRAM["seed"] + 1000 * rank + 17 * b)
        batches.append((torch.as_tensor(tokens).to(dev), torch.as_tensor(cu).to(dev), int(cu[-1])))
    R, k, n_min, n_max = workloads.NGRAM["R"], 7, 5, 5
    out = torch.empty((R, k), dtype=torch.int32, device=dev)
    num = torch.empty((R,), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    h = sv.spec_verify_create(R, k, 1, device=dev.index, flags=LAUNCH_FLAGS)
    lib = sv.load_library()
    built = [sv.build_ngram_args(token_ids=t, cu_num_tokens=c, draft_token_ids=out, num_draft_tokens=num,
                                 min_ngram=n_min, max_ngram=n_max, max_model_len=1 << 20, status=status)
             for t, c, _ in batches]
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def step(i):
        if lib.spec_verify_ngram_propose(ctypes.c_void_p(h), ctypes.byref(built[i % NGRAM_BATCHES]), sptr) != 0:
            raise RuntimeError(lib.spec_verify_last_error().decode())

    K = max(NGRAM_BATCHES, min(args.steps, args.ngram_steps))
    ms = _timed_launches(step, K, max(args.warmup, NGRAM_BATCHES), stream, dev, dist)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    proposed = num.cpu().numpy()
    sv.spec_verify_destroy(h)
    total = float(np.mean([n for _, _, n in batches]))
    alg = 4 * total + 8 * R + 4 * R * (k + 1)
    peak, src = measured_peak()
    traffic, _ = stored_traffic("ngram_propose_histories", NGRAM_KERNEL_SOURCES)
    return {"value": world * R / (ms / 1e3), "unit": "requests/s", "ms_per_step": ms, "steps": K,
            "history_tokens_per_s": world * total / (ms / 1e3),
            "config": {"workload": f"ngram: R={R} histories of 1024..16384 tokens (mean {int(total) // R}), "
                                   f"vocab 151936, half the segments repeated; min/max n-gram {n_min}/{n_max}, "
                                   f"k={k}", "l2": f"no flush: launch k reads history batch k mod {NGRAM_BATCHES} "
                                                   f"({NGRAM_BATCHES} batches, {NGRAM_BATCHES * 4 * total / 1e6:.0f} MB "
                                                   "together, > 126 MB L2), launches back to back"},
            "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": alg / (ms / 1e3) / 1e9 / peak, "traffic": traffic, "peak_source": src,
                         "algorithmic_bytes_per_launch": alg,
                         "kernel_source_sha": kernel_source_hash(NGRAM_KERNEL_SOURCES)},
            "proposed_fraction_last_batch": float((proposed > 0).mean()), "gpu_launches": K}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, world)
    return run_ours(args, world, rank, local_rank)


def run_ours(args, world, rank, local_rank):
    import numpy as np
    import torch

    import speculative_decoding_token_rejection_gb300 as sv
    import workloads

    assert sv.SV_FLAG_SERIAL_LAUNCH == 4
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist:
            dist.barrier()

    from speculative_decoding_token_rejection_gb300 import _build
    if rank == 0:
        _build.build()
    barrier()

    # weak scaling: every rank verifies its own batch of 512 requests
    w = workloads.make(WORKLOAD, seed=3 + 1000 * rank, test_mode=False, N=args.requests or None)
    N, G, V, T = w["N"], w["gamma"], w["V"], w["T"]
    gammas = workloads.gammas_of(w)
    t = workloads.as_torch(w, dev)
    ver = sv.Verifier(N, G, V, device=local_rank, cluster_ctas=args.cluster, flags=LAUNCH_FLAGS)
    lib = sv.load_library()
    out = torch.empty((N, G + 1), dtype=torch.int32, device=dev)
    K, W = args.steps, args.warmup
    nacc_hist = torch.empty((K + W, N), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ncomp = t["num_computed_tokens"].clone()
    slots = t["slot_mapping"].clone()
    a = sv.build_args(entry="probs", draft_ids=t["draft_ids"], target=t["target"], draft=t["draft"],
                      temperature=t["temperature"], out_tokens=out, num_accepted=nacc_hist[0],
                      num_computed_tokens=ncomp, slot_mapping=slots, status=status, seed=20240601,
                      rng_request_base=rank * N)
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    handle = ctypes.c_void_p(ver.handle)
    run = lib.spec_verify_run
    nacc_base = nacc_hist.data_ptr()
    nacc_stride = N * 4

    def step(k):
        a.offset = k
        a.num_accepted = nacc_base + k * nacc_stride
        rc = run(handle, ctypes.byref(a), sptr)
        if rc != 0:
            raise RuntimeError(lib.spec_verify_last_error().decode())

    for k in range(W):
        step(k)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.5)
    # two events around the K launches, which run back to back as a serving
    # loop issues them (an event between launches would keep each launch from
    # being scheduled while the previous one finishes)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ev[0].record(stream)
    for k in range(K):
        step(W + k)
    ev[1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    logits = None if args.no_logits else time_logits_entry(args, sv, lib, dev, world, rank, dist, stream)
    if logits:
        # the same rows under two other common settings (fewer launches)
        wl = logits.pop("_w")
        logits["other_settings"] = {}
        for name, kk, pp in (("top_p_0.9_alone", 0, 0.9), ("temperature_alone", 0, 1.0)):
            o = time_logits_entry(args, sv, lib, dev, world, rank, dist, stream, top_k=kk, top_p=pp,
                                  steps=args.logits_variant_steps, w=wl)
            o.pop("_w")
            logits["other_settings"][name] = {k: o[k] for k in ("value", "ms_per_step", "steps", "config")}
            logits["other_settings"][name]["roofline_frac"] = o["roofline"]["frac"]
            logits["gpu_launches"] += o["gpu_launches"]
    ngram = None if args.no_ngram else time_ngram(args, sv, dev, world, rank, dist, stream)
    nxt = {}
    if not args.no_next:
        nxt["synthetic_acceptance"] = time_synthetic(args, sv, lib, dev, world, rank, dist, stream, t, gammas,
                                                     N, G, V, T)
        if logits:
            nxt["logits_processors"] = time_processors(args, sv, lib, dev, world, rank, dist, stream, wl)
            nxt["draft_sampler"] = time_sampler(args, sv, dev, world, rank, dist, stream, wl, write_q=False)
            nxt["draft_sampler_with_q_rows"] = time_sampler(args, sv, dev, world, rank, dist, stream, wl,
                                                            write_q=True)
    clocks.stop()
    total_ms = ev[0].elapsed_time(ev[1])
    launch_ms = total_ms / K  # this rank's mean launch duration
    if dist:
        tt = torch.tensor([total_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_per_step = total_ms / K
    value = world * T * K / (total_ms / 1e3)

    nacc_np = nacc_hist[W:].cpu().numpy()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    alg = [algorithmic_bytes(nacc_np[k], gammas, V, G) for k in range(K)]
    alg_mean = float(np.mean(alg))
    achieved = alg_mean / (launch_ms / 1e3) / 1e9
    peak, peak_src = measured_peak()
    full_bytes = (T + N) * V * 4 + T * V * 4
    traffic, traffic_sha = stored_traffic()
    if traffic is not None and N != 512:
        traffic = None  # the stored counters are scaled to a 512-request launch
    acc = nacc_np.astype(np.int64)
    e2e, e2e_fc = (None, None) if args.no_e2e else run_e2e(args, w, t, ver, sv, dev, world, dist)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, args.cpu_seconds)
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: N={N} gamma={G} V={V} fp32 rows (T=0.8, top-k 50, top-p 0.9), "
                               "production Philox",
                   "entry": "probs", "l2": "no flush: ~0.6 GB of rows per step >> 126 MB L2",
                   "cluster_ctas": args.cluster or "auto",
                   "launch": "serial" if LAUNCH_FLAGS else "programmatic (back-to-back kernels may be scheduled "
                                                           "early; each waits for the previous grid first)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": alg_mean, "launch_ms": launch_ms,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "full_tensor_bytes": full_bytes,
                     "full_tensor_equiv_gbs": full_bytes / (launch_ms / 1e3) / 1e9,
                     "full_tensor_equiv_of_peak": full_bytes / (launch_ms / 1e3) / 1e9 / peak,
                     "kernel_source_sha": kernel_source_hash(), "traffic_source_sha": traffic_sha},
        "acceptance": {"rate": float(acc.sum() / (gammas.sum() * K)),
                       "mean_accepted": float(acc.mean()),
                       "committed_tokens_per_s": world * float((acc + 1).sum()) / (total_ms / 1e3),
                       "A_hist": np.bincount(acc.reshape(-1), minlength=G + 1).tolist()},
        "gpu_launches": K,
        "clocks": clocks.summary(t0, t1),
    }
    if e2e:
        line["e2e"] = e2e
        line["e2e_full_copy"] = e2e_fc
    if cpu:
        line["cpu_baseline"] = cpu
    # the other kernels' full objects, then a compact summary of every kernel
    # as the line's last key (the end of the line is what short log tails keep)
    if ngram:
        line["ngram_proposer"] = ngram
    line.update(nxt)
    if logits:
        line["logits_entry"] = logits
    line["summary"] = summary_of(line)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def summary_of(line):
    """Per kernel: ms per call, roofline fraction of the measured peak and
    DRAM traffic over algorithmic bytes (when counters match the source)."""
    def one(o):
        r = o["roofline"]
        t = r.get("traffic")
        return {"ms": round(o["ms_per_step"], 4), "frac": round(r["frac"], 3),
                "traffic_x": None if t is None else round(t / r["algorithmic_bytes_per_launch"], 3)}
    out = {"verify_probs": one(dict(line, ms_per_step=line["roofline"]["launch_ms"]))}
    for key in ("synthetic_acceptance", "ngram_proposer", "draft_sampler", "draft_sampler_with_q_rows",
                "logits_processors", "logits_entry"):
        if key in line:
            out[key] = one(line[key])
    if "logits_entry" in line:
        for name, o in line["logits_entry"].get("other_settings", {}).items():
            out["logits_" + name] = {"ms": round(o["ms_per_step"], 4), "frac": round(o["roofline_frac"], 3)}
    return out


def run_e2e(args, w, t, ver, sv, dev, world, dist):
    """The same metric through the public API with inputs in pinned host
    memory; the timed region of every step includes moving that step's inputs
    to the GPU and reading its results back.

    Zero-copy (reported as ``e2e``): the probability rows stay in pinned host
    memory and the kernel reads only the rows it needs over NVLink-C2C; ids,
    temperatures and the KV bookkeeping are copied.  Full copy (reported as
    ``e2e_full_copy``): every input tensor is copied to HBM first."""
    import numpy as np
    import torch
    import workloads
    h = workloads.as_torch({k: w[k] for k in ("draft_ids", "target", "draft", "temperature",
                                               "num_computed_tokens", "slot_mapping")}, "cpu", pin=True)
    N, G, V, T = w["N"], w["gamma"], w["V"], w["T"]
    gam = workloads.gammas_of(w)
    small = ("draft_ids", "temperature", "num_computed_tokens", "slot_mapping")
    d_in = {k: torch.empty_like(v, device=dev) for k, v in h.items()}
    out = torch.empty((N, G + 1), dtype=torch.int32, device=dev)
    steps = max(1, args.e2e_steps)
    nacc = torch.empty((steps + 1, N), dtype=torch.int32, device=dev)
    h_out = torch.empty((N, G + 1), dtype=torch.int32, pin_memory=True)
    h_nacc = torch.empty((N,), dtype=torch.int32, pin_memory=True)
    h_ncomp = torch.empty_like(h["num_computed_tokens"], pin_memory=True)
    h_slots = torch.empty_like(h["slot_mapping"], pin_memory=True)
    d2h = sum(v.numel() * v.element_size() for v in (h_out, h_nacc, h_ncomp, h_slots))

    def step(k, zero_copy):
        keys = small if zero_copy else tuple(h)
        for key in keys:
            d_in[key].copy_(h[key], non_blocking=True)
        rows = dict(target=h["target"], draft=h["draft"], host_rows=True, device=dev) if zero_copy else \
            dict(target=d_in["target"], draft=d_in["draft"])
        sv.spec_verify_run(ver.handle, entry="probs", draft_ids=d_in["draft_ids"], temperature=d_in["temperature"],
                           out_tokens=out, num_accepted=nacc[k % (steps + 1)],
                           num_computed_tokens=d_in["num_computed_tokens"], slot_mapping=d_in["slot_mapping"],
                           seed=7, offset=k, **rows)
        h_out.copy_(out, non_blocking=True)
        h_nacc.copy_(nacc[k % (steps + 1)], non_blocking=True)
        h_ncomp.copy_(d_in["num_computed_tokens"], non_blocking=True)
        h_slots.copy_(d_in["slot_mapping"], non_blocking=True)

    def timed(zero_copy):
        step(0, zero_copy)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            step(k + 1, zero_copy)
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
        if dist:
            tt = torch.tensor([el], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            el = float(tt.item())
        return el

    el_zc = timed(True)
    na = nacc[1:steps + 1].cpu().numpy()
    rows_read = float(np.mean([algorithmic_bytes(na[k], gam, V, G) for k in range(steps)]))
    small_b = sum(h[k].numel() * h[k].element_size() for k in small)
    zc = {"value": world * T * steps / el_zc, "unit": UNIT,
          "h2d_bytes_per_step": int(small_b + rows_read), "d2h_bytes_per_step": int(d2h),
          "steps": steps, "ms_per_step": el_zc / steps * 1e3,
          "mode": "probability rows read in place from pinned host memory over NVLink-C2C (only the rows the "
                  "verifier needs cross the link); ids, temperatures and KV bookkeeping copied each step; "
                  "outputs and KV bookkeeping read back each step"}
    el_fc = timed(False)
    full_h2d = sum(v.numel() * v.element_size() for v in h.values())
    fc = {"value": world * T * steps / el_fc, "unit": UNIT, "h2d_bytes_per_step": int(full_h2d),
          "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": el_fc / steps * 1e3,
          "mode": "every input tensor copied host->HBM each step, outputs read back"}
    return zc, fc


def oracle_threads() -> int:
    """Host threads for the oracle: every core this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_parallel(w, req_range, threads, **kw):
    """The oracle over the requests [a, b), split into contiguous ranges run by
    ``threads`` host threads.  The C oracle keeps no global state and ctypes
    releases the GIL during each call, so the ranges run in parallel; each
    call is the oracle as it stands."""
    import numpy as np
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    a, b = req_range
    cuts = np.linspace(a, b, min(threads, b - a) + 1).astype(int)
    ranges = [(int(x), int(y)) for x, y in zip(cuts[:-1], cuts[1:]) if y > x]
    if len(ranges) == 1:
        oracle.verify(w, req_range=ranges[0], **kw)
        return
    with ThreadPoolExecutor(len(ranges)) as ex:
        list(ex.map(lambda r: oracle.verify(w, req_range=r, **kw), ranges))


def cpu_baseline(w, seconds):
    """The CPU oracle, as it stands, on a bounded sample of the same batch:
    on every host core (requests split over threads), and on one thread."""
    import oracle
    oracle.build()
    N = w["N"]
    gam = w["gamma"]
    threads = oracle_threads()

    def timed(nthreads):
        t0 = time.perf_counter()
        passes = 0
        while True:
            oracle_parallel(w, (0, N), nthreads, production=True, seed=1, offset=passes, with_diag=False)
            passes += 1
            if time.perf_counter() - t0 >= seconds:
                break
        return passes, time.perf_counter() - t0

    p1, e1 = timed(1)
    one = {"value": p1 * N * gam / e1, "cores": 1,
           "sample": f"{p1} full passes over the N={N} batch (production Philox), {e1:.1f} s, one thread"}
    if threads == 1:
        return dict(one, unit=UNIT, kind="oracle")
    pn, en = timed(threads)
    return {"value": pn * N * gam / en, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{pn} full passes over the N={N} batch (production Philox), {en:.1f} s, requests split "
                      f"over {threads} threads",
            "one_thread": one}


def run_reference(args, world):
    """The oracle timed as the reference arm: each step verifies a bounded slice
    of the same batch on the host cores (requests split over threads), sized
    so the whole run stays within --reference-seconds."""
    import oracle
    import workloads
    oracle.build()
    w = workloads.make(WORKLOAD, seed=3, test_mode=False)
    N, G = w["N"], w["gamma"]
    threads = oracle_threads()
    probe = min(N, 4 * threads)
    t0 = time.perf_counter()
    oracle_parallel(w, (0, probe), threads, production=True, seed=1, offset=0, with_diag=False)
    per_req = max((time.perf_counter() - t0) / probe, 1e-6)
    K, W = args.steps, args.warmup
    budget = args.reference_seconds / max(1, K + W)
    n = int(min(N, max(1, budget / per_req)))
    for k in range(W):
        s0 = (k * n) % N
        oracle_parallel(w, (s0, min(N, s0 + n)), threads, production=True, seed=1, offset=k, with_diag=False)
    done = 0
    t0 = time.perf_counter()
    for k in range(K):
        s0 = ((W + k) * n) % N
        s1 = min(N, s0 + n)
        oracle_parallel(w, (s0, s1), threads, production=True, seed=1, offset=W + k, with_diag=False)
        done += (s1 - s0) * G
    el = time.perf_counter() - t0
    value = done / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": el / K * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD}: N={N} gamma={G} V={w['V']} fp32 probability rows, production "
                                   "Philox", "entry": "probs"},
            "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": threads,
                             "sample": f"{n} requests of the N={N} batch per step, split over {threads} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
