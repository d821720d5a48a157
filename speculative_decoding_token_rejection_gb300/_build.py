"""Compile the native verifier library (libspec_verify.so) in-tree for sm_103a.

Each CUDA translation unit is compiled in parallel with nvcc, then linked into
one shared object next to this file.  The CUDA runtime is linked statically,
so the library loads on a machine without a GPU (for symbol checks) and needs
nothing beyond the NVIDIA driver on a GPU machine.
"""
from __future__ import annotations

import os
import pathlib
import shutil
import subprocess
import tempfile

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB_NAME = "libspec_verify.so"
LIB_PATH = PKG / LIB_NAME
SOURCES = ["sv_api.cu", "sv_probs.cu", "sv_logits.cu", "sv_logits_bf16.cu", "sv_logits_f32.cu", "sv_logits_bf16_proc.cu",
           "sv_logits_f32_proc.cu", "sv_sample_bf16.cu", "sv_sample_f32.cu", "sv_sample_bf16_proc.cu",
           "sv_sample_f32_proc.cu", "sv_stream_bf16.cu", "sv_stream_f32.cu",
           "sv_stream_bf16_proc.cu", "sv_stream_f32_proc.cu", "sv_ngram.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I", str(INCLUDE), "-I", str(CSRC)]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (needed to build the verifier library)")
    return cand


def _inputs():
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + \
        list(INCLUDE.glob("*.h")) + [pathlib.Path(__file__)]


def up_to_date() -> bool:
    if not LIB_PATH.exists():
        return False
    t = LIB_PATH.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> pathlib.Path:
    """Build (or reuse) libspec_verify.so and return its path."""
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    objdir = PKG / "_build"
    objdir.mkdir(exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    procs = []
    objs = []
    for src in SOURCES:
        obj = objdir / (pathlib.Path(src).stem + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_info or p.returncode != 0):
            print(out, end="", flush=True)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=PKG)
    os.close(fd)
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *map(str, objs)]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
