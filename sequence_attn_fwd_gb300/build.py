"""Builds libseqattn.so in-tree with nvcc for sm_103a (GB300).

    python sequence_attn_fwd_gb300/build.py [--force]

(run as a script: importing the package loads the library, so the build
cannot go through the package import).

Each translation unit is compiled in parallel, then linked into
``sequence_attn_fwd_gb300/lib/libseqattn.so`` (the CUDA runtime is linked
statically; the driver's tensor-map encoder is looked up at run time, so the
library needs no libcuda at link time). ptxas resource usage of every kernel
is written to ``lib/ptxas.log``.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libseqattn.so")
SOURCES = ["attn_kernel.cu", "lse_merge.cu", "api.cu"]
HEADERS = ["ptx.cuh", "kernels.h", "attn_common.cuh", "attn_bwd.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "seqattn.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                    "-Xcompiler", "-fPIC", "-Xptxas", "-v", "-I", os.path.join(ROOT, "include")]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(LIBDIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc()] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    log = []
    failed = []
    for src, cmd, p in procs:
        out, _ = p.communicate()
        log.append(f"==== {src}\n{out}")
        if p.returncode != 0:
            failed.append((src, cmd, out))
    with open(os.path.join(LIBDIR, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    if failed:
        msg = "\n".join(f"nvcc failed on {s}:\n{' '.join(c)}\n{o}" for s, c, o in failed)
        raise RuntimeError(msg)
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, LIB)
    if verbose:
        print("\n".join(log))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
