"""Build libattn_decode.so in-tree with nvcc for sm_103a.

The translation units (one C-ABI unit plus one kernel unit per head_dim) are
compiled in parallel; ptxas statistics (registers, spills, shared memory) of
every kernel are written next to the objects in ``_build/ptxas_*.txt``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn_decode.so")

SOURCES = ["attn_api.cu", "attn_noalloc.cu"] + [
    "attn_kernels_hd%d_%s.cu" % (hd, t) for hd in (8, 64, 128, 256) for t in ("f16", "bf16")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build")
    return cand


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
           "-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(BUILD, "ptxas_" + src.replace(".cu", ".txt")), "w") as f:
        f.write(res.stderr)
    if res.returncode != 0:
        sys.stderr.write(res.stderr)
        raise RuntimeError("nvcc failed on %s" % src)
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(ROOT, "include", "attn_decode.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False) -> str:
    """Compile (if sources changed) and return the path of libattn_decode.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def spill_report() -> dict:
    """Per-kernel 'bytes stack frame / spill stores / spill loads' from the last build."""
    out = {}
    for src in SOURCES:
        path = os.path.join(BUILD, "ptxas_" + src.replace(".cu", ".txt"))
        if not os.path.exists(path):
            continue
        fn = None
        for line in open(path):
            if "Compiling entry function" in line:
                fn = line.split("'")[1]
            elif "spill stores" in line and fn:
                parts = line.replace(",", "").split()
                out[fn] = {"stack": int(parts[0]), "spill_stores": int(parts[4]),
                           "spill_loads": int(parts[8])}
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
