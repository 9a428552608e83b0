"""Build libgdn.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit compiles in parallel into ``_build/`` at the repo
root; the objects link into ``hybrid_gated_deltanet_gb300/libgdn.so`` with the
CUDA runtime linked statically.  Usage: ``python -m hybrid_gated_deltanet_gb300.build``.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgdn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["gdn_api.cu", "gdn_decode.cu", "gdn_prefill.cu", "gdn_chunk16.cu", "gdn_noalloc.cu", "gdn_proj.cu",
           "gdn_attn.cu"]
HEADERS = ["gdn_common.cuh", "gdn_internal.h", "gdn_prefill_common.cuh", "gdn_tc.cuh", "gdn_tma.cuh"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                   "-I", os.path.join(ROOT, "include")] + list(extra)


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "gdn.h"),
                                                                   os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths)


# ELF e_machine of the host, so that a library built on another architecture is never taken as current.
_ELF_MACHINE = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}


def _built_here(path: str) -> bool:
    want = _ELF_MACHINE.get(platform.machine().lower())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    return want is None or int.from_bytes(head[18:20], "little") == want


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libgdn.so; skipped when the library exists, was built for this
    host's architecture and is newer than every source, header and this script."""
    if not force and os.path.exists(LIB) and _built_here(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + _flags(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results] + ["-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
