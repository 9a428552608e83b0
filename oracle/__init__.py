"""CPU fp64 oracle for the Gated DeltaNet layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path (the CUDA library and its
binding) never imports, links or calls anything here, and nothing here imports
the product path: the two share only the seeded input arrays.

Contents
--------
* ``gdn_oracle.c`` -- the oracle proper: plain token-by-token fp64 evaluation
  (conv + SiLU, L2 norm, gates, gated delta rule, gated RMSNorm).  This module
  builds it with gcc and calls it through ctypes, one (sequence, v-head) unit per
  call, spread over host threads (ctypes releases the GIL during the call).
* ``twin.py`` -- an independent pure-numpy token loop for small cases; it
  cross-checks the C code.
* ``chunk_form.py`` -- the chunkwise (WY / UT-transform) evaluation in fp64,
  the secondary CPU reference that pins the chunk algebra before any kernel.

Parity pins for all three live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")

RAW_QKV = 1
NO_L2NORM = 2
GATES_DIRECT = 4
NO_OUTNORM = 8


class OracleGeom(ctypes.Structure):
    _fields_ = [
        ("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
        ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32), ("d_conv", ctypes.c_int32),
        ("mutant", ctypes.c_int32),
        ("q_scale", ctypes.c_double), ("l2_eps", ctypes.c_double), ("norm_eps", ctypes.c_double),
        ("flags", ctypes.c_uint32),
    ]


def _native(path: str) -> bool:
    """True if the shared object at `path` is an ELF file for this host's machine type."""
    machine = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine().lower())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    return machine is None or int.from_bytes(head[18:20], "little") == machine


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math), unless a library for this
    host's architecture, newer than the source, is already there."""
    if (force or not os.path.exists(_LIB) or not _native(_LIB)
            or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_lib_lock = threading.Lock()


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            lib.gdn_oracle_head.restype = ctypes.c_int
            lib.gdn_oracle_head.argtypes = [ctypes.POINTER(OracleGeom), ctypes.c_int32, ctypes.c_int64,
                                            d, d, d, d, d, d, d, d, d, d, d, d]
            lib.gdn_oracle_conv_silu.restype = None
            lib.gdn_oracle_conv_silu.argtypes = [ctypes.POINTER(OracleGeom), ctypes.c_int64, d, d, d, d,
                                                 ctypes.c_int64, ctypes.c_int64, d]
            lib.gdn_oracle_conv_final.restype = None
            lib.gdn_oracle_conv_final.argtypes = [ctypes.POINTER(OracleGeom), ctypes.c_int64, d, d, d]
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def make_geom(geom, q_scale: float = 1.0, l2_eps: float = 1e-6, norm_eps: float = 1e-6,
              flags: int = 0, mutant: int = 0) -> OracleGeom:
    return OracleGeom(geom.n_k_heads, geom.n_v_heads, geom.d_k, geom.d_v, geom.d_conv, mutant,
                      q_scale, l2_eps, norm_eps, flags)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def run_sequence(geom, x, z, a, b, conv_w, A_log, norm_w, *, s0=None, conv0=None, conv_b=None,
                 dt_bias=None, heads: Optional[Sequence[int]] = None, q_scale: float = 1.0,
                 l2_eps: float = 1e-6, norm_eps: float = 1e-6, flags: int = 0, mutant: int = 0,
                 threads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Evaluate one sequence token by token in fp64.

    x [T, C_ch], z [T, H_v*d_v], a, b [T, H_v]; s0 [H_v, d_v, d_k] or None (zeros);
    conv0 [d_conv-1, C_ch] or None (zeros).  ``heads`` restricts the work to some
    v-heads (outputs of the others are NaN, their states are s0).
    Returns y [T, H_v*d_v], S [H_v, d_v, d_k] and conv [d_conv-1, C_ch].
    """
    lib = _load()
    g = make_geom(geom, q_scale, l2_eps, norm_eps, flags, mutant)
    x, z, a, b = _f64(x), _f64(z), _f64(a), _f64(b)
    conv_w, A_log, norm_w = _f64(conv_w), _f64(A_log), _f64(norm_w)
    conv0, conv_b, dt_bias = _f64(conv0), _f64(conv_b), _f64(dt_bias)
    T = x.shape[0]
    Hv, dv, dk = geom.n_v_heads, geom.d_v, geom.d_k
    S = np.zeros((Hv, dv, dk)) if s0 is None else np.array(s0, dtype=np.float64, copy=True)
    y = np.full((T, Hv * dv), np.nan)
    heads = list(range(Hv)) if heads is None else list(heads)
    outs = {}

    def one(j):
        Sj = np.ascontiguousarray(S[j])
        yj = np.empty((T, dv))
        rc = lib.gdn_oracle_head(ctypes.byref(g), j, T, _ptr(x), _ptr(conv0), _ptr(conv_w), _ptr(conv_b),
                                 _ptr(z), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w),
                                 _ptr(Sj), _ptr(yj))
        if rc != 0:
            raise RuntimeError(f"oracle head {j} failed ({rc})")
        outs[j] = (Sj, yj)

    nthr = min(len(heads), threads or default_threads())
    if nthr <= 1:
        for j in heads:
            one(j)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(one, heads))
    for j in heads:
        S[j], y[:, j * dv:(j + 1) * dv] = outs[j]
    conv = np.empty((geom.d_conv - 1, geom.conv_channels))
    lib.gdn_oracle_conv_final(ctypes.byref(g), T, _ptr(x), _ptr(conv0), _ptr(conv))
    return {"y": y, "S": S, "conv": conv}


def conv_silu(geom, x, conv_w, conv0=None, conv_b=None, mutant: int = 0) -> np.ndarray:
    """silu(causal depthwise conv) over all channels: [T, C_ch]."""
    lib = _load()
    g = make_geom(geom, mutant=mutant)
    x, conv_w, conv0, conv_b = _f64(x), _f64(conv_w), _f64(conv0), _f64(conv_b)
    T, C = x.shape
    u = np.empty((T, C))
    lib.gdn_oracle_conv_silu(ctypes.byref(g), T, _ptr(x), _ptr(conv0), _ptr(conv_w), _ptr(conv_b), 0, C,
                             _ptr(u))
    return u


def conv_final(geom, x, conv0=None, mutant: int = 0) -> np.ndarray:
    lib = _load()
    g = make_geom(geom, mutant=mutant)
    x, conv0 = _f64(x), _f64(conv0)
    out = np.empty((geom.d_conv - 1, geom.conv_channels))
    lib.gdn_oracle_conv_final(ctypes.byref(g), x.shape[0], _ptr(x), _ptr(conv0), _ptr(out))
    return out
