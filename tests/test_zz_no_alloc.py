"""gdn_chunk_prefill_noalloc: the chunked prefill for callers that cannot allocate
device memory when they run it -- a runtime that owns the whole device memory budget
through its own allocator, code running while its stream is captured into a CUDA
graph (where cudaMalloc/cudaFree are not allowed), or a latency-critical path that
cannot pay for cudaFree's device-wide synchronisation.  Its workspace is a static
64 MiB device array inside libgdn instead of a caller-provided buffer.

The entry point is called through the C ABI and must give bit for bit what
gdn_chunk_prefill gives with a caller-owned workspace (the prefill kernels reduce
in a fixed order), for two calls in a row with different inputs and lengths, so
that a second call that read anything stale from the shared array would show; the
outputs are also held to the fp64 oracle.  The largest T whose workspace fits the
array is accepted and one more token is refused.  This file is collected last on
purpose; it passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, host, make_case, oracle_kwargs, params_dev, rel_fro, tol_for

pytestmark = pytest.mark.gpu

SCRATCH = 64 << 20


def _inputs(stream, T):
    geom, act, r, p, tok = make_case("prefill4b", stream, T)
    S0 = synth.make_state(geom, 1, r, std=0.1)
    C0 = synth.make_conv_state(geom, 1, r, act, std=0.1)
    return geom, act, p, tok, S0, C0


def _outputs(cfg, T):
    s = torch.empty((cfg.n_v_heads, cfg.d_v, cfg.d_k), device="cuda")
    c = torch.empty((cfg.d_conv - 1, cfg.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    y = torch.empty((T, cfg.n_v_heads * cfg.d_v), dtype=cfg.torch_dtype, device="cuda")
    return s, c, y


def _call_noalloc_c_abi(cfg, prm, x, z, a, b, s0, c0, s, c, y):
    lib = gb.load()
    cc, pp = cfg.c(), prm.c()
    return lib.gdn_chunk_prefill_noalloc(ctypes.byref(cc), ctypes.byref(pp), x.data_ptr(), z.data_ptr(),
                                         a.data_ptr(), b.data_ptr(), x.shape[0], s0.data_ptr(), c0.data_ptr(),
                                         s.data_ptr(), c.data_ptr(), y.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)


def _largest_fitting_T(cfg):
    lib = gb.load()
    cc = cfg.c()
    lo, hi = 1, 1 << 20
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if lib.gdn_workspace_size(ctypes.byref(cc), gb.OP_CHUNK_PREFILL, mid, 1) <= SCRATCH:
            lo = mid
        else:
            hi = mid - 1
    return lo


def _run_both(stream, T):
    """(noalloc outputs, workspace-prefill outputs, inputs) for one seeded case."""
    geom, act, p, tok, S0, C0 = _inputs(stream, T)
    cfg = config(geom, act)
    prm = params_dev(p)
    x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
    s0, c0 = dev(S0)[0], dev(C0)[0]
    s_ref, c_ref, y_ref = _outputs(cfg, T)
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, T), dtype=torch.uint8, device="cuda")
    gb.gdn_chunk_prefill(cfg, prm, x, z, a, b, s0, c0, s_ref, c_ref, y_ref, ws)
    s_na, c_na, y_na = _outputs(cfg, T)
    st = _call_noalloc_c_abi(cfg, prm, x, z, a, b, s0, c0, s_na, c_na, y_na)
    assert st == 0, gb.load().gdn_last_error().decode()
    torch.cuda.synchronize()
    return (s_na, c_na, y_na), (s_ref, c_ref, y_ref), (geom, act, p, tok, S0, C0)


def test_noalloc_prefill_equals_workspace_prefill_two_calls():
    for stream, T in ((501, 440), (502, 300)):
        (s_na, c_na, y_na), (s_ref, c_ref, y_ref), (geom, act, p, tok, S0, C0) = _run_both(stream, T)
        assert torch.equal(y_na, y_ref) and torch.equal(s_na, s_ref) and torch.equal(c_na, c_ref)
        ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, s0=S0.f64[0],
                                  conv0=C0.f64[0], **oracle_kwargs(p))
        tol = tol_for(act)
        errs = {"y": rel_fro(host(y_na), ref["y"]), "S": rel_fro(host(s_na), ref["S"])}
        assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], (T, fmt(errs))
        np.testing.assert_array_equal(host(c_na), ref["conv"])
    assert gb.gdn_device_status() == 0


def test_noalloc_accepts_the_largest_fitting_T_and_refuses_one_more():
    geom, act, p, tok, S0, C0 = _inputs(503, 1)
    cfg = config(geom, act)
    T = _largest_fitting_T(cfg)
    assert T > 1000  # the Qwen3.5-4B geometry: 1727 tokens fit 64 MiB
    (s_na, c_na, y_na), (s_ref, c_ref, y_ref), _ = _run_both(504, T)
    assert torch.equal(y_na, y_ref) and torch.equal(s_na, s_ref) and torch.equal(c_na, c_ref)
    T1 = T + 1
    x = torch.zeros((T1, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    s, c, y = _outputs(cfg, T1)
    st = _call_noalloc_c_abi(cfg, params_dev(p), x, x, x, x, s, c, s, c, y)
    assert st == -6
    msg = gb.load().gdn_last_error().decode()
    need = gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, T1)
    assert "static scratch" in msg and str(SCRATCH) in msg and str(need) in msg
