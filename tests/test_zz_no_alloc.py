"""gdn_chunk_prefill_noalloc: the chunked prefill for callers that cannot
allocate device memory (a runtime that owns the device memory budget, code
running under stream capture, paths that cannot afford cudaFree's device-wide
synchronisation).  Its workspace is a static 64 MiB device array inside
libgdn instead of a caller-provided buffer.

The entry point is called through the C ABI and compared with
gdn_chunk_prefill (caller-owned workspace) on the same inputs, for two calls
in a row with different inputs and lengths, so that a second call that read
anything stale from the shared array would show.  This file is collected last
on purpose; it passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_gb300 import binding as gb
from gdn_cases import config, dev, fmt, host, make_case, params_dev, rel_fro, tol_for

pytestmark = pytest.mark.gpu


def _inputs(stream, T):
    geom, act, r, p, tok = make_case("prefill4b", stream, T)
    from hybrid_gated_deltanet_gb300 import synth
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
    st = lib.gdn_chunk_prefill_noalloc(ctypes.byref(cc), ctypes.byref(pp), x.data_ptr(), z.data_ptr(), a.data_ptr(),
                                       b.data_ptr(), x.shape[0], s0.data_ptr(), c0.data_ptr(), s.data_ptr(),
                                       c.data_ptr(), y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.gdn_last_error().decode()


def test_noalloc_prefill_matches_workspace_prefill_two_calls():
    for stream, T in ((501, 440), (502, 300)):
        geom, act, p, tok, S0, C0 = _inputs(stream, T)
        cfg = config(geom, act)
        prm = params_dev(p)
        x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
        s0, c0 = dev(S0)[0], dev(C0)[0]
        # existing entry point, caller-owned workspace
        s_ref, c_ref, y_ref = _outputs(cfg, T)
        ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, T), dtype=torch.uint8, device="cuda")
        gb.gdn_chunk_prefill(cfg, prm, x, z, a, b, s0, c0, s_ref, c_ref, y_ref, ws)
        # the entry point without a workspace argument
        s_na, c_na, y_na = _outputs(cfg, T)
        _call_noalloc_c_abi(cfg, prm, x, z, a, b, s0, c0, s_na, c_na, y_na)
        torch.cuda.synchronize()
        tol = tol_for(act)
        errs = {"y": rel_fro(host(y_na), host(y_ref)), "S": rel_fro(host(s_na), host(s_ref))}
        assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], (T, fmt(errs))
        np.testing.assert_array_equal(host(c_na), host(c_ref))


def test_noalloc_rejects_a_workspace_beyond_the_static_scratch():
    geom, act, p, tok, S0, C0 = _inputs(503, 1)
    cfg = config(geom, act)
    T = 4096  # 4096 x 33,024 B of workspace > 64 MiB
    x = torch.empty((T, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    s, c, y = _outputs(cfg, T)
    lib = gb.load()
    cc, pp = cfg.c(), params_dev(p).c()
    st = lib.gdn_chunk_prefill_noalloc(ctypes.byref(cc), ctypes.byref(pp), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                       x.data_ptr(), T, None, None, s.data_ptr(), c.data_ptr(), y.data_ptr(), None)
    assert st == -6
    msg = lib.gdn_last_error().decode()
    assert "static scratch" in msg and str(64 << 20) in msg
