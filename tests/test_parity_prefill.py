"""GPU parity of gdn_chunk_prefill against the token-by-token fp64 oracle.

The chunkwise prefill is an exact reformulation of the token recurrence, so its
outputs and final state are compared with the oracle's token loop ("Strata"
chapter 6, section 6.9: prefill is the decode path one token at a time).
Sizes span several chunks and a ragged tail; the full 8192-token Qwen3.5-4B
prefill is checked on a sample of v-heads (the oracle computes heads
independently), in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import (config, dev, fmt, head_cols, host, make_case, oracle_kwargs, params_dev, rel_fro,
                       sample_heads, tol_for)

pytestmark = pytest.mark.gpu


def run_prefill(cfg, p, tok, s0=None, conv0=None, T=None):
    geom_T = tok["x"].shape[0] if T is None else T
    H = cfg.n_v_heads
    x, z, a, b = (dev(tok[k])[:geom_T] for k in ("x", "z", "a", "b"))
    s_fin = torch.empty((H, cfg.d_v, cfg.d_k), device="cuda")
    c_fin = torch.empty((cfg.d_conv - 1, cfg.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    y = torch.full((geom_T, H * cfg.d_v), float("nan"), dtype=cfg.torch_dtype, device="cuda")
    ws = torch.empty(max(1, gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, geom_T)), dtype=torch.uint8,
                     device="cuda")
    gb.gdn_chunk_prefill(cfg, params_dev(p), x, z, a, b, s0, conv0, s_fin, c_fin, y, ws)
    torch.cuda.synchronize()
    return host(y), host(s_fin), host(c_fin)


@pytest.mark.parametrize("chunk,T", [(16, 64), (16, 45), (32, 64), (64, 64), (64, 100), (16, 1)])
def test_prefill_tiny_fp32(chunk, T):
    geom, act, r, p, tok = make_case("tiny", 10 + T, T)
    cfg = config(geom, act, chunk=chunk)
    y, s, c = run_prefill(cfg, p, tok)
    ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, **oracle_kwargs(p))
    errs = {"y": rel_fro(y, ref["y"]), "S": rel_fro(s, ref["S"])}
    assert errs["y"] <= 1e-4 and errs["S"] <= 1e-4, fmt(errs)
    np.testing.assert_array_equal(c, ref["conv"])


@pytest.mark.parametrize("T", [1000, 130])
def test_prefill_qwen35_4b_all_heads(T):
    """16/32 heads, d = 128, bf16, chunk 64: several chunks and a ragged tail."""
    geom, act, r, p, tok = make_case("prefill4b", 20 + T, T)
    cfg = config(geom, act)
    y, s, c = run_prefill(cfg, p, tok)
    ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, **oracle_kwargs(p))
    errs = {"y": rel_fro(y, ref["y"]), "S": rel_fro(s, ref["S"])}
    tol = tol_for(act)
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    np.testing.assert_array_equal(c, ref["conv"])


def test_prefill_long_memory_gates():
    """Gates that keep a long memory.  The workloads' A_log ~ U(0, ln 16) gives a mean
    alpha of about 0.2 to 0.5, so the state forgets within a few tokens and rounding in
    the state products cannot build up.  Here A_log runs from -6 to 0 over the v-heads
    (mean alpha from about 0.998 down to 0.5, i.e. memories of up to ~500 tokens), over
    2000 tokens, on the tcgen05 path."""
    T = 2000
    geom, act, r, p, tok = make_case("prefill4b", 60, T)
    p = dict(p, A_log=synth.store(np.linspace(-6.0, 0.0, geom.n_v_heads), synth.F32))
    cfg = config(geom, act)
    y, s, c = run_prefill(cfg, p, tok)
    ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, **oracle_kwargs(p))
    errs = {"y": rel_fro(y, ref["y"]), "S": rel_fro(s, ref["S"])}
    tol = tol_for(act)
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    # the longest memories on their own, where any build-up would show first
    long = list(range(4))
    errs_long = {"S": rel_fro(s[long], ref["S"][long])}
    assert errs_long["S"] <= tol["S"], fmt(errs_long)
    np.testing.assert_array_equal(c, ref["conv"])


def test_prefill_qwen35_4b_full_size_sampled_heads():
    """T = 8192 (the benchmarked prefill), final state and outputs of 6 v-heads."""
    T = 8192
    geom, act, r, p, tok = make_case("prefill4b", 0, T)
    cfg = config(geom, act)
    y, s, c = run_prefill(cfg, p, tok)
    heads = sample_heads(geom.n_v_heads, 6, seed=1)
    ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, heads=heads,
                              **oracle_kwargs(p))
    cols = head_cols(heads, geom.d_v)
    errs = {"y": rel_fro(y[:, cols], ref["y"][:, cols]), "S": rel_fro(s[heads], ref["S"][heads])}
    tol = tol_for(act)
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    np.testing.assert_array_equal(c, ref["conv"])
    assert np.all(np.isfinite(y))


def test_prefill_with_initial_state_and_split_invariance():
    """prefill(T1) then prefill(T - T1) from the carried states == prefill(T) == oracle."""
    T, T1 = 300, 77
    geom, act, r, p, tok = make_case("prefill4b", 55, T)
    cfg = config(geom, act)
    S0 = synth.make_state(geom, 1, r, std=0.1)
    C0 = synth.make_conv_state(geom, 1, r, act, std=0.1)
    y_full, s_full, c_full = run_prefill(cfg, p, tok, s0=dev(S0)[0], conv0=dev(C0)[0])
    ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, s0=S0.f64[0],
                              conv0=C0.f64[0], **oracle_kwargs(p))
    tol = tol_for(act)
    errs = {"y": rel_fro(y_full, ref["y"]), "S": rel_fro(s_full, ref["S"])}
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    np.testing.assert_array_equal(c_full, ref["conv"])
    # split: first T1 tokens, then the rest with the carried (device) states, in place
    x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
    s_buf = dev(S0)[0].clone()
    c_buf = dev(C0)[0].clone()
    ys = []
    for lo, hi in ((0, T1), (T1, T)):
        y = torch.empty((hi - lo, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
        ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, hi - lo), dtype=torch.uint8, device="cuda")
        gb.gdn_chunk_prefill(cfg, params_dev(p), x[lo:hi], z[lo:hi], a[lo:hi], b[lo:hi], s_buf, c_buf, s_buf, c_buf,
                             y, ws)
        ys.append(y)
    torch.cuda.synchronize()
    errs = {"y": rel_fro(host(torch.cat(ys)), ref["y"]), "S": rel_fro(host(s_buf), ref["S"])}
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    np.testing.assert_array_equal(host(c_buf), ref["conv"])


def test_prefill_equals_decode_steps():
    """T decode steps and one prefill of the same T tokens agree (both vs oracle)."""
    T = 40
    geom, act, r, p, tok = make_case("prefill4b", 66, T)
    cfg = config(geom, act)
    y_pf, s_pf, c_pf = run_prefill(cfg, p, tok)
    sp = torch.zeros((1, geom.n_v_heads, geom.d_v, geom.d_k), device="cuda")
    cp = torch.zeros((1, geom.d_conv - 1, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
    sl = torch.zeros(1, dtype=torch.int32, device="cuda")
    prm = params_dev(p)
    ys = []
    for t in range(T):
        y = torch.empty((1, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
        gb.gdn_decode_step(cfg, prm, x[t:t + 1], z[t:t + 1], a[t:t + 1], b[t:t + 1], cp, sp, sl, y)
        ys.append(y)
    torch.cuda.synchronize()
    y_dec, s_dec = host(torch.cat(ys)), host(sp)[0]
    tol = tol_for(act)
    assert rel_fro(y_pf, y_dec) <= tol["y"] and rel_fro(s_pf, s_dec) <= tol["S"]
    np.testing.assert_array_equal(c_pf, host(cp)[0])


def test_prefill_closed_forms_on_gpu():
    """Direct mode (raw q/k/v, direct gates, no norms) against the oracle with
    orthonormal keys, alpha = 1, beta = 1: retrieval S_T k_i = v_i holds on the GPU."""
    geom = synth.Geometry(1, 1, 64, 64, 4)
    T = 48
    rng = np.random.Generator(np.random.PCG64(8))
    k = synth.orthonormal_rows(rng, T, 64)
    q = rng.standard_normal((T, 64))
    v = rng.standard_normal((T, 64))
    x = synth.store(np.concatenate([q, k, v], axis=1), synth.F32)
    flags = gb.RAW_QKV | gb.NO_L2NORM | gb.GATES_DIRECT | gb.NO_OUTNORM
    cfg = config(geom, synth.F32, chunk=16, flags=flags)
    tok = {"x": x, "z": synth.store(np.zeros((T, 64)), synth.F32), "a": synth.store(np.zeros((T, 1)), synth.F32),
           "b": synth.store(np.ones((T, 1)), synth.F32)}
    p = {"conv_w": synth.store(np.zeros((192, 4)), synth.F32), "A_log": synth.store(np.zeros(1), synth.F32),
         "norm_w": synth.store(np.ones(64), synth.F32)}
    y, s, c = run_prefill(cfg, p, tok)
    for i in range(T):
        np.testing.assert_allclose(s[0] @ k[i], v[i], atol=2e-4)
    ref = oracle.run_sequence(geom, x.f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, flags=flags,
                              **oracle_kwargs(p))
    assert rel_fro(y, ref["y"]) <= 1e-4 and rel_fro(s, ref["S"]) <= 1e-4


def test_prefill_empty_sequence_keeps_state():
    geom, act, r, p, tok = make_case("prefill4b", 77, 1)
    cfg = config(geom, act)
    S0 = synth.make_state(geom, 1, r, std=0.1)
    C0 = synth.make_conv_state(geom, 1, r, act, std=0.1)
    x = dev(tok["x"])[:0]
    s_fin = torch.empty((geom.n_v_heads, 128, 128), device="cuda")
    c_fin = torch.empty((3, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_chunk_prefill(cfg, params_dev(p), x, x, x, x, dev(S0)[0], dev(C0)[0], s_fin, c_fin, x, None)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(s_fin), S0.f64[0])
    np.testing.assert_array_equal(host(c_fin), C0.f64[0])


@pytest.mark.parametrize("T", [45 * 64, 4096 + 37])  # 45 and 65 chunks: 3 segments each
def test_segmented_single_sequence_is_bitwise_one_chain(T):
    """A long single sequence runs as segments (the prep of the next segment beside the
    chain of this one, the state handed over in s_final); a one-sequence varlen call of
    the same tokens runs one chain.  Both must agree bit for bit, with and without an
    initial state."""
    geom, act, r, p, tok = make_case("prefill4b", 300 + T, T)
    cfg = config(geom, act)
    H = cfg.n_v_heads
    prm = params_dev(p)
    x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
    S0 = synth.make_state(geom, 1, r, std=0.1)
    C0 = synth.make_conv_state(geom, 1, r, act, std=0.1)
    for init in (False, True):
        s_fin = torch.empty((H, cfg.d_v, cfg.d_k), device="cuda")
        c_fin = torch.empty((cfg.d_conv - 1, cfg.conv_channels), dtype=cfg.torch_dtype, device="cuda")
        y1 = torch.empty((T, H * cfg.d_v), dtype=cfg.torch_dtype, device="cuda")
        ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_CHUNK_PREFILL, T), dtype=torch.uint8, device="cuda")
        s0 = dev(S0)[0].contiguous() if init else None
        c0 = dev(C0)[0].contiguous() if init else None
        gb.gdn_chunk_prefill(cfg, prm, x, z, a, b, s0, c0, s_fin, c_fin, y1, ws)
        sp, cp = dev(S0), dev(C0)
        y2 = torch.empty_like(y1)
        ws2 = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, T, 1), dtype=torch.uint8, device="cuda")
        cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
        sl = torch.zeros(1, dtype=torch.int32, device="cuda")
        hi = torch.tensor([1 if init else 0], dtype=torch.uint8, device="cuda")
        gb.gdn_varlen_prefill(cfg, prm, x, z, a, b, cu, sl, hi, cp, sp, y2, ws2)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), f"y differs (init={init})"
        assert torch.equal(s_fin, sp[0]), f"S differs (init={init})"
        assert torch.equal(c_fin, cp[0]), f"conv differs (init={init})"
    assert gb.gdn_device_status() == 0
