"""GPU parity of gdn_decode_step against the fp64 oracle (through the C ABI).

Tolerances (relative Frobenius error vs the oracle): fp32 inputs 1e-4 on y and
S; bf16 inputs 2e-2 on y and 1e-3 on the fp32 state.  Conv states hold raw
inputs and must match bit for bit.
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


def _pool_case(wl_name, B, stream, pool_factor=4, s0_std=0.1, conv_std=0.1, n_tok=1, act=None, geom=None):
    geom, act, r, p, tok = make_case(wl_name, stream, B * n_tok, act_dtype=act, geom=geom)
    n_slots = pool_factor * B
    S = synth.make_state(geom, n_slots, r, std=s0_std)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=conv_std)
    slots = r.permutation(n_slots)[:B].astype(np.int32)
    return geom, act, p, tok, S, CS, slots


def _oracle_slot(geom, p, tok, S, CS, slot, rows, heads=None, **kw):
    return oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows], tok["b"].f64[rows],
                               s0=S.f64[slot], conv0=CS.f64[slot], heads=heads, **oracle_kwargs(p), **kw)


def _check_decode_step(B, stream, act=None):
    geom, act, p, tok, S, CS, slots = _pool_case("decode4b", B, stream=stream, act=act)
    cfg = config(geom, act)
    sp = dev(S)
    cp = dev(CS)
    y = torch.full((B, geom.value_dim), float("nan"), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_decode_step(cfg, params_dev(p), dev(tok["x"]), dev(tok["z"]), dev(tok["a"]), dev(tok["b"]), cp, sp,
                       torch.from_numpy(slots).cuda(), y)
    torch.cuda.synchronize()
    s_got, c_got, y_got = host(sp), host(cp), host(y)
    ys, yr, ss, sr = [], [], [], []
    for b in range(B):
        ref = _oracle_slot(geom, p, tok, S, CS, slots[b], slice(b, b + 1))
        ys.append(y_got[b]); yr.append(ref["y"][0]); ss.append(s_got[slots[b]]); sr.append(ref["S"])
        np.testing.assert_array_equal(c_got[slots[b]], ref["conv"])
    errs = {"y": rel_fro(ys, yr), "S": rel_fro(ss, sr)}
    tol = tol_for(act)
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    untouched = np.setdiff1d(np.arange(S.shape[0]), slots)
    np.testing.assert_array_equal(s_got[untouched], S.f64[untouched])
    np.testing.assert_array_equal(c_got[untouched], CS.f64[untouched])
    assert gb.gdn_device_status() == 0  # no bounded wait gave up


@pytest.mark.parametrize("B", [1, 4, 16, 64])
def test_decode_step_qwen35_4b(B):
    _check_decode_step(B, stream=B)


def test_decode_step_fp32_activations_at_a_persistent_batch():
    """fp32 activations at B = 24 (768 slot-heads: a batch that bf16 activations run on the
    persistent kernel, whose three stages of fp32 inputs would not fit in shared memory)."""
    _check_decode_step(24, stream=24, act=synth.F32)


@pytest.mark.parametrize("slices", ["1", "2", "4"])
def test_decode_row_slices(slices, monkeypatch):
    """The state rows of a v-head split over 1, 2 or 4 CTAs of a cluster (output
    norm through distributed shared memory) give the same parity."""
    monkeypatch.setenv("GDN_DECODE_SLICES", slices)
    geom, act, p, tok, S, CS, slots = _pool_case("decode4b", 8, stream=77)
    cfg = config(geom, act)
    sp, cp = dev(S), dev(CS)
    y = torch.empty((8, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_decode_step(cfg, params_dev(p), dev(tok["x"]), dev(tok["z"]), dev(tok["a"]), dev(tok["b"]), cp, sp,
                       torch.from_numpy(slots).cuda(), y)
    torch.cuda.synchronize()
    s_got, c_got, y_got = host(sp), host(cp), host(y)
    ys, yr, ss, sr = [], [], [], []
    for b in range(8):
        ref = _oracle_slot(geom, p, tok, S, CS, slots[b], slice(b, b + 1))
        ys.append(y_got[b]); yr.append(ref["y"][0]); ss.append(s_got[slots[b]]); sr.append(ref["S"])
        np.testing.assert_array_equal(c_got[slots[b]], ref["conv"])
    errs = {"y": rel_fro(ys, yr), "S": rel_fro(ss, sr)}
    assert errs["y"] <= 2e-2 and errs["S"] <= 1e-3, fmt(errs)


@pytest.mark.parametrize("wl_name,B", [("decode4b", 64), ("wide", 32)])
def test_decode_persistent_path_with_invalid_slots(wl_name, B):
    """Batches large enough for the persistent pipelined kernel (>= 4 items per
    SM), with a few out-of-range slot indices that must be skipped, on the
    2- and 3-v-heads-per-k-head geometries."""
    geom, act, p, tok, S, CS, slots = _pool_case(wl_name, B, stream=400 + B, pool_factor=2)
    bad = np.array([1, B // 2, B - 1])
    slots = slots.copy()
    slots[bad] = [-3, S.shape[0], 10 ** 6]
    cfg = config(geom, act)
    sp, cp = dev(S), dev(CS)
    y = torch.zeros((B, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_decode_step(cfg, params_dev(p), dev(tok["x"]), dev(tok["z"]), dev(tok["a"]), dev(tok["b"]), cp, sp,
                       torch.from_numpy(slots).cuda(), y)
    torch.cuda.synchronize()
    s_got, c_got, y_got = host(sp), host(cp), host(y)
    good = [b for b in range(B) if b not in set(bad.tolist())]
    ys, yr, ss, sr = [], [], [], []
    for b in good[:12]:
        ref = _oracle_slot(geom, p, tok, S, CS, slots[b], slice(b, b + 1))
        ys.append(y_got[b]); yr.append(ref["y"][0]); ss.append(s_got[slots[b]]); sr.append(ref["S"])
        np.testing.assert_array_equal(c_got[slots[b]], ref["conv"])
    errs = {"y": rel_fro(ys, yr), "S": rel_fro(ss, sr)}
    assert errs["y"] <= 2e-2 and errs["S"] <= 1e-3, fmt(errs)
    assert np.all(y_got[bad] == 0)  # skipped entries leave y untouched
    used = set(slots[good].tolist())
    untouched = np.array([i for i in range(S.shape[0]) if i not in used])
    np.testing.assert_array_equal(s_got[untouched], S.f64[untouched])
    np.testing.assert_array_equal(c_got[untouched], CS.f64[untouched])
    assert gb.gdn_device_status() == 0


def test_decode_16_consecutive_steps():
    """16 decode steps on 4 slots == the oracle over the 16 tokens of each slot."""
    B, T = 4, 16
    geom, act, p, tok, S, CS, slots = _pool_case("decode4b", B, stream=101, n_tok=T)
    cfg = config(geom, act)
    sp, cp = dev(S), dev(CS)
    x, z, a, b = (dev(tok[k]).view(B, T, -1) for k in ("x", "z", "a", "b"))
    y = torch.empty((B, T, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    prm = params_dev(p)
    sl = torch.from_numpy(slots).cuda()
    for t in range(T):
        yt = torch.empty((B, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
        gb.gdn_decode_step(cfg, prm, x[:, t].contiguous(), z[:, t].contiguous(), a[:, t].contiguous(),
                           b[:, t].contiguous(), cp, sp, sl, yt)
        y[:, t] = yt
    torch.cuda.synchronize()
    s_got, c_got, y_got = host(sp), host(cp), host(y)
    ys, yr, ss, sr = [], [], [], []
    for bi in range(B):
        rows = slice(bi * T, (bi + 1) * T)
        ref = _oracle_slot(geom, p, tok, S, CS, slots[bi], rows)
        ys.append(y_got[bi]); yr.append(ref["y"]); ss.append(s_got[slots[bi]]); sr.append(ref["S"])
        np.testing.assert_array_equal(c_got[slots[bi]], ref["conv"])
    errs = {"y": rel_fro(ys, yr), "S": rel_fro(ss, sr)}
    tol = tol_for(act)
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)


@pytest.mark.parametrize("q_scale", [1.0, 32 ** -0.5])
def test_decode_tiny_fp32_token_by_token(q_scale):
    """The tiny fp32 workload run as 64 decode steps equals the oracle (1e-4)."""
    geom, act, r, p, tok = make_case("tiny", 7, 64)
    cfg = config(geom, act, q_scale=q_scale)
    sp = torch.zeros((1, geom.n_v_heads, geom.d_v, geom.d_k), device="cuda")
    cp = torch.zeros((1, geom.d_conv - 1, geom.conv_channels), device="cuda")
    prm = params_dev(p)
    x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
    sl = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = []
    for t in range(64):
        y = torch.empty((1, geom.value_dim), device="cuda")
        gb.gdn_decode_step(cfg, prm, x[t:t + 1], z[t:t + 1], a[t:t + 1], b[t:t + 1], cp, sp, sl, y)
        ys.append(y)
    torch.cuda.synchronize()
    ref = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, q_scale=q_scale,
                              **oracle_kwargs(p))
    errs = {"y": rel_fro(host(torch.cat(ys)), ref["y"]), "S": rel_fro(host(sp)[0], ref["S"])}
    assert errs["y"] <= 1e-4 and errs["S"] <= 1e-4, fmt(errs)
    np.testing.assert_array_equal(host(cp)[0], ref["conv"])


def test_decode_closed_form_beta0_on_gpu():
    """beta = 0 with direct gates: S_T = exp(sum g) S0 exactly in the GPU path too."""
    geom = synth.Geometry(2, 4, 64, 64, 4)
    r = np.random.Generator(np.random.PCG64(5))
    B, T = 3, 5
    cfg = config(geom, synth.F32, flags=gb.GATES_DIRECT | gb.NO_OUTNORM)
    S = synth.make_state(geom, B, r, std=1.0)
    sp = dev(S)
    cp = torch.zeros((B, 3, geom.conv_channels), device="cuda")
    g = -r.uniform(0, 0.3, (T, B, geom.n_v_heads))
    prm = gb.Params(conv_w=dev(synth.store(r.uniform(-.5, .5, (geom.conv_channels, 4)), synth.F32)), A_log=None,
                    norm_w=None)
    sl = torch.arange(B, dtype=torch.int32, device="cuda")
    for t in range(T):
        x = torch.randn((B, geom.conv_channels), device="cuda")
        y = torch.empty((B, geom.value_dim), device="cuda")
        gb.gdn_decode_step(cfg, prm, x, x[:, :geom.value_dim].contiguous(),
                           torch.from_numpy(g[t].astype(np.float32)).cuda(),
                           torch.zeros((B, geom.n_v_heads), device="cuda"), cp, sp, sl, y)
    torch.cuda.synchronize()
    expect = np.exp(g.sum(0))[:, :, None, None] * S.f64
    assert rel_fro(host(sp), expect) <= 1e-6


def test_decode_invalid_slot_is_skipped_and_B0_is_noop():
    geom, act, p, tok, S, CS, slots = _pool_case("decode4b", 2, stream=9)
    cfg = config(geom, act)
    sp, cp = dev(S), dev(CS)
    slots = torch.tensor([-1, S.shape[0]], dtype=torch.int32, device="cuda")
    y = torch.zeros((2, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_decode_step(cfg, params_dev(p), dev(tok["x"]), dev(tok["z"]), dev(tok["a"]), dev(tok["b"]), cp, sp, slots,
                       y)
    gb.gdn_decode_step(cfg, params_dev(p), dev(tok["x"])[:0], dev(tok["z"])[:0], dev(tok["a"])[:0],
                       dev(tok["b"])[:0], cp, sp, slots[:0], y[:0])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(sp), S.f64)
    np.testing.assert_array_equal(host(cp), CS.f64)
    assert torch.count_nonzero(y).item() == 0


def test_conv_state_update_entry_point():
    """gdn_conv_state_update: silu(conv) of every channel and the rolled conv state."""
    geom, act, r, p, tok = make_case("decode4b", 33, 3 * 5)
    cfg = config(geom, act)
    n_seq, n_tok, n_slots = 3, 5, 6
    CS = synth.make_conv_state(geom, n_slots, r, act)
    slots = np.array([4, 0, 2], dtype=np.int32)
    cp = dev(CS)
    u = torch.empty((n_seq * n_tok, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_conv_state_update(cfg, params_dev(p), dev(tok["x"]), cp, torch.from_numpy(slots).cuda(), n_tok, u)
    torch.cuda.synchronize()
    for s in range(n_seq):
        rows = slice(s * n_tok, (s + 1) * n_tok)
        ref_u = oracle.conv_silu(geom, tok["x"].f64[rows], p["conv_w"].f64, conv0=CS.f64[slots[s]])
        # u is rounded to bf16 on output: at most half an ulp, 2^-8 relative, per element
        assert rel_fro(host(u)[rows], ref_u) <= 2.0 ** -8 + 1e-6
        np.testing.assert_array_equal(host(cp)[slots[s]], oracle.conv_final(geom, tok["x"].f64[rows],
                                                                            conv0=CS.f64[slots[s]]))
