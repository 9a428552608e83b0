"""GPU parity of the projections (gdn_proj_gemm) and of the whole layer with
them (gdn_layer_decode, gdn_layer_varlen_prefill) against the fp64 oracle.

Tolerances: a projection output is one bf16 rounding (relative error at most
2^-8) of an fp32 sum whose error is at most k 2^-24 sum_k |act w| (a loose
bound of the accumulation); each element is held to the sum of the two.  The
layer's outputs are held to the bf16 tolerances of the layer (2e-2 on out and
y, 1e-3 on the fp32 state); its conv state stores the in-projection's bf16
values, which may differ from the oracle's rounding by one bf16 step where the
fp32 sum lies next to a rounding boundary."""
import numpy as np
import pytest
import torch

from oracle import projections as pj
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, host, params_dev, rel_fro, tol_for

pytestmark = pytest.mark.gpu


def _ws(n_tok, n_out, k):
    n = gb.gdn_proj_workspace_size(n_tok, n_out, k)
    return torch.empty(n, dtype=torch.uint8, device="cuda") if n else None


def _check_gemm(act64, w64, got, rows=None):
    ref = pj.project(act64 if rows is None else act64[rows], w64)
    mag = pj.project(np.abs(act64 if rows is None else act64[rows]), np.abs(w64))
    k = act64.shape[1]
    bound = 2.0 ** -8 * np.abs(ref) + k * 2.0 ** -24 * mag * 1.01 + 1e-30
    g = got if rows is None else got[rows]
    bad = np.abs(g - ref) > bound
    assert not bad.any(), f"{bad.sum()} elements outside the bound, worst {np.max(np.abs(g - ref) - bound)}"
    assert rel_fro(g, ref) <= 4e-3


@pytest.mark.parametrize("n_tok,n_out,k", [
    (1, 1, 8), (1, 200, 64), (4, 2560, 4096), (37, 300, 136), (64, 12352, 2560), (65, 129, 72),
    (100, 256, 1024), (257, 640, 520), (1000, 384, 512), (3000, 2560, 256)])
def test_proj_gemm_shapes(n_tok, n_out, k):
    r = synth.rng_for(50, n_tok * 7 + n_out + k)
    act = synth.store(r.standard_normal((n_tok, k)), synth.BF16)
    w = synth.store(r.standard_normal((n_out, k)) / np.sqrt(k), synth.BF16)
    out = torch.full((n_tok, n_out + 3), 7.0, dtype=torch.bfloat16, device="cuda")
    gb.gdn_proj_gemm(dev(act), dev(w), out, _ws(n_tok, n_out, k))
    torch.cuda.synchronize()
    got = host(out)
    _check_gemm(act.f64[:], w.f64[:], got[:, :n_out])
    assert np.all(got[:, n_out:] == 7.0)  # columns past n_out untouched


@pytest.mark.parametrize("n_tok,n_out,k,ctas", [(64, 12352, 2560, 600), (33, 1000, 1024, 4000),
                                                  (300, 640, 2048, 400)])
def test_proj_gemm_forced_split(monkeypatch, n_tok, n_out, k, ctas):
    """K split over many CTAs per tile (the split factor forced through its tuning
    override): the partial sums and their reduction give the same bound."""
    monkeypatch.setenv("GDN_PROJ_SPLIT_CTAS", str(ctas))
    assert gb.gdn_proj_workspace_size(n_tok, n_out, k) > 0
    r = synth.rng_for(53, n_tok + n_out)
    act = synth.store(r.standard_normal((n_tok, k)), synth.BF16)
    w = synth.store(r.standard_normal((n_out, k)) / np.sqrt(k), synth.BF16)
    out = torch.empty((n_tok, n_out), dtype=torch.bfloat16, device="cuda")
    gb.gdn_proj_gemm(dev(act), dev(w), out, _ws(n_tok, n_out, k))
    torch.cuda.synchronize()
    _check_gemm(act.f64[:], w.f64[:], host(out))


def test_proj_gemm_empty_and_errors():
    w = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    act = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((0, 16), dtype=torch.bfloat16, device="cuda")
    gb.gdn_proj_gemm(act, w, out)
    with pytest.raises(gb.GdnError, match="workspace: found NULL"):
        gb.gdn_proj_gemm(torch.zeros((4, 4096), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((2560, 4096), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((4, 2560), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(gb.GdnError, match="k: found 60"):
        gb.gdn_proj_gemm(torch.zeros((2, 60), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((16, 60), dtype=torch.bfloat16, device="cuda"),
                         torch.zeros((2, 16), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("which", ["in", "out"])
def test_proj_full_size_sampled(which):
    """The prefill projections of a T = 8192 sequence at hidden 2560 (the launch
    shape the layer uses), 96 sampled token rows checked in full."""
    geom = synth.QWEN35_4B
    r = synth.rng_for(51, 0 if which == "in" else 1)
    T = 8192
    pw = synth.make_proj(geom, synth.HIDDEN, r)
    w = pw["w_in"] if which == "in" else pw["w_out"]
    k = w.shape[1]
    act = synth.store(r.standard_normal((T, k)), synth.BF16)
    out = torch.empty((T, w.shape[0]), dtype=torch.bfloat16, device="cuda")
    gb.gdn_proj_gemm(dev(act), dev(w), out, _ws(T, w.shape[0], k))
    torch.cuda.synchronize()
    rows = np.sort(r.choice(T, 96, replace=False))
    rows[-1] = T - 1
    got = np.zeros((T, w.shape[0]))
    got[rows] = host(out[torch.from_numpy(rows).cuda()])
    _check_gemm(act.f64[:], w.f64[:], got, rows=rows)


def _layer_case(stream, n_tok):
    wl = synth.WORKLOADS["decode4b"]
    geom = wl.geom
    r = synth.rng_for(52, stream)
    p = synth.make_params(geom, r, synth.BF16)
    pw = synth.make_proj(geom, synth.HIDDEN, r)
    h = synth.make_hidden(n_tok, synth.HIDDEN, r)
    return geom, r, p, pw, h


def _okw(p):
    return dict(conv_w=p["conv_w"].f64, A_log=p["A_log"].f64, norm_w=p["norm_w"].f64)


def _conv_close(got, ref, h_seq, w_in, geom):
    """conv rows hold bf16 in-projection values x of the sequence's last d_conv-1
    tokens (rows carried over from the old conv state are exact): each may sit one
    bf16 rounding from the oracle's, plus the fp32 accumulation bound
    k 2^-24 sum_k |h w| of its sum."""
    wx = np.abs(np.asarray(w_in[:geom.conv_channels]))
    k = wx.shape[1]
    mag = np.zeros_like(ref)
    n_new = min(len(h_seq), ref.shape[0])
    if n_new:
        mag[-n_new:] = pj.project(np.abs(np.asarray(h_seq[-n_new:])), wx)
    bound = 2.0 ** -7 * np.abs(ref) + k * 2.0 ** -24 * mag * 1.01
    diff = np.abs(got - ref)
    assert np.all(diff <= bound), f"worst excess {np.max(diff - bound)}"
    assert np.mean(diff > 0) < 0.01


@pytest.mark.parametrize("B", [4, 64])
def test_layer_decode_steps(B):
    steps = 3 if B == 4 else 1
    geom, r, p, pw, h = _layer_case(B, B * steps)
    cfg = config(geom, synth.BF16)
    n_slots = 2 * B
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, synth.BF16, std=0.1)
    slots = r.permutation(n_slots)[:B].astype(np.int32)
    sp, cp = dev(S), dev(CS)
    prm = params_dev(p)
    proj = gb.Proj(dev(pw["w_in"]), dev(pw["w_out"]))
    hd = dev(h).view(steps, B, synth.HIDDEN)
    out = torch.empty((steps, B, synth.HIDDEN), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gb.gdn_layer_workspace_size(cfg, gb.OP_LAYER_DECODE, B, 1, synth.HIDDEN), dtype=torch.uint8,
                     device="cuda")
    si = torch.from_numpy(slots).cuda()
    for s in range(steps):
        gb.gdn_layer_decode(cfg, prm, proj, hd[s], cp, sp, si, out[s], ws)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    got_out, got_S, got_C = host(out), host(sp), host(cp)
    hf = h.f64[:].reshape(steps, B, synth.HIDDEN)
    w_in64, w_out64 = pw["w_in"].f64[:], pw["w_out"].f64[:]
    outs, outr, ss, sr = [], [], [], []
    for i, slot in enumerate(slots):
        ref = pj.layer_sequence(geom, hf[:, i], w_in64, w_out64, s0=S.f64[slot],
                                conv0=CS.f64[slot], **_okw(p))
        outs.append(got_out[:, i].ravel()); outr.append(ref["out"].ravel())
        ss.append(got_S[slot].ravel()); sr.append(ref["S"].ravel())
        _conv_close(got_C[slot], ref["conv"], hf[:, i], w_in64, geom)
    tol = tol_for(synth.BF16)
    e_out = rel_fro(np.concatenate(outs), np.concatenate(outr))
    e_s = rel_fro(np.concatenate(ss), np.concatenate(sr))
    assert e_out <= tol["y"] and e_s <= tol["S"], (e_out, e_s)
    rest = np.setdiff1d(np.arange(n_slots), slots)
    np.testing.assert_array_equal(got_S[rest], S.f64[rest])


def test_layer_varlen_prefill():
    lens = [100, 64, 1, 130]
    geom, r, p, pw, h = _layer_case(7, sum(lens))
    cfg = config(geom, synth.BF16)
    n_slots = 6
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, synth.BF16, std=0.1)
    slots, has_init = [4, 0, 2, 5], [1, 0, 1, 0]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    sp, cp = dev(S), dev(CS)
    out = torch.full((N, synth.HIDDEN), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gb.gdn_layer_workspace_size(cfg, gb.OP_LAYER_VARLEN_PREFILL, N, len(lens), synth.HIDDEN),
                     dtype=torch.uint8, device="cuda")
    gb.gdn_layer_varlen_prefill(cfg, params_dev(p), gb.Proj(dev(pw["w_in"]), dev(pw["w_out"])), dev(h),
                                torch.from_numpy(cu).cuda(), torch.from_numpy(np.asarray(slots, np.int32)).cuda(),
                                torch.from_numpy(np.asarray(has_init, np.uint8)).cuda(), cp, sp, out, ws)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    got_out, got_S, got_C = host(out), host(sp), host(cp)
    hf = h.f64[:]
    w_in64, w_out64 = pw["w_in"].f64[:], pw["w_out"].f64[:]
    outs, outr, ss, sr = [], [], [], []
    for s in range(len(lens)):
        rows = slice(int(cu[s]), int(cu[s + 1]))
        init = bool(has_init[s])
        ref = pj.layer_sequence(geom, hf[rows], w_in64, w_out64,
                                s0=S.f64[slots[s]] if init else None, conv0=CS.f64[slots[s]] if init else None,
                                **_okw(p))
        outs.append(got_out[rows].ravel()); outr.append(ref["out"].ravel())
        ss.append(got_S[slots[s]].ravel()); sr.append(ref["S"].ravel())
        _conv_close(got_C[slots[s]], ref["conv"], hf[rows], w_in64, geom)
    tol = tol_for(synth.BF16)
    e_out = rel_fro(np.concatenate(outs), np.concatenate(outr))
    e_s = rel_fro(np.concatenate(ss), np.concatenate(sr))
    assert e_out <= tol["y"] and e_s <= tol["S"], (e_out, e_s)


def test_layer_prefill_then_decode_steps():
    """gdn_layer_varlen_prefill of a 150-token prompt into a pool slot, then 2
    gdn_layer_decode steps from that slot: out of every token and the final state
    against the oracle layer run over the whole sequence."""
    T, steps = 150, 2
    geom, r, p, pw, h = _layer_case(11, T + steps)
    cfg = config(geom, synth.BF16)
    n_slots = 3
    sp = torch.zeros((n_slots, geom.n_v_heads, geom.d_v, geom.d_k), device="cuda")
    cp = torch.zeros((n_slots, geom.d_conv - 1, geom.conv_channels), dtype=torch.bfloat16, device="cuda")
    slot = 1
    proj = gb.Proj(dev(pw["w_in"]), dev(pw["w_out"]))
    prm = params_dev(p)
    hd = dev(h)
    outs = torch.empty((T + steps, synth.HIDDEN), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gb.gdn_layer_workspace_size(cfg, gb.OP_LAYER_VARLEN_PREFILL, T, 1, synth.HIDDEN),
                     dtype=torch.uint8, device="cuda")
    gb.gdn_layer_varlen_prefill(cfg, prm, proj, hd[:T], torch.tensor([0, T], dtype=torch.int32).cuda(),
                                torch.tensor([slot], dtype=torch.int32).cuda(), None, cp, sp, outs[:T], ws)
    wsd = torch.empty(gb.gdn_layer_workspace_size(cfg, gb.OP_LAYER_DECODE, 1, 1, synth.HIDDEN), dtype=torch.uint8,
                      device="cuda")
    si = torch.tensor([slot], dtype=torch.int32).cuda()
    for s in range(steps):
        gb.gdn_layer_decode(cfg, prm, proj, hd[T + s:T + s + 1], cp, sp, si, outs[T + s:T + s + 1], wsd)
    torch.cuda.synchronize()
    ref = pj.layer_sequence(geom, h.f64[:], pw["w_in"].f64[:], pw["w_out"].f64[:], **_okw(p))
    tol = tol_for(synth.BF16)
    assert rel_fro(host(outs), ref["out"]) <= tol["y"]
    assert rel_fro(host(sp)[slot], ref["S"]) <= tol["S"]
