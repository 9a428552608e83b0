"""GDN_DEBUG: the device-side check of slot indices.

With GDN_DEBUG set, decode, verify, commit and varlen prefill check their slot
indices on the device first (every index in [0, n_slots), none twice).  A bad
batch is refused with GDN_ERR_RANGE, the message naming the position and the
value, before any kernel touches the pools; GDN_DEV_BAD_SLOT is set in the
device status.  A valid batch gives exactly the result of the same call without
the check.  The pages describe no such mode: it is a debugging aid.
"""
import numpy as np
import pytest
import torch

from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, make_case, params_dev

pytestmark = pytest.mark.gpu

ERR_RANGE = -5
DEV_BAD_SLOT = 2


def _pools(geom, act, r, n_slots):
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=0.1)
    return dev(S), dev(CS)


def _decode(cfg, prm, tok, sp, cp, slots):
    B = len(slots)
    y = torch.zeros((B, cfg.n_v_heads * cfg.d_v), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_decode_step(cfg, prm, dev(tok["x"])[:B], dev(tok["z"])[:B], dev(tok["a"])[:B], dev(tok["b"])[:B], cp, sp,
                       torch.tensor(slots, dtype=torch.int32, device="cuda"), y)
    return y


def _refused(fn, *words):
    with pytest.raises(gb.GdnError) as ei:
        fn()
    assert ei.value.status == ERR_RANGE
    for w in words:
        assert w in str(ei.value), str(ei.value)
    assert gb.gdn_device_status() & DEV_BAD_SLOT


@pytest.fixture
def decode_case():
    geom, act, r, p, tok = make_case("decode4b", 41, 8)
    return geom, act, r, p, tok, config(geom, act)


def test_debug_refuses_repeated_and_out_of_range_decode_slots(decode_case, monkeypatch):
    geom, act, r, p, tok, cfg = decode_case
    prm = params_dev(p)
    sp, cp = _pools(geom, act, r, 16)
    s_before, c_before = sp.clone(), cp.clone()
    gb.gdn_device_status()
    monkeypatch.setenv("GDN_DEBUG", "1")
    _refused(lambda: _decode(cfg, prm, tok, sp, cp, [3, 5, 9, 5]), "slot_idx[1]", "slot_idx[3]", "slot 5 twice")
    _refused(lambda: _decode(cfg, prm, tok, sp, cp, [3, 16, 9]), "slot_idx[1]", "found slot 16", "0..15")
    _refused(lambda: _decode(cfg, prm, tok, sp, cp, [-2, 1]), "slot_idx[0]", "found slot -2")
    torch.cuda.synchronize()
    assert torch.equal(sp, s_before) and torch.equal(cp, c_before)  # refused before any kernel ran
    assert gb.gdn_device_status() == 0  # the bit was read and cleared above


def test_debug_off_values_disable_the_check(decode_case, monkeypatch):
    geom, act, r, p, tok, cfg = decode_case
    prm = params_dev(p)
    sp, cp = _pools(geom, act, r, 16)
    for v in ("0", ""):
        monkeypatch.setenv("GDN_DEBUG", v)
        _decode(cfg, prm, tok, sp, cp, [3, 16])  # out of range is skipped by the kernels, not refused
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0


def test_debug_valid_decode_is_bitwise_the_unchecked_call(decode_case, monkeypatch):
    geom, act, r, p, tok, cfg = decode_case
    prm = params_dev(p)
    slots = [11, 2, 7, 0, 15, 4, 9, 13]
    sp1, cp1 = _pools(geom, act, r, 16)
    sp2, cp2 = sp1.clone(), cp1.clone()
    monkeypatch.delenv("GDN_DEBUG", raising=False)
    y1 = _decode(cfg, prm, tok, sp1, cp1, slots)
    monkeypatch.setenv("GDN_DEBUG", "1")
    y2 = _decode(cfg, prm, tok, sp2, cp2, slots)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(sp1, sp2) and torch.equal(cp1, cp2)
    assert gb.gdn_device_status() == 0


def test_debug_verify_and_commit_check_slots_and_snapshots_together(monkeypatch):
    B, rr = 2, 3
    geom, act, r, p, tok = make_case("tiny", 43, B * rr)
    cfg = config(geom, act)
    prm = params_dev(p)
    sp, cp = _pools(geom, act, r, 12)
    s_before = sp.clone()
    x, z, a, b = (dev(tok[k]).view(B, rr, -1) for k in ("x", "z", "a", "b"))
    y = torch.zeros((B, rr, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    sl = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    sn_bad = torch.tensor([[2, 3, 4], [5, 1, 7]], dtype=torch.int32, device="cuda")  # live slot 1 reused as snapshot
    sn_ok = torch.tensor([[2, 3, 4], [5, 6, 7]], dtype=torch.int32, device="cuda")
    gb.gdn_device_status()
    monkeypatch.setenv("GDN_DEBUG", "1")
    _refused(lambda: gb.gdn_verify_rows(cfg, prm, x, z, a, b, cp, sp, sl, sn_bad, y),
             "slot_idx[1]", "snap_idx[4]", "slot 1 twice")
    acc = torch.tensor([2, 1], dtype=torch.int32, device="cuda")
    _refused(lambda: gb.gdn_commit_rows(cfg, cp, sp, sl, sn_bad, acc), "snap_idx[4]")
    torch.cuda.synchronize()
    assert torch.equal(sp, s_before)
    gb.gdn_verify_rows(cfg, prm, x, z, a, b, cp, sp, sl, sn_ok, y)
    gb.gdn_commit_rows(cfg, cp, sp, sl, sn_ok, acc)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0


def test_debug_varlen_prefill_refuses_a_slot_given_twice(monkeypatch):
    lens = [5, 70, 9]
    geom, act, r, p, tok = make_case("serving", 44, sum(lens))
    cfg = config(geom, act)
    sp, cp = _pools(geom, act, r, 6)
    s_before = sp.clone()
    N = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    x, z, a, b = (dev(tok[k])[:N] for k in ("x", "z", "a", "b"))
    y = torch.zeros((N, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    ws = torch.empty(max(1, gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, N, len(lens))), dtype=torch.uint8,
                     device="cuda")
    gb.gdn_device_status()
    monkeypatch.setenv("GDN_DEBUG", "1")
    bad = torch.tensor([4, 1, 4], dtype=torch.int32, device="cuda")
    _refused(lambda: gb.gdn_varlen_prefill(cfg, params_dev(p), x, z, a, b, cu, bad, None, cp, sp, y, ws),
             "slot_idx[0]", "slot_idx[2]", "slot 4 twice")
    torch.cuda.synchronize()
    assert torch.equal(sp, s_before)
    good = torch.tensor([4, 1, 0], dtype=torch.int32, device="cuda")
    gb.gdn_varlen_prefill(cfg, params_dev(p), x, z, a, b, cu, good, None, cp, sp, y, ws)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0


def test_debug_under_graph_capture_only_sets_the_status_bit(decode_case, monkeypatch):
    """A capturing stream cannot wait for the check: the call is captured with it,
    and a replay over an out-of-range slot (which the kernels skip) reports
    GDN_DEV_BAD_SLOT."""
    geom, act, r, p, tok, cfg = decode_case
    prm = params_dev(p)
    sp, cp = _pools(geom, act, r, 16)
    B = 4
    x, z, a, b = (dev(tok[k])[:B] for k in ("x", "z", "a", "b"))
    y = torch.zeros((B, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    slots = torch.tensor([1, 2, 3, 4], dtype=torch.int32, device="cuda")
    monkeypatch.setenv("GDN_DEBUG", "1")
    stream = torch.cuda.Stream()
    gb.gdn_device_status()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        gb.gdn_decode_step(cfg, prm, x, z, a, b, cp, sp, slots, y, stream=stream)
    graph.replay()
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    slots.copy_(torch.tensor([1, 2, 99, 4], dtype=torch.int32))
    graph.replay()
    torch.cuda.synchronize()
    assert gb.gdn_device_status() & DEV_BAD_SLOT
