"""GPU parity of gdn_verify_rows / gdn_commit_rows against the fp64 oracle.

A verify of r rows writes the state (and conv state) after row i of entry b to
pool slot snap_idx[b, i]; accepting a rows selects snapshot a-1 (a = 0 keeps
the original slot), which must equal the oracle run over the a accepted
tokens ("Forge: how I wrote my own inference engine", entry of 27 August:
sequential rows with shadow snapshots, rollback = copy of a snapshot).
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, host, make_case, oracle_kwargs, params_dev, rel_fro, tol_for

pytestmark = pytest.mark.gpu


def _verify_case(wl_name, B, r_rows, stream):
    geom, act, r, p, tok = make_case(wl_name, stream, B * r_rows)
    n_slots = B * (r_rows + 2)
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=0.1)
    perm = r.permutation(n_slots).astype(np.int32)
    slots = perm[:B]
    snaps = perm[B:B + B * r_rows].reshape(B, r_rows)
    return geom, act, r, p, tok, S, CS, slots, snaps


@pytest.mark.parametrize("wl_name,B,r_rows", [("wide", 4, 4), ("decode4b", 3, 2), ("tiny", 2, 5)])
def test_verify_rows_snapshots_and_commit(wl_name, B, r_rows):
    geom, act, r, p, tok, S, CS, slots, snaps = _verify_case(wl_name, B, r_rows, stream=200 + B)
    cfg = config(geom, act)
    sp, cp = dev(S), dev(CS)
    x, z, a, b = (dev(tok[k]).view(B, r_rows, -1) for k in ("x", "z", "a", "b"))
    y = torch.empty((B, r_rows, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    sl, sn = torch.from_numpy(slots).cuda(), torch.from_numpy(snaps).cuda()
    gb.gdn_verify_rows(cfg, params_dev(p), x, z, a, b, cp, sp, sl, sn, y)
    torch.cuda.synchronize()
    s_got, c_got, y_got = host(sp), host(cp), host(y)
    tol = tol_for(act)
    ys, yr, ss, sr = [], [], [], []
    for bi in range(B):
        rows = slice(bi * r_rows, (bi + 1) * r_rows)
        # the original slot is read, not written
        np.testing.assert_array_equal(s_got[slots[bi]], S.f64[slots[bi]])
        np.testing.assert_array_equal(c_got[slots[bi]], CS.f64[slots[bi]])
        for i in range(r_rows):
            sub = slice(bi * r_rows, bi * r_rows + i + 1)
            ref = oracle.run_sequence(geom, tok["x"].f64[sub], tok["z"].f64[sub], tok["a"].f64[sub],
                                      tok["b"].f64[sub], s0=S.f64[slots[bi]], conv0=CS.f64[slots[bi]],
                                      **oracle_kwargs(p))
            ss.append(s_got[snaps[bi, i]]); sr.append(ref["S"])
            np.testing.assert_array_equal(c_got[snaps[bi, i]], ref["conv"])
        ys.append(y_got[bi]); yr.append(ref["y"])
    errs = {"y": rel_fro(ys, yr), "S": rel_fro(ss, sr)}
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)

    # commit by copy: accepted a in {0..r}
    acc = r.integers(0, r_rows + 1, size=B).astype(np.int32)
    acc[0] = 0
    acc[-1] = r_rows
    gb.gdn_commit_rows(cfg, cp, sp, sl, sn, torch.from_numpy(acc).cuda())
    torch.cuda.synchronize()
    s2, c2 = host(sp), host(cp)
    for bi in range(B):
        src = slots[bi] if acc[bi] == 0 else snaps[bi, acc[bi] - 1]
        expect_s = S.f64[slots[bi]] if acc[bi] == 0 else s_got[src]
        expect_c = CS.f64[slots[bi]] if acc[bi] == 0 else c_got[src]
        np.testing.assert_array_equal(s2[slots[bi]], expect_s)
        np.testing.assert_array_equal(c2[slots[bi]], expect_c)


def test_verify_one_row_equals_decode():
    """verify with r = 1 writes exactly what a decode step writes in place."""
    geom, act, r, p, tok, S, CS, slots, snaps = _verify_case("decode4b", 2, 1, stream=300)
    cfg = config(geom, act)
    prm = params_dev(p)
    sp1, cp1, sp2, cp2 = dev(S), dev(CS), dev(S), dev(CS)
    x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
    y1 = torch.empty((2, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    y2 = torch.empty_like(y1)
    sl = torch.from_numpy(slots).cuda()
    gb.gdn_decode_step(cfg, prm, x, z, a, b, cp1, sp1, sl, y1)
    gb.gdn_verify_rows(cfg, prm, x.view(2, 1, -1), z.view(2, 1, -1), a.view(2, 1, -1), b.view(2, 1, -1), cp2, sp2,
                       sl, torch.from_numpy(snaps).cuda(), y2.view(2, 1, -1))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    for bi in range(2):
        assert torch.equal(sp1[slots[bi]], sp2[snaps[bi, 0]])
        assert torch.equal(cp1[slots[bi]], cp2[snaps[bi, 0]])
