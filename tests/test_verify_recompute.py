"""Verify without snapshots + commit by recompute (gdn_verify_rows_nosnap,
gdn_commit_rows_recompute) against the snapshot path ("Forge: how I wrote my
own inference engine", 27 August: rows verified in sequence, rollback by
copying a snapshot).  The recompute runs the verify's arithmetic in the same
order, so the committed state and conv state must equal the snapshot path's
bit for bit, y of the verify likewise, and a verify without snapshots must
leave the pools untouched.  The snapshot path itself is held to the oracle in
test_parity_verify and test_workload_wide_verify; one case here also checks
the committed states against the oracle directly."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, host, make_case, oracle_kwargs, params_dev, rel_fro, sample_heads, tol_for

pytestmark = pytest.mark.gpu


def _case(wl, stream, B, r, geom=None, act=None):
    geom_, act_, rng, p, tok = make_case(wl, stream, B * r, act_dtype=act, geom=geom)
    n_slots = B * (2 + r)
    S = synth.make_state(geom_, n_slots, rng, std=0.1)
    CS = synth.make_conv_state(geom_, n_slots, rng, act_, std=0.1)
    perm = rng.permutation(n_slots).astype(np.int32)
    slots, snaps = perm[:B], perm[B:B * (1 + r)].reshape(B, r)
    accept = rng.integers(0, r + 1, size=B).astype(np.int32)
    accept[0], accept[-1] = 0, r  # both ends always present
    return geom_, act_, p, tok, S, CS, slots, snaps, accept


def _compare(wl, stream, B, r, geom=None, act=None, oracle_heads=None):
    geom, act, p, tok, S, CS, slots, snaps, accept = _case(wl, stream, B, r, geom, act)
    cfg = config(geom, act)
    prm = params_dev(p)
    x, z, a, b = (dev(tok[k]).view(B, r, -1) for k in ("x", "z", "a", "b"))
    sl, sn, acc = (torch.from_numpy(v).cuda() for v in (slots, snaps, accept))
    # snapshot path
    sa, ca = dev(S), dev(CS)
    ya = torch.empty((B, r, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_verify_rows(cfg, prm, x, z, a, b, ca, sa, sl, sn, ya)
    gb.gdn_commit_rows(cfg, ca, sa, sl, sn, acc)
    # recompute path
    sb, cb = dev(S), dev(CS)
    yb = torch.empty((B, r, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    gb.gdn_verify_rows_nosnap(cfg, prm, x, z, a, b, cb, sb, sl, yb)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(sb), S.f64)  # nothing written by the verify
    np.testing.assert_array_equal(host(cb), CS.f64)
    gb.gdn_commit_rows_recompute(cfg, prm, x, a, b, cb, sb, sl, acc)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    np.testing.assert_array_equal(host(yb), host(ya))
    sA, sB, cA, cB = host(sa), host(sb), host(ca), host(cb)
    np.testing.assert_array_equal(sB[slots], sA[slots])
    np.testing.assert_array_equal(cB[slots], cA[slots])
    others = np.setdiff1d(np.arange(S.raw.shape[0]), slots)
    np.testing.assert_array_equal(sB[others], S.f64[others])  # the recompute path touches no other slot
    if oracle_heads is not None:
        # y of every verified row against the oracle on all r rows
        cols = np.concatenate([np.arange(jh * geom.d_v, (jh + 1) * geom.d_v) for jh in oracle_heads])
        yg, ys, yr = host(yb), [], []
        for i in range(B):
            rows = np.arange(i * r, (i + 1) * r)
            ref = oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows],
                                      tok["b"].f64[rows], s0=S.f64[slots[i]], conv0=CS.f64[slots[i]],
                                      heads=oracle_heads, **oracle_kwargs(p))
            ys.append(yg[i][:, cols].ravel()); yr.append(ref["y"][:, cols].ravel())
        err = rel_fro(np.concatenate(ys), np.concatenate(yr))
        assert err <= tol_for(act)["y"], fmt({"y": err})
        ss, sr = [], []
        for i in range(B):
            n = int(accept[i])
            if n == 0:  # nothing accepted: the slot keeps its state
                np.testing.assert_array_equal(sB[slots[i]], S.f64[slots[i]])
                continue
            rows = np.arange(i * r, i * r + n)
            ref = oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows],
                                      tok["b"].f64[rows], s0=S.f64[slots[i]], conv0=CS.f64[slots[i]],
                                      heads=oracle_heads, **oracle_kwargs(p))
            ss.append(sB[slots[i]][oracle_heads].ravel()); sr.append(ref["S"][oracle_heads].ravel())
            np.testing.assert_array_equal(cB[slots[i]], ref["conv"])
        err = rel_fro(np.concatenate(ss), np.concatenate(sr))
        assert err <= tol_for(act)["S"], fmt({"S": err})


@pytest.mark.parametrize("B,r", [(8, 4), (3, 16), (5, 1)])
def test_recompute_equals_snapshot_path_4b(B, r):
    _compare("decode4b", 31 + B, B, r)


def test_recompute_equals_snapshot_path_wide_gva_and_oracle():
    _compare("wide", 41, 4, 4, oracle_heads=sample_heads(48, 3, seed=9))


def test_recompute_tiny_fp32():
    _compare("tiny", 51, 6, 5, oracle_heads=[0, 1])


# larger batches (B x H_v above the SM count) and r up to 16
@pytest.mark.parametrize("B,r", [(24, 4), (20, 16), (40, 1)])
def test_recompute_equals_snapshot_path_large_batch_4b(B, r):
    _compare("decode4b", 61 + r, B, r, oracle_heads=sample_heads(32, 2, seed=B))


def test_recompute_equals_snapshot_path_large_batch_wide():
    _compare("wide", 71, 16, 4, oracle_heads=sample_heads(48, 2, seed=4))
