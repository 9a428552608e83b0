"""Prefix snapshots of the chunked prefill (gdn_varlen_prefill_ckpt): the state
and conv state after every ckpt_every tokens of each sequence land in the pool
slots the caller names ("Hybrid transformers under load ...", braintools.ru,
sections 3 and 4.2: prefix reuse needs a saved copy of the state at the prefix
end; a snapshot at each block boundary).  Each snapshot must equal the fp64
oracle run on the prefix alone, and a decode resumed from a snapshot slot must
equal the oracle on the prefix plus the new tokens."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, host, make_case, oracle_kwargs, params_dev, rel_fro, sample_heads, tol_for

pytestmark = pytest.mark.gpu


def _run(cfg, p, tok, lens, slots, has_init, S, CS, every, ck_counts, ck_slots):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    sp, cp = dev(S), dev(CS)
    x, z, a, b = (dev(tok[k])[:N] for k in ("x", "z", "a", "b"))
    y = torch.empty((N, cfg.n_v_heads * cfg.d_v), dtype=cfg.torch_dtype, device="cuda")
    ws = torch.empty(max(1, gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, N, len(lens))), dtype=torch.uint8,
                     device="cuda")
    off = np.concatenate([[0], np.cumsum(ck_counts)]).astype(np.int32)
    hi = None if has_init is None else torch.from_numpy(np.asarray(has_init, np.uint8)).cuda()
    gb.gdn_varlen_prefill_ckpt(cfg, params_dev(p), x, z, a, b, torch.from_numpy(cu).cuda(),
                               torch.from_numpy(np.asarray(slots, np.int32)).cuda(), hi, cp, sp, y, every,
                               torch.from_numpy(off).cuda(), torch.from_numpy(np.asarray(ck_slots, np.int32)).cuda(), ws)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    return cu, off, host(sp), host(cp), sp, cp


def _check_snapshots(geom, act, p, tok, cu, off, lens, slots, has_init, S, CS, every, ck_slots, s_got, c_got, heads,
                     tol_S):
    written = set()
    ss, sr = [], []
    for s, L in enumerate(lens):
        rows0 = int(cu[s])
        init = has_init is not None and has_init[s]
        n_ck = min(L // every, int(off[s + 1] - off[s]))
        for k in range(n_ck):
            slot = int(ck_slots[off[s] + k])
            P = (k + 1) * every
            rows = slice(rows0, rows0 + P)
            ref = oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows],
                                      tok["b"].f64[rows], s0=S.f64[slots[s]] if init else None,
                                      conv0=CS.f64[slots[s]] if init else None, heads=heads, **oracle_kwargs(p))
            hs = heads if heads is not None else list(range(geom.n_v_heads))
            ss.append(s_got[slot][hs].ravel())
            sr.append(ref["S"][hs].ravel())
            np.testing.assert_array_equal(c_got[slot], ref["conv"])
            written.add(slot)
    err = rel_fro(np.concatenate(ss), np.concatenate(sr))
    assert err <= tol_S, fmt({"S": err})
    return written


def test_snapshots_tcgen05_path_varlen_mixed_init():
    lens = [700, 300, 1100]
    geom, act, r, p, tok = make_case("serving", 21, sum(lens))
    cfg = config(geom, act)
    n_slots = 14
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=0.1)
    slots, has_init = [0, 1, 2], [1, 0, 0]
    every = 256
    counts = [L // every for L in lens]            # 2, 1, 4
    ck_slots = [5, 3, 12, 4, 6, 7, 8]
    cu, off, s_got, c_got, _, _ = _run(cfg, p, tok, lens, slots, has_init, S, CS, every, counts, ck_slots)
    heads = sample_heads(geom.n_v_heads, 3, seed=5)
    written = _check_snapshots(geom, act, p, tok, cu, off, lens, slots, has_init, S, CS, every, ck_slots, s_got,
                               c_got, heads, tol_for(act)["S"])
    assert written == set(ck_slots)
    rest = np.setdiff1d(np.arange(n_slots), list(written) + slots)
    np.testing.assert_array_equal(s_got[rest], S.f64[rest])
    np.testing.assert_array_equal(c_got[rest], CS.f64[rest])


def test_snapshots_fallback_path_fp32_and_fewer_slots_than_boundaries():
    lens = [64, 45, 100]
    geom, act, r, p, tok = make_case("tiny", 22, sum(lens))
    cfg = config(geom, act, chunk=16)
    n_slots = 10
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=0.1)
    slots, has_init = [0, 1, 2], [0, 1, 1]
    every = 32
    counts = [2, 1, 2]  # sequence 2 has 3 boundaries (32, 64, 96) but only 2 slots: the third is not written
    ck_slots = [3, 4, 5, 6, 9]
    cu, off, s_got, c_got, _, _ = _run(cfg, p, tok, lens, slots, has_init, S, CS, every, counts, ck_slots)
    written = _check_snapshots(geom, act, p, tok, cu, off, lens, slots, has_init, S, CS, every, ck_slots, s_got,
                               c_got, None, tol_for(act)["S"])
    assert written == set(ck_slots)
    rest = [7, 8]
    np.testing.assert_array_equal(s_got[rest], S.f64[rest])
    np.testing.assert_array_equal(c_got[rest], CS.f64[rest])


def test_decode_resumes_from_a_snapshot_slot():
    """A second request sharing the first 512 tokens of a prefix continues from
    the snapshot: 4 decode steps there equal the oracle on the prefix + 4 tokens."""
    L, every, extra = 900, 256, 4
    geom, act, r, p, tok = make_case("serving", 23, L + extra)
    cfg = config(geom, act)
    n_slots = 6
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=0.1)
    ck_slots = [3, 4, 5]  # after 256, 512, 768 tokens
    tok_pf = {k: tok[k] for k in ("x", "z", "a", "b")}
    cu, off, s_got, c_got, sp, cp = _run(cfg, p, tok_pf, [L], [0], None, S, CS, every, [3], ck_slots)
    P = 512
    slot = torch.tensor([4], dtype=torch.int32, device="cuda")
    prm = params_dev(p)
    ys = []
    for t in range(extra):  # the new request's own tokens after the shared prefix
        x, z, a, b = (dev(tok[k])[L + t:L + t + 1] for k in ("x", "z", "a", "b"))
        y = torch.empty((1, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
        gb.gdn_decode_step(cfg, prm, x, z, a, b, cp, sp, slot, y)
        ys.append(host(y)[0])
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(P), np.arange(L, L + extra)])
    heads = sample_heads(geom.n_v_heads, 3, seed=6)
    ref = oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows], tok["b"].f64[rows],
                              heads=heads, **oracle_kwargs(p))
    s_after = host(sp)[4]
    cols = np.concatenate([np.arange(j * geom.d_v, (j + 1) * geom.d_v) for j in heads])
    errs = {"y": rel_fro(np.stack(ys)[:, cols], ref["y"][P:, cols]), "S": rel_fro(s_after[heads], ref["S"][heads])}
    tol = tol_for(act)
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    np.testing.assert_array_equal(host(cp)[4], ref["conv"])
