"""The wide-GVA workload at its stated length: 16 k-heads / 48 v-heads, 10240 conv
channels (Strata chapter 6, section 6.2), a prefill of 32768 tokens into 4 pool slots,
then 8 speculative verify steps of 4 rows per slot, each followed by a commit of a
seeded number of accepted rows (0..4, rollback when 0) by copying the snapshot back
("Forge: how I wrote my own inference engine", 27 August: verify rows with shadow
snapshots, rollback = copy).

The 4 slots are prefilled with the same 32768-token sequence, packed 4 times into one
varlen call (4 x 32768 tokens of prefill work, 512 chunks per sequence); the 4 copies
must agree bit for bit.  One sampled v-head is given a long memory (A_log = -6, mean
alpha about 0.998), where any build-up of rounding over 512 chunks would show first.
The oracle evaluates each sampled v-head on that head's own channels (q and k of its
k-head, its v, z, a and b), once over the prefix and then per slot over the accepted
rows from the prefix's state."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, host, oracle_kwargs, params_dev, rel_fro, tol_for

pytestmark = pytest.mark.gpu

L, N_SEQ, STEPS, R_ROWS = 32768, 4, 8, 4
HEADS = [0, 23, 47]  # 47 keeps a long memory
LONG = 47


def _head_inputs(geom, p, tok, j, rows):
    """The channels of v-head j (k-head j // G) as a 1-k-head, 1-v-head layer."""
    G, D, Hk = geom.n_v_heads // geom.n_k_heads, geom.d_v, geom.n_k_heads
    h = j // G
    ch = np.concatenate([np.arange(h * D, (h + 1) * D), np.arange((Hk + h) * D, (Hk + h + 1) * D),
                         np.arange(2 * Hk * D + j * D, 2 * Hk * D + (j + 1) * D)])
    r = np.arange(tok["x"].shape[0])[rows]  # decode only the rows and columns asked for
    x = tok["x"].f64[np.ix_(r, ch)]
    z = tok["z"].f64[np.ix_(r, np.arange(j * D, (j + 1) * D))]
    a = tok["a"].f64[np.ix_(r, [j])]
    b = tok["b"].f64[np.ix_(r, [j])]
    prm = dict(conv_w=p["conv_w"].f64[ch], A_log=p["A_log"].f64[j:j + 1], norm_w=p["norm_w"].f64)
    return x, z, a, b, prm


def test_wide_32768_prefill_4_slots_then_verify_with_rollback():
    wl = synth.WORKLOADS["wide"]
    geom, act = wl.geom, wl.act_dtype
    sub = synth.Geometry(1, 1, geom.d_k, geom.d_v, geom.d_conv)
    rng = synth.rng_for(wl.seed, 11)
    p = synth.make_params(geom, rng, act)
    a_log = p["A_log"].f64[:].copy()
    a_log[LONG] = -6.0
    p = dict(p, A_log=synth.store(a_log, synth.F32))
    seq = synth.make_tokens(geom, L, rng, act)
    ver = synth.make_tokens(geom, STEPS * N_SEQ * R_ROWS, rng, act)  # [step][slot][row]
    accept = rng.integers(0, R_ROWS + 1, size=(STEPS, N_SEQ)).astype(np.int32)
    cfg = config(geom, act)
    prm = params_dev(p)
    n_slots = N_SEQ * (1 + R_ROWS)
    slots = np.arange(N_SEQ, dtype=np.int32)
    snaps = (N_SEQ + np.arange(N_SEQ * R_ROWS, dtype=np.int32)).reshape(N_SEQ, R_ROWS)
    sp = torch.zeros((n_slots, geom.n_v_heads, geom.d_v, geom.d_k), device="cuda")
    cp = torch.zeros((n_slots, geom.d_conv - 1, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")

    # prefill: the sequence 4 times, into slots 0..3
    x, z, a, b = (dev(seq[k]).repeat(N_SEQ, 1) for k in ("x", "z", "a", "b"))
    cu = torch.tensor(np.arange(N_SEQ + 1) * L, dtype=torch.int32, device="cuda")
    y_pre = torch.empty((N_SEQ * L, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, N_SEQ * L, N_SEQ), dtype=torch.uint8,
                     device="cuda")
    gb.gdn_varlen_prefill(cfg, prm, x, z, a, b, cu, torch.from_numpy(slots).cuda(), None, cp, sp, y_pre, ws)
    torch.cuda.synchronize()
    del x, z, a, b, ws
    s_pre = host(sp[:N_SEQ])
    y_pre_h = y_pre.view(N_SEQ, L, -1)
    for s in range(1, N_SEQ):  # the copies agree bit for bit
        assert torch.equal(y_pre_h[s], y_pre_h[0])
        np.testing.assert_array_equal(s_pre[s], s_pre[0])
    y0 = host(y_pre_h[0])
    del y_pre, y_pre_h

    # verify steps with commit / rollback
    vx, vz, va, vb = (dev(ver[k]).view(STEPS, N_SEQ, R_ROWS, -1) for k in ("x", "z", "a", "b"))
    sl, sn = torch.from_numpy(slots).cuda(), torch.from_numpy(snaps).cuda()
    y_acc = {s: [] for s in range(N_SEQ)}
    kept = {s: [] for s in range(N_SEQ)}
    for st in range(STEPS):
        y = torch.empty((N_SEQ, R_ROWS, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
        gb.gdn_verify_rows(cfg, prm, vx[st].contiguous(), vz[st].contiguous(), va[st].contiguous(),
                           vb[st].contiguous(), cp, sp, sl, sn, y)
        gb.gdn_commit_rows(cfg, cp, sp, sl, sn, torch.from_numpy(accept[st]).cuda())
        yh = host(y)
        for s in range(N_SEQ):
            n_acc = int(accept[st, s])
            base = (st * N_SEQ + s) * R_ROWS
            kept[s].extend(range(base, base + n_acc))
            y_acc[s].append(yh[s, :n_acc])
    torch.cuda.synchronize()
    s_got = host(sp[:N_SEQ])
    assert gb.gdn_device_status() == 0

    tol = tol_for(act)
    D = geom.d_v
    pre_y, pre_yr, pre_s, pre_sr, fin_s, fin_sr, acc_y, acc_yr = [], [], [], [], [], [], [], []
    long_s, long_sr = [], []
    for j in HEADS:
        xh, zh, ah, bh, kw = _head_inputs(geom, p, seq, j, slice(0, L))
        ref = oracle.run_sequence(sub, xh, zh, ah, bh, **kw)
        pre_y.append(y0[:, j * D:(j + 1) * D].ravel()); pre_yr.append(ref["y"].ravel())
        pre_s.append(s_pre[0][j].ravel()); pre_sr.append(ref["S"][0].ravel())
        if j == LONG:
            long_s.append(s_pre[0][j].ravel()); long_sr.append(ref["S"][0].ravel())
        for s in range(N_SEQ):
            kr = np.array(kept[s], dtype=np.int64)
            if len(kr):
                xv, zv, av, bv, _ = _head_inputs(geom, p, ver, j, kr)
                r2 = oracle.run_sequence(sub, xv, zv, av, bv, s0=ref["S"], conv0=ref["conv"], **kw)
                acc_y.append(np.concatenate(y_acc[s])[:, j * D:(j + 1) * D].ravel()); acc_yr.append(r2["y"].ravel())
                sref = r2["S"][0]
            else:
                sref = ref["S"][0]
            fin_s.append(s_got[s][j].ravel()); fin_sr.append(sref.ravel())
    cat = np.concatenate
    errs = {"prefill y": rel_fro(cat(pre_y), cat(pre_yr)), "prefill S": rel_fro(cat(pre_s), cat(pre_sr)),
            "long-memory S": rel_fro(cat(long_s), cat(long_sr)),
            "verify y": rel_fro(cat(acc_y), cat(acc_yr)), "committed S": rel_fro(cat(fin_s), cat(fin_sr))}
    assert errs["prefill y"] <= tol["y"] and errs["verify y"] <= tol["y"], fmt(errs)
    assert errs["prefill S"] <= tol["S"] and errs["long-memory S"] <= tol["S"] and errs["committed S"] <= tol["S"], \
        fmt(errs)
    assert accept.min() == 0 and accept.max() == R_ROWS  # both rollback and full accept happened
