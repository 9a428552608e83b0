"""The wide-GVA workload end to end on the GPU: 16 k-heads / 48 v-heads,
10240 conv channels (Strata chapter 6, section 6.2).  A prefill of 32768
tokens packed as 4 sequences of 8192 fills 4 pool slots; then 8 speculative
verify steps of 4 rows per slot run, each followed by a commit of a seeded
number of accepted rows (0..4, rollback when 0) by copying the snapshot back
("Forge: how I wrote my own inference engine", 27 August: verify rows with
shadow snapshots, rollback = copy).  Every slot's committed state and conv
state, and the outputs of every accepted row, must equal the fp64 oracle run
on only the tokens that were accepted (checked on 3 of the 48 v-heads, which
the oracle evaluates independently)."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, head_cols, host, oracle_kwargs, params_dev, rel_fro, sample_heads, tol_for

pytestmark = pytest.mark.gpu


def test_wide_prefill_then_verify_with_rollback():
    wl = synth.WORKLOADS["wide"]
    geom, act = wl.geom, wl.act_dtype
    n_seq, L, steps, r_rows = 4, 8192, 8, 4
    rng = synth.rng_for(wl.seed, 1)
    p = synth.make_params(geom, rng, act)
    pre = synth.make_tokens(geom, n_seq * L, rng, act)
    ver = synth.make_tokens(geom, steps * n_seq * r_rows, rng, act)  # [step][slot][row]
    accept = rng.integers(0, r_rows + 1, size=(steps, n_seq)).astype(np.int32)
    cfg = config(geom, act)
    prm = params_dev(p)
    n_slots = n_seq * (1 + r_rows)
    slots = np.arange(n_seq, dtype=np.int32)
    snaps = (n_seq + np.arange(n_seq * r_rows, dtype=np.int32)).reshape(n_seq, r_rows)
    sp = torch.zeros((n_slots, geom.n_v_heads, geom.d_v, geom.d_k), device="cuda")
    cp = torch.zeros((n_slots, geom.d_conv - 1, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")

    # prefill: 4 sequences into slots 0..3
    cu = torch.tensor(np.arange(n_seq + 1) * L, dtype=torch.int32, device="cuda")
    y_pre = torch.empty((n_seq * L, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
    ws = torch.empty(gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, n_seq * L, n_seq), dtype=torch.uint8,
                     device="cuda")
    gb.gdn_varlen_prefill(cfg, prm, dev(pre["x"]), dev(pre["z"]), dev(pre["a"]), dev(pre["b"]), cu,
                          torch.from_numpy(slots).cuda(), None, cp, sp, y_pre, ws)

    # verify steps
    vx, vz, va, vb = (dev(ver[k]).view(steps, n_seq, r_rows, -1) for k in ("x", "z", "a", "b"))
    sl, sn = torch.from_numpy(slots).cuda(), torch.from_numpy(snaps).cuda()
    y_acc = {s: [] for s in range(n_seq)}
    kept_rows = {s: [] for s in range(n_seq)}  # indices into `ver`
    for st in range(steps):
        y = torch.empty((n_seq, r_rows, geom.value_dim), dtype=cfg.torch_dtype, device="cuda")
        gb.gdn_verify_rows(cfg, prm, vx[st].contiguous(), vz[st].contiguous(), va[st].contiguous(),
                           vb[st].contiguous(), cp, sp, sl, sn, y)
        gb.gdn_commit_rows(cfg, cp, sp, sl, sn, torch.from_numpy(accept[st]).cuda())
        yh = host(y)
        for s in range(n_seq):
            a = int(accept[st, s])
            base = (st * n_seq + s) * r_rows
            kept_rows[s].extend(range(base, base + a))
            y_acc[s].append(yh[s, :a])
    torch.cuda.synchronize()
    s_got, c_got = host(sp), host(cp)

    heads = sample_heads(geom.n_v_heads, 3, seed=3)
    cols = head_cols(heads, geom.d_v)
    tol = tol_for(act)
    ys, yr, ss, sr = [], [], [], []
    for s in range(n_seq):
        rows = np.arange(s * L, (s + 1) * L)
        kr = np.array(kept_rows[s], dtype=np.int64)
        x = np.concatenate([pre["x"].f64[rows], ver["x"].f64[kr]]) if len(kr) else pre["x"].f64[rows]
        z = np.concatenate([pre["z"].f64[rows], ver["z"].f64[kr]]) if len(kr) else pre["z"].f64[rows]
        a_ = np.concatenate([pre["a"].f64[rows], ver["a"].f64[kr]]) if len(kr) else pre["a"].f64[rows]
        b_ = np.concatenate([pre["b"].f64[rows], ver["b"].f64[kr]]) if len(kr) else pre["b"].f64[rows]
        ref = oracle.run_sequence(geom, x, z, a_, b_, heads=heads, **oracle_kwargs(p))
        ss.append(s_got[s][heads].ravel()); sr.append(ref["S"][heads].ravel())
        if len(kr):
            ys.append(np.concatenate(y_acc[s])[:, cols].ravel()); yr.append(ref["y"][L:, cols].ravel())
        np.testing.assert_array_equal(c_got[s], ref["conv"])
    errs = {"S": rel_fro(np.concatenate(ss), np.concatenate(sr)),
            "y": rel_fro(np.concatenate(ys), np.concatenate(yr))}
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    assert accept.min() == 0 and accept.max() == r_rows  # both rollback and full accept happened
    assert gb.gdn_device_status() == 0
