"""The serving mix's decode batch: 256 slots, chosen at random without repeats from a
pool of 1024 (16 k-heads / 32 v-heads, d = 128, bf16 activations, fp32 states of 2 MiB
a slot), two consecutive decode steps through the C ABI.  Slots 0 .. 1023 not in the
batch hold zeros and must stay zero; 16 sampled batch slots are compared with the fp64
oracle run on their two tokens from their initial state, and every batch slot's conv
state must hold its last d_conv - 1 raw inputs."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, host, oracle_kwargs, params_dev, rel_fro, tol_for

pytestmark = pytest.mark.gpu


def test_serving_decode_256_of_1024_random_slots_two_steps():
    wl = synth.WORKLOADS["serving"]
    geom, act = wl.geom, wl.act_dtype
    B, n_slots, steps = 256, 1024, 2
    rng = synth.rng_for(wl.seed, 21)
    p = synth.make_params(geom, rng, act)
    tok = synth.make_tokens(geom, steps * B, rng, act)  # [step][batch]
    S = synth.make_state(geom, B, rng, std=0.1)          # initial states of the batch slots
    CS = synth.make_conv_state(geom, B, rng, act, std=0.1)
    slots = rng.choice(n_slots, B, replace=False).astype(np.int32)
    cfg = config(geom, act)
    prm = params_dev(p)
    sp = torch.zeros((n_slots, geom.n_v_heads, geom.d_v, geom.d_k), device="cuda")
    cp = torch.zeros((n_slots, geom.d_conv - 1, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    idx = torch.from_numpy(slots).long().cuda()
    sp[idx] = dev(S)
    cp[idx] = dev(CS)
    sl = torch.from_numpy(slots).cuda()
    ys = []
    for st in range(steps):
        rows = slice(st * B, (st + 1) * B)
        y = torch.full((B, geom.value_dim), float("nan"), dtype=cfg.torch_dtype, device="cuda")
        gb.gdn_decode_step(cfg, prm, dev(tok["x"])[rows].contiguous(), dev(tok["z"])[rows].contiguous(),
                           dev(tok["a"])[rows].contiguous(), dev(tok["b"])[rows].contiguous(), cp, sp, sl, y)
        ys.append(y)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    # slots outside the batch are untouched
    rest = torch.ones(n_slots, dtype=torch.bool, device="cuda")
    rest[idx] = False
    assert float(sp[rest].abs().sum()) == 0.0 and float(cp[rest].float().abs().sum()) == 0.0
    s_got, c_got = host(sp[idx]), host(cp[idx])
    y_got = [host(y) for y in ys]
    check = sorted(set([0, B - 1] + list(rng.choice(B, 14, replace=False))))
    yv, yr, sv, sr = [], [], [], []
    for b in check:
        rows = np.array([st * B + b for st in range(steps)])
        ref = oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows],
                                  tok["b"].f64[rows], s0=S.f64[b], conv0=CS.f64[b], **oracle_kwargs(p))
        yv.append(np.stack([y_got[st][b] for st in range(steps)])); yr.append(ref["y"])
        sv.append(s_got[b]); sr.append(ref["S"])
        np.testing.assert_array_equal(c_got[b], ref["conv"])
    tol = tol_for(act)
    errs = {"y": rel_fro(np.stack(yv), np.stack(yr)), "S": rel_fro(np.stack(sv), np.stack(sr))}
    assert len(check) >= 16
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
