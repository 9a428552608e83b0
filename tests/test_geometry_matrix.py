"""Every entry point on geometries beyond the pages' two models: d_k = d_v in
{32, 64, 128}, GVA group sizes G = 1, 2, 3, conv widths d_conv = 2, 3, 4, bf16
and fp32 activations.  Per geometry: a prefill of an odd length (several
chunks and a ragged tail), three decode steps continuing from it, then a
verify of 3 rows with a commit of 2 -- all against the fp64 oracle run on the
same accepted tokens (the layer's definition: "Hybrid transformers under load
...", braintools.ru, section 3, as a token recurrence)."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import config, dev, fmt, host, oracle_kwargs, params_dev, rel_fro, tol_for

pytestmark = pytest.mark.gpu

CASES = [
    # (H_k, H_v, d, d_conv, act, chunk)
    (4, 8, 64, 4, synth.BF16, 64),
    (2, 6, 64, 3, synth.F32, 32),
    (3, 3, 32, 2, synth.BF16, 16),
    (2, 4, 128, 3, synth.BF16, 64),   # the tcgen05 prefill path with a 3-tap conv
    (1, 3, 128, 2, synth.BF16, 64),   # tcgen05 path, G = 3, 2-tap conv
]


@pytest.mark.parametrize("hk,hv,d,K,act,chunk", CASES)
def test_prefill_decode_verify_commit(hk, hv, d, K, act, chunk):
    geom = synth.Geometry(hk, hv, d, d, K)
    rng = synth.rng_for(77, hk * 100 + hv * 10 + K)
    p = synth.make_params(geom, rng, act)
    T, steps, r, acc = 150, 3, 3, 2
    tok = synth.make_tokens(geom, T + steps + r, rng, act)
    cfg = config(geom, act, chunk=chunk)
    prm = params_dev(p)
    n_slots = 1 + r
    S = torch.zeros((n_slots, hv, d, d), device="cuda")
    Cp = torch.zeros((n_slots, K - 1, geom.conv_channels), dtype=cfg.torch_dtype, device="cuda")
    x, z, a, b = (dev(tok[k]) for k in ("x", "z", "a", "b"))
    # prefill into slot 0 (varlen, one sequence)
    y_pf = torch.empty((T, hv * d), dtype=cfg.torch_dtype, device="cuda")
    ws = torch.empty(max(1, gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, T, 1)), dtype=torch.uint8,
                     device="cuda")
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    sl = torch.zeros(1, dtype=torch.int32, device="cuda")
    gb.gdn_varlen_prefill(cfg, prm, x[:T], z[:T], a[:T], b[:T], cu, sl, None, Cp, S, y_pf, ws)
    # decode steps
    ys = []
    for t in range(T, T + steps):
        y = torch.empty((1, hv * d), dtype=cfg.torch_dtype, device="cuda")
        gb.gdn_decode_step(cfg, prm, x[t:t + 1], z[t:t + 1], a[t:t + 1], b[t:t + 1], Cp, S, sl, y)
        ys.append(y)
    # verify r rows with snapshots into slots 1..r, commit acc of them
    v0 = T + steps
    yv = torch.empty((1, r, hv * d), dtype=cfg.torch_dtype, device="cuda")
    snaps = torch.arange(1, 1 + r, dtype=torch.int32, device="cuda").view(1, r)
    gb.gdn_verify_rows(cfg, prm, x[v0:v0 + r].view(1, r, -1).contiguous(), z[v0:v0 + r].view(1, r, -1).contiguous(),
                       a[v0:v0 + r].view(1, r, -1).contiguous(), b[v0:v0 + r].view(1, r, -1).contiguous(), Cp, S, sl,
                       snaps, yv)
    gb.gdn_commit_rows(cfg, Cp, S, sl, snaps, torch.tensor([acc], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    n_tot = v0 + acc
    ref = oracle.run_sequence(geom, tok["x"].f64[:n_tot], tok["z"].f64[:n_tot], tok["a"].f64[:n_tot],
                              tok["b"].f64[:n_tot], **oracle_kwargs(p))
    ref_v = oracle.run_sequence(geom, tok["x"].f64[:v0 + r], tok["z"].f64[:v0 + r], tok["a"].f64[:v0 + r],
                                tok["b"].f64[:v0 + r], **oracle_kwargs(p))
    y_got = np.concatenate([host(y_pf), np.concatenate([host(y) for y in ys]), host(yv)[0]])
    errs = {"y": rel_fro(y_got, ref_v["y"]), "S": rel_fro(host(S)[0], ref["S"])}
    tol = tol_for(act)
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)
    np.testing.assert_array_equal(host(Cp)[0], ref["conv"])
