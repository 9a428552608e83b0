"""GPU parity of gdn_varlen_prefill (packed sequences, pool slots) against the
oracle run on each sequence separately.  Chunks restart at every sequence
start; sequences with has_init = 1 continue from their slot's states."""
import numpy as np
import pytest
import torch

import oracle
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import (config, dev, fmt, head_cols, host, make_case, oracle_kwargs, params_dev, rel_fro,
                       sample_heads, tol_for)

pytestmark = pytest.mark.gpu


def run_varlen(cfg, p, tok, lens, slots, has_init, S, CS):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    sp, cp = dev(S), dev(CS)
    x, z, a, b = (dev(tok[k])[:N] for k in ("x", "z", "a", "b"))
    y = torch.full((N, cfg.n_v_heads * cfg.d_v), float("nan"), dtype=cfg.torch_dtype, device="cuda")
    ws = torch.empty(max(1, gb.gdn_workspace_size(cfg, gb.OP_VARLEN_PREFILL, N, len(lens))), dtype=torch.uint8,
                     device="cuda")
    hi = None if has_init is None else torch.from_numpy(np.asarray(has_init, np.uint8)).cuda()
    gb.gdn_varlen_prefill(cfg, params_dev(p), x, z, a, b, torch.from_numpy(cu).cuda(),
                          torch.from_numpy(np.asarray(slots, np.int32)).cuda(), hi, cp, sp, y, ws)
    torch.cuda.synchronize()
    return cu, host(y), host(sp), host(cp)


def check_seqs(geom, act, p, tok, cu, y, s_got, c_got, slots, has_init, S, CS, seqs, heads=None):
    tol = tol_for(act)
    ys, yr, ss, sr = [], [], [], []
    cols = None if heads is None else head_cols(heads, geom.d_v)
    for s in seqs:
        rows = slice(int(cu[s]), int(cu[s + 1]))
        init = has_init is not None and has_init[s]
        ref = oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows],
                                  tok["b"].f64[rows], s0=S.f64[slots[s]] if init else None,
                                  conv0=CS.f64[slots[s]] if init else None, heads=heads, **oracle_kwargs(p))
        if heads is None:
            ys.append(y[rows].ravel()); yr.append(ref["y"].ravel())
            ss.append(s_got[slots[s]].ravel()); sr.append(ref["S"].ravel())
        else:
            ys.append(y[rows][:, cols].ravel()); yr.append(ref["y"][:, cols].ravel())
            ss.append(s_got[slots[s]][heads].ravel()); sr.append(ref["S"][heads].ravel())
        np.testing.assert_array_equal(c_got[slots[s]], ref["conv"])
    errs = {"y": rel_fro(np.concatenate(ys), np.concatenate(yr)), "S": rel_fro(np.concatenate(ss), np.concatenate(sr))}
    assert errs["y"] <= tol["y"] and errs["S"] <= tol["S"], fmt(errs)


def test_varlen_small_mixed_init():
    lens = [1, 17, 64, 100, 3, 0, 129]
    geom, act, r, p, tok = make_case("serving", 1, sum(lens))
    cfg = config(geom, act)
    n_slots = 12
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=0.1)
    slots = [3, 0, 7, 11, 5, 2, 9]
    has_init = [1, 0, 1, 0, 1, 1, 0]
    cu, y, s_got, c_got = run_varlen(cfg, p, tok, lens, slots, has_init, S, CS)
    check_seqs(geom, act, p, tok, cu, y, s_got, c_got, slots, has_init, S, CS, range(len(lens)))
    # slots not named are untouched
    rest = np.setdiff1d(np.arange(n_slots), slots)
    np.testing.assert_array_equal(s_got[rest], S.f64[rest])
    np.testing.assert_array_equal(c_got[rest], CS.f64[rest])


def test_varlen_mixed_lengths_and_init():
    """Sequences of 200, 1, 64, 130 and 63 tokens (full chunks, a one-token
    sequence, exact and ragged tails) with mixed initial states, through one
    varlen call."""
    lens = [200, 1, 64, 130, 63]
    geom, act, r, p, tok = make_case("serving", 4, sum(lens))
    cfg = config(geom, act)
    S = synth.make_state(geom, 8, r, std=0.1)
    CS = synth.make_conv_state(geom, 8, r, act, std=0.1)
    slots, has_init = [6, 1, 0, 3, 4], [1, 0, 1, 0, 1]
    cu, y, s_got, c_got = run_varlen(cfg, p, tok, lens, slots, has_init, S, CS)
    check_seqs(geom, act, p, tok, cu, y, s_got, c_got, slots, has_init, S, CS, range(len(lens)))


def test_varlen_tiny_fp32_equals_single_prefill():
    lens = [64, 45, 16, 3]
    geom, act, r, p, tok = make_case("tiny", 2, sum(lens))
    cfg = config(geom, act, chunk=16)
    S = synth.make_state(geom, 4, r, std=0.1)
    CS = synth.make_conv_state(geom, 4, r, act, std=0.1)
    slots, has_init = [0, 1, 2, 3], [0, 1, 0, 1]
    cu, y, s_got, c_got = run_varlen(cfg, p, tok, lens, slots, has_init, S, CS)
    for s in range(4):
        rows = slice(int(cu[s]), int(cu[s + 1]))
        ref = oracle.run_sequence(geom, tok["x"].f64[rows], tok["z"].f64[rows], tok["a"].f64[rows],
                                  tok["b"].f64[rows], s0=S.f64[s] if has_init[s] else None,
                                  conv0=CS.f64[s] if has_init[s] else None, **oracle_kwargs(p))
        errs = {"y": rel_fro(y[rows], ref["y"]), "S": rel_fro(s_got[s], ref["S"])}
        assert errs["y"] <= 1e-4 and errs["S"] <= 1e-4, (s, fmt(errs))


def test_varlen_serving_mix_full_size_sampled():
    """20 sequences, lengths floor(exp(U(ln 500, ln 30000))) (~144K tokens), pool of
    1024 slots; checked on 3 sequences (the longest, the shortest, one more) x 4 heads."""
    wl = synth.WORKLOADS["serving"]
    rl = synth.rng_for(wl.seed, 999)
    lens = synth.log_uniform_lengths(rl, 20, 500, 30000)
    geom, act, r, p, tok = make_case("serving", 3, sum(lens))
    cfg = config(geom, act)
    n_slots = 1024
    S = synth.make_state(geom, n_slots, r, std=0.1)
    CS = synth.make_conv_state(geom, n_slots, r, act, std=0.1)
    slots = r.permutation(n_slots)[:20].astype(np.int32)
    cu, y, s_got, c_got = run_varlen(cfg, p, tok, lens, slots, None, S, CS)
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 7})
    heads = sample_heads(geom.n_v_heads, 4, seed=2)
    check_seqs(geom, act, p, tok, cu, y, s_got, c_got, slots, None, S, CS, seqs, heads=heads)
    assert np.all(np.isfinite(y))
