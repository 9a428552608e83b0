"""Shared helpers for the GPU parity tests: the same seeded inputs go to the
CUDA path (as device tensors in their storage dtype) and to the oracle (as the
exactly decoded fp64 values)."""
from __future__ import annotations

import numpy as np
import torch

from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth

# tolerances stated for the layer: relative Frobenius error against the fp64 oracle
TOL_F32 = {"y": 1e-4, "S": 1e-4}
TOL_BF16 = {"y": 2e-2, "S": 1e-3}


def tol_for(act_dtype):
    return TOL_F32 if act_dtype == synth.F32 else TOL_BF16


def rel_fro(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def dev(stored: synth.Stored, device="cuda") -> torch.Tensor:
    if stored.dtype == synth.BF16:
        return torch.from_numpy(np.ascontiguousarray(stored.raw).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(stored.raw)).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def config(geom: synth.Geometry, act_dtype: str, chunk=64, q_scale=1.0, flags=0, l2_eps=1e-6, norm_eps=1e-6):
    return gb.Config(geom.n_k_heads, geom.n_v_heads, geom.d_k, geom.d_v, geom.d_conv, chunk,
                     gb.BF16 if act_dtype == synth.BF16 else gb.F32, q_scale, l2_eps, norm_eps, flags)


def params_dev(p, device="cuda"):
    return gb.Params(conv_w=dev(p["conv_w"], device), A_log=dev(p["A_log"], device), norm_w=dev(p["norm_w"], device))


def oracle_kwargs(p):
    return dict(conv_w=p["conv_w"].f64, A_log=p["A_log"].f64, norm_w=p["norm_w"].f64)


def act_empty(cfg: gb.Config, *shape, device="cuda"):
    return torch.empty(*shape, dtype=cfg.torch_dtype, device=device)


def make_case(wl_name: str, stream: int, n_tok: int, act_dtype=None, geom=None):
    wl = synth.WORKLOADS[wl_name]
    geom = geom or wl.geom
    act = act_dtype or wl.act_dtype
    r = synth.rng_for(wl.seed, stream)
    p = synth.make_params(geom, r, act)
    tok = synth.make_tokens(geom, n_tok, r, act)
    return geom, act, r, p, tok


def sample_heads(Hv: int, n: int, seed: int = 0):
    if n >= Hv:
        return list(range(Hv))
    rs = np.random.Generator(np.random.PCG64(seed))
    return sorted(set([0, Hv - 1] + list(rs.choice(Hv, n - 2, replace=False))))


def head_cols(heads, dv):
    return np.concatenate([np.arange(j * dv, (j + 1) * dv) for j in heads])


def fmt(errs):
    return ", ".join(f"{k}={v:.2e}" for k, v in errs.items())


def isclose_tol(errs, tol):
    return all(errs[k] <= tol[k.split(":")[0]] for k in errs)

