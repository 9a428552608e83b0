"""fp64 projections either side of the layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this module; the product path never imports it.

The layer sits between two dense projections of the model's hidden states
("Forge: how I wrote my own inference engine and overtook llama.cpp",
24 August: the matrix projections take 59% of its hybrid prefill; its opening
formulas: decode time is the weight bytes read per token over the memory
bandwidth):

* in-projection: u = h W_in^T, u = [x | z | a | b] (rows of W_in in that order:
  the C_ch conv-input channels, the H_v*d_v gate channels z, H_v values a, H_v
  values b);
* out-projection: out = y W_out^T.

Reading taken where the pages are silent: the layer's inputs and outputs are
stored in bf16 between the steps (the pages' configurations feed the layer
bf16 x and z and return bf16 y), so u and y are rounded to bf16 (round to
nearest even) before the next step consumes them.  Everything else is fp64.
"""
from __future__ import annotations

from typing import Dict

import numpy as np

from . import run_sequence


def project(act, w) -> np.ndarray:
    """out[t, n] = sum_k act[t, k] w[n, k] in fp64 (w in the nn.Linear layout
    [n_out, k]); the matrix product is the library primitive."""
    return np.asarray(act, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T


def round_bf16(v) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even (bf16 keeps the top 16 bits
    of the fp32 pattern), returned as fp64.  Values are first rounded to fp32;
    for the sums here that double rounding is below the comparison tolerances."""
    f = np.ascontiguousarray(np.asarray(v, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (((u + 0x7FFF + lsb) >> 16) << 16).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def split_in(geom, u: np.ndarray):
    """[x | z | a | b] column blocks of the in-projection output."""
    C, V, H = geom.conv_channels, geom.n_v_heads * geom.d_v, geom.n_v_heads
    return u[:, :C], u[:, C:C + V], u[:, C + V:C + V + H], u[:, C + V + H:C + V + 2 * H]


def layer_sequence(geom, h, w_in, w_out, conv_w, A_log, norm_w, **kw) -> Dict[str, np.ndarray]:
    """One sequence through in-projection, the layer (the token-by-token oracle)
    and out-projection.  ``kw`` goes to ``run_sequence`` (s0, conv0, heads, ...).
    Returns out [T, hidden] (fp64 product of the bf16 y), y, S, conv and the
    layer inputs x, z, a, b (bf16 values)."""
    u = round_bf16(project(h, w_in))
    x, z, a, b = (np.ascontiguousarray(p) for p in split_in(geom, u))
    ref = run_sequence(geom, x, z, a, b, conv_w, A_log, norm_w, **kw)
    y16 = round_bf16(ref["y"])
    return {"out": project(y16, w_out), "y": ref["y"], "S": ref["S"], "conv": ref["conv"],
            "x": x, "z": z, "a": a, "b": b}
