"""The per-v-head slicing that the full-length wide-geometry test feeds the oracle:
v-head j evaluated as a layer of 1 k-head and 1 v-head on its own channels must equal
v-head j of the full layer (the recurrence of a v-head reads only its k-head's q and k
and its own v, z, a and b)."""
import numpy as np

import oracle
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import oracle_kwargs
from test_workload_wide_full_length import _head_inputs


def test_one_head_layer_equals_the_full_layer_head():
    wl = synth.WORKLOADS["wide"]
    geom = wl.geom
    sub = synth.Geometry(1, 1, geom.d_k, geom.d_v, geom.d_conv)
    rng = synth.rng_for(wl.seed, 99)
    p = synth.make_params(geom, rng, wl.act_dtype)
    tok = synth.make_tokens(geom, 12, rng, wl.act_dtype)
    heads = [0, 20, 47]  # first, middle and last k-head groups (G = 3)
    full = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, heads=heads,
                               **oracle_kwargs(p))
    D = geom.d_v
    for j in heads:
        x, z, a, b, kw = _head_inputs(geom, p, tok, j, slice(0, 12))
        one = oracle.run_sequence(sub, x, z, a, b, **kw)
        np.testing.assert_allclose(one["y"], full["y"][:, j * D:(j + 1) * D], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(one["S"][0], full["S"][j], rtol=1e-12, atol=1e-12)
