"""Pins of the oracle's projections (oracle/projections.py) against things
other than themselves: a brute-force triple loop for the product and its
orientation, exact bf16 rounding cases and torch's CPU bf16 cast, and the
layer composition reduced by identity projections to the pinned layer oracle."""
import numpy as np
import torch

import oracle
from oracle import projections as pj
from hybrid_gated_deltanet_gb300 import synth


def test_project_equals_brute_force_loop():
    r = np.random.Generator(np.random.PCG64(7))
    act = r.standard_normal((3, 5))
    w = r.standard_normal((4, 5))
    got = pj.project(act, w)
    assert got.shape == (3, 4)
    for t in range(3):
        for n in range(4):
            ref = 0.0
            for k in range(5):
                ref += act[t, k] * w[n, k]
            assert abs(got[t, n] - ref) <= 1e-13 * (1 + abs(ref))


def test_round_bf16_exact_cases():
    u = 2.0 ** -7  # bf16 spacing on [1, 2)
    cases = {1.0: 1.0, 1 + u / 2: 1.0, 1 + 3 * u / 2: 1 + 2 * u, 1 + u: 1 + u, 1 + 0.51 * u: 1 + u,
             -(1 + u / 2): -1.0, 3.0: 3.0, 0.0: 0.0, 2.0 ** -130: 2.0 ** -130}
    got = pj.round_bf16(np.array(list(cases)))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))


def test_round_bf16_matches_torch_cast():
    r = np.random.Generator(np.random.PCG64(8))
    v = (r.standard_normal(20000) * np.exp(r.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(pj.round_bf16(v), ref)


def test_identity_projections_reduce_to_the_layer():
    """W_in = I: x, z, a, b are h's column blocks in that order; W_out = [I; 0]:
    out = (bf16 y, 0).  Everything else equals the token-by-token oracle."""
    geom = synth.TINY
    r = synth.rng_for(0, 77)
    n_in = geom.conv_channels + geom.value_dim + 2 * geom.n_v_heads
    T = 9
    h = synth.store(r.standard_normal((T, n_in)), synth.BF16).f64[:]
    p = synth.make_params(geom, r, synth.F32)
    kw = dict(conv_w=p["conv_w"].f64, A_log=p["A_log"].f64, norm_w=p["norm_w"].f64)
    w_out = np.zeros((n_in, geom.value_dim))
    w_out[:geom.value_dim] = np.eye(geom.value_dim)
    got = pj.layer_sequence(geom, h, np.eye(n_in), w_out, **kw)
    C, V, H = geom.conv_channels, geom.value_dim, geom.n_v_heads
    ref = oracle.run_sequence(geom, h[:, :C], h[:, C:C + V], h[:, C + V:C + V + H], h[:, C + V + H:], **kw)
    np.testing.assert_array_equal(got["y"], ref["y"])
    np.testing.assert_array_equal(got["S"], ref["S"])
    np.testing.assert_array_equal(got["out"][:, :V], pj.round_bf16(ref["y"]))
    assert not np.any(got["out"][:, V:])
