"""Pins of the fp64 CPU oracle against things other than itself.

Each pin is a function ``pin_*(mutant) -> None`` that raises AssertionError on
a mismatch.  With ``mutant=0`` every pin must pass; ``test_every_mutant_is_caught``
plants each known mistake in the oracle (on the CPU) and checks that at least one
pin fails, so the pins are shown to be sensitive to dropped terms, wrong signs,
wrong operands and wrong indices.

Sources of the pinned facts:
* closed forms of the gated delta rule S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T)
  + beta_t v_t k_t^T, o_t = S_t q_t (the mechanism of "Hybrid transformers under
  load: where Gated DeltaNet loses to full attention", section 3: a gate that
  partly erases the state and a delta-rule corrective write);
* textbook routines (torch conv1d, softplus, sigmoid, SiLU, np.linalg.norm);
* exact byte counts printed on the pages (tests/golden/state_geometry.txt).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import GATES_DIRECT, NO_L2NORM, NO_OUTNORM, RAW_QKV
from oracle import chunk_form, twin
from hybrid_gated_deltanet_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "state_geometry.txt")
DIRECT = RAW_QKV | NO_L2NORM | GATES_DIRECT | NO_OUTNORM


def _rng(s):
    return np.random.Generator(np.random.PCG64(1000 + s))


def _unit_rows(r, n, d):
    m = r.standard_normal((n, d))
    return m / np.linalg.norm(m, axis=1, keepdims=True)


def _direct_inputs(geom, q, k, v):
    """x = [q | k | v] for the RAW_QKV mode (q, k per k-head; v per v-head)."""
    T = q.shape[0]
    return np.concatenate([q.reshape(T, -1), k.reshape(T, -1), v.reshape(T, -1)], axis=1)


def _dummy_params(geom):
    return dict(conv_w=np.zeros((geom.conv_channels, geom.d_conv)), A_log=np.zeros(geom.n_v_heads),
                norm_w=np.ones(geom.d_v))


# -----------------------------------------------------------------------------
# pins
# -----------------------------------------------------------------------------
def pin_beta0_pure_decay(mutant=0):
    """beta = 0: S_T = exp(sum g) S0 and o_t = exp(gamma_t) S0 q_t (no write ever)."""
    geom = synth.Geometry(2, 4, 8, 8, 4)
    r = _rng(1)
    T = 12
    q = r.standard_normal((T, 2, 8)); k = r.standard_normal((T, 2, 8)); v = r.standard_normal((T, 4, 8))
    g = -r.uniform(0.0, 0.5, (T, 4)); beta = np.zeros((T, 4))
    s0 = r.standard_normal((4, 8, 8))
    out = oracle.run_sequence(geom, _direct_inputs(geom, q, k, v), np.zeros((T, 32)), g, beta,
                              s0=s0, flags=DIRECT, mutant=mutant, **_dummy_params(geom))
    gam = np.cumsum(g, axis=0)
    for j in range(4):
        np.testing.assert_allclose(out["S"][j], math.exp(gam[-1, j]) * s0[j], rtol=1e-12, atol=1e-14)
        for t in range(T):
            o = math.exp(gam[t, j]) * s0[j] @ q[t, j // 2]
            np.testing.assert_allclose(out["y"][t, j * 8:(j + 1) * 8], o, rtol=1e-11, atol=1e-13)


def pin_orthonormal_retrieval(mutant=0):
    """alpha = 1, beta = 1, orthonormal keys: S_T k_i = v_i exactly and
    S_t = S0 (I - sum_{i<=t} k_i k_i^T) + sum_{i<=t} v_i k_i^T."""
    geom = synth.Geometry(1, 2, 16, 16, 4)
    r = _rng(2)
    T = 10
    kk = synth.orthonormal_rows(r, T, 16)
    k = kk[:, None, :]
    q = r.standard_normal((T, 1, 16))
    v = r.standard_normal((T, 2, 16))
    s0 = r.standard_normal((2, 16, 16))
    out = oracle.run_sequence(geom, _direct_inputs(geom, q, k, v), np.zeros((T, 32)), np.zeros((T, 2)),
                              np.ones((T, 2)), s0=s0, flags=DIRECT, mutant=mutant, **_dummy_params(geom))
    for j in range(2):
        for i in range(T):
            np.testing.assert_allclose(out["S"][j] @ kk[i], v[i, j], rtol=0, atol=1e-12)
        P = np.zeros((16, 16)); Acc = np.zeros((16, 16))
        for t in range(T):
            P += np.outer(kk[t], kk[t]); Acc += np.outer(v[t, j], kk[t])
            St = s0[j] @ (np.eye(16) - P) + Acc
            np.testing.assert_allclose(out["y"][t, j * 16:(j + 1) * 16], St @ q[t, 0], rtol=0, atol=1e-11)


def _brute_force_states(s0, k, v, alpha, beta):
    """S_t = S0 prod_{s<=t} alpha_s (I - beta_s k_s k_s^T)
           + sum_{i<=t} beta_i v_i k_i^T prod_{i<s<=t} alpha_s (I - beta_s k_s k_s^T),
    built from explicit matrix products (no recurrence)."""
    T, d = k.shape
    E = [alpha[s] * (np.eye(d) - beta[s] * np.outer(k[s], k[s])) for s in range(T)]
    states = []
    for t in range(T):
        M = np.eye(d)
        for s in range(t + 1):
            M = M @ E[s]
        St = s0 @ M
        for i in range(t + 1):
            R = np.eye(d)
            for s in range(i + 1, t + 1):
                R = R @ E[s]
            St = St + beta[i] * np.outer(v[i], k[i]) @ R
        states.append(St)
    return states


def pin_brute_force_small(mutant=0):
    """T <= 8 tokens: the oracle equals the explicit product expansion, with and
    without an initial state, for every v-head of a 2 -> 4 GVA geometry."""
    geom = synth.Geometry(2, 4, 6, 5, 4)
    r = _rng(3)
    for T, zero_init in ((8, True), (7, False), (1, False)):
        q = r.standard_normal((T, 2, 6)); k = _unit_rows(r, T * 2, 6).reshape(T, 2, 6)
        v = r.standard_normal((T, 4, 5))
        g = -r.uniform(0.05, 1.5, (T, 4)); beta = r.uniform(0.0, 1.0, (T, 4))
        s0 = np.zeros((4, 5, 6)) if zero_init else r.standard_normal((4, 5, 6))
        out = oracle.run_sequence(geom, _direct_inputs(geom, q, k, v), np.zeros((T, 20)), g, beta,
                                  s0=None if zero_init else s0, flags=DIRECT, mutant=mutant,
                                  **_dummy_params(geom))
        for j in range(4):
            h = j // 2
            states = _brute_force_states(s0[j], k[:, h], v[:, j], np.exp(g[:, j]), beta[:, j])
            np.testing.assert_allclose(out["S"][j], states[-1], rtol=1e-11, atol=1e-12)
            for t in range(T):
                np.testing.assert_allclose(out["y"][t, j * 5:(j + 1) * 5], states[t] @ q[t, h],
                                           rtol=1e-10, atol=1e-12)


def pin_conv_textbook(mutant=0):
    """conv + SiLU equals torch's grouped conv1d (fp64) followed by SiLU, with the
    conv state as left context; the stored conv state is the last d_conv-1 raw
    inputs; and the oracle's per-head path consumes exactly those activations."""
    geom = synth.Geometry(2, 2, 8, 8, 4)
    r = _rng(4)
    T, C = 9, geom.conv_channels
    x = r.standard_normal((T, C)); w = r.uniform(-0.5, 0.5, (C, 4)); bias = r.standard_normal(C)
    conv0 = r.standard_normal((3, C))
    xt = torch.from_numpy(np.concatenate([conv0, x]).T[None].copy())
    ref = torch.nn.functional.conv1d(xt, torch.from_numpy(w[:, None, :].copy()), torch.from_numpy(bias),
                                     groups=C)[0].T
    ref = torch.nn.functional.silu(ref).numpy()
    u = oracle.conv_silu(geom, x, w, conv0=conv0, conv_b=bias, mutant=mutant)
    np.testing.assert_allclose(u, ref, rtol=1e-12, atol=1e-13)
    fin = oracle.conv_final(geom, x, conv0=conv0, mutant=mutant)
    np.testing.assert_array_equal(fin, x[-3:])
    fin2 = oracle.conv_final(geom, x[:2], conv0=conv0, mutant=mutant)  # T < d_conv - 1
    np.testing.assert_array_equal(fin2, np.concatenate([conv0[2:], x[:2]]))
    # per-head path: beta = 0, alpha = 1 => o_t = S0 q_t with q_t = the conv activations
    s0 = r.standard_normal((2, 8, 8))
    out = oracle.run_sequence(geom, x, np.zeros((T, 16)), np.zeros((T, 2)), np.zeros((T, 2)), conv_w=w,
                              A_log=np.zeros(2), norm_w=np.ones(8), conv0=conv0, conv_b=bias, s0=s0,
                              flags=NO_L2NORM | GATES_DIRECT | NO_OUTNORM, mutant=mutant)
    for j in range(2):
        np.testing.assert_allclose(out["y"][:, j * 8:(j + 1) * 8], ref[:, j * 8:(j + 1) * 8] @ s0[j].T,
                                   rtol=1e-11, atol=1e-12)


def pin_gates_special_values(mutant=0):
    """alpha = exp(-exp(A_log) softplus(a)), beta = sigmoid(b): a = 0, A_log = 0 gives
    alpha = 1/2 exactly; a = ln(e - 1) gives softplus = 1; b = 0 gives beta = 1/2.
    Checked through the state: with v = 0 and k = 0 the state only decays."""
    geom = synth.Geometry(1, 3, 4, 4, 4)
    T = 3
    a = np.array([[0.0, math.log(math.e - 1.0), -2.0]] * T)
    A_log = np.array([0.0, math.log(3.0), 0.7])
    b = np.zeros((T, 3))
    s0 = np.ones((3, 4, 4))
    x = np.zeros((T, geom.conv_channels))
    out = oracle.run_sequence(geom, x, np.zeros((T, 12)), a, b, conv_w=np.zeros((geom.conv_channels, 4)),
                              A_log=A_log, norm_w=np.ones(4), s0=s0, flags=RAW_QKV | NO_OUTNORM,
                              mutant=mutant)
    sp = torch.nn.functional.softplus(torch.tensor(-2.0, dtype=torch.float64)).item()
    expect = [0.5 ** T, math.exp(-3.0 * T), math.exp(-math.exp(0.7) * sp * T)]
    for j in range(3):
        np.testing.assert_allclose(out["S"][j], expect[j] * s0[j], rtol=1e-12)
    # beta through a write: one token, S0 = 0, k unit, v = 1, alpha = 1/2  =>  S = beta v k^T
    x = np.zeros((1, geom.conv_channels))
    x[0, 4:8] = [1.0, 0.0, 0.0, 0.0]            # k of k-head 0
    x[0, 8:20] = 1.0                             # v of the three v-heads
    b1 = np.array([[0.0, 1.3, -0.4]])
    out = oracle.run_sequence(geom, x, np.zeros((1, 12)), np.zeros((1, 3)), b1,
                              conv_w=np.zeros((geom.conv_channels, 4)), A_log=np.zeros(3),
                              norm_w=np.ones(4), flags=RAW_QKV | NO_L2NORM | NO_OUTNORM, mutant=mutant)
    sig = torch.sigmoid(torch.from_numpy(b1[0])).numpy()
    for j in range(3):
        np.testing.assert_allclose(out["S"][j][:, 0], sig[j] * np.ones(4), rtol=1e-13)
        np.testing.assert_allclose(out["S"][j][:, 1:], 0.0, atol=0)


def pin_norms_special_values(mutant=0):
    """L2 norm: q = (3, 4, 0, 0) -> (0.6, 0.8, 0, 0) with eps 0; RMSNorm of a constant
    vector c 1 is sign(c) 1, so y = norm_w sign(c) silu(z); and against
    np.linalg.norm on random vectors."""
    geom = synth.Geometry(1, 1, 4, 4, 4)
    # o = S0 q^ with S0 rows = c e_1 and q^ = (0.6, 0.8, 0, 0) => o = 0.6 c 1
    c = -2.5
    s0 = np.zeros((1, 4, 4)); s0[0, :, 0] = c
    x = np.zeros((1, geom.conv_channels)); x[0, 0:4] = [3.0, 4.0, 0.0, 0.0]; x[0, 4:8] = [0, 0, 1.0, 0]
    z = np.array([[0.3, -1.2, 2.0, 0.0]])
    norm_w = np.array([1.0, 0.5, -2.0, 3.0])
    out = oracle.run_sequence(geom, x, z, np.zeros((1, 1)), np.zeros((1, 1)), conv_w=np.zeros((12, 4)),
                              A_log=np.zeros(1), norm_w=norm_w, s0=s0, l2_eps=0.0, norm_eps=0.0,
                              flags=RAW_QKV | GATES_DIRECT, mutant=mutant)
    silu_z = torch.nn.functional.silu(torch.from_numpy(z[0])).numpy()
    np.testing.assert_allclose(out["y"][0], norm_w * np.sign(c) * silu_z, rtol=1e-14, atol=1e-15)
    # random vectors against the library norm; q_scale applied after normalising
    geom = synth.Geometry(1, 1, 8, 8, 4)
    r = _rng(5)
    x = r.standard_normal((1, geom.conv_channels)); s0 = r.standard_normal((1, 8, 8)); z = r.standard_normal((1, 8))
    out = oracle.run_sequence(geom, x, z, np.zeros((1, 1)), np.zeros((1, 1)), conv_w=np.zeros((24, 4)),
                              A_log=np.zeros(1), norm_w=np.ones(8), s0=s0, q_scale=0.25, l2_eps=0.0,
                              norm_eps=0.0, flags=RAW_QKV | GATES_DIRECT, mutant=mutant)
    qh = 0.25 * x[0, :8] / np.linalg.norm(x[0, :8])
    o = s0[0] @ qh
    rms = np.linalg.norm(o) / math.sqrt(8)
    np.testing.assert_allclose(out["y"][0], o / rms * torch.nn.functional.silu(torch.from_numpy(z[0])).numpy(),
                               rtol=1e-12)


def pin_linearity(mutant=0):
    """With the gates and keys fixed and no output norm, o and S are linear in (S0, V)."""
    geom = synth.Geometry(1, 2, 6, 6, 4)
    r = _rng(6)
    T = 11
    q = r.standard_normal((T, 1, 6)); k = _unit_rows(r, T, 6)[:, None, :]
    g = -r.uniform(0, 1, (T, 2)); beta = r.uniform(0, 1, (T, 2))
    va, vb = r.standard_normal((T, 2, 6)), r.standard_normal((T, 2, 6))
    sa, sb = r.standard_normal((2, 6, 6)), r.standard_normal((2, 6, 6))

    def run(v, s0):
        return oracle.run_sequence(geom, _direct_inputs(geom, q, k, v), np.zeros((T, 12)), g, beta, s0=s0,
                                   flags=DIRECT, mutant=mutant, **_dummy_params(geom))

    ra, rb, rab = run(va, sa), run(vb, sb), run(va + 2.0 * vb, sa + 2.0 * sb)
    np.testing.assert_allclose(rab["y"], ra["y"] + 2.0 * rb["y"], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(rab["S"], ra["S"] + 2.0 * rb["S"], rtol=1e-10, atol=1e-11)


def pin_contraction_bound(mutant=0):
    """||I - beta k k^T||_2 = 1 for unit k and beta in [0, 1], hence
    ||S_t||_2 <= alpha_t ||S_{t-1}||_2 + beta_t ||v_t||, stepping one token at a time."""
    geom = synth.Geometry(1, 1, 8, 8, 4)
    r = _rng(7)
    S = r.standard_normal((1, 8, 8))
    for t in range(40):
        q = r.standard_normal((1, 1, 8)); k = _unit_rows(r, 1, 8)[:, None, :]; v = r.standard_normal((1, 1, 8))
        g = np.array([[-r.uniform(0, 0.2)]]); beta = np.array([[r.uniform(0.5, 1.0)]])
        out = oracle.run_sequence(geom, _direct_inputs(geom, q, k, v), np.zeros((1, 8)), g, beta, s0=S,
                                  flags=DIRECT, mutant=mutant, **_dummy_params(geom))
        bound = math.exp(g[0, 0]) * np.linalg.norm(S[0], 2) + beta[0, 0] * np.linalg.norm(v[0, 0])
        assert np.linalg.norm(out["S"][0], 2) <= bound * (1 + 1e-12), (t, bound)
        S = out["S"]


def pin_split_invariance(mutant=0):
    """Running T tokens at once equals running T1 then T - T1 with the state and
    the conv state carried; the stored state's size does not depend on T."""
    wl = synth.WORKLOADS["tiny"]
    geom = wl.geom
    r = synth.rng_for(77)
    p = synth.make_params(geom, r, synth.F32)
    tok = synth.make_tokens(geom, 40, r, synth.F32)
    kw = dict(conv_w=p["conv_w"].f64, A_log=p["A_log"].f64, norm_w=p["norm_w"].f64, mutant=mutant)
    full = oracle.run_sequence(geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, **kw)
    T1 = 13
    first = oracle.run_sequence(geom, tok["x"].f64[:T1], tok["z"].f64[:T1], tok["a"].f64[:T1],
                                tok["b"].f64[:T1], **kw)
    second = oracle.run_sequence(geom, tok["x"].f64[T1:], tok["z"].f64[T1:], tok["a"].f64[T1:],
                                 tok["b"].f64[T1:], s0=first["S"], conv0=first["conv"], **kw)
    np.testing.assert_allclose(np.concatenate([first["y"], second["y"]]), full["y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(second["S"], full["S"], rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(second["conv"], full["conv"])
    assert first["S"].shape == full["S"].shape and first["conv"].shape == full["conv"].shape


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split()
                vals[key] = int(val)
    return vals


def pin_golden_geometry(mutant=0):
    """The oracle's stored state at the Qwen3.5-4B geometry is exactly the bytes the
    braintools.ru page prints (32 x 128 x 128 fp32 + 3 bf16 conv rows x 8192 ch),
    and the wide geometry has the Strata ModelGeometry's 10240 conv channels."""
    gold = _golden()
    geom = synth.QWEN35_4B
    x = np.zeros((1, geom.conv_channels))
    out = oracle.run_sequence(geom, x, np.zeros((1, geom.value_dim)), np.zeros((1, 32)), np.zeros((1, 32)),
                              conv_w=np.zeros((geom.conv_channels, 4)), A_log=np.zeros(32),
                              norm_w=np.ones(128), heads=[0], mutant=mutant)
    assert out["S"].size * 4 == gold["qwen35_4b.ssm_state_bytes"]
    assert out["conv"].size * 2 == gold["qwen35_4b.conv_state_bytes"]
    assert out["S"].size * 4 + out["conv"].size * 2 == gold["qwen35_4b.layer_state_bytes"]
    assert round(gold["qwen35_4b.layer_state_bytes"] / 2 ** 20 * 100) == gold["qwen35_4b.state_mib_x100"]
    assert geom.state_bytes_per_slot() == gold["qwen35_4b.ssm_state_bytes"]
    assert geom.conv_state_bytes_per_slot(synth.BF16) == gold["qwen35_4b.conv_state_bytes"]
    w = synth.WIDE_GVA
    assert (w.d_k, w.n_k_heads, w.n_v_heads, w.d_conv) == (gold["wide.ssm_state_size"], gold["wide.n_k_heads"],
                                                           gold["wide.n_v_heads"], gold["wide.d_conv"])
    assert w.conv_channels == gold["wide.conv_channels"] and w.value_dim == gold["wide.value_dim"]
    out = oracle.conv_final(w, np.zeros((5, w.conv_channels)), mutant=mutant)
    assert out.shape == (w.d_conv - 1, gold["wide.conv_channels"])


PINS = [pin_beta0_pure_decay, pin_orthonormal_retrieval, pin_brute_force_small, pin_conv_textbook,
        pin_gates_special_values, pin_norms_special_values, pin_linearity, pin_contraction_bound,
        pin_split_invariance, pin_golden_geometry]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(0)


MUTANTS = {1: "error measured against the undecayed state", 2: "write sign flipped",
           3: "output read before the write", 4: "output reads with k instead of q",
           5: "conv taps reversed", 6: "interleaved GVA groups", 7: "softplus dropped from the gate",
           8: "RMS uses the sum instead of the mean", 9: "silu(z) replaced by z",
           11: "conv state stores activated values"}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: f"m{m}")
def test_every_mutant_is_caught(mutant):
    caught = []
    for pin in PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passes every pin"


# -----------------------------------------------------------------------------
# cross-checks: the numpy twin and the fp64 chunk form against the C oracle
# -----------------------------------------------------------------------------
def _tiny_case(seed, T=64, s0_std=0.0, conv_std=0.0):
    wl = synth.WORKLOADS["tiny"]
    geom = wl.geom
    r = synth.rng_for(wl.seed, seed)
    p = synth.make_params(geom, r, wl.act_dtype)
    tok = synth.make_tokens(geom, T, r, wl.act_dtype)
    s0 = synth.make_state(geom, 1, r, std=s0_std).f64[0] if s0_std else None
    c0 = synth.make_conv_state(geom, 1, r, wl.act_dtype, std=conv_std).f64[0] if conv_std else None
    return geom, p, tok, s0, c0


@pytest.mark.parametrize("q_scale", [1.0, 32 ** -0.5])
def test_twin_matches_c_oracle(q_scale):
    geom, p, tok, s0, c0 = _tiny_case(1, s0_std=0.1, conv_std=0.1)
    args = (geom, tok["x"].f64, tok["z"].f64, tok["a"].f64, tok["b"].f64, p["conv_w"].f64, p["A_log"].f64,
            p["norm_w"].f64)
    a = oracle.run_sequence(*args, s0=s0, conv0=c0, q_scale=q_scale)
    b = twin.run(*args, s0=s0, conv0=c0, q_scale=q_scale)
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(a["S"], b["S"], rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(a["conv"], b["conv"])


@pytest.mark.parametrize("chunk,T", [(1, 20), (16, 64), (16, 45), (64, 150), (64, 64)])
def test_chunk_form_equals_token_form(chunk, T):
    geom = synth.Geometry(2, 4, 16, 16, 4)
    r = _rng(100 + chunk + T)
    q = _unit_rows(r, T * 2, 16).reshape(T, 2, 16)
    k = _unit_rows(r, T * 2, 16).reshape(T, 2, 16)
    v = r.standard_normal((T, 4, 16))
    g = -np.exp(r.uniform(0, math.log(16), 4))[None, :] * np.logaddexp(0, r.standard_normal((T, 4)))
    beta = 1 / (1 + np.exp(-r.standard_normal((T, 4))))
    s0 = 0.1 * r.standard_normal((4, 16, 16))
    ref = oracle.run_sequence(geom, _direct_inputs(geom, q, k, v), np.zeros((T, 64)), g, beta, s0=s0,
                              flags=DIRECT, **_dummy_params(geom))
    for j in range(4):
        o, S = chunk_form.run_head(q[:, j // 2], k[:, j // 2], v[:, j], g[:, j], beta[:, j], s0[j], chunk)
        np.testing.assert_allclose(o, ref["y"][:, j * 16:(j + 1) * 16], rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(S, ref["S"][j], rtol=1e-10, atol=1e-11)


def test_padding_rows_leave_state_unchanged():
    """q = k = v = 0, beta = 0, g = 0 rows are exact no-ops on the state."""
    geom = synth.Geometry(1, 1, 8, 8, 4)
    r = _rng(9)
    s0 = r.standard_normal((1, 8, 8))
    T = 5
    out = oracle.run_sequence(geom, np.zeros((T, 24)), np.zeros((T, 8)), np.zeros((T, 1)), np.zeros((T, 1)),
                              s0=s0, flags=DIRECT, **_dummy_params(geom))
    np.testing.assert_array_equal(out["S"], s0)


def test_gate_underflow_is_benign():
    """alpha down to e^-49 (the configs' extreme) gives finite states and outputs."""
    geom = synth.Geometry(1, 1, 8, 8, 4)
    r = _rng(10)
    T = 16
    x = r.standard_normal((T, 24))
    out = oracle.run_sequence(geom, x, r.standard_normal((T, 8)), np.full((T, 1), 3.0), np.zeros((T, 1)),
                              conv_w=r.uniform(-.5, .5, (24, 4)), A_log=np.full(1, math.log(16.0)),
                              norm_w=np.ones(8), s0=r.standard_normal((1, 8, 8)))
    assert np.all(np.isfinite(out["y"])) and np.all(np.isfinite(out["S"]))
