"""Pure-numpy token loop -- TEST INFRASTRUCTURE (small cases only).

An independent second implementation of the token-by-token layer, written
vectorised over heads with numpy, sharing no code with ``gdn_oracle.c``.  It
exists to cross-check the C oracle on tiny inputs (agreement to ~1e-12); the
oracle's own pins are the closed forms in ``tests/test_oracle_pins.py``.

The layer (gated delta rule with GVA, conv + SiLU, L2-normalised q/k, gated
RMSNorm) is the one described on "Hybrid transformers under load: where Gated
DeltaNet loses to full attention" (braintools.ru), section 3, with the geometry
of its section 4.1 and of Strata chapter 6, section 6.2.
"""
from __future__ import annotations

import numpy as np

from . import GATES_DIRECT, NO_L2NORM, NO_OUTNORM, RAW_QKV


def _silu(x):
    return x / (1.0 + np.exp(-x))


def run(geom, x, z, a, b, conv_w, A_log, norm_w, s0=None, conv0=None, conv_b=None, dt_bias=None,
        q_scale=1.0, l2_eps=1e-6, norm_eps=1e-6, flags=0):
    x = np.asarray(x, np.float64)
    T, C = x.shape
    K = geom.d_conv
    Hk, Hv, dk, dv = geom.n_k_heads, geom.n_v_heads, geom.d_k, geom.d_v
    G = Hv // Hk
    hist = np.zeros((K - 1, C)) if conv0 is None else np.asarray(conv0, np.float64)
    padded = np.concatenate([hist, x], axis=0)
    if flags & RAW_QKV:
        u = x.copy()
    else:
        w = np.asarray(conv_w, np.float64)
        c = np.zeros((T, C)) if conv_b is None else np.tile(np.asarray(conv_b, np.float64), (T, 1))
        for tap in range(K):
            c = c + padded[tap:tap + T] * w[:, tap][None, :]
        u = _silu(c)
    q = u[:, :Hk * dk].reshape(T, Hk, dk)
    k = u[:, Hk * dk:2 * Hk * dk].reshape(T, Hk, dk)
    v = u[:, 2 * Hk * dk:].reshape(T, Hv, dv)
    if flags & NO_L2NORM:
        q = q * q_scale
    else:
        q = q * (q_scale / np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + l2_eps))
        k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True) + l2_eps)
    # contiguous GVA groups: v-head j reads k-head j // G
    qh = np.repeat(q, G, axis=1)
    kh = np.repeat(k, G, axis=1)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if flags & GATES_DIRECT:
        g, beta = a, b
    else:
        dt = 0.0 if dt_bias is None else np.asarray(dt_bias, np.float64)[None, :]
        g = -np.exp(np.asarray(A_log, np.float64))[None, :] * np.logaddexp(0.0, a + dt)
        beta = 1.0 / (1.0 + np.exp(-b))
    alpha = np.exp(g)
    S = np.zeros((Hv, dv, dk)) if s0 is None else np.array(s0, np.float64, copy=True)
    o = np.empty((T, Hv, dv))
    for t in range(T):
        S = S * alpha[t][:, None, None]
        err = v[t] - np.einsum("jik,jk->ji", S, kh[t])
        S = S + beta[t][:, None, None] * err[:, :, None] * kh[t][:, None, :]
        o[t] = np.einsum("jik,jk->ji", S, qh[t])
    if flags & NO_OUTNORM:
        y = o
    else:
        zz = np.asarray(z, np.float64).reshape(T, Hv, dv)
        rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + norm_eps)
        y = np.asarray(norm_w, np.float64)[None, None, :] * (o / rms) * _silu(zz)
    conv = padded[T:T + K - 1].copy() if T >= 0 else None
    return {"y": y.reshape(T, Hv * dv), "S": S, "conv": conv}
