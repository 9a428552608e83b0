"""Chunkwise (WY / UT-transform) evaluation in fp64 -- TEST INFRASTRUCTURE.

The secondary CPU reference: it evaluates the gated delta rule a chunk of C
tokens at a time, using the exact reformulation that the prefill kernels use,
so that the algebra is pinned against the token-by-token oracle before any
kernel exists.  The pages state the recurrence only in words ("Hybrid
transformers under load ...", braintools.ru, section 3) and name a chunked
prefill kernel without its algebra ("Forge: how I wrote my own inference
engine", entry of 25 August); the derivation below is ours.

Derivation (per v-head, inside one chunk, S0 the state entering it):
  b_t = prod_{s<=t} alpha_s = exp(gamma_t), gamma_t = sum_{s<=t} g_s.
  With u_t = beta_t (v_t - alpha_t S_{t-1} k_t) the recurrence reads
  S_t = alpha_t S_{t-1} + u_t k_t^T, hence by induction
      S_t = b_t S0 + sum_{i<=t} (b_t / b_i) u_i k_i^T.
  Substituting into u_t gives, in matrix form over the chunk rows,
      (I + A) U = diag(beta) V - diag(beta b) K S0^T,
      A_ti = beta_t exp(gamma_t - gamma_i) k_t.k_i  for i < t (else 0).
  So with T = (I + A)^{-1}:  W = T diag(beta b) K,  U~ = T diag(beta) V,
      U   = U~ - W S0^T
      O   = diag(b) Q S0^T + (Q K^T o Gamma o M_incl) U
      S_C = b_C S0 + U^T diag(exp(gamma_C - gamma)) K
  where Gamma_ti = exp(gamma_t - gamma_i) and M_incl keeps i <= t.
Only exponents gamma_t - gamma_i with i <= t (never positive) are evaluated.
Tail chunks are padded with q = k = v = 0, beta = 0, g = 0 rows, which leave
the state unchanged exactly.
"""
from __future__ import annotations

import numpy as np


def run_head(q, k, v, g, beta, s0, chunk):
    """One v-head: q, k [T, d_k] (already normalised/scaled), v [T, d_v], g, beta [T].

    Returns (o [T, d_v], S_final [d_v, d_k]).
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if s0 is None else np.array(s0, np.float64, copy=True)
    out = np.empty((T, dv))
    C = int(chunk)
    lower_strict = np.tril(np.ones((C, C), dtype=bool), -1)
    lower_incl = np.tril(np.ones((C, C), dtype=bool), 0)
    for start in range(0, T, C):
        n = min(C, T - start)
        Qc = np.zeros((C, dk)); Qc[:n] = q[start:start + n]
        Kc = np.zeros((C, dk)); Kc[:n] = k[start:start + n]
        Vc = np.zeros((C, dv)); Vc[:n] = v[start:start + n]
        gc = np.zeros(C); gc[:n] = g[start:start + n]
        bc = np.zeros(C); bc[:n] = beta[start:start + n]
        gam = np.cumsum(gc)
        diff = gam[:, None] - gam[None, :]
        Gam = np.where(lower_incl, np.exp(np.where(lower_incl, diff, 0.0)), 0.0)
        A = np.where(lower_strict, bc[:, None] * Gam * (Kc @ Kc.T), 0.0)
        Tm = np.linalg.solve(np.eye(C) + A, np.eye(C))
        eg = np.exp(gam)
        W = Tm @ ((bc * eg)[:, None] * Kc)
        Ut = Tm @ (bc[:, None] * Vc)
        U = Ut - W @ S.T
        P = np.where(lower_incl, (Qc @ Kc.T) * Gam, 0.0)
        O = eg[:, None] * (Qc @ S.T) + P @ U
        out[start:start + n] = O[:n]
        S = eg[-1] * S + U.T @ (np.exp(gam[-1] - gam)[:, None] * Kc)
    return out, S
