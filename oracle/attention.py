"""fp64 decode attention of the hybrid's full-attention layers -- TEST
INFRASTRUCTURE (only tests/, smoke() and bench.py's CPU leg use it).

Grouped-query attention for one new token per sequence ("Forge: how I wrote
my own inference engine and overtook llama.cpp", architecture section: the
hybrid's non-DeltaNet layers are ordinary GQA attention with a KV cache, 4
kv-heads of 256 dims): query head h reads kv-head floor(h / G),
G = n_q_heads / n_kv_heads (contiguous groups; the pages do not spell the
mapping out, this is the reading taken), and

    o_h = sum_t softmax_t(scale q_h . k_t) v_t

over all tokens of the sequence, the new one included (it is the last row of
K and V here).  The paging of the cache is storage, not arithmetic: the
oracle takes each sequence's K and V in token order.
"""
from __future__ import annotations

import numpy as np


def decode_attention(q, K, V, scale: float) -> np.ndarray:
    """q [Hq, D]; K, V [L, Hkv, D] (tokens in order, L >= 1).  Returns o [Hq, D]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq, Hkv = q.shape[0], K.shape[1]
    G = Hq // Hkv
    o = np.empty_like(q)
    for h in range(Hq):
        kvh = h // G
        s = scale * (K[:, kvh, :] @ q[h])
        p = np.exp(s - s.max())
        o[h] = (p @ V[:, kvh, :]) / p.sum()
    return o


def prefill_attention(q, K, V, ctx_len: int, scale: float) -> np.ndarray:
    """Chunk of n new tokens after ctx_len cached ones: q [n, Hq, D]; K, V [ctx_len + n,
    Hkv, D] (all tokens of the sequence in order).  New token i sits at position
    ctx_len + i and attends to positions 0 .. ctx_len + i.  Returns o [n, Hq, D]."""
    q = np.asarray(q, dtype=np.float64)
    return np.stack([decode_attention(q[i], K[:ctx_len + i + 1], V[:ctx_len + i + 1], scale)
                     for i in range(q.shape[0])])
