"""Pins of the attention oracle (oracle/attention.py): a brute-force loop with
the softmax written out, the library routine (torch scaled_dot_product_attention
in fp64 on the CPU, key/value heads repeated per group), and closed forms
(one token returns its value; equal keys return the mean of the values; a
dominant score returns its value)."""
import math

import numpy as np
import torch

from oracle import attention as at


def _rng(s):
    return np.random.Generator(np.random.PCG64(2000 + s))


def test_brute_force_loop():
    r = _rng(1)
    Hq, Hkv, D, L = 4, 2, 8, 5
    q, K, V = r.standard_normal((Hq, D)), r.standard_normal((L, Hkv, D)), r.standard_normal((L, Hkv, D))
    got = at.decode_attention(q, K, V, 0.3)
    for h in range(Hq):
        kvh = h // 2
        w = [math.exp(0.3 * sum(q[h, d] * K[t, kvh, d] for d in range(D))) for t in range(L)]
        for d in range(D):
            ref = sum(w[t] * V[t, kvh, d] for t in range(L)) / sum(w)
            assert abs(got[h, d] - ref) <= 1e-12 * (1 + abs(ref))


def test_matches_torch_sdpa():
    r = _rng(2)
    Hq, Hkv, D, L = 12, 2, 16, 37
    q, K, V = r.standard_normal((Hq, D)), r.standard_normal((L, Hkv, D)), r.standard_normal((L, Hkv, D))
    got = at.decode_attention(q, K, V, 1 / math.sqrt(D))
    G = Hq // Hkv
    kq = torch.from_numpy(np.repeat(K.transpose(1, 0, 2), G, axis=0))  # [Hq, L, D]
    vq = torch.from_numpy(np.repeat(V.transpose(1, 0, 2), G, axis=0))
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], kq, vq)[:, 0, :]
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_closed_forms():
    r = _rng(3)
    D = 8
    q, k, v = r.standard_normal((2, D)), r.standard_normal((1, 1, D)), r.standard_normal((1, 1, D))
    np.testing.assert_allclose(at.decode_attention(q, k, v, 0.5), np.repeat(v[0], 2, axis=0), rtol=1e-14)
    K = np.repeat(r.standard_normal((1, 1, D)), 6, axis=0)
    V = r.standard_normal((6, 1, D))
    np.testing.assert_allclose(at.decode_attention(q, K, V, 0.5), np.repeat(V.mean(axis=0), 2, axis=0), rtol=1e-12)
    K = np.zeros((6, 1, D))
    K[4, 0, 0] = 1.0
    q1 = np.zeros((1, D))
    q1[0, 0] = 800.0
    np.testing.assert_allclose(at.decode_attention(q1, K, V, 1.0), V[4], rtol=1e-12)


def test_group_mapping_is_contiguous():
    """G = 2: query heads 0, 1 read kv-head 0 and heads 2, 3 read kv-head 1."""
    r = _rng(4)
    D, L = 8, 3
    qh = r.standard_normal(D)
    q = np.stack([qh] * 4)
    K, V = r.standard_normal((L, 2, D)), r.standard_normal((L, 2, D))
    o = at.decode_attention(q, K, V, 1.0)
    np.testing.assert_allclose(o[0], o[1])
    np.testing.assert_allclose(o[2], o[3])
    assert not np.allclose(o[1], o[2])
    np.testing.assert_allclose(o[1], at.decode_attention(qh[None], K[:, :1], V[:, :1], 1.0)[0])


def test_prefill_matches_torch_sdpa_with_bottom_right_mask():
    """The chunk form against torch SDPA with an explicit mask: new token i (after
    ctx cached tokens) sees keys 0 .. ctx + i."""
    r = _rng(5)
    Hq, Hkv, D, ctx, n = 8, 2, 16, 7, 5
    q = r.standard_normal((n, Hq, D))
    K, V = r.standard_normal((ctx + n, Hkv, D)), r.standard_normal((ctx + n, Hkv, D))
    got = at.prefill_attention(q, K, V, ctx, 0.25)
    G = Hq // Hkv
    kq = torch.from_numpy(np.repeat(K.transpose(1, 0, 2), G, axis=0))
    vq = torch.from_numpy(np.repeat(V.transpose(1, 0, 2), G, axis=0))
    mask = torch.from_numpy(np.arange(ctx + n)[None, :] <= ctx + np.arange(n)[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q.transpose(1, 0, 2)), kq, vq,
                                                           attn_mask=mask, scale=0.25)
    np.testing.assert_allclose(got, ref.numpy().transpose(1, 0, 2), rtol=1e-12, atol=1e-12)
