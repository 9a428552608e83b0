"""GPU parity of gdn_attn_prefill (a chunk of new tokens per sequence against a
paged KV cache, causal with the mask aligned at the bottom right) against the
fp64 oracle.  The tensor cores take bf16 q, K, V exactly and accumulate in
fp32; P is rounded to bf16 (2^-8 relative per weight, the sum of the weights
uses the same rounded values) and o is rounded to bf16, so the relative
Frobenius error of o is held to 8e-3."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as at
from hybrid_gated_deltanet_gb300 import binding as gb
from hybrid_gated_deltanet_gb300 import synth
from gdn_cases import dev, host, rel_fro

pytestmark = pytest.mark.gpu


def _bf16(r, shape):
    return synth.store(r.standard_normal(shape), synth.BF16)


def run_case(Hq, Hkv, D, page, seqs, seed, holes=()):
    """seqs: (cached tokens, new tokens) per sequence."""
    r = synth.rng_for(61, seed)
    n_seq = len(seqs)
    cfg = gb.AttnConfig(Hq, Hkv, D, page)
    need = [math.ceil((c + n) / page) for c, n in seqs]
    max_pages = max(need)
    n_pages = sum(need) + 2
    perm = r.permutation(n_pages).astype(np.int32)
    table = np.full((n_seq, max_pages), -1, np.int32)
    o0 = 0
    for s, nd in enumerate(need):
        table[s, :nd] = perm[o0:o0 + nd]
        o0 += nd
    for s, pg in holes:
        table[s, pg] = n_pages + 3
    news = [n for _, n in seqs]
    cu = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    N = int(cu[-1])
    ctx = np.asarray([c for c, _ in seqs], np.int32)
    q = _bf16(r, (N, Hq, D))
    kn, vn = _bf16(r, (N, Hkv, D)), _bf16(r, (N, Hkv, D))
    kp, vp = _bf16(r, (n_pages, Hkv, page, D)), _bf16(r, (n_pages, Hkv, page, D))
    kpd, vpd = dev(kp), dev(vp)
    o = torch.full((N, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    gb.gdn_attn_prefill(cfg, dev(q), dev(kn), dev(vn), kpd, vpd, torch.from_numpy(table).cuda(),
                        torch.from_numpy(cu).cuda(), torch.from_numpy(ctx).cuda(), o)
    torch.cuda.synchronize()
    assert gb.gdn_device_status() == 0
    got = host(o)
    kp64, vp64, kn64, vn64, q64 = kp.f64[:], vp.f64[:], kn.f64[:], vn.f64[:], q.f64[:]
    kp_want, vp_want = kp64.copy(), vp64.copy()
    refs = []
    for s, (c, n) in enumerate(seqs):
        rows = slice(int(cu[s]), int(cu[s + 1]))
        Ks, Vs, keep = [], [], []
        for t in range(c + n):
            pid = table[s, t // page]
            inside = 0 <= pid < n_pages
            if t < c:
                Ks.append(kp64[pid, :, t % page] if inside else np.zeros((Hkv, D)))
                Vs.append(vp64[pid, :, t % page] if inside else np.zeros((Hkv, D)))
            else:
                Ks.append(kn64[cu[s] + t - c])
                Vs.append(vn64[cu[s] + t - c])
                if inside:
                    kp_want[pid, :, t % page] = kn64[cu[s] + t - c]
                    vp_want[pid, :, t % page] = vn64[cu[s] + t - c]
            keep.append(inside)
        K, V, keep = np.stack(Ks), np.stack(Vs), np.asarray(keep)
        out = np.empty((n, Hq, D))
        for i in range(n):  # keys on missing pages are left out
            sel = np.nonzero(keep[:c + i + 1])[0]
            out[i] = at.decode_attention(q64[rows][i], K[sel], V[sel], 1 / math.sqrt(D))
        refs.append(out)
    ref = np.concatenate(refs)
    err = rel_fro(got, ref)
    assert err <= 8e-3, err
    np.testing.assert_array_equal(host(kpd), kp_want)
    np.testing.assert_array_equal(host(vpd), vp_want)
    return err


def test_attn_prefill_qwen35_4b_mixed():
    """16 query / 4 kv heads of 256 (32 tokens x 4 heads per 128-row tile), pages of 16:
    fresh prompts, continuations after cached tokens, one token, ragged tails."""
    run_case(16, 4, 256, 16, [(0, 1), (0, 37), (5, 64), (100, 200), (0, 300), (527, 130)], 1)


def test_attn_prefill_wide_gqa_pages_528():
    """24 query / 2 kv heads (10 tokens x 12 heads per tile), pages of 528."""
    run_case(24, 2, 256, 528, [(0, 45), (600, 33), (1000, 130)], 2)


@pytest.mark.parametrize("Hq,Hkv,D,page", [(8, 8, 128, 8), (4, 2, 128, 32), (32, 4, 128, 64)])
def test_attn_prefill_small_groups_and_d128(Hq, Hkv, D, page):
    run_case(Hq, Hkv, D, page, [(0, 20), (70, 150), (3, 1)], 3)


def test_attn_prefill_long_prompt():
    """One 2048-token prompt (16 key tiles for the last rows)."""
    run_case(16, 4, 256, 16, [(0, 2048)], 4)


def test_attn_prefill_page_outside_pool_is_left_out():
    run_case(16, 4, 256, 16, [(64, 40), (16, 100)], 5, holes=[(0, 1), (1, 0)])


def test_prefill_then_decode_continue_the_cache():
    """A 300-token prompt through gdn_attn_prefill, then 3 decode steps through
    gdn_attn_decode on the same pages: every step against the oracle over all tokens
    so far (the cache written by one call is what the next one reads)."""
    Hq, Hkv, D, page = 16, 4, 256, 16
    r = synth.rng_for(62, 0)
    cfg = gb.AttnConfig(Hq, Hkv, D, page)
    T, steps = 300, 3
    n_pages = math.ceil((T + steps) / page) + 1
    table = torch.from_numpy(r.permutation(n_pages)[:n_pages - 1].astype(np.int32)).view(1, -1).cuda()
    kp = torch.zeros((n_pages, Hkv, page, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    q, k, v = (_bf16(r, (T + steps, H, D)) for H in (Hq, Hkv, Hkv))
    q64, k64, v64 = q.f64[:], k.f64[:], v.f64[:]
    qd, kd, vd = dev(q), dev(k), dev(v)
    o = torch.empty((T, Hq, D), dtype=torch.bfloat16, device="cuda")
    gb.gdn_attn_prefill(cfg, qd[:T], kd[:T], vd[:T], kp, vp, table, torch.tensor([0, T], dtype=torch.int32).cuda(),
                        torch.zeros(1, dtype=torch.int32).cuda(), o)
    torch.cuda.synchronize()
    ref = at.prefill_attention(q64[:T], k64[:T], v64[:T], 0, 1 / math.sqrt(D))
    assert rel_fro(host(o), ref) <= 8e-3
    for s in range(steps):
        t = T + s
        od = torch.empty((1, Hq, D), dtype=torch.bfloat16, device="cuda")
        nws = gb.gdn_attn_workspace_size(cfg, 1, t + 1)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda") if nws else None
        gb.gdn_attn_decode(cfg, qd[t:t + 1], kd[t:t + 1], vd[t:t + 1], kp, vp, table,
                           torch.tensor([t], dtype=torch.int32).cuda(), t + 1, od, ws)
        torch.cuda.synchronize()
        refd = at.decode_attention(q64[t], k64[:t + 1], v64[:t + 1], 1 / math.sqrt(D))
        assert rel_fro(host(od)[0], refd) <= 4e-3, s
