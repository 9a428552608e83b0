"""GPU parity of gdn_attn_decode (paged KV cache, grouped query heads) against
the fp64 oracle, on the oracle's own gather of each sequence's tokens from the
pages.  Tolerance: q, K, V are bf16 and exact in both; the kernel scores and
accumulates in fp32 (errors near 1e-6 relative) and rounds o to bf16 (at most
2^-8 relative per element, 2^-8/sqrt(3) in the root mean square), so the
relative Frobenius error of o is held to 4e-3, and each element to
2^-8 |ref| + 1e-3 max|V|.  The tensor-core path (G = 8, 12, 16) also rounds
q scale and the softmax weights to bf16 (2^-9 relative each, unbiased): a score
then moves by at most 2^-9 of sum |q_i k_i|, and a weight by 2^-9 of itself,
both well inside the same bounds at these value ranges."""
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


def run_case(Hq, Hkv, D, page, lens, seed, holes=()):
    r = synth.rng_for(60, seed)
    B = len(lens)
    cfg = gb.AttnConfig(Hq, Hkv, D, page)
    need = [math.ceil((L + 1) / page) for L in lens]
    max_pages = max(need)
    n_pages = sum(need) + 3
    perm = r.permutation(n_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, np.int32)
    o0 = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[o0:o0 + n]
        o0 += n
    for b, pg in holes:  # a page index outside the pool: its tokens are left out
        table[b, pg] = n_pages + 5
    q = _bf16(r, (B, Hq, D))
    kn, vn = _bf16(r, (B, Hkv, D)), _bf16(r, (B, Hkv, D))
    kp, vp = _bf16(r, (n_pages, Hkv, page, D)), _bf16(r, (n_pages, Hkv, page, D))
    max_seq = max(lens) + 1
    kpd, vpd = dev(kp), dev(vp)
    o = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    n_ws = gb.gdn_attn_workspace_size(cfg, B, max_seq)
    ws = torch.empty(n_ws, dtype=torch.uint8, device="cuda") if n_ws else None
    gb.gdn_attn_decode(cfg, dev(q), dev(kn), dev(vn), kpd, vpd, torch.from_numpy(table).cuda(),
                       torch.from_numpy(np.asarray(lens, np.int32)).cuda(), max_seq, o, ws)
    torch.cuda.synchronize()
    got = host(o)
    kp64, vp64, kn64, vn64, q64 = kp.f64[:], vp.f64[:], kn.f64[:], vn.f64[:], q.f64[:]
    refs = []
    scale = 1 / math.sqrt(D)
    for b, L in enumerate(lens):
        rows_k, rows_v = [], []
        for t in range(L):
            pid = table[b, t // page]
            if 0 <= pid < n_pages:
                rows_k.append(kp64[pid, :, t % page])
                rows_v.append(vp64[pid, :, t % page])
        rows_k.append(kn64[b])
        rows_v.append(vn64[b])
        refs.append(at.decode_attention(q64[b], np.stack(rows_k), np.stack(rows_v), scale))
    ref = np.stack(refs)
    assert rel_fro(got, ref) <= 4e-3, rel_fro(got, ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.max(np.abs(vp64))
    assert np.all(np.abs(got - ref) <= bound)
    # the new tokens were appended to their pages; nothing else changed
    kp_got, vp_got = host(kpd), host(vpd)
    kp_want, vp_want = kp64.copy(), vp64.copy()
    for b, L in enumerate(lens):
        pid = table[b, L // page]
        if 0 <= pid < n_pages:
            kp_want[pid, :, L % page] = kn64[b]
            vp_want[pid, :, L % page] = vn64[b]
    np.testing.assert_array_equal(kp_got, kp_want)
    np.testing.assert_array_equal(vp_got, vp_want)
    return gb.gdn_attn_workspace_size(cfg, B, max_seq)


def test_attn_qwen35_4b_mixed_lengths_split():
    """16 query heads over 4 kv-heads of 256 (G = 4), pages of 16 tokens; the
    longest context makes the kernel split the context and combine."""
    assert run_case(16, 4, 256, 16, [0, 1, 7, 8, 9, 100, 527, 528, 529, 3000], 1) > 0


def test_attn_wide_gqa_large_pages():
    """24 query heads over 2 kv-heads (G = 12: the tensor-core kernel, all 12 heads of a
    kv-head as MMA rows of one CTA), pages of 528 tokens."""
    run_case(24, 2, 256, 528, [5, 600, 1056, 2000], 2)


@pytest.mark.parametrize("Hq,Hkv,D,page", [(8, 8, 128, 8), (4, 2, 128, 32), (32, 4, 128, 16)])
def test_attn_small_groups_and_d128(Hq, Hkv, D, page):
    run_case(Hq, Hkv, D, page, [3, 64, 65, 0, 200], 3)


@pytest.mark.parametrize("Hq,Hkv,D,page", [(16, 2, 128, 8), (32, 2, 256, 24), (24, 3, 128, 40)])
def test_attn_wide_gqa_pages_of_8_rows(Hq, Hkv, D, page):
    """The tensor-core kernel (G = 8, 16) on pages that are not a multiple of 16 tokens:
    a group of 16 tokens is then two runs of 8 page rows, each loaded on its own, and
    the runs of a group can sit on different pages."""
    run_case(Hq, Hkv, D, page, [1, 8, 15, 16, 17, 100, 333, 1000], 6)


def test_attn_many_sequences_no_split():
    r = np.random.Generator(np.random.PCG64(5))
    lens = [int(v) for v in r.integers(0, 60, 200)]
    assert run_case(16, 4, 256, 16, lens, 4) == 0


def test_attn_page_outside_pool_is_left_out():
    run_case(16, 4, 256, 16, [40, 100], 5, holes=[(0, 1), (1, 0)])


def test_attn_empty_batch():
    cfg = gb.AttnConfig(16, 4, 256, 16)
    z = torch.zeros((0, 16, 256), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((1, 4, 16, 256), dtype=torch.bfloat16, device="cuda")
    gb.gdn_attn_decode(cfg, z, z[:, :4], z[:, :4], pool, pool, torch.zeros((0, 1), dtype=torch.int32, device="cuda"),
                       torch.zeros(0, dtype=torch.int32, device="cuda"), 1, z)
