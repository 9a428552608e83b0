// gdn_attn.cu -- decode attention of the hybrid's full-attention layers over a
// paged KV cache, with grouped query heads (GQA).
//
// "Forge: how I wrote my own inference engine and overtook llama.cpp": the
// hybrid's other layers are ordinary GQA attention with a KV cache (its
// architecture section: 48 of 64 layers DeltaNet, 16 GQA attention, 4 kv-heads
// of 256 dims); its decode kernel splits the context over CTAs (split-KV, its
// 25-26 August entry) and packs the query heads of a kv-head into one CTA so
// that every kv-head is read once.  "Hybrid transformers under load ..."
// (braintools.ru, section 4.1): an attention page holds the K and V of
// block_size tokens of one layer, 4 kv-heads x 256 values in bf16 per token for
// Qwen3.5-4B.
//
// Decode is HBM-bound (1 KB of K and V per token and kv-head at d = 256 against
// 4 flops per byte for a group of 4 query heads), so the kernel runs on the
// CUDA cores: one CTA per (context split, kv-head, sequence), each warp streams
// groups of 8 tokens straight from the pages (lane = d/32 consecutive dims, one
// 16-byte load per token row), scores the group's query heads, keeps a running
// max and sum per head (online softmax) and accumulates P V in registers.  The
// warps of a CTA, then the splits, are merged by their maxima.
#include <cuda_bf16.h>

#include <cstdlib>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

constexpr int kAtWarps = 4;
constexpr int kTJ = 8;  // tokens per warp step

struct AttnArgs {
    const __nv_bfloat16* q;      // [B][Hq][D]
    const __nv_bfloat16* k_new;  // [B][Hkv][D]
    const __nv_bfloat16* v_new;
    __nv_bfloat16* k_pool;  // [n_pages][Hkv][page][D]
    __nv_bfloat16* v_pool;
    const int32_t* block_table;  // [B][max_pages]
    const int32_t* seq_lens;     // [B] tokens in the cache before this step
    __nv_bfloat16* o;            // [B][Hq][D]
    float* part;                 // [B][Hq][n_split][D + 2]: unnormalised o, max, sum
    int B, Hq, Hkv, page, max_pages, n_pages, n_split, span;  // span: tokens per split (multiple of kTJ)
    float scale;
};

template <int DPL>
struct Row;
template <>
struct Row<8> {
    using T = uint4;
};
template <>
struct Row<4> {
    using T = uint2;
};

template <int DPL>
__device__ __forceinline__ void unpack_row(const typename Row<DPL>::T& u, float f[DPL]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) {
        const float2 v = __bfloat1622float2(h[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

// 32 partial sums per lane -> lane l holds the full sum of value l (31 shuffles)
__device__ __forceinline__ float transpose_reduce32(float v[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = lane & s;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

// one CTA: GC (1, 2 or 4) query heads of kv-head kvh, tokens of one split.
// Each warp owns a ring of kStages shared-memory stages; a stage holds the K
// and V rows of one group of 8 tokens, which lie contiguously on one page
// (page size and group start are multiples of 8), so lane 0 fetches them with
// two bulk copies completing on the stage's mbarrier.
constexpr int kStages = 2;  // 2 stages x 4 warps x 8 KB: 3 CTAs per SM (12 warps) measured faster than 3 stages

template <int D>
struct AtLay {
    static constexpr int ROWS = kTJ * D * 2;        // bytes of 8 rows of K (or V)
    static constexpr int STAGE = 2 * ROWS;          // K then V
    static constexpr int RING = kStages * STAGE;    // per warp
    static constexpr int SMEM = kAtWarps * RING + kAtWarps * kStages * 8;  // + mbarriers
};

template <int D, int GC>
__global__ void __launch_bounds__(32 * kAtWarps) k_attn_decode(const __grid_constant__ AttnArgs A) {
    constexpr int DPL = D / 32;
    using RowT = typename Row<DPL>::T;
    using Lay = AtLay<D>;
    const int G = A.Hq / A.Hkv, hg = G / GC;
    const int split = blockIdx.x, kvh = blockIdx.y / hg, h0 = kvh * G + (blockIdx.y % hg) * GC, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = A.seq_lens[b];  // cached tokens; the new one is token L
    if (L < 0 || L >= A.max_pages * A.page) return;  // nothing to read or write for b
    const int n_tok = L + 1;
    const int t_begin = split * A.span;
    const int t_end = min(n_tok, t_begin + A.span);

    extern __shared__ __align__(128) unsigned char at_smem[];
    unsigned char* ring = at_smem + warp * Lay::RING;
    uint64_t* full = reinterpret_cast<uint64_t*>(at_smem + kAtWarps * Lay::RING) + warp * kStages;
    __shared__ float s_m[kAtWarps][GC], s_l[kAtWarps][GC], s_alpha[kAtWarps][GC];
    __shared__ __align__(16) float s_p[kAtWarps][32];

    // the new token's K and V go to the pool (every reader takes token L from
    // k_new / v_new): the last split's first head group writes them
    if (split == A.n_split - 1 && (blockIdx.y % hg) == 0 && tid < D / 8) {
        const int pg = L / A.page;
        const int page_id = (pg < A.max_pages) ? A.block_table[(size_t)b * A.max_pages + pg] : -1;
        if (page_id >= 0 && page_id < A.n_pages) {
            const size_t dst = (((size_t)page_id * A.Hkv + kvh) * A.page + L % A.page) * D + tid * 8;
            const size_t src = ((size_t)b * A.Hkv + kvh) * D + tid * 8;
            *reinterpret_cast<uint4*>(A.k_pool + dst) = *reinterpret_cast<const uint4*>(A.k_new + src);
            *reinterpret_cast<uint4*>(A.v_pool + dst) = *reinterpret_cast<const uint4*>(A.v_new + src);
        }
    }

    // groups of this warp: t0 = t_begin + 8 (warp + kAtWarps i); their validity
    // (bit j: token t0 + j is in the cache on a page of the pool, or is token L)
    const int first = t_begin + warp * kTJ;
    const int step = kAtWarps * kTJ;
    const int n_groups = (first < t_end) ? (t_end - first + step - 1) / step : 0;
    auto group_mask = [&](int t0, bool& pool_rows) -> unsigned {
        const int pg = t0 / A.page;
        const int page_id = (pg < A.max_pages) ? A.block_table[(size_t)b * A.max_pages + pg] : -1;
        pool_rows = page_id >= 0 && page_id < A.n_pages;
        unsigned m = 0;
#pragma unroll
        for (int j = 0; j < kTJ; ++j) {
            const int t = t0 + j;
            if ((t < L && pool_rows) || t == L) m |= 1u << j;
        }
        return m;
    };
    auto issue = [&](int gi) {  // lane 0: the pool rows of group gi into stage gi % kStages
        const int t0 = first + gi * step;
        const int pg = t0 / A.page;
        const int page_id = (pg < A.max_pages) ? A.block_table[(size_t)b * A.max_pages + pg] : -1;
        uint64_t* bar = full + gi % kStages;
        if (page_id >= 0 && page_id < A.n_pages && t0 < L) {
            const size_t off = (((size_t)page_id * A.Hkv + kvh) * A.page + t0 % A.page) * D;
            unsigned char* st = ring + (gi % kStages) * Lay::STAGE;
            mbar_arrive_expect_tx(bar, 2 * Lay::ROWS);
            bulk_g2s(st, A.k_pool + off, Lay::ROWS, bar);
            bulk_g2s(st + Lay::ROWS, A.v_pool + off, Lay::ROWS, bar);
        } else {
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
        }
    };
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(full + s, 1);
        fence_mbar_init();
        for (int gi = 0; gi < kStages && gi < n_groups; ++gi) issue(gi);
    }
    if (lane < GC) {
        s_m[warp][lane] = -INFINITY;
        s_l[warp][lane] = 0.f;
    }
    float o[GC][DPL];
#pragma unroll
    for (int g = 0; g < GC; ++g)
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[g][d] = 0.f;
    // this lane's dims of the CTA's query heads, scaled
    float qv[GC][DPL];
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        const RowT u = *reinterpret_cast<const RowT*>(A.q + ((size_t)b * A.Hq + h0 + g) * D + lane * DPL);
        unpack_row<DPL>(u, qv[g]);
#pragma unroll
        for (int d = 0; d < DPL; ++d) qv[g][d] *= A.scale;
    }
    const size_t new_row = ((size_t)b * A.Hkv + kvh) * D + lane * DPL;
    bool ok = true;
    __syncwarp();

    for (int gi = 0; gi < n_groups; ++gi) {
        const int t0 = first + gi * step;
        bool pool_rows;
        const unsigned vmask = group_mask(t0, pool_rows);
        const int ls = gi % kStages;
        const unsigned char* st = ring + ls * Lay::STAGE;
        const bool w = mbar_wait(full + ls, (uint32_t)((gi / kStages) & 1));
        ok = ok && w;
        // partial scores: value (hh, j) = 8 hh + j; heads hh >= GC are padding
        float sv[32];
#pragma unroll
        for (int j = 0; j < kTJ; ++j) {
            float kf[DPL];
            RowT u = RowT{};
            if (t0 + j == L) u = *reinterpret_cast<const RowT*>(A.k_new + new_row);
            else if ((vmask >> j) & 1u) u = *reinterpret_cast<const RowT*>(st + (size_t)j * D * 2 + lane * DPL * 2);
            unpack_row<DPL>(u, kf);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                float acc = 0.f;
                if (hh < GC) {
#pragma unroll
                    for (int d = 0; d < DPL; ++d) acc = fmaf(qv[hh][d], kf[d], acc);
                }
                sv[hh * 8 + j] = acc;
            }
        }
        float s = transpose_reduce32(sv, lane);
        const int hh = lane >> 3, j = lane & 7;
        const bool valid = ((vmask >> j) & 1u) && hh < GC;
        s = valid ? s : -INFINITY;
        float mb = s;
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
        const float m_old = (hh < GC) ? s_m[warp][hh] : -INFINITY;
        const float m_new = fmaxf(m_old, mb);
        const float p = (s == -INFINITY) ? 0.f : __expf(s - m_new);
        const float alpha = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
        float ps = p;
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        __syncwarp();
        s_p[warp][lane] = p;
        if (j == 0 && hh < GC) {
            s_l[warp][hh] = s_l[warp][hh] * alpha + ps;
            s_m[warp][hh] = m_new;
            s_alpha[warp][hh] = alpha;
        }
        __syncwarp();
        // o = alpha o + sum_j p_j v_j over the valid rows (others may hold anything)
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const float al = s_alpha[warp][g];
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[g][d] *= al;
        }
#pragma unroll
        for (int jj = 0; jj < kTJ; ++jj) {
            if (!((vmask >> jj) & 1u)) continue;
            RowT u;
            if (t0 + jj == L) u = *reinterpret_cast<const RowT*>(A.v_new + new_row);
            else u = *reinterpret_cast<const RowT*>(st + Lay::ROWS + (size_t)jj * D * 2 + lane * DPL * 2);
            float vf[DPL];
            unpack_row<DPL>(u, vf);
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                const float pj = s_p[warp][g * 8 + jj];
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[g][d] = fmaf(pj, vf[d], o[g][d]);
            }
        }
        // the stage is read: refill it with group gi + kStages
        __syncwarp();
        if (lane == 0 && gi + kStages < n_groups) {
            fence_proxy_async_smem();
            issue(gi + kStages);
        }
    }
    if (!ok && lane == 0) report_device_status(kDevWaitTimeout);

    // ---- merge the warps: rescale each warp's o and sum to the CTA maximum ------------
    __syncthreads();  // every warp's ring is idle: reuse it for the partial o
    float* s_o = reinterpret_cast<float*>(at_smem);  // [kAtWarps][GC][D]
#pragma unroll
    for (int g = 0; g < GC; ++g)
#pragma unroll
        for (int d = 0; d < DPL; ++d) s_o[((size_t)warp * GC + g) * D + lane * DPL + d] = o[g][d];
    __syncthreads();
    for (int idx = tid; idx < GC * D; idx += 32 * kAtWarps) {
        const int g = idx / D, d = idx % D;
        float m = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kAtWarps; ++w2) m = fmaxf(m, s_m[w2][g]);
        float acc = 0.f, l = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kAtWarps; ++w2) {
            const float f = (s_m[w2][g] == -INFINITY) ? 0.f : __expf(s_m[w2][g] - m);
            acc = fmaf(f, s_o[((size_t)w2 * GC + g) * D + d], acc);
            l = fmaf(f, s_l[w2][g], l);
        }
        const int h = h0 + g;
        if (A.n_split == 1) {
            A.o[((size_t)b * A.Hq + h) * D + d] = __float2bfloat16_rn(l > 0.f ? acc / l : 0.f);
        } else {
            float* pr = A.part + (((size_t)b * A.Hq + h) * A.n_split + split) * (D + 2);
            pr[d] = acc;
            if (d == 0) {
                pr[D] = m;
                pr[D + 1] = l;
            }
        }
    }
}

// the splits of one (sequence, query head): o = sum_i e^(m_i - M) o_i / sum_i e^(m_i - M) l_i
template <int D>
__global__ void __launch_bounds__(D) k_attn_combine(const __grid_constant__ AttnArgs A) {
    const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const int L = A.seq_lens[b];
    if (L < 0 || L >= A.max_pages * A.page) return;
    const float* pr = A.part + ((size_t)b * A.Hq + h) * A.n_split * (D + 2);
    float m = -INFINITY;
    for (int i = 0; i < A.n_split; ++i) m = fmaxf(m, pr[(size_t)i * (D + 2) + D]);
    float acc = 0.f, l = 0.f;
    for (int i = 0; i < A.n_split; ++i) {
        const float mi = pr[(size_t)i * (D + 2) + D];
        const float f = (mi == -INFINITY) ? 0.f : __expf(mi - m);
        acc = fmaf(f, pr[(size_t)i * (D + 2) + d], acc);
        l = fmaf(f, pr[(size_t)i * (D + 2) + D + 1], l);
    }
    A.o[((size_t)b * A.Hq + h) * D + d] = __float2bfloat16_rn(l > 0.f ? acc / l : 0.f);
}

template <int D, int GC>
cudaError_t launch_decode(const AttnArgs& A, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_attn_decode<D, GC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             AtLay<D>::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int hg = (A.Hq / A.Hkv) / GC;
    const dim3 grid((unsigned)A.n_split, (unsigned)(A.Hkv * hg), (unsigned)A.B);
    k_attn_decode<D, GC><<<grid, 32 * kAtWarps, AtLay<D>::SMEM, st>>>(A);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || A.n_split == 1) return e;
    k_attn_combine<D><<<dim3((unsigned)A.Hq, (unsigned)A.B), D, 0, st>>>(A);
    return cudaGetLastError();
}

// query heads per kv-head G: 1 or 2 in one CTA, multiples of 4 in CTAs of 4
// heads (the kv-head's K and V are then read by G/4 CTAs side by side, the
// later reads mostly from L2)
template <int D>
cudaError_t launch_decode_d(const AttnArgs& A, int G, cudaStream_t st) {
    if (G == 1) return launch_decode<D, 1>(A, st);
    if (G == 2) return launch_decode<D, 2>(A, st);
    if (G % 4 == 0) return launch_decode<D, 4>(A, st);
    return cudaErrorInvalidValue;
}

}  // namespace

// Splits of the context: about kAttnCtas CTAs over all (sequence, kv-head,
// head group) triples, each split at least 128 tokens (a multiple of 8);
// shapes only, so the workspace is known without a device.
constexpr int kAttnCtas = 1216;  // 8 waves of 152: short CTAs balance the load (fewer, longer ones measured slower)

AttnPlan attn_plan(int B, int Hq, int Hkv, int max_seq_len) {
    AttnPlan p;
    const int G = Hq / Hkv;
    const int64_t pairs = (int64_t)B * Hkv * (G >= 4 ? G / 4 : 1);
    const int max_tok = max_seq_len > 1 ? max_seq_len : 1;
    int target = kAttnCtas;
    if (const char* e = std::getenv("GDN_ATTN_CTAS")) {  // tuning override
        const int v = std::atoi(e);
        if (v >= 1 && v <= 1 << 20) target = v;
    }
    int ns = pairs > 0 ? (int)((target + pairs - 1) / pairs) : 1;
    const int max_ns = (max_tok + 127) / 128;
    if (ns > max_ns) ns = max_ns;
    if (ns < 1) ns = 1;
    int span = (max_tok + ns - 1) / ns;
    span = (span + kTJ - 1) / kTJ * kTJ;
    ns = (max_tok + span - 1) / span;
    p.n_split = ns;
    p.span = span;
    return p;
}

size_t attn_workspace_bytes(int B, int Hq, int Hkv, int D, int max_seq_len) {
    const AttnPlan p = attn_plan(B, Hq, Hkv, max_seq_len);
    return p.n_split > 1 ? (size_t)B * Hq * p.n_split * (D + 2) * 4 : 0;
}

cudaError_t launch_attn_decode(const AttnJob& j, cudaStream_t st) {
    if (j.B == 0) return cudaSuccess;
    const AttnPlan p = attn_plan(j.B, j.Hq, j.Hkv, j.max_seq_len);
    AttnArgs A;
    A.q = static_cast<const __nv_bfloat16*>(j.q);
    A.k_new = static_cast<const __nv_bfloat16*>(j.k_new);
    A.v_new = static_cast<const __nv_bfloat16*>(j.v_new);
    A.k_pool = static_cast<__nv_bfloat16*>(j.k_pool);
    A.v_pool = static_cast<__nv_bfloat16*>(j.v_pool);
    A.block_table = j.block_table;
    A.seq_lens = j.seq_lens;
    A.o = static_cast<__nv_bfloat16*>(j.o);
    A.part = static_cast<float*>(j.ws);
    A.B = j.B;
    A.Hq = j.Hq;
    A.Hkv = j.Hkv;
    A.page = j.page;
    A.max_pages = j.max_pages;
    A.n_pages = j.n_pages;
    A.n_split = p.n_split;
    A.span = p.span;
    A.scale = j.scale;
    const int G = j.Hq / j.Hkv;
    if (j.D == 256) return launch_decode_d<256>(A, G, st);
    if (j.D == 128) return launch_decode_d<128>(A, G, st);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
