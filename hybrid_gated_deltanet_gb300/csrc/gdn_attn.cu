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

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"
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
    int B, Hq, Hkv, page, max_pages, n_pages, n_split, span;  // span: tokens per split (multiple of 16)
    int box_rows;  // tensor-core kernel: page rows per K/V box, gcd(page, 16)
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
    griddep_wait();  // launched with programmatic serialization
    griddep_launch_dependents();
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
    // page of group gi (-1: past the cache or outside the pool).  Lane i of the warp
    // holds the page of group base + i of a 32-group window: one coalesced lookup per
    // 32 groups, read out with a shuffle (warp-collective).  Two windows: the groups
    // being issued run kStages ahead of the groups being scored.
    auto lookup = [&](int gi) -> int {
        const int t0 = first + gi * step;
        if (gi >= n_groups || t0 >= L) return -1;
        const int pg = t0 / A.page;
        const int pid = (pg < A.max_pages) ? __ldg(A.block_table + (size_t)b * A.max_pages + pg) : -1;
        return (pid >= 0 && pid < A.n_pages) ? pid : -1;
    };
    int win_issue = -1, pid_issue = -1, win_score = -1, pid_score = -1;
    auto page_of = [&](int gi, int& win, int& held) -> int {
        const int base = gi & ~31;
        if (base != win) {
            win = base;
            held = lookup(base + lane);
        }
        return __shfl_sync(0xffffffffu, held, gi & 31);
    };
    auto group_mask = [&](int t0, int page_id) -> unsigned {
        unsigned m = 0;
#pragma unroll
        for (int j = 0; j < kTJ; ++j) {
            const int t = t0 + j;
            if ((t < L && page_id >= 0) || t == L) m |= 1u << j;
        }
        return m;
    };
    auto issue = [&](int gi, int page_id) {  // lane 0: the pool rows of group gi into stage gi % kStages
        const int t0 = first + gi * step;
        uint64_t* bar = full + gi % kStages;
        if (page_id >= 0) {
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
    }
    for (int gi = 0; gi < kStages && gi < n_groups; ++gi) {
        const int pid = page_of(gi, win_issue, pid_issue);
        if (lane == 0) issue(gi, pid);
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
        const unsigned vmask = group_mask(t0, page_of(gi, win_score, pid_score));
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
        if (gi + kStages < n_groups) {
            const int pid = page_of(gi + kStages, win_issue, pid_issue);
            __syncwarp();
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(gi + kStages, pid);
            }
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
    griddep_wait();
    griddep_launch_dependents();
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
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = raise_smem_limit(k_attn_decode<D, GC>, AtLay<D>::SMEM, smem_set);
    if (e != cudaSuccess) return e;
    const int hg = (A.Hq / A.Hkv) / GC;
    const dim3 grid((unsigned)A.n_split, (unsigned)(A.Hkv * hg), (unsigned)A.B);
    e = launch_pdl(k_attn_decode<D, GC>, grid, dim3(32 * kAtWarps), AtLay<D>::SMEM, st, A);
    if (e != cudaSuccess || A.n_split == 1) return e;
    return launch_pdl(k_attn_combine<D>, dim3((unsigned)A.Hq, (unsigned)A.B), dim3(D), 0, st, A);
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 at_encode_fn();

// ---- tensor-core decode for wide groups (8 to 16 query heads per kv-head) ---------
// One CTA per (context split, kv-head, sequence) scores all G heads of the kv-head at
// once, so K and V are read once: the heads are the 16 rows (zero past G) of warp-level
// bf16 MMAs (m16n8k16, fp32 accumulation).  The split's tokens come in groups of 16
// and warp w takes groups w, w + 4, ... whole: S = Q K^T, an online softmax per row in
// registers (its reference maximum moves in steps of at least 8), O += P V over all d
// columns with P as the A operand straight from the score accumulators.  Each warp fills its own ring of NSW stages (16 K rows, then 16
// V rows): a group is one or two runs of rows of a page (splits start on multiples of
// 16 tokens, pages hold a multiple of 8), each run loaded by tensor TMA in boxes of
// 64 columns with the 128-byte swizzle, so the 8-row fragment loads are free of bank
// conflicts; the page of a run is fetched one group before its copy.  The four warps'
// (maximum, sum, O) are merged once at the end through shared memory.  The new token L
// (its row in the pool is written by this launch) is added from k_new / v_new by
// warp 0 of the split that holds it.
__device__ __forceinline__ void ldsm_x4_b16(uint32_t r[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(tc::smem_addr(p)));
}

__device__ __forceinline__ void ldsm_x4_trans_b16(uint32_t r[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(tc::smem_addr(p)));
}

__device__ __forceinline__ void mma_bf16_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a in the low half
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}

template <int D>
struct AtTcLay {
    static constexpr int NCH = D / 64;         // 128-byte column chunks of a row
    static constexpr int TILE = NCH * 2048;    // 16 rows of K (or V): chunk-major, 128-byte swizzled
    static constexpr int STAGE = 2 * TILE;     // K tile, then V tile
    static constexpr int NSW = 3;              // stages per warp
    static constexpr int NST = 4 * NSW;
    static constexpr int QS = D * 2 + 16;      // padded row stride of Q (bytes)
    static constexpr int Q_OFF = NST * STAGE;  // Q of the 16 rows, scaled, bf16
    static constexpr int BAR_OFF = Q_OFF + 16 * QS;
    static constexpr int SMEM = BAR_OFF + NST * 8 + NST * 4;  // + mbarriers, token masks
    static constexpr int SMEM_ALLOC = SMEM + 1024;             // base rounded up to a swizzle atom
    // the merge overlays the rings: per warp 16 rows of O (OS floats) and (m, l) per row
    static constexpr int OS = D + 4;
    static_assert(4 * 16 * OS * 4 + 4 * 16 * 2 * 4 <= NST * STAGE, "merge area");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(128, 1)
    k_attn_decode_tc(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     const __grid_constant__ AttnArgs A) {
    using Lay = AtTcLay<D>;
    constexpr int KS = D / 16;  // k-steps of Q K^T
    constexpr int NT = D / 8;   // n8 tiles of O
    constexpr int NSW = Lay::NSW;
    static_assert(KS % 2 == 0, "k-steps in pairs");
    griddep_wait();  // launched with programmatic serialization
    griddep_launch_dependents();
    const int G = A.Hq / A.Hkv;
    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int h0 = kvh * G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, t4 = lane & 3;
    const int L = A.seq_lens[b];  // cached tokens; the new one is token L
    if (L < 0 || L >= A.max_pages * A.page) return;  // nothing to read or write for b
    const int n_tok = L + 1;
    const int t_begin = split * A.span;
    const int t_end = min(n_tok, t_begin + A.span);
    const int lim = min(t_end, L);  // tokens from the pool: t_begin .. lim - 1
    const int n_groups = lim > t_begin ? (lim - t_begin + 15) / 16 : 0;
    const int my_groups = n_groups > warp ? (n_groups - warp + 3) / 4 : 0;  // groups warp, warp + 4, ...

    extern __shared__ __align__(128) unsigned char at_dyn[];
    unsigned char* at_smem = at_dyn + ((1024u - (smem_u32(at_dyn) & 1023u)) & 1023u);
    unsigned char* ring = at_smem + warp * NSW * Lay::STAGE;
    unsigned char* q_s = at_smem + Lay::Q_OFF;
    uint64_t* full = reinterpret_cast<uint64_t*>(at_smem + Lay::BAR_OFF) + warp * NSW;
    volatile uint32_t* smask = reinterpret_cast<uint32_t*>(at_smem + Lay::BAR_OFF + Lay::NST * 8) + warp * NSW;
    const int R = A.box_rows, n_seg = 16 / R;  // runs of page rows per group

    // the new token's K and V go to the pool (every reader takes token L from k_new / v_new)
    if (split == A.n_split - 1 && tid < D / 8) {
        const int pg = L / A.page;
        const int page_id = (pg < A.max_pages) ? A.block_table[(size_t)b * A.max_pages + pg] : -1;
        if (page_id >= 0 && page_id < A.n_pages) {
            const size_t dst = (((size_t)page_id * A.Hkv + kvh) * A.page + L % A.page) * D + tid * 8;
            const size_t src = ((size_t)b * A.Hkv + kvh) * D + tid * 8;
            *reinterpret_cast<uint4*>(A.k_pool + dst) = *reinterpret_cast<const uint4*>(A.k_new + src);
            *reinterpret_cast<uint4*>(A.v_pool + dst) = *reinterpret_cast<const uint4*>(A.v_new + src);
        }
    }
    // Q of the G heads, scaled in fp32 and rounded to bf16; rows past G are zero
    for (int i = tid; i < 16 * (D / 8); i += 128) {
        const int r = i / (D / 8), c = i % (D / 8);
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < G) {
            const uint4 raw = *reinterpret_cast<const uint4*>(A.q + ((size_t)b * A.Hq + h0 + r) * D + 8 * c);
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
            float2 f = __bfloat1622float2(h[0]);
            u.x = pack_bf2(f.x * A.scale, f.y * A.scale);
            f = __bfloat1622float2(h[1]);
            u.y = pack_bf2(f.x * A.scale, f.y * A.scale);
            f = __bfloat1622float2(h[2]);
            u.z = pack_bf2(f.x * A.scale, f.y * A.scale);
            f = __bfloat1622float2(h[3]);
            u.w = pack_bf2(f.x * A.scale, f.y * A.scale);
        }
        *reinterpret_cast<uint4*>(q_s + r * Lay::QS + 16 * c) = u;
    }
    if (lane == 0) {
        for (int s = 0; s < NSW; ++s) mbar_init(full + s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // token t of the pool: its page, or -1 (outside the cache or the pool)
    auto page_of = [&](int t) -> int {
        if (t < t_begin || t >= lim) return -1;
        const int pg = t / A.page;
        const int pid = (pg < A.max_pages) ? __ldg(A.block_table + (size_t)b * A.max_pages + pg) : -1;
        return (pid >= 0 && pid < A.n_pages) ? pid : -1;
    };
    // lane l < n_seg: run l (rows l R .. l R + R - 1) of this warp's j-th group; a run
    // whose first token is in the pool is loaded whole (its rows past lim lie on the
    // same page and are masked)
    auto row_page = [&](int j) -> int {
        return lane < n_seg ? page_of(t_begin + 16 * (warp + 4 * j) + lane * R) : -1;
    };
    auto issue = [&](int j, int pid) {
        const int s = j % NSW, t0 = t_begin + 16 * (warp + 4 * j);
        const unsigned live = __ballot_sync(0xffffffffu, pid >= 0);
        if (lane == 0) {
            const unsigned runs = (R == 16) ? ((live & 1u) ? 0xffffu : 0u)
                                            : (((live & 1u) ? 0x00ffu : 0u) | ((live & 2u) ? 0xff00u : 0u));
            const int nv = lim - t0;  // tokens of the group before lim (at least 1)
            smask[s] = nv >= 16 ? runs : (runs & ((1u << nv) - 1u));  // tokens of the group to score
            const uint32_t bytes = (uint32_t)__popc(live) * (uint32_t)(2 * Lay::NCH * R * 128);
            if (bytes) mbar_arrive_expect_tx(full + s, bytes);
            else asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(full + s)) : "memory");
        }
        __syncwarp();
        if (pid >= 0) {
            const int y = (t0 + lane * R) % A.page;
            unsigned char* kt = ring + s * Lay::STAGE + lane * R * 128;
#pragma unroll
            for (int ch = 0; ch < Lay::NCH; ++ch) {
                tma_load_4d(kt + ch * 2048, &tk, 64 * ch, y, kvh, pid, full + s);
                tma_load_4d(kt + Lay::TILE + ch * 2048, &tv, 64 * ch, y, kvh, pid, full + s);
            }
        }
    };
    {
        int pid0[NSW];
#pragma unroll
        for (int j = 0; j < NSW; ++j) pid0[j] = j < my_groups ? row_page(j) : -1;
#pragma unroll
        for (int j = 0; j < NSW; ++j)
            if (j < my_groups) issue(j, pid0[j]);
    }
    int pf = NSW < my_groups ? row_page(NSW) : -1;  // the page of the next copy, one group ahead

    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq, gq + 8
    bool ok = true;
    const unsigned char* qb = q_s + (lane & 15) * Lay::QS + (lane >> 4) * 16;
    // A tile as TMA writes it with the 128-byte swizzle: 16-byte unit u of row r sits in
    // chunk u / 8 (2 KB each), row r (128 bytes), at unit (u % 8) ^ (r % 8).  Per-lane
    // parts of the fragment addresses: K row (lane & 7) + 8 (lane >> 4) at unit
    // 2 ks + ((lane >> 3) & 1); V row lane & 15 at unit n + (lane >> 4) for even n.
    const int k_row = (lane & 7) + ((lane >> 4) << 3), k_x = ((lane >> 3) & 1) ^ (lane & 7);
    const int v_row = lane & 15, v_x = (lane >> 4) ^ (lane & 7);

    for (int j = 0; j < my_groups; ++j) {
        const int s = j % NSW;
        unsigned char* st = ring + s * Lay::STAGE;
        ok = mbar_wait(full + s, (uint32_t)((j / NSW) & 1)) && ok;
        // rows never loaded hold anything: their scores are masked, their V rows zeroed
        const unsigned valid = smask[s];
        if (valid != 0xffffu) {
            for (int i = lane; i < 16 * (D / 8); i += 32) {  // whole rows: the swizzle does not matter
                const int r = i / (D / 8), c = i % (D / 8);
                if (!((valid >> r) & 1u))
                    *reinterpret_cast<uint4*>(st + Lay::TILE + (c >> 3) * 2048 + r * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        // S = Q K^T: tokens 0..7 and 8..15, even and odd k-steps apart (shorter chains)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const unsigned char* kb = st + k_row * 128;
#pragma unroll
            for (int ks = 0; ks < KS; ks += 2) {
                uint32_t qa[4], qc[4], bk[4], bl[4];
                ldsm_x4_b16(qa, qb + ks * 32);
                ldsm_x4_b16(bk, kb + (ks >> 2) * 2048 + (((2 * ks) & 7) ^ k_x) * 16);
                ldsm_x4_b16(qc, qb + ks * 32 + 32);
                ldsm_x4_b16(bl, kb + ((ks + 1) >> 2) * 2048 + (((2 * ks + 2) & 7) ^ k_x) * 16);
                mma_bf16_16816(sa, qa, bk[0], bk[1]);
                mma_bf16_16816(sb, qa, bk[2], bk[3]);
                mma_bf16_16816(sc, qc, bl[0], bl[1]);
                mma_bf16_16816(sd, qc, bl[2], bl[3]);
            }
        }
        // online softmax per row (a quad holds a row's 16 scores)
        const int j0 = 2 * t4, j1 = 8 + 2 * t4;
        auto pick = [&](int t, float x) { return ((valid >> t) & 1u) ? x : -INFINITY; };
        const float v00 = pick(j0, sa[0] + sc[0]), v01 = pick(j0 + 1, sa[1] + sc[1]);
        const float v02 = pick(j1, sb[0] + sd[0]), v03 = pick(j1 + 1, sb[1] + sd[1]);
        const float v10 = pick(j0, sa[2] + sc[2]), v11 = pick(j0 + 1, sa[3] + sc[3]);
        const float v12 = pick(j1, sb[2] + sd[2]), v13 = pick(j1 + 1, sb[3] + sd[3]);
        float mx0 = fmaxf(fmaxf(v00, v01), fmaxf(v02, v03)), mx1 = fmaxf(fmaxf(v10, v11), fmaxf(v12, v13));
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // the reference maximum of a row moves only when the row's maximum passes it by
        // more than 8 (p then stays below e^8, well inside bf16 and fp32), so O is
        // rescaled in few groups
        const bool up0 = mx0 > m0 + 8.f, up1 = mx1 > m1 + 8.f;
        const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
        const bool moved = __any_sync(0xffffffffu, up0 || up1);
        const float a0 = !up0 ? 1.f : (m0 == -INFINITY) ? 0.f : __expf(m0 - mn0);
        const float a1 = !up1 ? 1.f : (m1 == -INFINITY) ? 0.f : __expf(m1 - mn1);
        auto ex = [](float v, float m) { return v == -INFINITY ? 0.f : __expf(v - m); };
        const float p00 = ex(v00, mn0), p01 = ex(v01, mn0), p02 = ex(v02, mn0), p03 = ex(v03, mn0);
        const float p10 = ex(v10, mn1), p11 = ex(v11, mn1), p12 = ex(v12, mn1), p13 = ex(v13, mn1);
        float ps0 = p00 + p01 + p02 + p03, ps1 = p10 + p11 + p12 + p13;
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
            ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
        }
        l0 = l0 * a0 + ps0;
        l1 = l1 * a1 + ps1;
        m0 = mn0;
        m1 = mn1;
        if (moved) {  // a reference maximum moved somewhere in the warp: rescale O
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
        }
        // O += P V, P as the A operand (rows gq, gq + 8; k = the 16 tokens)
        const uint32_t pa[4] = {pack_bf2(p00, p01), pack_bf2(p10, p11), pack_bf2(p02, p03), pack_bf2(p12, p13)};
        {
            const unsigned char* vb = st + Lay::TILE + v_row * 128;
#pragma unroll
            for (int n = 0; n < NT; n += 2) {
                uint32_t bv[4];
                ldsm_x4_trans_b16(bv, vb + (n >> 3) * 2048 + ((n & 7) ^ v_x) * 16);
                mma_bf16_16816(o[n], pa, bv[0], bv[1]);
                mma_bf16_16816(o[n + 1], pa, bv[2], bv[3]);
            }
        }
        // the stage is read (and its V rows written) by this warp: refill it
        __syncwarp();
        if (j + NSW < my_groups) {
            fence_proxy_async_smem();
            issue(j + NSW, pf);
            pf = j + NSW + 1 < my_groups ? row_page(j + NSW + 1) : -1;
        }
    }

    // the new token L, from k_new / v_new, by warp 0 of the split that holds it
    if (warp == 0 && L >= t_begin && L < t_end) {
        const __nv_bfloat16* kn = A.k_new + ((size_t)b * A.Hkv + kvh) * D;
        const __nv_bfloat16* vn = A.v_new + ((size_t)b * A.Hkv + kvh) * D;
        float d0 = 0.f, d1 = 0.f;  // q . k_new for rows gq, gq + 8 over this lane's dims
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const int d = 8 * i + 2 * t4;
            const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kn + d));
            const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(q_s + gq * Lay::QS + 2 * d));
            const float2 f1 =
                __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(q_s + (gq + 8) * Lay::QS + 2 * d));
            d0 = fmaf(f0.x, kf.x, fmaf(f0.y, kf.y, d0));
            d1 = fmaf(f1.x, kf.x, fmaf(f1.y, kf.y, d1));
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            d0 += __shfl_xor_sync(0xffffffffu, d0, off);
            d1 += __shfl_xor_sync(0xffffffffu, d1, off);
        }
        const float mn0 = fmaxf(m0, d0), mn1 = fmaxf(m1, d1);
        const float a0 = (m0 == -INFINITY) ? 0.f : __expf(m0 - mn0), a1 = (m1 == -INFINITY) ? 0.f : __expf(m1 - mn1);
        const float pn0 = __expf(d0 - mn0), pn1 = __expf(d1 - mn1);
        l0 = l0 * a0 + pn0;
        l1 = l1 * a1 + pn1;
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vn + 8 * n + 2 * t4));
            o[n][0] = fmaf(pn0, vf.x, o[n][0] * a0);
            o[n][1] = fmaf(pn0, vf.y, o[n][1] * a0);
            o[n][2] = fmaf(pn1, vf.x, o[n][2] * a1);
            o[n][3] = fmaf(pn1, vf.y, o[n][3] * a1);
        }
    }

    // ---- merge of the four warps (over the rings, all copies landed) and out --------
    if (__syncthreads_or(!ok)) {  // a wait gave up: copies may still land in the rings
        if (tid == 0) report_device_status(kDevWaitTimeout);
        return;
    }
    float* ob = reinterpret_cast<float*>(at_smem);          // [warp][16][OS]
    float* ml = ob + 4 * 16 * Lay::OS;                      // [warp][16][2]: maximum, sum
    {
        float* w0 = ob + (warp * 16 + gq) * Lay::OS + 2 * t4;
        float* w1 = w0 + 8 * Lay::OS;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            *reinterpret_cast<float2*>(w0 + 8 * n) = make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2*>(w1 + 8 * n) = make_float2(o[n][2], o[n][3]);
        }
        if (t4 == 0) {
            ml[(warp * 16 + gq) * 2] = m0;
            ml[(warp * 16 + gq) * 2 + 1] = l0;
            ml[(warp * 16 + gq + 8) * 2] = m1;
            ml[(warp * 16 + gq + 8) * 2 + 1] = l1;
        }
    }
    __syncthreads();
    for (int i = tid; i < G * (D / 2); i += 128) {
        const int r = i / (D / 2), c = 2 * (i % (D / 2));
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, ml[(w * 16 + r) * 2]);
        float l = 0.f, ox = 0.f, oy = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float mw = ml[(w * 16 + r) * 2];
            const float sw = (mw == -INFINITY) ? 0.f : __expf(mw - M);
            const float2 v = *reinterpret_cast<const float2*>(ob + (w * 16 + r) * Lay::OS + c);
            l = fmaf(sw, ml[(w * 16 + r) * 2 + 1], l);
            ox = fmaf(sw, v.x, ox);
            oy = fmaf(sw, v.y, oy);
        }
        const int h = h0 + r;
        if (A.n_split == 1) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            *reinterpret_cast<__nv_bfloat162*>(A.o + ((size_t)b * A.Hq + h) * D + c) =
                __floats2bfloat162_rn(ox * inv, oy * inv);
        } else {
            float* pr = A.part + (((size_t)b * A.Hq + h) * A.n_split + split) * (D + 2);
            pr[c] = ox;
            pr[c + 1] = oy;
            if (c == 0) {
                pr[D] = M;
                pr[D + 1] = l;
            }
        }
    }
}

template <int D>
cudaError_t launch_decode_tc(const AttnArgs& A0, cudaStream_t st) {
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = raise_smem_limit(k_attn_decode_tc<D>, AtTcLay<D>::SMEM_ALLOC, smem_set);
    if (e != cudaSuccess) return e;
    PFN_cuTensorMapEncodeTiled_v12000 enc = at_encode_fn();
    if (!enc) return cudaErrorInvalidValue;
    AttnArgs A = A0;
    A.box_rows = (A.page % 16 == 0) ? 16 : 8;  // the page size is a multiple of 8
    CUtensorMap mk, mv;
    for (int w = 0; w < 2; ++w) {  // [n_pages][Hkv][page][D] bf16, boxes of box_rows x 64
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)A.page, (cuuint64_t)A.Hkv, (cuuint64_t)A.n_pages};
        const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)A.page * D * 2,
                                       (cuuint64_t)A.Hkv * A.page * D * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)A.box_rows, 1, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(w == 0 ? &mk : &mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w == 0 ? A.k_pool : A.v_pool, dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)A.n_split, (unsigned)A.Hkv, (unsigned)A.B);
    e = launch_pdl(k_attn_decode_tc<D>, grid, dim3(128), AtTcLay<D>::SMEM_ALLOC, st, mk, mv, A);
    if (e != cudaSuccess || A.n_split == 1) return e;
    return launch_pdl(k_attn_combine<D>, dim3((unsigned)A.Hq, (unsigned)A.B), dim3(D), 0, st, A);
}

// query heads per kv-head G: 1 or 2 in one CTA of the CUDA-core kernel, 4 in one CTA
// of 4 heads; 8, 12 or 16 on the tensor-core kernel (one CTA per kv-head, the heads
// as MMA rows); more in CTAs of 4 heads of the CUDA-core kernel (the kv-head's K and V
// are then read by G/4 CTAs side by side, the later reads mostly from L2)
template <int D>
cudaError_t launch_decode_d(const AttnArgs& A, int G, cudaStream_t st) {
    if (G == 1) return launch_decode<D, 1>(A, st);
    if (G == 2) return launch_decode<D, 2>(A, st);
    if (G % 4 != 0) return cudaErrorInvalidValue;
    if (G > 4 && G <= 16) return launch_decode_tc<D>(A, st);
    return launch_decode<D, 4>(A, st);
}

// ---------------------------------------------------------------------------
// Prefill (chunk) attention: n_s new tokens of sequence s at positions
// P_s .. P_s + n_s - 1 attend causally to the sequence's tokens 0 .. own position
// (the bottom-right aligned mask of forge's 27 August entry: row i sees
// 0 .. kv0 + i).  The new K and V are first appended to their pages
// (k_attn_append), then every key comes from the pool.
//
// k_attn_prefill: one CTA per (tile of TQ = 128 / G new tokens of one sequence,
// kv-head); the tile's 128 MMA rows are (token, query head) pairs of that kv-head,
// so K and V of a kv-head are read once for its G heads.  Per tile of 128 keys:
//   S = Q K^T   (tcgen05, M = 128, N = 128, K = d: d/16 instructions, S in TMEM)
//   softmax rows on 4 warps (thread = row), P in bf16 -> shared memory
//   O += P V    (M = 128, N = d, K = 128: 8 instructions, V read MN-major)
// with an online softmax whose reference maximum moves only when a row's
// maximum grows by more than 8 / scale (O is then rescaled in TMEM), so the
// common step never touches O.  Warp 0 drives the TMA loads (Q once; K and V
// per key tile, a box per run of page rows), warp 1 issues the MMAs.
// ---------------------------------------------------------------------------
struct AttnPfArgs {
    const int32_t* block_table;  // [n_seq][max_pages]
    const int32_t* cu_seqlens;   // [n_seq + 1] new tokens
    const int32_t* ctx_lens;     // [n_seq] cached tokens before the new ones
    __nv_bfloat16* o;            // [N][Hq][D]
    int n_seq, Hq, Hkv, G, TQ, page, R, max_pages, n_pages;
    int64_t n_slots;  // q tiles: N / TQ + n_seq + 1 slots (slot of tile c of sequence s: cu[s] / TQ + s + c)
    float scale_log2;  // scale * log2(e)
};

// all `count` threads of named barrier `id` agree on `pred` (logical and)
__device__ __forceinline__ bool named_bar_and(int id, int count, bool pred) {
    int r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n barrier.red.and.pred q, %2, %3, p;\n selp.s32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((int)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// 2^x on the SFU (the PTX ex2 instruction; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 128 consecutive TMEM columns of this warp's lanes: 8 loads, one wait
__device__ __forceinline__ void ld_row128(uint32_t ta, float v[128]) {
    uint32_t r[128];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[16 * q + 0]), "=r"(r[16 * q + 1]), "=r"(r[16 * q + 2]), "=r"(r[16 * q + 3]),
              "=r"(r[16 * q + 4]), "=r"(r[16 * q + 5]), "=r"(r[16 * q + 6]), "=r"(r[16 * q + 7]),
              "=r"(r[16 * q + 8]), "=r"(r[16 * q + 9]), "=r"(r[16 * q + 10]), "=r"(r[16 * q + 11]),
              "=r"(r[16 * q + 12]), "=r"(r[16 * q + 13]), "=r"(r[16 * q + 14]), "=r"(r[16 * q + 15])
            : "r"(ta + 16 * q));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr, uint32_t lbo) {
    // 128-byte swizzled MN-major operand: atoms of 64 (MN) x 8 (K) elements; lbo =
    // byte stride between atoms along MN, 1024 = stride between 8-row groups along K
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}

template <int D>
struct PfLay {
    static constexpr int ATOM = 128 * 128;  // 128 rows x 128 bytes
    static constexpr int Q = 0;             // [128 rows][D] K-major: D / 64 atoms
    static constexpr int K = Q + (D / 64) * ATOM;
    static constexpr int V = K + (D / 64) * ATOM;  // [128 keys][D] MN-major: D / 64 atoms of 128 keys
    static constexpr int P = V + (D / 64) * ATOM;  // [128 rows][128 keys] K-major: 2 atoms
    static constexpr int BAR = P + 2 * ATOM;
    static constexpr int SMEM = BAR + 16 * 8;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    static constexpr int TMEM_COLS = D == 256 ? 512 : 256;  // S [0, 128), O [TMEM_COLS - D, TMEM_COLS)
    static constexpr int O_COL = TMEM_COLS - D;
};

__device__ __forceinline__ int pf_slot_seq(const AttnPfArgs& A, int64_t slot) {
    int lo = 0, hi = A.n_seq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)A.cu_seqlens[mid] / A.TQ + mid <= slot) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int D>
__global__ void __launch_bounds__(224, 1)
    k_attn_prefill(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ AttnPfArgs A) {
    using Ly = PfLay<D>;
    constexpr int NA = D / 64;  // 64-wide atoms along d
    griddep_wait();  // launched with programmatic serialization: the appended rows are visible
    griddep_launch_dependents();
    const int64_t slot = A.n_slots - 1 - blockIdx.x;  // late (long) tiles first
    const int kvh = blockIdx.y;
    const int s = pf_slot_seq(A, slot);
    const int cu0 = A.cu_seqlens[s], n_s = A.cu_seqlens[s + 1] - cu0;
    const int P = A.ctx_lens[s];
    const int t0 = (int)(slot - ((int64_t)cu0 / A.TQ + s)) * A.TQ;  // first new token of the tile
    if (t0 < 0 || t0 >= n_s || P < 0) return;
    const int nq = min(A.TQ, n_s - t0);
    const int L = P + n_s;                                // keys of the sequence
    const int n_kv = (P + t0 + nq + 127) / 128;           // key tiles the tile's last row needs
    if ((int64_t)(L + A.page - 1) / A.page > A.max_pages) return;  // pages past the block table

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::BAR);
    uint64_t *full_q = bars, *full_k = bars + 1, *full_v = bars + 2, *s_done = bars + 3, *s_read = bars + 4,
             *p_ready = bars + 5, *pv_done = bars + 6;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);
    if (tid == 0) {
        mbar_init(full_q, 1);
        mbar_init(full_k, 1);
        mbar_init(full_v, 1);
        mbar_init(s_done, 1);
        mbar_init(s_read, 4);   // one arrival per softmax warp
        mbar_init(p_ready, 1);
        mbar_init(pv_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc(tslot, Ly::TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;
    bool ok = true;

    // key tile j: lane i (< 128 / R) looks up the page of its run of R rows, all lanes
    // at once (one load latency per tile, issued a tile ahead); -1: past the
    // sequence or a page outside the pool
    const int nseg = 128 / A.R;
    auto lane_page = [&](int j) -> int {
        const int pos = j * 128 + lane * A.R;
        if (lane >= nseg || j >= n_kv || pos >= L) return -1;
        const int pid = __ldg(A.block_table + (size_t)s * A.max_pages + pos / A.page);
        return (pid >= 0 && pid < A.n_pages) ? pid : -1;
    };

    if (warp == 0) {
        // Q of the tile: tokens cu0 + t0 .., heads kvh G ..; rows past the tile are other
        // tokens or zeros (never stored)
        if (lane == 0) {
            mbar_arrive_expect_tx(full_q, (uint32_t)(NA * A.TQ * A.G * 128));
            for (int a = 0; a < NA; ++a) tma_load_3d(sm + Ly::Q + a * Ly::ATOM, &tq, a * 64, kvh * A.G, cu0 + t0, full_q);
        }
        int last_k = -1;
        int pid_next = lane_page(0);
        for (int j = 0; j < n_kv && ok; ++j) {
            const int k0 = j * 128;
            const int pid = pid_next;
            pid_next = lane_page(j + 1);
            const unsigned have = __ballot_sync(0xffffffffu, pid >= 0);
            const uint32_t bytes = (uint32_t)__popc(have) * NA * A.R * 128;
            // K_j once S_{j-1} has read K_{j-1}
            if (j > 0 && !mbar_wait(s_done, (uint32_t)((j - 1) & 1))) ok = false;
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) mbar_arrive_expect_tx(full_k, bytes);
            __syncwarp();
            if (pid >= 0)  // lane i issues its run's boxes
                for (int a = 0; a < NA; ++a)
                    tma_load_4d(sm + Ly::K + a * Ly::ATOM + lane * A.R * 128, &tk, a * 64, (k0 + lane * A.R) % A.page,
                                kvh, pid, full_k);
            last_k = j;
        }
        // copies still in flight land before the CTA leaves
        if (last_k >= 0) mbar_wait(full_k, (uint32_t)(last_k & 1));
        if (!mbar_wait(full_q, 0)) ok = false;
    } else if (warp == 6) {
        // ---- V producer: V_j once PV_{j-1} has read V_{j-1} (its own warp, so that the
        // K loads of the next tile never queue behind a V load that waits for PV) ------
        int last_v = -1;
        int pid_next = lane_page(0);
        for (int j = 0; j < n_kv && ok; ++j) {
            const int k0 = j * 128;
            const int pid = pid_next;
            pid_next = lane_page(j + 1);
            const unsigned have = __ballot_sync(0xffffffffu, pid >= 0);
            const uint32_t bytes = (uint32_t)__popc(have) * NA * A.R * 128;
            if (j > 0 && !mbar_wait(pv_done, (uint32_t)((j - 1) & 1))) ok = false;
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) mbar_arrive_expect_tx(full_v, bytes);
            __syncwarp();
            if (pid >= 0)
                for (int a = 0; a < NA; ++a)
                    tma_load_4d(sm + Ly::V + a * Ly::ATOM + lane * A.R * 128, &tv, a * 64, (k0 + lane * A.R) % A.page,
                                kvh, pid, full_v);
            last_v = j;
        }
        if (last_v >= 0) mbar_wait(full_v, (uint32_t)(last_v & 1));
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(128 >> 3) << 17) |
                                         ((uint32_t)(128 >> 4) << 24);
            constexpr uint32_t idesc_o = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                         ((uint32_t)(D >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
            const uint32_t q0 = tc::smem_addr(sm + Ly::Q), kk0 = tc::smem_addr(sm + Ly::K);
            const uint32_t v0 = tc::smem_addr(sm + Ly::V), p0 = tc::smem_addr(sm + Ly::P);
            ok = mbar_wait(full_q, 0);
            for (int j = 0; j < n_kv && ok; ++j) {
                // S_j = Q K_j^T once K_j has landed and the softmax has read S_{j-1}
                if (!mbar_wait(full_k, (uint32_t)(j & 1))) { ok = false; break; }
                if (j > 0 && !mbar_wait(s_read, (uint32_t)((j - 1) & 1))) { ok = false; break; }
                tc::fence_after();
                for (int kd = 0; kd < D / 16; ++kd) {
                    const uint32_t off = (uint32_t)((kd >> 2) * Ly::ATOM + (kd & 3) * 32);
                    mma_f16(tm, tc::sdesc(q0 + off), tc::sdesc(kk0 + off), idesc_s, kd > 0 ? 1u : 0u);
                }
                tc::commit(s_done);
                // O += P_j V_j once P_j is written and V_j has landed
                if (!mbar_wait(p_ready, (uint32_t)(j & 1))) { ok = false; break; }
                if (!mbar_wait(full_v, (uint32_t)(j & 1))) { ok = false; break; }
                tc::fence_after();
                for (int kk = 0; kk < 8; ++kk) {  // 16 keys per instruction
                    const uint32_t pa = p0 + (uint32_t)((kk >> 2) * Ly::ATOM + (kk & 3) * 32);
                    const uint32_t vb = v0 + (uint32_t)(kk * 16 * 128);
                    mma_f16(tm + Ly::O_COL, tc::sdesc(pa), sdesc_mn(vb, Ly::ATOM), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(pv_done);
            }
        }
    } else if (warp < 6) {
        // ---- softmax and epilogue: thread = row r of the tile (TMEM lane r) ----------------
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const int tl = r / A.G, g = r % A.G;      // token in the tile, head in the group
        const bool row_ok = tl < nq;              // rows past the tile's tokens are never stored
        const int qpos = P + t0 + tl;             // the row's position in the sequence
        float m_ref = -INFINITY, l = 0.f;
        unsigned char* prow = sm + Ly::P + r * 128;
        int pid_next = lane_page(0);
        for (int j = 0; j < n_kv; ++j) {
            const int k0 = j * 128;
            bool w = mbar_wait(s_done, (uint32_t)(j & 1));
            if (!named_bar_and(1, 128, w)) { ok = false; break; }
            tc::fence_after();
            float sv[128];
            ld_row128(tc::taddr(tm, 32 * q4, 0), sv);
            tc::fence_before();
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(s_read)) : "memory");
            // keys on pages outside the pool, per run of R page rows (bit c of dead[c / 32]);
            // runs with no key (past the sequence) are bit seg of gone
            const int pid = pid_next;
            pid_next = lane_page(j + 1);
            const unsigned hole = __ballot_sync(0xffffffffu, lane < nseg && k0 + lane * A.R < L && pid < 0);
            const unsigned gone = __ballot_sync(0xffffffffu, lane < nseg && pid < 0);
            uint32_t dead[4] = {0u, 0u, 0u, 0u};
            if (hole) {
                for (int sg = 0; sg < nseg; ++sg) {
                    if (!((hole >> sg) & 1u)) continue;
                    const int r0 = sg * A.R;
                    for (int c = r0; c < r0 + A.R; c += 32) {
                        const int n = min(32, r0 + A.R - c);
                        dead[c >> 5] |= (n == 32 ? 0xffffffffu : ((1u << n) - 1u)) << (c & 31);
                    }
                }
            }
            // mask: causal (which also keeps the key inside the sequence) and on a page of the
            // pool; a tile below the diagonal of every row of the warp, with no hole, needs none
            float mt = -INFINITY;
            const bool full_tile = __all_sync(0xffffffffu, row_ok && k0 + 127 <= qpos) && !hole;
            if (full_tile) {
#pragma unroll
                for (int c = 0; c < 128; ++c) mt = fmaxf(mt, sv[c]);
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const int pos = k0 + c;
                    const bool v = row_ok && pos <= qpos && !((dead[c >> 5] >> (c & 31)) & 1u);
                    sv[c] = v ? sv[c] : -INFINITY;
                    mt = fmaxf(mt, sv[c]);
                }
            }
            // move a row's reference maximum when its maximum grew by more than 2^8 in the
            // exponent (its O and l are then rescaled by f)
            float f = 1.f;
            if (mt > -INFINITY && (m_ref == -INFINITY || (mt - m_ref) * A.scale_log2 > 8.f)) {
                if (j > 0 && m_ref > -INFINITY) {
                    f = exp2f((m_ref - mt) * A.scale_log2);
                    l *= f;
                }
                m_ref = mt;
            }
            // p = 2^((s - m_ref) scale log2 e) in bf16, packed in registers while PV_{j-1}
            // still runs; the sum takes the rounded values, like the product
            uint32_t pk[64];
            const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref * A.scale_log2;  // a masked s gives 2^-inf = 0
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                const float p0 = ex2_approx(fmaf(sv[2 * e], A.scale_log2, neg_m));
                const float p1 = ex2_approx(fmaf(sv[2 * e + 1], A.scale_log2, neg_m));
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                const float2 back = __bfloat1622float2(h2);
                l += back.x + back.y;
                pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            // P_j may replace P_{j-1}, and O be rescaled, once PV_{j-1} is done
            w = (j == 0) || mbar_wait(pv_done, (uint32_t)((j - 1) & 1));
            if (!named_bar_and(1, 128, w)) { ok = false; break; }
            tc::fence_after();
            // TMEM loads and stores are warp-collective: the warp rescales together when any
            // of its rows needs it (the others by 1)
            if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float ov[16];
                    tc::ld16(tc::taddr(tm, 32 * q4, Ly::O_COL + c0), ov);
#pragma unroll
                    for (int c = 0; c < 16; ++c) ov[c] *= f;
                    tc::st16(tc::taddr(tm, 32 * q4, Ly::O_COL + c0), ov);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            // P row (128-byte swizzle, K-major)
#pragma unroll
            for (int c8 = 0; c8 < 16; ++c8) {
                const int atom = c8 >> 3, ch = c8 & 7;
                *reinterpret_cast<uint4*>(prow + atom * Ly::ATOM + ((ch ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
            }
            // V rows with no key behind them (past the sequence or on a missing page) -> 0,
            // so that 0 x garbage never reaches O
            w = mbar_wait(full_v, (uint32_t)(j & 1));
            if (!named_bar_and(1, 128, w)) { ok = false; break; }
            {
                const int key = r;  // thread r clears V row r when its run has no key
                if ((gone >> (key / A.R)) & 1u) {
#pragma unroll
                    for (int a = 0; a < NA; ++a) {
                        uint4* vr = reinterpret_cast<uint4*>(sm + Ly::V + a * Ly::ATOM + key * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) vr[c] = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            fence_proxy_async_smem();
            tc::fence_before();
            named_bar_sync(1, 128);
            if (tid == 64) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(p_ready)) : "memory");
        }
        // ---- epilogue: o = O / l (TMEM loads by the whole warp, stores by rows in the tile)
        bool w = ok && mbar_wait(pv_done, (uint32_t)((n_kv - 1) & 1));
        w = named_bar_and(1, 128, w);
        if (!w) ok = false;
        tc::fence_after();
        if (w) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* dst = A.o + ((size_t)(cu0 + t0 + tl) * A.Hq + kvh * A.G + g) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 16) {
                float ov[16];
                tc::ld16(tc::taddr(tm, 32 * q4, Ly::O_COL + c0), ov);
                uint4 pk[2];
                __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
                for (int c = 0; c < 8; ++c) h[c] = __floats2bfloat162_rn(ov[2 * c] * inv, ov[2 * c + 1] * inv);
                if (row_ok) {
                    reinterpret_cast<uint4*>(dst + c0)[0] = pk[0];
                    reinterpret_cast<uint4*>(dst + c0)[1] = pk[1];
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (!ok && lane == 0) report_device_status(kDevWaitTimeout);
    if (warp == 1) tc::dealloc(tm, Ly::TMEM_COLS);
}

// new K and V rows of every token into their pages: thread = 16 bytes of a row
__global__ void k_attn_append(const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
                              __nv_bfloat16* k_pool, __nv_bfloat16* v_pool, const int32_t* block_table,
                              const int32_t* cu_seqlens, const int32_t* ctx_lens, int n_seq, int64_t n_tokens,
                              int Hkv, int D, int page, int max_pages, int n_pages) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t tok = blockIdx.x;
    if (tok >= n_tokens) return;
    int lo = 0, hi = n_seq - 1;  // the sequence holding token tok
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu_seqlens[mid] <= tok) lo = mid;
        else hi = mid - 1;
    }
    const int P = ctx_lens[lo];
    if (P < 0) return;
    const int64_t pos = P + (tok - cu_seqlens[lo]);
    if (pos / page >= max_pages) return;
    const int pid = block_table[(size_t)lo * max_pages + pos / page];
    if (pid < 0 || pid >= n_pages) return;
    const int per_row = D / 8;
    for (int i = threadIdx.x; i < Hkv * per_row; i += blockDim.x) {
        const int h = i / per_row, c = i % per_row;
        const size_t src = ((size_t)tok * Hkv + h) * D + c * 8;
        const size_t dst = (((size_t)pid * Hkv + h) * page + pos % page) * D + c * 8;
        *reinterpret_cast<uint4*>(k_pool + dst) = *reinterpret_cast<const uint4*>(k_new + src);
        *reinterpret_cast<uint4*>(v_pool + dst) = *reinterpret_cast<const uint4*>(v_new + src);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 at_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <int D>
cudaError_t launch_prefill_attn(const AttnPfJob& j, cudaStream_t st) {
    using Ly = PfLay<D>;
    static std::atomic<uint64_t> smem_set{0};
    {
        const cudaError_t e = raise_smem_limit(k_attn_prefill<D>, Ly::SMEM_ALLOC, smem_set);
        if (e != cudaSuccess) return e;
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = at_encode_fn();
    if (!enc) return cudaErrorInvalidValue;
    const int G = j.Hq / j.Hkv;
    AttnPfArgs A;
    A.block_table = j.block_table;
    A.cu_seqlens = j.cu_seqlens;
    A.ctx_lens = j.ctx_lens;
    A.o = static_cast<__nv_bfloat16*>(j.o);
    A.n_seq = j.n_seq;
    A.Hq = j.Hq;
    A.Hkv = j.Hkv;
    A.G = G;
    A.TQ = 128 / G;
    A.page = j.page;
    int R = 128;
    while (j.page % R) R >>= 1;  // rows per K/V box: gcd(page, 128)
    A.R = R;
    A.max_pages = j.max_pages;
    A.n_pages = j.n_pages;
    A.n_slots = j.n_tokens / A.TQ + j.n_seq + 1;
    A.scale_log2 = j.scale * 1.4426950408889634f;
    CUtensorMap mq, mk, mv;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)j.Hq, (cuuint64_t)j.n_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)j.Hq * D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)A.TQ};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(j.q), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    for (int w = 0; w < 2; ++w) {
        const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)j.page, (cuuint64_t)j.Hkv, (cuuint64_t)j.n_pages};
        const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)j.page * D * 2,
                                       (cuuint64_t)j.Hkv * j.page * D * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)R, 1, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(w == 0 ? &mk : &mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w == 0 ? j.k_pool : j.v_pool, dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaError_t e = launch_pdl(k_attn_append, dim3((unsigned)j.n_tokens), dim3(128), 0, st,
                               static_cast<const __nv_bfloat16*>(j.k_new), static_cast<const __nv_bfloat16*>(j.v_new),
                               static_cast<__nv_bfloat16*>(j.k_pool), static_cast<__nv_bfloat16*>(j.v_pool),
                               j.block_table, j.cu_seqlens, j.ctx_lens, j.n_seq, j.n_tokens, j.Hkv, D, j.page,
                               j.max_pages, j.n_pages);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_attn_prefill<D>, dim3((unsigned)A.n_slots, (unsigned)j.Hkv), dim3(224), Ly::SMEM_ALLOC, st,
                      mq, mk, mv, A);
}

}  // namespace

// Splits of the context: about kAttnCtas CTAs over all (sequence, kv-head,
// head group) triples, each split at least 128 tokens (a multiple of 16);
// shapes only, so the workspace is known without a device.  A head group is the
// kv-head's G query heads, except for G > 16 (CTAs of 4 heads).  The tensor-core
// kernel (G = 8, 12, 16) holds one CTA per SM and aims at kAttnCtasTc CTAs: its
// fixed cost per CTA (Q, first copies, merge) made more, shorter CTAs slower.
constexpr int kAttnCtas = 1216;   // 8 waves of 152: short CTAs balance the load (fewer, longer ones measured slower)
constexpr int kAttnCtasTc = 152;  // one wave at one CTA per SM

AttnPlan attn_plan(int B, int Hq, int Hkv, int max_seq_len) {
    AttnPlan p;
    const int G = Hq / Hkv;
    const int64_t pairs = (int64_t)B * Hkv * (G > 16 ? G / 4 : 1);
    const int max_tok = max_seq_len > 1 ? max_seq_len : 1;
    const bool tc = G > 4 && G <= 16 && G % 4 == 0;
    int target = tc ? kAttnCtasTc : kAttnCtas;
    if (const char* e = std::getenv("GDN_ATTN_CTAS")) {  // tuning override
        const int v = std::atoi(e);
        if (v >= 1 && v <= 1 << 20) target = v;
    }
    int ns = pairs > 0 ? (int)((target + pairs - 1) / pairs) : 1;
    const int max_ns = (max_tok + 127) / 128;
    if (ns > max_ns) ns = max_ns;
    if (ns < 1) ns = 1;
    int span = (max_tok + ns - 1) / ns;
    span = (span + 15) / 16 * 16;
    ns = (max_tok + span - 1) / span;
    p.n_split = ns;
    p.span = span;
    return p;
}

size_t attn_workspace_bytes(int B, int Hq, int Hkv, int D, int max_seq_len) {
    const AttnPlan p = attn_plan(B, Hq, Hkv, max_seq_len);
    return p.n_split > 1 ? (size_t)B * Hq * p.n_split * (D + 2) * 4 : 0;
}

cudaError_t launch_attn_prefill(const AttnPfJob& j, cudaStream_t st) {
    if (j.n_tokens == 0 || j.n_seq == 0) return cudaSuccess;
    if (j.D == 256) return launch_prefill_attn<256>(j, st);
    if (j.D == 128) return launch_prefill_attn<128>(j, st);
    return cudaErrorInvalidValue;
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
