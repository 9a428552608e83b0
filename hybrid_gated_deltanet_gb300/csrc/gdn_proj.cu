// gdn_proj.cu -- the two projections either side of the layer, on the
// tcgen05 tensor cores: out[t][n] = sum_k act[t][k] w[n][k] with bf16 operands,
// fp32 accumulation in TMEM and a bf16 result (round to nearest even).
//
// The in-projection turns the model's hidden states into the layer's inputs
// [x | z | a | b] and the out-projection maps the gated-RMSNorm output y back to
// the model width.  "Forge: how I wrote my own inference engine and overtook
// llama.cpp" (24 August) measures the matrix projections at 59% of its hybrid
// prefill and bounds decode by the weight bytes read per token (its opening
// formulas): prefill needs them on the tensor cores, decode needs them to
// stream the weights at HBM speed.
//
// Kernel (one CTA = 6 warps): a 128-row block of w is the MMA's M side (TMEM
// lane = output channel) and a block of BT tokens is its N side, so one
// kernel covers decode (a few tokens, N = 64) and prefill (N = 256).
//   warp 0      TMA producer: 64-wide K blocks of w and act into a ring of
//               stages (128-byte swizzle, the tensor core's K-major layout)
//   warp 1      MMA issuer (one thread): 4 MMAs of K = 16 per stage into one
//               of two TMEM accumulators, tcgen05.commit frees the stage
//   warps 2..5  epilogue: accumulator -> registers -> bf16 -> global, one
//               output channel per thread, 32 consecutive channels per warp
//               store; the other accumulator takes the next tile meanwhile
// Many tokens: a persistent grid walks the (weight block, token block) tiles.
// Few tokens (decode): too few tiles to fill the GPU, so K is split over ks
// independent CTAs per tile; each writes its fp32 partial block to the
// caller's workspace and a second small kernel adds the ks blocks and rounds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdlib>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

constexpr int kPjThreads = 192;
constexpr int kBM = 128;  // weight rows per tile: MMA M, TMEM lanes
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle atom of bf16

// a stage holds KBOX consecutive 64-wide K blocks (each a 128-byte swizzle atom) of W and act
template <int BT, int STAGES, int KBOX>
struct PjLay {
    static constexpr int A_ATOM = kBM * kBK * 2;
    static constexpr int B_ATOM = BT * kBK * 2;
    static constexpr int A_BYTES = KBOX * A_ATOM;
    static constexpr int B_BYTES = KBOX * B_ATOM;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int BAR_OFF = STAGES * STAGE;  // full[S], empty[S], acc_full[2], acc_empty[2], TMEM address
    static constexpr int SMEM = BAR_OFF + (2 * STAGES + 4) * 8 + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;
    static constexpr int TMEM_COLS = 2 * BT;
    static_assert(BT % 16 == 0 && BT >= 32 && BT <= 256, "MMA N");
};

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

struct ProjSeg {
    void* out;   // bf16 [n_tok][ld]
    int64_t ld;  // row stride in elements
    int32_t n0;  // weight rows [n0, n1) -> columns [0, n1 - n0) of out
    int32_t n1;
};

struct ProjArgs {
    int32_t n_out, k;
    int64_t n_tok;
    int32_t tiles_n;  // 128-row weight blocks
    int32_t tiles_t;  // token blocks
    int32_t token_fast;  // tile order: token blocks fastest (1) or weight blocks fastest (0)
    int64_t n_tiles;  // tiles_n x tiles_t
    int32_t kb;       // 64-wide K blocks
    int32_t ks;       // K split over ks CTAs per tile (1: persistent grid, no split)
    float* part;      // split: fp32 partial blocks [tile][rank][bt columns][128 rows]
    int32_t bt;       // tokens per tile
    int32_t nseg;
    ProjSeg seg[4];
};

// tile -> (weight block, token block).  The tiles in flight on the grid sweep the
// fastest index while sharing a few blocks of the other, so the operand of the
// fastest index is re-read once per sweep and must stay in L2: the smaller operand
// goes fastest.  Measured on the 8192-token in-projection (weights 63 MB, tokens
// 42 MB): weight-fastest order read 477 MB from DRAM, token-fastest 121 MB.
__device__ __forceinline__ void tile_coords(const ProjArgs& P, int64_t tile, int& wn, int& tt) {
    if (P.token_fast) {
        wn = (int)(tile / P.tiles_t);
        tt = (int)(tile % P.tiles_t);
    } else {
        wn = (int)(tile % P.tiles_n);
        tt = (int)(tile / P.tiles_n);
    }
}

template <int BT, int STAGES, int KBOX>
__global__ void __launch_bounds__(kPjThreads, 2)
    k_proj(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap ta,
           const __grid_constant__ ProjArgs P) {
    using L = PjLay<BT, STAGES, KBOX>;
    griddep_wait();  // launched with programmatic serialization: the previous kernel's results are visible
    griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool split = P.ks > 1;
    const int rank = split ? (int)(blockIdx.x % P.ks) : 0;
    // K blocks of this CTA
    const int kb0 = split ? (int)((int64_t)rank * P.kb / P.ks) : 0;
    const int kb1 = split ? (int)((int64_t)(rank + 1) * P.kb / P.ks) : P.kb;
    const int64_t tile0 = split ? blockIdx.x / P.ks : blockIdx.x;
    const int64_t tstep = split ? P.n_tiles : gridDim.x;  // split: exactly one tile per CTA

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, 4);  // one arrival per epilogue warp
        }
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc(tslot, L::TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;
    bool ok = true;

    if (warp == 0) {
        // ---- TMA producer ------------------------------------------------------------
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tw)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ta)) : "memory");
            uint32_t it = 0;
            for (int64_t tile = tile0; tile < P.n_tiles && ok; tile += tstep) {
                int wn, tt;
                tile_coords(P, tile, wn, tt);
                for (int kb = kb0; kb < kb1; kb += KBOX, ++it) {
                    const int s = (int)(it % STAGES);
                    if (!mbar_wait(empty + s, ((it / STAGES) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    unsigned char* st = sm + s * L::STAGE;
                    const int nbox = (kb1 - kb < KBOX) ? kb1 - kb : KBOX;
                    mbar_arrive_expect_tx(full + s, (uint32_t)(nbox * (L::A_ATOM + L::B_ATOM)));
                    for (int a = 0; a < nbox; ++a)
                        tma_load_2d(st + a * L::A_ATOM, &tw, (kb + a) * kBK, wn * kBM, full + s);
                    for (int a = 0; a < nbox; ++a)
                        tma_load_2d(st + L::A_BYTES + a * L::B_ATOM, &ta, (kb + a) * kBK, tt * BT, full + s);
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer --------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kBM, BT);
            uint32_t it = 0, use = 0;
            for (int64_t tile = tile0; tile < P.n_tiles && ok; tile += tstep, ++use) {
                const uint32_t buf = use & 1u;
                if (!mbar_wait(acc_empty + buf, ((use >> 1) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint32_t d = tm + buf * BT;
                for (int kb = kb0; kb < kb1; kb += KBOX, ++it) {
                    const int s = (int)(it % STAGES);
                    if (!mbar_wait(full + s, (it / STAGES) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t a0 = tc::smem_addr(sm + s * L::STAGE);
                    const uint32_t b0 = a0 + L::A_BYTES;
                    const int nbox = (kb1 - kb < KBOX) ? kb1 - kb : KBOX;
                    for (int a = 0; a < nbox; ++a)
#pragma unroll
                        for (int k16 = 0; k16 < kBK / 16; ++k16)
                            mma_bf16(d, tc::sdesc(a0 + a * L::A_ATOM + k16 * 32),
                                     tc::sdesc(b0 + a * L::B_ATOM + k16 * 32), idesc,
                                     (kb > kb0 || a > 0 || k16 > 0) ? 1u : 0u);
                    tc::commit(empty + s);  // the stage is free once these MMAs have read it
                }
                if (!ok) break;
                tc::commit(acc_full + buf);
            }
        }
    } else {
        // ---- epilogue: warps 2..5 own TMEM lane quadrants 2, 3, 0, 1 ----------------------
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;  // weight row inside the tile
        uint32_t use = 0;
        for (int64_t tile = tile0; tile < P.n_tiles; tile += tstep, ++use) {
            const uint32_t buf = use & 1u;
            int wn, tt;
            tile_coords(P, tile, wn, tt);
            const bool w = mbar_wait(acc_full + buf, (use >> 1) & 1u);
            ok = ok && w;
            if (!__all_sync(0xffffffffu, w)) break;
            tc::fence_after();
            const uint32_t ta_acc = tc::taddr(tm, 32 * q4, (int)(buf * BT));
            const int n = wn * kBM + row;
            // destination of this thread's output channel
            unsigned char* dst = nullptr;
            int64_t ld = 0;
#pragma unroll
            for (int sgi = 0; sgi < 4; ++sgi)
                if (sgi < P.nseg && n >= P.seg[sgi].n0 && n < P.seg[sgi].n1) {
                    dst = static_cast<unsigned char*>(P.seg[sgi].out) + (size_t)(n - P.seg[sgi].n0) * 2;
                    ld = P.seg[sgi].ld;
                }
            const int64_t t0 = (int64_t)tt * BT;
            if (!split) {
                const int ncol = (int)((P.n_tok - t0) < BT ? (P.n_tok - t0) : BT);
#pragma unroll 1
                for (int c0 = 0; c0 < ncol; c0 += 16) {
                    float v[16];
                    tc::ld16(ta_acc + c0, v);
                    if (dst) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int64_t t = t0 + c0 + c;
                            if (t < P.n_tok)
                                *reinterpret_cast<__nv_bfloat16*>(dst + (size_t)t * ld * 2) = __float2bfloat16_rn(v[c]);
                        }
                    }
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(acc_empty + buf)) : "memory");
            }
            // split: the one accumulator goes to the workspace below
        }
    }

    if (split && warp >= 2 && __all_sync(0xffffffffu, ok)) {  // TMEM loads are warp-collective
        // this CTA's partial block -> workspace, column-major (a warp stores 32
        // consecutive rows of one column: 128 contiguous bytes); columns past the
        // last token are skipped
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        int wn0, tt;
        tile_coords(P, tile0, wn0, tt);
        (void)wn0;
        const int64_t t0 = (int64_t)tt * BT;
        const int ncol = (int)((P.n_tok - t0) < BT ? (P.n_tok - t0) : BT);
        float* dst = P.part + ((size_t)tile0 * P.ks + rank) * BT * kBM + row;
        const uint32_t ta_acc = tc::taddr(tm, 32 * q4, 0);
#pragma unroll 1
        for (int c0 = 0; c0 < ncol; c0 += 16) {
            float v[16];
            tc::ld16(ta_acc + c0, v);
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (c0 + c < ncol) dst[(size_t)(c0 + c) * kBM] = v[c];
        }
    }
    tc::fence_before();
    __syncthreads();
    if (!ok && (lane == 0)) report_device_status(kDevWaitTimeout);
    if (warp == 1) tc::dealloc(tm, L::TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// bf16 [rows][k] row-major, boxes of 64 (k) x box_rows, 128-byte swizzle,
// reads past the end filled with zeros
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int k, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}



// fp32 partial blocks of a split tile -> bf16 outputs.  One warp per (tile,
// column = token): lane l adds rows 4l .. 4l+3 of the ks partial blocks (16-byte
// loads, all ranks' loads issued before the adds) in rank order and stores the 4
// bf16 results, which sit side by side in the output row of that token.
constexpr int kRedWarps = 8;
__global__ void __launch_bounds__(32 * kRedWarps) k_proj_reduce(const __grid_constant__ ProjArgs P) {
    griddep_wait();
    griddep_launch_dependents();
    const int BT = P.bt;
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * kRedWarps + (threadIdx.x >> 5);  // tile * BT + column
    const int64_t tile = item / BT;
    const int c = (int)(item % BT);
    if (tile >= P.n_tiles) return;
    int wn, tt;
    tile_coords(P, tile, wn, tt);
    const int64_t t = (int64_t)tt * BT + c;
    if (t >= P.n_tok) return;
    const float4* src = reinterpret_cast<const float4*>(P.part + ((size_t)tile * P.ks * BT + c) * kBM) + lane;
    const size_t rstride = (size_t)BT * kBM / 4;  // float4s between ranks
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int r = 0;
    for (; r + 4 <= P.ks; r += 4) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = src[(size_t)(r + q) * rstride];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc.x += v[q].x;
            acc.y += v[q].y;
            acc.z += v[q].z;
            acc.w += v[q].w;
        }
    }
    for (; r < P.ks; ++r) {
        const float4 v = src[(size_t)r * rstride];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    const float o4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int n = wn * kBM + 4 * lane + e;
#pragma unroll
        for (int sgi = 0; sgi < 4; ++sgi)
            if (sgi < P.nseg && n >= P.seg[sgi].n0 && n < P.seg[sgi].n1)
                static_cast<__nv_bfloat16*>(P.seg[sgi].out)[(size_t)t * P.seg[sgi].ld + (n - P.seg[sgi].n0)] =
                    __float2bfloat16_rn(o4[e]);
    }
}

template <int BT, int STAGES, int KBOX>
cudaError_t launch_tiles(const CUtensorMap& mw, const CUtensorMap& ma, const ProjArgs& P, int ctas_per_sm,
                         cudaStream_t st) {
    using L = PjLay<BT, STAGES, KBOX>;
    static std::atomic<uint64_t> smem_set{0};
    {
        const cudaError_t e = raise_smem_limit(k_proj<BT, STAGES, KBOX>, L::SMEM_ALLOC, smem_set);
        if (e != cudaSuccess) return e;
    }
    const int64_t slots = (int64_t)sm_count() * ctas_per_sm;
    const int64_t grid = P.ks > 1 ? P.n_tiles * P.ks : (P.n_tiles < slots ? P.n_tiles : slots);
    cudaError_t e = launch_pdl(k_proj<BT, STAGES, KBOX>, dim3((unsigned)grid), dim3(kPjThreads), L::SMEM_ALLOC, st,
                               mw, ma, P);
    if (e != cudaSuccess || P.ks == 1) return e;
    const int64_t items = P.n_tiles * BT;
    return launch_pdl(k_proj_reduce, dim3((unsigned)((items + kRedWarps - 1) / kRedWarps)), dim3(32 * kRedWarps), 0,
                      st, P);
}

}  // namespace

cudaError_t take_device_status_proj(unsigned* out) { return take_device_status_tu(out); }

// The launch shape depends on the shapes only (so the workspace a call needs is
// known without a device): up to 64 tokens use 64-token tiles (1 CTA per SM),
// more use 256-token tiles (1 CTA per SM, persistent).  When the tiles would
// leave most of the GPU idle, K is split over ks CTAs per tile so that about
// kSplitCtas CTAs run, each with at least 2 K blocks; their fp32 partials take
// ks x BT x 128 x 4 bytes per tile of workspace.  An MMA instruction costs
// about the same at N = 64 as at N = 256, so a decode projection is bound by
// its instruction count per SM as much as by its weight bytes: splitting until
// about one CTA runs per SM (not two) measured fastest, the extra partial
// traffic and the reduction launch costing more beyond that.
constexpr int kSplitCtas = 148;

ProjPlan proj_plan(int32_t n_out, int32_t k, int64_t n_tok) {
    ProjPlan p;
    p.bt = n_tok <= 64 ? 64 : 256;
    const int64_t tiles_n = (n_out + kBM - 1) / kBM;
    p.n_tiles = tiles_n * ((n_tok + p.bt - 1) / p.bt);
    const int kb = (k + kBK - 1) / kBK;
    p.ks = 1;
    int target = kSplitCtas;
    if (const char* e = std::getenv("GDN_PROJ_SPLIT_CTAS")) {  // tuning override: CTAs a split aims at
        const int v = std::atoi(e);
        if (v >= 2 && v <= 4096) target = v;
    }
    if (p.n_tiles > 0 && p.n_tiles * 2 <= target) {
        int ks = (int)(target / p.n_tiles);
        if (ks > 16) ks = 16;
        while (ks > 1 && kb / ks < 2) --ks;
        p.ks = ks;
    }
    p.ws_bytes = p.ks > 1 ? (size_t)p.n_tiles * p.ks * p.bt * kBM * 4 : 0;
    return p;
}

cudaError_t launch_proj(const ProjJob& job, cudaStream_t st) {
    if (job.n_tok == 0 || job.n_out == 0) return cudaSuccess;
    const ProjPlan plan = proj_plan(job.n_out, job.k, job.n_tok);
    if (plan.ws_bytes > 0 && (job.ws == nullptr || job.ws_bytes < plan.ws_bytes)) return cudaErrorInvalidValue;
    ProjArgs P = {};
    P.n_out = job.n_out;
    P.k = job.k;
    P.n_tok = job.n_tok;
    P.tiles_n = (job.n_out + kBM - 1) / kBM;
    P.tiles_t = (int32_t)((job.n_tok + plan.bt - 1) / plan.bt);
    P.token_fast = job.n_tok < job.n_out ? 1 : 0;  // the token operand is the smaller one
    P.kb = (job.k + kBK - 1) / kBK;
    P.n_tiles = plan.n_tiles;
    P.ks = plan.ks;
    P.bt = plan.bt;
    P.part = static_cast<float*>(job.ws);
    P.nseg = job.nseg;
    for (int i = 0; i < job.nseg; ++i) P.seg[i] = ProjSeg{job.seg[i].out, job.seg[i].ld, job.seg[i].n0, job.seg[i].n1};
    CUtensorMap mw, ma;
    if (!make_map(&mw, job.w, job.n_out, job.k, kBM) || !make_map(&ma, job.act, job.n_tok, job.k, plan.bt))
        return cudaErrorInvalidValue;
    // few tokens: 3 stages of 2 K blocks (48 KB), one CTA per SM; under graph replay this
    // measured 16.1 us for the 64-token in-projection against 18.4 us for 4 stages of one
    // K block at two CTAs per SM (4 K blocks per stage: 17.0 us)
    if (plan.bt == 64) return launch_tiles<64, 3, 2>(mw, ma, P, 1, st);
    return launch_tiles<256, 4, 1>(mw, ma, P, 1, st);
}

}  // namespace gdn
