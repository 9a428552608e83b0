// gdn_chunk16.cu -- chunkwise (WY / UT-transform) prefill for d_k = d_v = 128,
// chunk 64 and bf16 activations, on tcgen05 tensor cores with fp16 operands
// and fp32 accumulation.
//
// The layer is the gated delta rule of "Hybrid transformers under load: where
// Gated DeltaNet loses to full attention" (braintools.ru, section 3): per
// v-head S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T and
// o_t = S_t q_t.  Over a chunk of C = 64 tokens with gamma = cumsum(log alpha)
// and the state S entering the chunk, the token loop is exactly
//     A   = strict-lower(diag(beta) (K K^T o Gamma)),  T = (I + A)^-1,
//     P   = lower-incl(Q K^T o Gamma),                 T' = T diag(beta),
//     W   = T' diag(e^gamma) K,   U~ = T' V,   U = U~ - W S^T,
//     O   = diag(e^gamma) Q S^T + P U = Q' S^T + X,  Q' = diag(e^gamma) Q - P W,
//                                                     X  = P U~,
//     S  <- e^gamma_C S + U^T diag(e^(gamma_C - gamma)) K,
// with Gamma_ti = e^(gamma_t - gamma_i).  Only the two products with S depend
// on the previous chunk; everything else is per chunk.
//
// Cost model (measured on GB300 with a probe): a tcgen05.mma instruction
// costs about 108 SM cycles to issue whatever its kind (f16, bf16, tf32), M
// (64 or 128) and N (up to 128); N = 256 costs about 155.  kind::f16 covers
// K = 16 per instruction where kind::tf32 covers 8, so fp16 operands halve the
// instruction count at TF32's precision (11-bit significands, rounded to
// nearest; fp32 accumulation).  A rounding emulation of this chain gives a
// relative state error of 3-5e-4 at T = 8192 for mean alpha 0.5 to 0.998,
// the same as TF32.  fp16 holds magnitudes below 65504: far above the
// activations and states of the layer (|S| stays near the scale of v).
//
// Two launches (the conv-state tail of gdn_prefill.cu follows):
//  1. k_prep16, one CTA per (chunk slot, k-head), all chunks at once:
//     conv + SiLU + L2 norm of the k-head's q and k -> [K^; Q^] (fp16) and the
//     Gram [K^ K^T; Q^ K^T] (one M = 128 product); K^ is stored for the chain.
//     Per v-head of the k-head's group: gates, gamma, the masks A and P, and
//     T' = (I + A)^-1 diag(beta): its diagonal 16 x 16 blocks by substitution
//     in fp32, the blocks below by T'_ab = -X_aa sum_c A_ac T'_cb on warp-level
//     fp16 MMAs (fp32 accumulation; a rounding emulation of the chain shows no
//     loss against an exact inverse).  Then [T'; PT'] = [I; P] T' and, in one
//     product over [K^; Q^] (K = 128), the chain's A operand
//         [-W; Q'] = [-[T'; PT'] diag(e^gamma) | 0; diag(e^gamma)] [K^; Q^],
//     and V = silu(conv(x)) of the v-head's channels (while the products run)
//     -> stored fp16 with e^gamma and e^(gamma_C - gamma).  Elementwise work
//     runs on paired fp32 instructions (two lanes per FFMA2 / FMUL2).
//  2. k_chain16, one CTA per (sequence, v-head), chunks in order; the fp32
//     state S^T lives in tensor memory for the whole sequence.  Per chunk:
//       PRE  [U~; X] = [T'; PT'] V                                   (4 MMAs)
//       RA   [U; O]  = [U~; X] + [-W; Q'] S^T                        (8 MMAs)
//       RB   S^T    <- e^gamma_C S^T + K^T (diag(e^(gamma_C - gamma)) U)  (4 MMAs)
//     RA accumulates onto the U~ / X columns that PRE wrote, so U and O come
//     out of tensor memory directly.  Warp roles: a producer lane (bulk
//     copies, every operand double-buffered and requested as soon as its
//     buffer is free), an MMA issuer lane, 8 warps for U' (lanes 0..63) and
//     the S operand after each state update (the chain's critical path), and
//     4 warps for the gated RMSNorm of O -> y.  They hand over through
//     mbarriers, one pair per hand-over (indexed by chunk parity), so that no
//     waiter can see a phase two chunks ahead.
// Every wait is bounded: a wait that gives up sets an abort flag, after which
// the CTA runs to its end without waiting (its results are then undefined)
// and reports kDevWaitTimeout in the device status word.  Reductions have a
// fixed order, so results are bitwise reproducible ("Forge: how I wrote my
// own inference engine", 25-26 August: chunked DeltaNet prefill with
// deterministic reduction).
#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prefill_common.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

namespace gdn {
namespace {

namespace c16 {
constexpr int C = 64, D = 128;
constexpr uint32_t kK = 16384;            // K^ fp16 [64 t][128 d_k]: 2 atoms of [64][64]
constexpr uint32_t kAop = 32768;          // [-W; Q'] fp16 [128][128] K-major SW128: 2 atoms of 128 rows
constexpr uint32_t kTP = 16384;           // [T'; PT'] fp16 [128][64] K-major SW128: 1 atom
constexpr uint32_t kV = 16384;            // V = silu(conv(x)) fp16, MN-major [64 tokens][128]: 2 atoms
constexpr uint32_t kGates = 512;          // e^gamma [64] | e^(gamma_C - gamma) [64], fp32
constexpr uint32_t kRecTP = kAop, kRecV = kAop + kTP, kRecG = kAop + kTP + kV;
constexpr uint32_t kRec = kAop + kTP + kV + kGates;  // per (chunk slot, v-head)

struct Args {
    Geom g;
    LayerParams p;
    PrefillJob J;
    unsigned char* kk;   // [ncs][Hk] kK
    unsigned char* rec;  // [ncs][Hv] kRec
    int64_t ncs;         // chunk slots
    int64_t cs_lo;       // k_prep16 covers chunk slots cs_lo .. cs_lo + grid - 1
    int c_lo, c_hi;      // k_chain16 runs chunks c_lo .. c_hi - 1 of each sequence
    int carry_in;        // k_chain16 starts from the state a previous segment left in s_final
    int prep_wait_end;   // k_prep16 ends with a wait for the grid before it in the stream
    int32_t* ord;        // [n_seq] or null: chain row y runs sequence ord[y] (longest first)
};

size_t align1024(size_t x) { return (x + 1023) & ~(size_t)1023; }

// Sequences a varlen call orders longest first for the chain (more are left in
// their given order: the ranking is one CTA's O(n_seq^2) loop).
constexpr int kOrdMax = 1024;

struct Ws {
    size_t kk, rec, ord, total;  // ord: 0 when there is no order region
    int64_t ncs;
};

Ws ws_layout(const Geom& g, int64_t N, int n_seq) {
    Ws L;
    L.ncs = N / C + n_seq + 1;
    L.kk = 0;
    L.rec = align1024((size_t)L.ncs * g.Hk * kK);
    L.total = align1024(L.rec + (size_t)L.ncs * g.Hv * kRec);
    L.ord = 0;
    if (n_seq > 1 && n_seq <= kOrdMax) {
        L.ord = L.total;
        L.total = align1024(L.ord + (size_t)n_seq * 4);
    }
    return L;
}

// 8 floats -> 8 fp16 in one 16-byte chunk
__device__ __forceinline__ uint4 pack8(const float* v) {
    return make_uint4(tc::pack_h2(v[0], v[1]), tc::pack_h2(v[2], v[3]), tc::pack_h2(v[4], v[5]),
                      tc::pack_h2(v[6], v[7]));
}

// ---------------------------------------------------------------------------
// 1. per-chunk preparation
// ---------------------------------------------------------------------------
// Packed fp32 pairs: sm_100's paired FMA / multiply / add (__ffma2_rn and kin)
// round each lane exactly like the scalar operation, at half the instructions.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {  // two bf16 (element 0 in the low half)
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float tanh_hw(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(x));
    return t;
}

__device__ __forceinline__ float ex2_hw(float x) {  // 2^x; x <= 0 here
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// silu of a pair through one hardware tanh each: x sigma(x) = h + h tanh(h), h = x / 2
__device__ __forceinline__ float2 silu2(float2 x) {
    const float2 hh = __fmul2_rn(x, make_float2(0.5f, 0.5f));
    return __ffma2_rn(hh, make_float2(tanh_hw(hh.x), tanh_hw(hh.y)), hh);
}

__device__ __forceinline__ uint4 pack8x2(const float2 v[4]) {
    return make_uint4(tc::pack_h2(v[0].x, v[0].y), tc::pack_h2(v[1].x, v[1].y), tc::pack_h2(v[2].x, v[2].y),
                      tc::pack_h2(v[3].x, v[3].y));
}

// warp-level fp16 tensor-core pieces of the triangular merges (m16n8k16, fp32
// accumulation): fragments straight from shared memory
__device__ __forceinline__ void ldsm_x4(uint32_t r[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(tc::smem_addr(p)));
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t r[2], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(tc::smem_addr(p)));
}

__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], const uint32_t b[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// 4-channel forms of the conv helpers (a thread owns 4 channels: two pairs)
__device__ __forceinline__ void unpack4x2(const uint2& u, float2 f[2]) {
    f[0] = bf2_to_f2(u.x);
    f[1] = bf2_to_f2(u.y);
}

__device__ __forceinline__ uint2 pack4x2(const float2 v[2]) {
    return make_uint2(tc::pack_h2(v[0].x, v[0].y), tc::pack_h2(v[1].x, v[1].y));
}

// conv + SiLU of NT tokens for 4 channels (two pairs); row(k) returns packed bf16 row k,
// rows i .. i+3 are the window of token i
template <int NT, typename Row, typename Emit>
__device__ __forceinline__ void conv4x2(Row row, const float2 w[4][2], const float2 bias[2], bool raw, Emit emit) {
    float2 win[4][2];
#pragma unroll
    for (int r = 1; r < 4; ++r) unpack4x2(row(r - 1), win[r]);
#pragma unroll
    for (int i = 0; i < NT; ++i) {
#pragma unroll
        for (int r = 0; r < 3; ++r)
#pragma unroll
            for (int c = 0; c < 2; ++c) win[r][c] = win[r + 1][c];
        unpack4x2(row(i + 3), win[3]);
        float2 u[2];
        if (raw) {
            u[0] = win[3][0];
            u[1] = win[3][1];
        } else {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float2 s = bias[c];
#pragma unroll
                for (int r = 0; r < 4; ++r) s = __ffma2_rn(w[r][c], win[r][c], s);
                u[c] = silu2(s);
            }
        }
        emit(i, u);
    }
}

// window-row weights of 4 channels from the [4][K] bf16 taps at `src` (8-byte aligned)
__device__ __forceinline__ void conv_weights4x2(const __nv_bfloat16* src, int K, float2 w[4][2]) {
    float f[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) f[r][c] = 0.f;
    const uint2* s2 = reinterpret_cast<const uint2*>(src);
    auto unpack_taps = [&](auto kk) {
        constexpr int KK = decltype(kk)::value;
        float t[4 * KK];
#pragma unroll
        for (int v = 0; v < KK; ++v) {
            const uint2 u = s2[v];
            const float2 a = bf2_to_f2(u.x), b = bf2_to_f2(u.y);
            t[4 * v] = a.x;
            t[4 * v + 1] = a.y;
            t[4 * v + 2] = b.x;
            t[4 * v + 3] = b.y;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int m = 0; m < KK; ++m) f[4 - KK + m][c] = t[c * KK + m];
    };
    if (K == 4) unpack_taps(std::integral_constant<int, 4>{});
    else if (K == 3) unpack_taps(std::integral_constant<int, 3>{});
    else unpack_taps(std::integral_constant<int, 2>{});
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        w[r][0] = make_float2(f[r][0], f[r][1]);
        w[r][1] = make_float2(f[r][2], f[r][3]);
    }
}

__device__ __forceinline__ void bias4x2(const LayerParams& p, int ch, float2 b[2]) {
    b[0] = b[1] = make_float2(0.f, 0.f);
    if (p.conv_b) {
        const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.conv_b) + ch);
        b[0] = bf2_to_f2(u.x);
        b[1] = bf2_to_f2(u.y);
    }
}

constexpr int P_THREADS = 256;
constexpr int kXRows = C + 3;                              // staged x rows: tokens t0-3 .. t0+63
constexpr uint32_t kStage = kXRows * 512;                  // q/k rows, or the v rows of 2 v-heads
constexpr uint32_t kStageV = kXRows * 256;                 // the v rows of one v-head
constexpr uint32_t P_KQ = 0;                               // [K^; Q^] fp16 [128][128], atoms of 128 rows
constexpr uint32_t P_SCR = 32768;                          // scratch of one v-head (staging before it):
constexpr uint32_t P_IP = P_SCR;                           //   [I; P] fp16 K-major [128][64]
constexpr uint32_t P_TB = P_IP + 16384;                    //   T' fp16 MN-major [64 (k)][64]
constexpr int kBLd = 24;                                   //   row stride (halves) of the 16 x 16 blocks
constexpr uint32_t kBlk = 16 * kBLd * 2;                   //   768 B per block
constexpr uint32_t P_A16 = P_TB + 8192;                    //   A's 6 blocks below the diagonal, fp16
constexpr int kA32Ld = 17;                                 //   (floats)
constexpr uint32_t P_A32 = P_A16 + 6 * kBlk;               //   A's diagonal 16 x 16 blocks fp32 [4][16][17]
constexpr uint32_t P_X16 = P_A32 + 4 * 16 * kA32Ld * 4;    //   (I + A)^-1's diagonal blocks fp16 [4] blocks
constexpr uint32_t P_Y = P_X16 + 4 * kBlk;                 //   a 16 x 8 fp16 tile per warp
constexpr uint32_t P_SCR_END = P_Y + 8 * 256;
constexpr uint32_t P_WA = P_SCR;                           //   later [-T'e, 0; -PT'e, diag(e^gamma)] [128][128]
constexpr uint32_t P_STG = P_SCR;                          //   before: the staged raw x rows
constexpr uint32_t P_WV = P_SCR_END;                       // conv taps of the 2 staged v-heads (2 x 1 KB)
constexpr uint32_t P_SMALL = P_WV + 2048;                  // gamma log2(e), beta, e^gamma, e^(gamma_C - gamma)
constexpr uint32_t P_SMEM = P_SMALL + 4 * C * 4 + 16;      //   [64] each; mbarrier; TMEM slot
constexpr uint32_t P_SMEM_ALLOC = P_SMEM + 1024;
constexpr uint32_t P_TMEM_COLS = 128;                      // Gram (0..63) | [T'; PT'] (64..127), then [-W; Q']
constexpr int P_CTAS_PER_SM = 3;
static_assert(P_WA + 32768 <= P_SCR_END && P_STG + kStage <= P_SCR_END, "overlays of the scratch");
static_assert((P_IP & 1023) == 0 && (P_TB & 1023) == 0 && (P_A16 & 15) == 0 && (P_X16 & 15) == 0 &&
                  (P_Y & 15) == 0 && (P_WV & 15) == 0,
              "operand alignment");
static_assert(P_CTAS_PER_SM * (P_SMEM_ALLOC + 1024) <= 233472, "three CTAs per SM");

// byte offset of row r, column c (fp16) of block b of the packed 16 x 16 blocks
__device__ __forceinline__ uint32_t blk_off(int b, int r, int c) { return (uint32_t)(b * kBlk + (r * kBLd + c) * 2); }
// packed index of A's block (a, c) below the diagonal (a > c)
__device__ __forceinline__ int low_blk(int a, int c) { return a * (a - 1) / 2 + c; }

__global__ void __launch_bounds__(P_THREADS, P_CTAS_PER_SM) k_prep16(const __grid_constant__ Args A) {
    using L = Act<__nv_bfloat16>;
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv, G = g.G, K = g.K, Cch = g.C_ch;
    const int h = blockIdx.x;
    const int64_t cs = A.cs_lo + (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
    if (cs >= A.ncs) return;
    // Sequences longest first for the chain (one CTA per sequence and v-head, one
    // per SM, so the longest should start first): rank by length, ties by index.
    if (A.ord && cs == 0 && h == 0) {
        const int ns = J.n_seq;
        for (int i = threadIdx.x; i < ns; i += P_THREADS) {
            const int li = J.cu_seqlens[i + 1] - J.cu_seqlens[i];
            int rk = 0;
            for (int k = 0; k < ns; ++k) {
                const int lk = __ldg(J.cu_seqlens + k + 1) - __ldg(J.cu_seqlens + k);
                rk += (lk > li || (lk == li && k < i)) ? 1 : 0;
            }
            A.ord[rk] = i;
        }
    }
    int sq, n;
    int64_t start, end, t0;
    if (!slot_chunk(J, cs, sq, start, end, t0, n)) return;  // a slot between two sequences' chunks
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hf = warp >> 2;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    unsigned char *sKQ = sm + P_KQ, *sSTG = sm + P_STG, *sIP = sm + P_IP, *sTB = sm + P_TB, *sWA = sm + P_WA;
    unsigned char *sA16 = sm + P_A16, *sX16 = sm + P_X16, *sY = sm + P_Y, *sWV = sm + P_WV;
    float* A32 = reinterpret_cast<float*>(sm + P_A32);
    float* gam2 = reinterpret_cast<float*>(sm + P_SMALL);
    float* bet = gam2 + C;
    float* eg = bet + C;
    float* erev = eg + C;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(erev + C);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 1);
    const bool raw = g.flags & kFlagRawQKV;
    const bool direct = g.flags & kFlagGatesDirect;
    int slot_ok;
    const __nv_bfloat16* cin = static_cast<const __nv_bfloat16*>(seq_conv_in(J, g, sq, slot_ok));
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(J.x);
    const __nv_bfloat16* cw = static_cast<const __nv_bfloat16*>(A.p.conv_w);

    // stage x rows tau = t0-3+r (r < kXRows), 32 chunks of 16 bytes per row: chunk ci
    // of row r goes to dst(r, ci) from channel ch (negative: not staged).  Rows before
    // the sequence come from its conv state (or are zero), rows past its end are zero.
    auto stage_rows = [&](auto dst, int ch) {
        const int ci = tid & 31;
        if (ch < 0) return;
        for (int r = tid >> 5; r < kXRows; r += P_THREADS / 32) {
            const int64_t tau = t0 - 3 + r;
            unsigned char* d = dst(r, ci);
            if (tau >= start && tau < end) cp_async16(d, x + (size_t)tau * Cch + ch);
            else if (tau < start && cin && tau - start >= -(K - 1))
                cp_async16(d, cin + (size_t)((K - 1) + (tau - start)) * Cch + ch);
            else *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
        }
    };
    // the v rows and conv taps of v-heads 2p and 2p + 1 of the group
    auto stage_pair = [&](int p) {
        const int u = (tid & 31) >> 4;
        const int jh = h * G + 2 * p + u;
        const bool live = 2 * p + u < G;
        stage_rows([&](int r, int ci) { return sSTG + (ci >> 4) * kStageV + r * 256 + (ci & 15) * 16; },
                   live ? 2 * Hk * D + jh * D + (tid & 15) * 8 : -1);
        if (!raw && tid < 2 * 16 * K) {  // 128 channels x K taps of each v-head: 16 K chunks of 16 bytes
            const int uu = tid / (16 * K), f = tid % (16 * K);
            if (2 * p + uu < G)
                cp_async16(sWV + uu * 1024 + f * 16, cw + (size_t)(2 * Hk * D + (h * G + 2 * p + uu) * D) * K + f * 8);
        }
        cp_async_commit();
    };

    // ---- prologue: stage the k-head's q and k rows (chunks 0..15 q, 16..31 k) -------------
    stage_rows([&](int r, int ci) { return sSTG + r * 512 + ci * 16; },
               ((tid & 31) < 16 ? h : Hk + h) * D + (tid & 15) * 8);
    cp_async_commit();
    if (warp == 0) tc::alloc(tslot, P_TMEM_COLS);
    if (tid == 0) {
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    // gate inputs of tokens lane and lane + 32 of the first v-head (warp 0)
    float ga[2] = {0.f, 0.f}, gb[2] = {0.f, 0.f};
    auto load_gates = [&](int j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = lane + 32 * e;
            if (t < n) {
                const size_t tok = (size_t)(t0 + t);
                ga[e] = L::ld(J.a, tok * Hv + j);
                gb[e] = L::ld(J.b, tok * Hv + j);
            }
        }
    };
    if (warp == 0) load_gates(h * G);
    // q/k thread: warps 0..3 q, 4..7 k; lane = 4 channels; warp & 3 = a block of 16 tokens
    const bool is_q = warp < 4;
    const int ch_qk = (is_q ? h : Hk + h) * D + lane * 4;
    float2 wqk[4][2], bqk[2];
    if (raw) {
#pragma unroll
        for (int r = 0; r < 4; ++r) wqk[r][0] = wqk[r][1] = make_float2(0.f, 0.f);
    } else {
        conv_weights4x2(cw + (size_t)ch_qk * K, K, wqk);
    }
    bias4x2(A.p, ch_qk, bqk);
    cp_async_wait_all();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;

    // ---- conv + SiLU + L2 norm of q and k -> rows 0..63 K^, 64..127 Q^ -------------------
    {
        const int tt0 = (warp & 3) * 16;
        const unsigned char* xr = sSTG + tt0 * 512 + (is_q ? 0 : 256) + lane * 8;
        const int d0 = lane * 4;
        unsigned char* atom = sKQ + (d0 >> 6) * 16384;
        const int cc = (d0 & 63) >> 3, sub = (d0 & 7) * 2;
        const float qs = is_q ? g.q_scale : 1.f;
        const bool l2 = !(g.flags & kFlagNoL2);
        conv4x2<16>([&](int k) { return *reinterpret_cast<const uint2*>(xr + k * 512); }, wqk, bqk, raw,
                    [&](int i, float2 u[2]) {
                        const int t = tt0 + i;
                        const float2 s2 = __ffma2_rn(u[1], u[1], __fmul2_rn(u[0], u[0]));
                        float ss = s2.x + s2.y;
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                        float scale = l2 ? qs * rsqrtf(ss + g.l2_eps) : qs;
                        if (t >= n) scale = 0.f;  // zero past the sequence end
                        float2 v[2] = {__fmul2_rn(u[0], make_float2(scale, scale)),
                                       __fmul2_rn(u[1], make_float2(scale, scale))};
                        *reinterpret_cast<uint2*>(atom + tc::h_off(is_q ? C + t : t, cc) + sub) = pack4x2(v);
                    });
    }
    fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    stage_pair(0);  // over the q/k rows, which are consumed
    if (tid == 0) {  // K^ for the chain: the first 64 rows of each atom
        unsigned char* dst = A.kk + ((size_t)cs * Hk + h) * kK;
        bulk_s2g(dst, sKQ, 8192);
        bulk_s2g(dst + 8192, sKQ + 16384, 8192);
        bulk_commit();
    }
    uint32_t phase = 0;
    bool ok = true;
    auto wait_mma = [&]() {
        bool w = true;
        if (warp == 0) {
            w = mbar_wait(mbar, phase);
            if (!w) w = mbar_wait(mbar, phase);
        }
        phase ^= 1u;
        ok = __syncthreads_and(ok && w);
        tc::fence_after();
    };
    // [K^ K^T; Q^ K^T] = [K^; Q^] K^T into columns 0..63 (B = the K^ rows of the same tile)
    auto issue_gram = [&]() {
        if (tid == 0) {
            tc::fence_after();
            if (ok) {
                const uint32_t a0 = tc::smem_addr(sKQ);
                for (int s = 0; s < D / 16; ++s) {
                    const uint64_t d = tc::sdesc_lbo(a0 + (uint32_t)((s >> 2) * 16384 + (s & 3) * 32), 16);
                    tc::mma_f16(tm, d, d, tc::idesc_f16(128, 64, false, false), s > 0 ? 1u : 0u);
                }
            }
            tc::commit(mbar);
        }
    };
    issue_gram();

    // V = silu(conv(x)) of v-head slot u (0, 1) of the staged pair, head j: thread = 4
    // channels x 8 tokens, straight to the record (MN-major [64 tokens][128] fp16)
    auto v_conv = [&](int u, int j) {
        const int cgp = tid & 31, tg = tid >> 5;
        float2 w[4][2], bias[2];
        if (raw) {
#pragma unroll
            for (int r = 0; r < 4; ++r) w[r][0] = w[r][1] = make_float2(0.f, 0.f);
        } else {
            conv_weights4x2(reinterpret_cast<const __nv_bfloat16*>(sWV + u * 1024) + cgp * 4 * K, K, w);
        }
        bias4x2(A.p, 2 * Hk * D + j * D + cgp * 4, bias);
        const unsigned char* xr = sSTG + u * kStageV + 8 * tg * 256 + cgp * 8;
        const int d0 = cgp * 4;
        unsigned char* vat = A.rec + ((size_t)cs * Hv + j) * kRec + kRecV + (d0 >> 6) * 8192;
        const int cc = (d0 & 63) >> 3, sub = (d0 & 7) * 2;
        conv4x2<8>([&](int k) { return *reinterpret_cast<const uint2*>(xr + k * 256); }, w, bias, raw,
                   [&](int i, float2 uu[2]) {
                       const int t = 8 * tg + i;
                       if (t >= n) uu[0] = uu[1] = make_float2(0.f, 0.f);  // zero past the sequence end
                       *reinterpret_cast<uint2*>(vat + tc::h_off(t, cc) + sub) = pack4x2(uu);
                   });
    };

    for (int jj = 0; jj < G; ++jj) {
        const int j = h * G + jj;
        unsigned char* rec = A.rec + ((size_t)cs * Hv + j) * kRec;
        // ---- V of the pair at its first v-head (the staged rows use the scratch) ----------
        if ((jj & 1) == 0) {
            if (jj > 0) {
                stage_pair(jj / 2);  // the scratch is free: the previous [-W; Q'] product is done
            }
            cp_async_wait_all();
            __syncthreads();
            v_conv(0, j);
            if (jj + 1 < G) v_conv(1, j + 1);
        }
        // ---- gates (warp 0): g, beta of tokens lane, lane + 32; gamma = cumsum(g) ----------
        if (warp == 0) {
            const float alog = direct ? 0.f : A.p.A_log[j];
            const float dtb = (!direct && A.p.dt_bias) ? A.p.dt_bias[j] : 0.f;
            float gl[2], be[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                gl[e] = 0.f;
                be[e] = 0.f;
                if (lane + 32 * e < n) gates(ga[e], gb[e], alog, dtb, direct, gl[e], be[e]);
            }
            if (jj + 1 < G) load_gates(j + 1);  // the next v-head's inputs, in flight meanwhile
            float run = 0.f;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = gl[e];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, v, off);
                    if (lane >= off) v += o;
                }
                gl[e] = v + run;
                run = __shfl_sync(0xffffffffu, gl[e], 31);
            }
            const float gC = run;
            float* rg = reinterpret_cast<float*>(rec + kRecG);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = lane + 32 * e;
                const float ev = expf(gl[e]), er = expf(gC - gl[e]);
                gam2[t] = gl[e] * 1.4426950408889634f;
                bet[t] = be[e];
                eg[t] = ev;
                erev[t] = er;
                rg[t] = ev;
                rg[C + t] = er;
            }
        }
        wait_mma();  // the Gram of this v-head (ends with a CTA barrier)
        // ---- masks from the Gram: A = strict-lower(beta_t Gamma o K^K^T) (TMEM lanes 0..63),
        // P = lower-incl(Gamma o Q^K^T) (lanes 64..127); Gamma_ti = 2^(gamma2_t - gamma2_i) ------
        for (int f = tid; f < C * 8; f += P_THREADS) {  // identity rows of [I; P]
            const int r = f >> 3, cc = f & 7;
            // fp16 1.0 at column r: word (r & 7) / 2 of chunk r / 8, high half for odd r
            const uint32_t one = (r >> 3) == cc ? ((r & 1) ? 0x3C000000u : 0x00003C00u) : 0u;
            const int wsel = (r & 7) >> 1;
            *reinterpret_cast<uint4*>(sIP + tc::h_off(r, cc)) =
                make_uint4(wsel == 0 ? one : 0u, wsel == 1 ? one : 0u, wsel == 2 ? one : 0u, wsel == 3 ? one : 0u);
        }
        {
            const bool isA = q4 < 2;
            const int rb = q4 & 1;             // row half: rows 32 rb .. 32 rb + 31
            const int t = 32 * rb + lane;
            if (hf > rb) {                     // above the diagonal: A unused, P zero
                if (!isA) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(sIP + tc::h_off(C + t, 4 * hf + k)) = make_uint4(0, 0, 0, 0);
                }
            } else {
                const float gt = gam2[t];
                const float bt = isA ? bet[t] : 1.f;
                const bool diag = hf == rb;
                const int tb = t >> 4;
                // one 16-column block at a time: 8 pairs
#pragma unroll 1
                for (int bq = 0; bq < 2; ++bq) {
                    const int cb = 2 * hf + bq;
                    float v[16];
                    tc::ld16(tc::taddr(tm, 32 * q4, 16 * cb), v);  // warp-collective: every lane loads
                    if (isA && cb > tb) continue;  // above the diagonal: unused
                    const float2* g2 = reinterpret_cast<const float2*>(gam2 + 16 * cb);
                    float2 m[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float2 d = __ffma2_rn(g2[c], make_float2(-1.f, -1.f), make_float2(gt, gt));
                        const float2 e = make_float2(ex2_hw(fminf(d.x, 0.f)), ex2_hw(fminf(d.y, 0.f)));
                        m[c] = __fmul2_rn(__fmul2_rn(e, make_float2(v[2 * c], v[2 * c + 1])), make_float2(bt, bt));
                        if (diag) {  // strictly below (A) or on / below (P) the diagonal
                            const int i0 = 16 * cb + 2 * c;
                            if (isA ? i0 >= t : i0 > t) m[c].x = 0.f;
                            if (isA ? i0 + 1 >= t : i0 + 1 > t) m[c].y = 0.f;
                        }
                    }
                    if (!isA) {
                        *reinterpret_cast<uint4*>(sIP + tc::h_off(C + t, 2 * cb)) = pack8x2(m);
                        *reinterpret_cast<uint4*>(sIP + tc::h_off(C + t, 2 * cb + 1)) = pack8x2(m + 4);
                    } else if (cb < tb) {  // below the diagonal -> fp16 block (tb, cb)
                        uint4* dst = reinterpret_cast<uint4*>(sA16 + blk_off(low_blk(tb, cb), t & 15, 0));
                        dst[0] = pack8x2(m);
                        dst[1] = pack8x2(m + 4);
                    } else {  // the diagonal block -> fp32 A32
                        float* dst = A32 + (tb * 16 + (t & 15)) * kA32Ld;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            dst[2 * c] = m[c].x;
                            dst[2 * c + 1] = m[c].y;
                        }
                    }
                }
            }
        }
        tc::fence_before();
        __syncthreads();
        // ---- T' = (I + A)^-1 diag(beta) -> sTB (MN-major: row k holds T'[k][0..63]) --------
        // diagonal 16 x 16 blocks by register-resident substitution (fp32): lane = column
        // jc of block b; once x_k is final, every later row takes -A_ik x_k.  The blocks
        // above the diagonal are zero.
        if (warp < 2) {
            const int b = 2 * warp + (lane >> 4), jc = lane & 15, lb = lane & 16;
            const float* ab = A32 + b * 16 * kA32Ld;
            float acol[16], xv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                acol[i] = ab[i * kA32Ld + jc];
                xv[i] = i == jc ? 1.f : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 15; ++k) {
#pragma unroll
                for (int i = k + 1; i < 16; ++i) xv[i] = fmaf(-__shfl_sync(0xffffffffu, acol[i], lb + k), xv[k], xv[i]);
            }
            const float bj = bet[16 * b + jc];
            const int col = 16 * b + jc;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                *reinterpret_cast<__half*>(sX16 + blk_off(b, i, jc)) = __float2half_rn(xv[i]);
                *reinterpret_cast<__half*>(sTB + tc::h_off(16 * b + i, col >> 3) + (col & 7) * 2) =
                    __float2half_rn(xv[i] * bj);
            }
        } else {
            // zeros above the diagonal blocks: row r, 16-byte chunk cc with cc / 2 > r / 16
            const int f = tid - 64;
            int r, cc;
            if (f < 96) {
                r = f / 6;
                cc = 2 + f % 6;
            } else if (f < 160) {
                r = 16 + (f - 96) / 4;
                cc = 4 + (f - 96) % 4;
            } else {
                r = 32 + (f - 160) / 2;
                cc = 6 + (f - 160) % 2;
            }
            *reinterpret_cast<uint4*>(sTB + tc::h_off(r, cc)) = make_uint4(0, 0, 0, 0);
        }
        __syncthreads();
        // the blocks below the diagonal, row block a = 1..3 after the rows above it:
        // T'_ab = -X_aa sum_{c=b}^{a-1} A_ac T'_cb, one 16 x 8 tile (b, column half nh)
        // per warp, fp16 operands with fp32 accumulation
#pragma unroll 1
        for (int a = 1; a < 4; ++a) {
            if (warp < 2 * a) {
                const int b = warp >> 1, nh = warp & 1;
                const int gq = lane >> 2, t4 = lane & 3;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int c = b; c < a; ++c) {
                    uint32_t af[4], bfr[2];
                    ldsm_x4(af, sA16 + blk_off(low_blk(a, c), lane & 15, (lane >> 4) * 8));
                    ldsm_x2_trans(bfr, sTB + tc::h_off(16 * c + (lane & 15), 2 * b + nh));
                    mma16816(acc, af, bfr);
                }
                uint32_t* yw = reinterpret_cast<uint32_t*>(sY + warp * 256);
                yw[gq * 4 + t4] = tc::pack_h2(acc[0], acc[1]);
                yw[(gq + 8) * 4 + t4] = tc::pack_h2(acc[2], acc[3]);
                __syncwarp();
                uint32_t xf[4], yf[2];
                ldsm_x4(xf, sX16 + blk_off(a, lane & 15, (lane >> 4) * 8));
                ldsm_x2_trans(yf, sY + warp * 256 + (lane & 15) * 16);
                float o[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(o, xf, yf);
                *reinterpret_cast<uint32_t*>(sTB + tc::h_off(16 * a + gq, 2 * b + nh) + 4 * t4) =
                    tc::pack_h2(-o[0], -o[1]);
                *reinterpret_cast<uint32_t*>(sTB + tc::h_off(16 * a + gq + 8, 2 * b + nh) + 4 * t4) =
                    tc::pack_h2(-o[2], -o[3]);
                __syncwarp();  // the scratch tile is rewritten at the next row block
            }
            __syncthreads();
        }
        fence_proxy_async_smem();
        tc::fence_before();
        __syncthreads();
        if (tid == 0) {  // [T'; PT'] = [I; P] T' (M = 128, N = 64, K = 64) into columns 64..127
            tc::fence_after();
            if (ok) {
                const uint32_t a0 = tc::smem_addr(sIP), b0 = tc::smem_addr(sTB);
                for (int s = 0; s < C / 16; ++s)
                    tc::mma_f16(tm + 64, tc::sdesc_lbo(a0 + (uint32_t)(s * 32), 16),
                                tc::sdesc_lbo(b0 + (uint32_t)(s * 2048), 8192), tc::idesc_f16(128, 64, false, true),
                                s > 0 ? 1u : 0u);
            }
            tc::commit(mbar);
        }
        wait_mma();
        {  // [T'; PT'] -> the record tile (K-major [128][64]); -[T'; PT'] diag(e^gamma) -> WA
            const int r = 32 * q4 + lane;
            unsigned char* rtp = rec + kRecTP;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float v[16];
                tc::ld16(tc::taddr(tm, 32 * q4, 64 + hf * 32 + 16 * hh), v);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int cc = 4 * hf + 2 * hh + k;
                    float2 p2[4], s2[4];
                    const float4 e0 = *reinterpret_cast<const float4*>(eg + 8 * cc);
                    const float4 e1 = *reinterpret_cast<const float4*>(eg + 8 * cc + 4);
                    const float2 en[4] = {make_float2(-e0.x, -e0.y), make_float2(-e0.z, -e0.w),
                                          make_float2(-e1.x, -e1.y), make_float2(-e1.z, -e1.w)};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        p2[c] = make_float2(v[8 * k + 2 * c], v[8 * k + 2 * c + 1]);
                        s2[c] = __fmul2_rn(p2[c], en[c]);
                    }
                    *reinterpret_cast<uint4*>(rtp + tc::h_off(r, cc)) = pack8x2(p2);
                    *reinterpret_cast<uint4*>(sWA + tc::h_off(r, cc)) = pack8x2(s2);
                    // the second atom (columns 64..127): zero, with e^gamma_t at column t of row 64 + t
                    uint32_t dw = 0u;
                    if (r >= C && ((r - C) >> 3) == cc) {
                        const uint32_t hb = __half_as_ushort(__float2half_rn(eg[r - C]));
                        dw = ((r - C) & 1) ? (hb << 16) : hb;
                    }
                    const int wsel = ((r - C) & 7) >> 1;
                    *reinterpret_cast<uint4*>(sWA + 16384 + tc::h_off(r, cc)) =
                        make_uint4(wsel == 0 ? dw : 0u, wsel == 1 ? dw : 0u, wsel == 2 ? dw : 0u, wsel == 3 ? dw : 0u);
                }
            }
        }
        fence_proxy_async_smem();
        tc::fence_before();
        __syncthreads();
        if (tid == 0) {  // [-W; Q'] = WA [K^; Q^] (M = 128, N = 128, K = 128) into columns 0..127
            tc::fence_after();
            if (ok) {
                const uint32_t a0 = tc::smem_addr(sWA), b0 = tc::smem_addr(sKQ);
                for (int s = 0; s < 2 * C / 16; ++s)
                    tc::mma_f16(tm, tc::sdesc_lbo(a0 + (uint32_t)((s >> 2) * 16384 + (s & 3) * 32), 16),
                                tc::sdesc_lbo(b0 + (uint32_t)(s * 2048), 16384),
                                tc::idesc_f16(128, 128, false, true), s > 0 ? 1u : 0u);
            }
            tc::commit(mbar);
        }
        wait_mma();
        {  // [-W; Q'] -> the record (K-major [128][128], atoms of 128 rows), from registers
            const int r = 32 * q4 + lane;
            unsigned char* aop = rec + hf * 16384;
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
                float v[16];
                tc::ld16(tc::taddr(tm, 32 * q4, hf * 64 + 16 * b), v);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float2 p2[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) p2[c] = make_float2(v[8 * k + 2 * c], v[8 * k + 2 * c + 1]);
                    *reinterpret_cast<uint4*>(aop + tc::h_off(r, 2 * b + k)) = pack8x2(p2);
                }
            }
        }
        tc::fence_before();
        __syncthreads();  // the columns are read before the next Gram, the scratch before the next staging
        if (jj + 1 < G) issue_gram();
    }
    if (tid == 0) bulk_wait_read_all();
    if (!ok && tid == 0) report_device_status(kDevWaitTimeout);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tm, P_TMEM_COLS);
    // a segment's prep launched beside the previous chain segment completes only after it,
    // so that the next chain segment, launched after this grid, follows both
    if (A.prep_wait_end && tid == 0) griddep_wait();
}

// ---------------------------------------------------------------------------
// 2. the state chain
// ---------------------------------------------------------------------------
constexpr int CH_THREADS = 512;  // 16 warps
// warps 0..7: critical group (TMEM quadrant warp % 4, column half warp / 4);
// 8: producer; 9: MMA issuer; 10, 11, 14, 15: y (quadrants 2, 3); 12, 13: idle
constexpr int W_PROD = 8, W_MMA = 9;
constexpr uint32_t S_K = 0;                         // 2 stages of K^ (16 KB)
constexpr uint32_t S_AS = 32768;                    // 2 stages of [-W; Q'] (32 KB): A of RA
constexpr uint32_t S_TP = S_AS + 2 * kAop;          // 2 stages of [T'; PT'] (16 KB): A of PRE
constexpr uint32_t S_V = S_TP + 2 * kTP;            // 2 stages of V (16 KB): B of PRE
constexpr uint32_t S_SOP = S_V + 2 * kV;            // B of RA: S fp16, MN-major [128 d_k][128 d_v] (32 KB)
constexpr uint32_t S_UP = S_SOP + 32768;            // B of RB: U' fp16, MN-major [64 t][128 d_v] (16 KB)
constexpr uint32_t S_GATES = S_UP + 16384;          // 2 stages of the gate block (512 B each)
constexpr uint32_t S_ORED = S_GATES + 2 * kGates;   // [2][2][64] fp32 half-row sums of squares of O
constexpr uint32_t S_NW = S_ORED + 1024;            // norm_w [128] bf16
constexpr uint32_t S_BAR = S_NW + 256;              // mbarriers
constexpr int NBAR = 24;
constexpr uint32_t S_SMEM = S_BAR + NBAR * 8 + 16;  // + TMEM slot and abort flag
constexpr uint32_t S_SMEM_ALLOC = S_SMEM + 1024;
static_assert(S_SMEM_ALLOC <= 232448, "chain shared memory");
// tensor memory columns: R0 / R1 ([U~; X], then [U; O], of even / odd chunks), S^T (the
// fp32 state, d_k lanes x d_v columns)
constexpr uint32_t T_R0 = 0, T_R1 = 128, T_S = 256, T_COLS = 512;
// barrier pairs (index + chunk parity)
enum {
    B_FULL_K = 0,    // K^ and the gates of a chunk landed (producer, tx)
    B_FULL_A = 2,    // [-W; Q'] landed
    B_FULL_TP = 4,   // [T'; PT'] landed
    B_FULL_V = 6,    // V landed
    B_EMPTY_K = 8,   // K^ and gate stage free (the commit after RB)
    B_PRE = 10,      // PRE complete (commit): [T'; PT'] and V stages free
    B_RA = 12,       // RA complete (commit): [-W; Q'] stage free, [U; O] ready
    B_UP = 14,       // U' written and S^T rescaled in tensor memory (critical group, 256)
    B_RB = 16,       // RB complete (commit)
    B_SOP = 18,      // S operand written (critical group, 256)
    B_OE = 20,       // O rows read from tensor memory (the 4 y warps, 128)
};

__global__ void __launch_bounds__(CH_THREADS, 1) k_chain16(const __grid_constant__ Args A) {
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv;
    const int j = blockIdx.x, seq = A.ord ? A.ord[blockIdx.y] : (int)blockIdx.y, h = j / g.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();  // a following prep segment may start beside this grid

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    unsigned char *sK = sm + S_K, *sAS = sm + S_AS, *sTP = sm + S_TP, *sV = sm + S_V;
    unsigned char *sSOP = sm + S_SOP, *sUP = sm + S_UP;
    float* sG = reinterpret_cast<float*>(sm + S_GATES);  // [2][128]: e^gamma [64] | e^(gamma_C - gamma) [64]
    float* ored = reinterpret_cast<float*>(sm + S_ORED);
    __nv_bfloat16* sNW = reinterpret_cast<__nv_bfloat16*>(sm + S_NW);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + NBAR);
    volatile int* abortp = reinterpret_cast<volatile int*>(tslot + 1);

    int64_t start, end;
    seq_bounds(J, seq, start, end);
    const int64_t T = end - start;
    // this launch's chunks of the sequence: c_lo .. c_hi - 1 (local index c = 0 .. nch - 1)
    const int nch_all = (int)((T + C - 1) / C);
    const int c_lo = A.c_lo, c_hi = A.c_hi < nch_all ? A.c_hi : nch_all;
    const int nch = c_hi > c_lo ? c_hi - c_lo : 0;
    const bool outnorm = !(g.flags & kFlagNoOutNorm);
    const float* Sin = nullptr;
    float* Sout = nullptr;
    if (!J.cu_seqlens) {
        Sout = J.s_final + (size_t)j * D * D;
        // a later segment continues from the state the previous one left in s_final
        Sin = A.carry_in ? Sout : (J.s0 ? J.s0 + (size_t)j * D * D : nullptr);
    } else {
        const int slot = J.slot_idx[seq];
        if (slot >= 0 && slot < J.n_slots) {
            Sout = J.state_pool + ((size_t)slot * Hv + j) * D * D;
            if (J.has_init && J.has_init[seq]) Sin = Sout;
        }
    }

    // ---- set-up: barriers, tensor memory, norm weights -------------------------------
    if (warp == 0) tc::alloc(tslot, T_COLS);
    if (tid == 0) {
        for (int p = 0; p < 2; ++p) {
            mbar_init(bar + B_FULL_K + p, 1);
            mbar_init(bar + B_FULL_A + p, 1);
            mbar_init(bar + B_FULL_TP + p, 1);
            mbar_init(bar + B_FULL_V + p, 1);
            mbar_init(bar + B_EMPTY_K + p, 1);
            mbar_init(bar + B_PRE + p, 1);
            mbar_init(bar + B_RA + p, 1);
            mbar_init(bar + B_UP + p, 256);
            mbar_init(bar + B_RB + p, 1);
            mbar_init(bar + B_SOP + p, 256);
            mbar_init(bar + B_OE + p, 128);
        }
        *abortp = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < D; i += CH_THREADS)
        sNW[i] = outnorm ? static_cast<const __nv_bfloat16*>(A.p.norm_w)[i] : __float2bfloat16(1.f);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;

    auto chunk_t0 = [&](int c) -> int64_t { return start + (int64_t)(c_lo + c) * C; };
    auto chunk_n = [&](int c) -> int {
        const int64_t left = end - chunk_t0(c);
        return (int)(left < C ? left : C);
    };
    auto chunk_slot = [&](int c) -> size_t { return (size_t)(start / C + seq + c_lo + c); };
    // bounded wait; after an abort every wait returns at once
    auto wait = [&](int b, int c) {
        if (*abortp) return;
        if (!mbar_wait(bar + b + (c & 1), (uint32_t)((c >> 1) & 1))) *abortp = 1;
    };
    auto test = [&](int b, int c) -> bool { return mbar_test(bar + b + (c & 1), (uint32_t)((c >> 1) & 1)); };

    if (warp == W_PROD) {
        // =============================== producer ===============================
        // four streams, each issued as soon as its stage is free, in chunk order
        if (lane == 0 && nch > 0) {
            int nk = 0, na = 0, ntp = 0, nv = 0;
            auto src_rec = [&](int c) { return A.rec + (chunk_slot(c) * Hv + j) * kRec; };
            long long t_start = clock64();
            while ((nk < nch || na < nch || ntp < nch || nv < nch) && !*abortp) {
                bool progress = false;
                if (nk < nch && (nk < 2 || test(B_EMPTY_K, nk - 2))) {
                    const int c = nk, s = c & 1;
                    mbar_arrive_expect_tx(bar + B_FULL_K + s, kK + kGates);
                    bulk_g2s(sK + s * kK, A.kk + (chunk_slot(c) * Hk + h) * kK, kK, bar + B_FULL_K + s);
                    bulk_g2s(sG + s * 128, src_rec(c) + kRecG, kGates, bar + B_FULL_K + s);
                    ++nk;
                    progress = true;
                }
                if (na < nch && (na < 2 || test(B_RA, na - 2))) {
                    const int c = na, s = c & 1;
                    mbar_arrive_expect_tx(bar + B_FULL_A + s, kAop);
                    bulk_g2s(sAS + s * kAop, src_rec(c), kAop, bar + B_FULL_A + s);
                    ++na;
                    progress = true;
                }
                if (ntp < nch && (ntp < 2 || test(B_PRE, ntp - 2))) {
                    const int c = ntp, s = c & 1;
                    mbar_arrive_expect_tx(bar + B_FULL_TP + s, kTP);
                    bulk_g2s(sTP + s * kTP, src_rec(c) + kRecTP, kTP, bar + B_FULL_TP + s);
                    ++ntp;
                    progress = true;
                }
                if (nv < nch && (nv < 2 || test(B_PRE, nv - 2))) {
                    const int c = nv, s = c & 1;
                    mbar_arrive_expect_tx(bar + B_FULL_V + s, kV);
                    bulk_g2s(sV + s * kV, src_rec(c) + kRecV, kV, bar + B_FULL_V + s);
                    ++nv;
                    progress = true;
                }
                if (progress) t_start = clock64();
                else if (clock64() - t_start > kWaitLimitCycles) *abortp = 1;
            }
            // no copy may land after the CTA has gone: wait for the last ones (bounded, even after an abort)
            auto drain = [&](int b, int n) {
                for (int c = n - 2 < 0 ? 0 : n - 2; c < n; ++c) mbar_wait(bar + b + (c & 1), (uint32_t)((c >> 1) & 1));
            };
            drain(B_FULL_K, nk);
            drain(B_FULL_A, na);
            drain(B_FULL_TP, ntp);
            drain(B_FULL_V, nv);
        }
    } else if (warp == W_MMA) {
        // =============================== MMA issuer ===============================
        if (lane == 0 && nch > 0) {
            const uint32_t aTP = tc::smem_addr(sTP), aV = tc::smem_addr(sV), aAS = tc::smem_addr(sAS);
            const uint32_t aSOP = tc::smem_addr(sSOP), aUP = tc::smem_addr(sUP), aK = tc::smem_addr(sK);
            constexpr uint32_t idPre = tc::idesc_f16(128, 128, false, true);
            constexpr uint32_t idRa = tc::idesc_f16(128, 128, false, true);
            constexpr uint32_t idRb = tc::idesc_f16(128, 128, true, true);
            uint64_t* last = nullptr;  // barrier of the last commit and its parity
            uint32_t last_par = 0;
            auto commit = [&](int b, int c) {
                tc::commit(bar + b + (c & 1));
                last = bar + b + (c & 1);
                last_par = (uint32_t)((c >> 1) & 1);
            };
            // PRE needs its operands and the [U; O] columns of chunk c-2 read by the y warps
            // (the U' warps read them before RB(c-2), issued earlier)
            auto pre_ready = [&](int c) -> bool {
                return test(B_FULL_TP, c) && test(B_FULL_V, c) && (c < 2 || test(B_OE, c - 2));
            };
            auto issue_pre = [&](int c) {  // [U~; X] = [T'; PT'] V into R(c)
                tc::fence_after();
                if (!*abortp) {
                    const uint32_t a0 = aTP + (uint32_t)((c & 1) * kTP), b0 = aV + (uint32_t)((c & 1) * kV);
                    const uint32_t dcol = (c & 1) ? T_R1 : T_R0;
                    for (int s = 0; s < C / 16; ++s)
                        tc::mma_f16(tm + dcol, tc::sdesc_lbo(a0 + (uint32_t)(s * 32), 16),
                                    tc::sdesc_lbo(b0 + (uint32_t)(s * 2048), 8192), idPre, s > 0 ? 1u : 0u);
                }
                commit(B_PRE, c);
            };
            auto issue_rb = [&](int c) {  // S^T += K^T U'
                tc::fence_after();
                if (!*abortp) {
                    const uint32_t k0 = aK + (uint32_t)((c & 1) * kK);
                    for (int s = 0; s < C / 16; ++s)
                        tc::mma_f16(tm + T_S, tc::sdesc_lbo(k0 + (uint32_t)(s * 2048), 8192),
                                    tc::sdesc_lbo(aUP + (uint32_t)(s * 2048), 8192), idRb, 1u);
                }
                commit(B_RB, c);
                tc::commit(bar + B_EMPTY_K + (c & 1));
            };
            int npre = 0;  // pre-products issued
            for (int c = 0; c < nch; ++c) {
                if (npre == c) {  // the pre-product of this chunk was not ready earlier
                    wait(B_FULL_TP, c);
                    wait(B_FULL_V, c);
                    if (c >= 2) wait(B_OE, c - 2);
                    issue_pre(c);
                    ++npre;
                }
                wait(B_FULL_A, c);
                wait(B_SOP, c);
                wait(B_FULL_K, c);
                tc::fence_after();
                if (!*abortp) {  // RA: [U; O] = [U~; X] + [-W; Q'] S^T
                    const uint32_t a0 = aAS + (uint32_t)((c & 1) * kAop);
                    const uint32_t dcol = (c & 1) ? T_R1 : T_R0;
                    for (int s = 0; s < D / 16; ++s)
                        tc::mma_f16(tm + dcol, tc::sdesc_lbo(a0 + (uint32_t)((s >> 2) * 16384 + (s & 3) * 32), 16),
                                    tc::sdesc_lbo(aSOP + (uint32_t)(s * 2048), 16384), idRa, 1u);
                }
                commit(B_RA, c);
                // RB of this chunk and PRE of the next, in the order their inputs arrive (RB first)
                bool rb_todo = true;
                const long long t_start = clock64();
                while (rb_todo || (npre == c + 1 && npre < nch)) {
                    if (*abortp) {  // keep every barrier's count: commit without MMAs
                        if (rb_todo) issue_rb(c);
                        break;
                    }
                    if (rb_todo && test(B_UP, c)) {
                        issue_rb(c);
                        rb_todo = false;
                    } else if (npre == c + 1 && npre < nch && pre_ready(npre)) {
                        issue_pre(npre);
                        ++npre;
                    } else if (clock64() - t_start > kWaitLimitCycles) {
                        *abortp = 1;
                    } else if (!rb_todo) {
                        break;  // the next chunk's pre-product waits at the top of the loop
                    }
                }
            }
            if (last) mbar_wait(last, last_par);  // every MMA has completed before the TMEM is freed
        }
    } else if (warp < 8) {
        // =============================== critical group ===============================
        // lanes 0..63 (quadrants 0, 1): U' after RA; all 128 lanes: the S epilogue
        // after RB.  The S epilogue writes the S operand first (what RA waits for),
        // then rescales S^T in tensor memory for RB and writes snapshots / the final
        // state from a re-read.
        const int q = warp & 3, half = warp >> 2;
        const int r = 32 * q + lane;  // the tensor-memory lane: d_k of S^T, row of R
        const bool lo = q < 2;
        const uint32_t t_s = tc::taddr(tm, 32 * q, T_S + half * 64);
        // state rows half*64 + 32 b .. + 32 at column r of a [d_v][d_k] fp32 matrix
        auto store_rows = [&](float* dst, int b, const float* v) {
            float* d = dst + (size_t)(half * 64 + 32 * b) * D + r;
#pragma unroll
            for (int i = 0; i < 32; ++i) d[(size_t)i * D] = v[i];
        };
        // S^T <- e S^T in tensor memory for 32 columns from 32 b (RB accumulates onto it)
        auto rescale = [&](int b, const float* v, float e) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float w16[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w16[i] = v[16 * k + i] * e;
                tc::st16_nowait(t_s + 32 * b + 16 * k, w16);
            }
        };
        // S operand rows (fp16, MN-major [d_k][d_v]) for 32 columns from 32 b
        auto put_sop = [&](int b, const float* v) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4*>(sSOP + half * 16384 + tc::h_off(r, 4 * b + k)) = pack8(v + 8 * k);
        };
        auto s_epilogue = [&](int c) {
            const bool more = c + 1 < nch;
            tc::fence_after();
            if (more) {
                uint32_t u[64];
                tc::ld32_nowait(t_s, u);
                tc::ld32_nowait(t_s + 32, u + 32);
                tc::ld_wait();
                put_sop(0, reinterpret_cast<const float*>(u));
                put_sop(1, reinterpret_cast<const float*>(u) + 32);
                fence_proxy_async_smem();
                mbar_arrive(bar + B_SOP + ((c + 1) & 1));
                wait(B_FULL_K, c + 1);
            }
            const float egC = more ? sG[((c + 1) & 1) * 128 + C - 1] : 0.f;
            const int ck = ckpt_after(J, seq, (int64_t)(c_lo + c + 1) * C, T);
            float* snap = ck >= 0 ? J.state_pool + ((size_t)ck * Hv + j) * D * D : nullptr;
#pragma unroll 1
            for (int b = 0; b < 2; ++b) {
                float v[32];
                tc::ld32(t_s + 32 * b, v);
                if (more) rescale(b, v, egC);
                if (snap) store_rows(snap, b, v);           // a prefix snapshot ends with this chunk
                if (!more && Sout) store_rows(Sout, b, v);  // the final state
            }
            if (more) {
                tc::st_wait();
                tc::fence_before();
            }
        };
        if (nch > 0) {  // the initial state: S operand of RA(0) and S^T for RB(0)
            wait(B_FULL_K, 0);
            const float egC = sG[C - 1];
            const float* sp = Sin ? Sin + (size_t)(half * 64) * D + r : nullptr;
#pragma unroll 1
            for (int b = 0; b < 2; ++b) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = sp ? sp[(size_t)(32 * b + i) * D] : 0.f;
                put_sop(b, v);
                rescale(b, v, egC);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar + B_SOP);
            tc::st_wait();
            tc::fence_before();
            if (!lo) mbar_arrive(bar + B_UP);  // S^T of chunk 0 is in place
        } else if (Sout && Sout != Sin) {  // an empty sequence keeps its state
#pragma unroll 1
            for (int b = 0; b < 2; ++b) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = Sin ? Sin[(size_t)(half * 64 + 32 * b + i) * D + r] : 0.f;
                store_rows(Sout, b, v);
            }
        }
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            if (lo) {  // U' = diag(e^(gamma_C - gamma)) U -> B operand of RB
                wait(B_RA, c);
                tc::fence_after();
                const float er = sG[s * 128 + C + r];
                uint32_t u[64];
                tc::ld32_nowait(tc::taddr(tm, 32 * q, (s ? T_R1 : T_R0) + half * 64), u);
                tc::ld32_nowait(tc::taddr(tm, 32 * q, (s ? T_R1 : T_R0) + half * 64 + 32), u + 32);
                tc::ld_wait();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(u[8 * k + i]) * er;
                    *reinterpret_cast<uint4*>(sUP + half * 8192 + tc::h_off(r, k)) = pack8(v);
                }
                fence_proxy_async_smem();
                tc::fence_before();
                mbar_arrive(bar + B_UP + s);
            }
            wait(B_RB, c);
            s_epilogue(c);
            if (!lo && c + 1 < nch) mbar_arrive(bar + B_UP + ((c + 1) & 1));  // S^T rescaled for RB(c+1)
        }
    } else if (warp == 10 || warp == 11 || warp == 14 || warp == 15) {
        // =============================== y warps ===============================
        const int q = warp & 3, half = (warp - 10) >> 2;
        const int r = 32 * q + lane;  // tensor-memory lane: a row of O
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            const int t = r - C, n = chunk_n(c);
            // z of this lane's output row, requested before any wait
            uint4 zr[8];
            const size_t row = (size_t)(chunk_t0(c) + (t < n ? t : 0)) * Hv * D + (size_t)j * D + half * 64;
            if (outnorm && t < n) {
                const uint4* zp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(J.z) + row);
#pragma unroll
                for (int k = 0; k < 8; ++k) zr[k] = zp[k];
            }
            wait(B_RA, c);
            tc::fence_after();
            const uint32_t t_o = tc::taddr(tm, 32 * q, (s ? T_R1 : T_R0) + half * 64);
            float part = 0.f;
#pragma unroll 1
            for (int b = 0; b < 2; ++b) {
                float o[32];
                tc::ld32(t_o + 32 * b, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) part = fmaf(o[i], o[i], part);
            }
            float* ob = ored + s * 128;  // [2][64] per chunk parity
            ob[half * C + t] = part;
            named_bar_sync(2, 128);
            const float rstd = outnorm ? rsqrtf((ob[t] + ob[C + t]) / (float)D + g.norm_eps) : 1.f;
            uint4* yp = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(J.y) + row);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float o[32];
                tc::ld32(t_o + 32 * b, o);  // warp-collective: every lane loads
                if (b == 1) {               // the O rows of this chunk have been read
                    tc::fence_before();
                    mbar_arrive(bar + B_OE + s);
                }
                if (t < n) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 pk;
                        uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
                        const __nv_bfloat162* zh = reinterpret_cast<const __nv_bfloat162*>(&zr[4 * b + k]);
                        const __nv_bfloat162* wh = reinterpret_cast<const __nv_bfloat162*>(sNW + half * 64 + 32 * b + 8 * k);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 8 * k + 2 * e;
                            float y0 = o[i] * rstd, y1 = o[i + 1] * rstd;
                            if (outnorm) {  // g = w silu(z) in bf16x2: silu(z) = h + h tanh(h), h = z/2
                                const __nv_bfloat162 hz = __hmul2(zh[e], __float2bfloat162_rn(0.5f));
                                __nv_bfloat162 th;
                                {
                                    uint32_t hi, ho;
                                    memcpy(&hi, &hz, 4);
                                    asm("tanh.approx.bf16x2 %0, %1;" : "=r"(ho) : "r"(hi));
                                    memcpy(&th, &ho, 4);
                                }
                                const float2 gf = __bfloat1622float2(__hmul2(__hfma2(hz, th, hz), wh[e]));
                                y0 *= gf.x;
                                y1 *= gf.y;
                            }
                            const __nv_bfloat162 yb = __floats2bfloat162_rn(y0, y1);
                            pw[e] = *reinterpret_cast<const uint32_t*>(&yb);
                        }
                        yp[4 * b + k] = pk;
                    }
                }
            }
        }
    }
    // ---- tear-down -----------------------------------------------------------------
    tc::fence_before();
    __syncthreads();
    if (*abortp && tid == 0) report_device_status(kDevWaitTimeout);
    if (warp == 0) tc::dealloc(tm, T_COLS);
}

}  // namespace c16
}  // namespace

bool chunk16_applies(const Geom& g) { return g.D == 128 && g.chunk == 64 && g.act_bf16; }

size_t chunk16_workspace_bytes(const Geom& g, int64_t n_tokens, int n_seq) {
    return n_tokens > 0 ? c16::ws_layout(g, n_tokens, n_seq).total : 0;
}

namespace {
cudaError_t launch_prep(const c16::Args& A, int64_t cs_lo, int64_t n_cs, bool beside, cudaStream_t st) {
    c16::Args B = A;
    B.cs_lo = cs_lo;
    B.prep_wait_end = beside ? 1 : 0;
    const int64_t ny = n_cs < 32768 ? n_cs : 32768;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)A.g.Hk, (unsigned)ny, (unsigned)((n_cs + ny - 1) / ny));
    cfg.blockDim = dim3(c16::P_THREADS);
    cfg.dynamicSmemBytes = c16::P_SMEM_ALLOC;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = beside ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, c16::k_prep16, B);
}

cudaError_t launch_chain(const c16::Args& A, int c_lo, int c_hi, bool carry_in, cudaStream_t st) {
    c16::Args B = A;
    B.c_lo = c_lo;
    B.c_hi = c_hi;
    B.carry_in = carry_in ? 1 : 0;
    k_chain16<<<dim3((unsigned)A.g.Hv, (unsigned)A.J.n_seq), c16::CH_THREADS, c16::S_SMEM_ALLOC, st>>>(B);
    return cudaGetLastError();
}
}  // namespace

cudaError_t chunk16_launch(const Geom& g, const LayerParams& p, const PrefillJob& J, cudaStream_t st) {
    using namespace c16;
    static std::atomic<uint64_t> smem_prep{0}, smem_chain{0};
    cudaError_t e = raise_smem_limit(k_prep16, (int)P_SMEM_ALLOC, smem_prep);
    if (e != cudaSuccess) return e;
    e = raise_smem_limit(k_chain16, (int)S_SMEM_ALLOC, smem_chain);
    if (e != cudaSuccess) return e;
    Args A;
    A.g = g;
    A.p = p;
    A.J = J;
    const Ws L = ws_layout(g, J.n_tokens, J.n_seq);
    unsigned char* ws = static_cast<unsigned char*>(J.workspace);
    A.kk = ws + L.kk;
    A.rec = ws + L.rec;
    A.ncs = L.ncs;
    A.cs_lo = 0;
    A.c_lo = 0;
    A.c_hi = 1 << 30;
    A.carry_in = 0;
    A.prep_wait_end = 0;
    A.ord = (L.ord && J.cu_seqlens) ? reinterpret_cast<int32_t*>(ws + L.ord) : nullptr;
    // One long sequence: its chain occupies one SM per v-head and leaves the rest of the
    // GPU idle while it walks the chunks.  The sequence is then cut into segments, all on
    // the caller's stream:  prep(0), chain(0), prep(1), chain(1), ...  Each chain segment
    // lets the next grid start once its CTAs are resident (programmatic dependent launch),
    // so the prep of segment k + 1 runs on the other SMs beside the chain of segment k and
    // waits for it only at its very end; the chain of segment k + 1, launched normally,
    // therefore follows both.  No kernel waits on another's data.  Each chain segment
    // leaves its state in s_final for the next, so the result is bit for bit that of one
    // chain launch.  A prep segment is sized to about one wave on the SMs the chain
    // leaves (P_CTAS_PER_SM per SM); it is faster per chunk than the chain (at
    // T = 8192: 6 segments of 22 chunks took 0.407 ms, 9 of 15 took 0.421 ms).
    const int64_t nch = J.n_tokens / C + (J.n_tokens % C ? 1 : 0);
    const int sms = sm_count();
    const int64_t per = std::max<int64_t>(4, (int64_t)(P_CTAS_PER_SM * (sms - g.Hv)) / g.Hk);
    const bool segmented = !J.cu_seqlens && 2 * g.Hv <= sms && nch >= 2 * per;
    if (J.n_tokens > 0 && segmented) {
        const int64_t nseg = std::min<int64_t>(32, (nch + per - 1) / per);
        const int64_t len = (nch + nseg - 1) / nseg;
        for (int64_t k = 0; k < nseg; ++k) {
            const int64_t c0 = k * len, c1 = std::min(nch, c0 + len);
            if (k == 0 && (e = launch_prep(A, c0, c1 - c0, false, st)) != cudaSuccess) return e;
            if ((e = launch_chain(A, (int)c0, (int)c1, k > 0, st)) != cudaSuccess) return e;
            const int64_t n0 = c1, n1 = std::min(nch, n0 + len);
            if (n0 < nch && (e = launch_prep(A, n0, n1 - n0, true, st)) != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (J.n_tokens > 0) {
        e = launch_prep(A, 0, L.ncs, false, st);
        if (e != cudaSuccess) return e;
    }
    return launch_chain(A, 0, 1 << 30, false, st);
}

cudaError_t take_device_status_chunk16(unsigned* out) { return take_device_status_tu(out); }

}  // namespace gdn
