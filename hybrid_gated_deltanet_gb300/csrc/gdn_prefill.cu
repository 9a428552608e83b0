// gdn_prefill.cu -- chunkwise (WY / UT-transform) prefill, single sequence and
// packed variable-length.
//
// Three launches on the caller's stream:
//  1. k_prologue  : conv + SiLU of every channel, L2 norm of q and k per k-head
//                   (q also times q_scale), gates g = log(alpha) and beta per
//                   v-head -> fp32 workspace.  Fully parallel over tokens.
//  2. k_conv_final: each sequence's new conv state = its last d_conv-1 raw
//                   inputs (after 1, so that an in-place conv state is never
//                   overwritten while 1 still reads it).
//  3. k_chunk     : one CTA per (sequence, v-head j, slice s of the d_v rows),
//                   a cluster of NS CTAs per (sequence, v-head); the CTA walks
//                   the sequence chunk by chunk with its fp32 state slice in
//                   shared memory and evaluates, per chunk of C tokens,
//                     gamma = cumsum(g), A = strict-lower(beta exp(gamma_t -
//                     gamma_i) K K^T), T = (I + A)^-1,
//                     U~ = T diag(beta) V, W = T diag(beta e^gamma) K,
//                     U = U~ - W S^T,
//                     O = diag(e^gamma) Q S^T + (Q K^T o Gamma o M_incl) U,
//                     S <- e^gamma_C S + U^T diag(e^(gamma_C - gamma)) K,
//                   then the gated RMSNorm of O (sum of squares over the head's
//                   d_v exchanged between the NS slices through distributed
//                   shared memory).  This is an exact reformulation of the token
//                   recurrence S_t = alpha_t S (I - beta_t k k^T) + beta_t v k^T,
//                   o_t = S_t q_t of "Hybrid transformers under load ..."
//                   (braintools.ru, section 3); its derivation is written out
//                   in the test infrastructure's chunk-form reference.
// The contractions run on the tensor cores through warp-level mma.sync with
// TF32 operands rounded to nearest (fp32 accumulate); fp32 activations use a
// three-pass hi/lo split so that the result keeps fp32 accuracy.  All
// reductions have a fixed order: results are bitwise reproducible ("Forge:
// how I wrote my own inference engine", 25-26 August: chunked DeltaNet
// prefill kernel with deterministic reduction).
#include <cooperative_groups.h>

#include <algorithm>
#include <cstdlib>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

namespace cg = cooperative_groups;

namespace gdn {
namespace {

// ---------------------------------------------------------------------------
// workspace layout (fp32, each section 256-byte aligned)
// ---------------------------------------------------------------------------
struct WsLayout {
    size_t qk, v, g, beta, total;  // byte offsets
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(const Geom& g, int64_t N) {
    WsLayout L;
    size_t off = 0;
    L.qk = off;
    off = align256(off + (size_t)N * 2 * g.Hk * g.D * 4);
    L.v = off;
    off = align256(off + (size_t)N * g.Hv * g.D * 4);
    L.g = off;
    off = align256(off + (size_t)N * g.Hv * 4);
    L.beta = off;
    off = align256(off + (size_t)N * g.Hv * 4);
    L.total = off;
    return L;
}

// Workspace of the tcgen05 chunk kernel (d = 128, chunk 64, 4 slices of 32
// state rows): ready-to-copy operand tiles, TF32-rounded and 128B-swizzled,
// one set per chunk slot.  Sequence s's chunk c sits in slot
// floor(start_s / 64) + s + c, which never collides with another sequence's.
//   per (slot, k-head): [K^; Q^] [128][128] | K^T [128][64]           (96 KB)
//   per (slot, v-head): V^T [128][64]                                  (32 KB)
//   per (slot, v-head): g [64], beta [64]                              (512 B)
//   per (slot, v-head): record written by the prep kernels             (161 KB)
//     [-W; Q'] [128][128] | per slice s of 32 state rows: U~_s, X_s fp32 [64][32] |
//     T diag(beta) [64][64] | P [64][64] | e^gamma [64], e^(gamma_C - gamma) [64]
constexpr size_t kTileQK = 3 * 32768, kTileV = 32768, kTileGB = 2 * 64 * 4;
constexpr size_t kRecA = 0, kRecUX = 65536, kRecTB = 131072, kRecP = 147456, kRecG = 163840, kTileRec = 164864;

struct TileWs {
    size_t qk, v, gb, rec, total;
    int64_t ncs;
};

size_t align1024(size_t x) { return (x + 1023) & ~(size_t)1023; }

TileWs tile_ws(const Geom& g, int64_t N, int n_seq) {
    TileWs L;
    L.ncs = N / 64 + n_seq + 1;
    size_t off = 0;
    L.qk = off;
    off = align1024(off + (size_t)L.ncs * g.Hk * kTileQK);
    L.v = off;
    off = align1024(off + (size_t)L.ncs * g.Hv * kTileV);
    L.gb = off;
    off = align1024(off + (size_t)L.ncs * g.Hv * kTileGB);
    L.rec = off;
    off = align1024(off + (size_t)L.ncs * g.Hv * kTileRec);
    L.total = off;
    return L;
}

struct PrefillArgs {
    Geom g;
    LayerParams p;
    PrefillJob J;
    float* qk;    // [N][2*Hk][D]  q^ (scaled) heads then k^ heads
    float* v;     // [N][Hv][D]
    float* gl;    // [N][Hv]       g = log(alpha)
    float* beta;  // [N][Hv]
    unsigned char* tqk;  // tile workspace (tcgen05 path), see TileWs
    unsigned char* tv;
    float* tgb;
    unsigned char* trec;  // chain records (prep kernel -> chain kernel)
    int64_t ncs;          // chunk slots of the tile workspace
    int tiles;           // 1: the prologue writes the tile workspace
    int NS;
};

// sequence bounds, clamped into [0, N]
__device__ __forceinline__ void seq_bounds(const PrefillJob& J, int s, int64_t& start, int64_t& end) {
    if (!J.cu_seqlens) {
        start = 0;
        end = J.n_tokens;
        return;
    }
    int64_t a = J.cu_seqlens[s], b = J.cu_seqlens[s + 1];
    a = a < 0 ? 0 : (a > J.n_tokens ? J.n_tokens : a);
    b = b < a ? a : (b > J.n_tokens ? J.n_tokens : b);
    start = a;
    end = b;
}

// sequence containing token n (largest s with cu[s] <= n, clamped)
__device__ __forceinline__ int find_seq(const PrefillJob& J, int64_t n) {
    if (!J.cu_seqlens) return 0;
    int lo = 0, hi = J.n_seq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)J.cu_seqlens[mid] <= n) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// sequence owning chunk slot cs: the largest s with floor(start_s / 64) + s <= cs
__device__ __forceinline__ int slot_seq(const PrefillJob& J, int64_t cs) {
    if (!J.cu_seqlens) return 0;
    int lo = 0, hi = J.n_seq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        int64_t st, en;
        seq_bounds(J, mid, st, en);
        if (st / 64 + mid <= cs) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// chunk of slot cs: its first token t0 and row count n; false for a slot
// between two sequences' chunks
__device__ __forceinline__ bool slot_chunk(const PrefillJob& J, int64_t cs, int64_t& t0, int& n) {
    const int sq = slot_seq(J, cs);
    int64_t start, end;
    seq_bounds(J, sq, start, end);
    t0 = (cs - (start / 64 + sq)) * 64 + start;
    if (t0 < start || t0 >= end) return false;
    n = (int)((end - t0) < 64 ? (end - t0) : 64);
    return true;
}

// pool slot of snapshot k of sequence s (the state after its first
// (k+1)*ckpt_every tokens), or -1 when none is to be written there
__device__ __forceinline__ int ckpt_slot(const PrefillJob& J, int s, int64_t k) {
    if (J.ckpt_every <= 0 || !J.ckpt_offset) return -1;
    const int64_t o0 = J.ckpt_offset[s], o1 = J.ckpt_offset[s + 1];
    if (k < 0 || k >= o1 - o0) return -1;
    const int slot = J.ckpt_slots[o0 + k];
    return (slot >= 0 && slot < J.n_slots) ? slot : -1;
}

// snapshot due after tokens [start, start + done) of a sequence of T tokens: its
// pool slot, or -1
__device__ __forceinline__ int ckpt_after(const PrefillJob& J, int s, int64_t done, int64_t T) {
    if (J.ckpt_every <= 0 || done > T || done % J.ckpt_every != 0) return -1;
    return ckpt_slot(J, s, done / J.ckpt_every - 1);
}

__device__ __forceinline__ const void* seq_conv_in(const PrefillJob& J, const Geom& g, int s, int& slot_ok) {
    if (!J.cu_seqlens) {
        slot_ok = 1;
        return J.conv0;
    }
    const int slot = J.slot_idx[s];
    slot_ok = slot >= 0 && slot < J.n_slots;
    if (!slot_ok || !J.has_init || !J.has_init[s]) return nullptr;
    const size_t elt = g.act_bf16 ? 2 : 4;
    return static_cast<const char*>(J.conv_pool) + (size_t)slot * (g.K - 1) * g.C_ch * elt;
}

// ---------------------------------------------------------------------------
// 1. prologue
// ---------------------------------------------------------------------------
// Thread = VEC consecutive channels (16 bytes of activations) x kProTok
// consecutive tokens.  The d_conv raw rows of the window stay in registers and
// slide by one row per token, so every x element is read once; taps that fall
// before a sequence start come from that sequence's conv state.  The L2 norm
// of a q/k head is a shuffle reduction over the D/VEC lanes that hold it.
constexpr int kProTok = 16;      // tokens per CTA
constexpr int kProThreads = 256;

template <typename TA>
struct Vec16;  // 16 bytes of activations
template <>
struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void load(const void* p, float* out) {
        const uint4 u = *static_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
};
template <>
struct Vec16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void load(const void* p, float* out) {
        const float4 f = *static_cast<const float4*>(p);
        out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
    }
};

template <int D, typename TA>
__global__ void __launch_bounds__(kProThreads, 2) k_prologue(const __grid_constant__ PrefillArgs A) {
    using L = Act<TA>;
    using V = Vec16<TA>;
    constexpr int VEC = V::N;
    constexpr int LPH = D / VEC;  // lanes per head
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv, K = g.K, C = g.C_ch;
    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.x * kProTok;
    const bool raw = g.flags & kFlagRawQKV;
    const bool direct = g.flags & kFlagGatesDirect;

    // gates of this CTA's tokens (first channel block only)
    if (blockIdx.y == 0) {
        for (int i = tid; i < kProTok * Hv; i += kProThreads) {
            const int64_t n = t0 + i / Hv;
            if (n >= J.n_tokens) break;
            const int j = i % Hv;
            float gl, be;
            gates(L::ld(J.a, (size_t)n * Hv + j), L::ld(J.b, (size_t)n * Hv + j), direct ? 0.f : A.p.A_log[j],
                  (!direct && A.p.dt_bias) ? A.p.dt_bias[j] : 0.f, direct, gl, be);
            A.gl[(size_t)n * Hv + j] = gl;
            A.beta[(size_t)n * Hv + j] = be;
        }
    }

    const int grp = blockIdx.y * kProThreads + tid;
    const int ch0 = grp * VEC;
    const bool active = ch0 < C;  // C is a multiple of VEC: a group is all in or all out
    const int ch = active ? ch0 : 0;
    // w[r][c]: weight of window row r (row n-3+r) for channel c; tap m of the
    // K taps multiplies row n-(K-1)+m, i.e. window row r = 4-K+m
    float w[4][VEC];
    float bias[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
        bias[c] = (!raw && A.p.conv_b) ? L::ld(A.p.conv_b, ch + c) : 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int m = r - (4 - K);
            w[r][c] = (!raw && m >= 0) ? L::ld(A.p.conv_w, (size_t)(ch + c) * K + m) : 0.f;
        }
    }
    // win[3] is row n, win[2] row n-1, ... (zeros before token 0); before the
    // first token win[1..3] hold rows t0-3 .. t0-1, shifted down at each token
    float win[4][VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) win[0][c] = 0.f;
#pragma unroll
    for (int m = 1; m < 4; ++m) {
        const int64_t tau = t0 - 4 + m;
        if (tau >= 0 && active) {
            V::load(static_cast<const TA*>(J.x) + (size_t)tau * C + ch, win[m]);
        } else {
#pragma unroll
            for (int c = 0; c < VEC; ++c) win[m][c] = 0.f;
        }
    }
    const bool is_q = ch0 < Hk * D, is_qk = ch0 < 2 * Hk * D;
    for (int tt = 0; tt < kProTok; ++tt) {
        const int64_t n = t0 + tt;
        if (n >= J.n_tokens) break;  // uniform over the CTA
        // slide: win[1..K-1] hold rows n-(K-1)..n-1; load row n into win[K]
#pragma unroll
        for (int m = 0; m < 3; ++m)
#pragma unroll
            for (int c = 0; c < VEC; ++c) win[m][c] = win[m + 1][c];
        if (active) V::load(static_cast<const TA*>(J.x) + (size_t)n * C + ch, win[3]);
        // with K < 4 the window's live rows are win[4-K .. 3]
        float u[VEC];
        const int s = find_seq(J, n);
        int64_t start, end;
        seq_bounds(J, s, start, end);
        if (raw) {
#pragma unroll
            for (int c = 0; c < VEC; ++c) u[c] = win[3][c];
        } else {
            int slot_ok;
            const void* cin = seq_conv_in(J, g, s, slot_ok);
#pragma unroll
            for (int c = 0; c < VEC; ++c) u[c] = bias[c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r < 4 - K) continue;  // not a tap
                const int64_t tau = n - 3 + r;
                if (tau >= start) {
#pragma unroll
                    for (int c = 0; c < VEC; ++c) u[c] = fmaf(w[r][c], win[r][c], u[c]);
                } else if (cin && tau - start >= -(K - 1) && active) {
                    float h[VEC];
                    V::load(static_cast<const TA*>(cin) + (size_t)((K - 1) + (tau - start)) * C + ch, h);
#pragma unroll
                    for (int c = 0; c < VEC; ++c) u[c] = fmaf(w[r][c], h[c], u[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < VEC; ++c) u[c] = siluf_(u[c]);
        }
        if (is_qk) {
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < VEC; ++c) ss = fmaf(u[c], u[c], ss);
#pragma unroll
            for (int off = LPH / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            float scale = is_q ? g.q_scale : 1.f;
            if (!(g.flags & kFlagNoL2)) scale *= rsqrtf(ss + g.l2_eps);
            if (active) {
                float4* dst = reinterpret_cast<float4*>(A.qk + (size_t)n * 2 * Hk * D + ch0);
#pragma unroll
                for (int c = 0; c < VEC; c += 4)
                    dst[c / 4] = make_float4(u[c] * scale, u[c + 1] * scale, u[c + 2] * scale, u[c + 3] * scale);
            }
        } else if (active) {
            float4* dst = reinterpret_cast<float4*>(A.v + (size_t)n * Hv * D + (ch0 - 2 * Hk * D));
#pragma unroll
            for (int c = 0; c < VEC; c += 4) dst[c / 4] = make_float4(u[c], u[c + 1], u[c + 2], u[c + 3]);
        }
    }
}

// ---------------------------------------------------------------------------
// 1b. tile prologue (tcgen05 path: d = 128, C = 64, bf16)
// ---------------------------------------------------------------------------
// One CTA per (chunk slot, unit): unit h < Hk builds k-head h's tiles -- the
// stacked [K^; Q^] (rows 0..63 k, 64..127 q of the chunk's tokens) and K^T --
// and unit Hk + j builds v-head j's V^T tile and gates.  A thread owns 8
// consecutive channels (one 16-byte load per row) of 8 (q/k) or 4 (v)
// consecutive tokens and loads all rows it needs (3 more for the conv
// window) before any arithmetic.  Rows are staged in shared memory, the
// transposed tile is built from them there, and every tile leaves with bulk
// stores.  Tokens past the sequence end give zero rows and columns, and zero
// gates, so no consumer has to mask the last chunk.
constexpr int kPtThreads = 256;
constexpr int kPtSmemAlloc = 98304 + 1024;

// conv window of one thread: rows tau0-3 .. tau0+NT-1 of its 8 channels
// (taps before the sequence start from its conv state), packed bf16
template <int NT>
__device__ __forceinline__ void load_window(const PrefillJob& J, int Cch, int K, int ch, int64_t tau0, int64_t start,
                                            int64_t end, const void* cin, uint4 rows[NT + 3]) {
#pragma unroll
    for (int r = 0; r < NT + 3; ++r) {
        const int64_t tau = tau0 - 3 + r;
        rows[r] = make_uint4(0, 0, 0, 0);
        if (tau >= start && tau < end) {
            rows[r] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(J.x) + (size_t)tau * Cch + ch);
        } else if (tau < start && cin && tau - start >= -(K - 1)) {
            rows[r] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(cin) +
                                                      (size_t)((K - 1) + (tau - start)) * Cch + ch);
        }
    }
}

__device__ __forceinline__ void unpack8(const uint4& u, float f[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __bfloat1622float2(h[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

// SiLU with the fast exponential and division (bf16 activations only: the
// difference to the exact form is far below their rounding)
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// conv + SiLU of the NT tokens of one thread's window (rows i .. i+3 are the
// taps of token i), through a sliding window of 4 unpacked rows; emit(i, u)
// receives token i's 8 channels
template <int NT, typename Emit>
__device__ __forceinline__ void conv_tokens(const uint4 rows[NT + 3], const float w[4][8], const float bias[8],
                                            int K, bool raw, Emit emit) {
    float win[4][8];
#pragma unroll
    for (int r = 1; r < 4; ++r) unpack8(rows[r - 1], win[r]);
#pragma unroll
    for (int i = 0; i < NT; ++i) {
#pragma unroll
        for (int r = 0; r < 3; ++r)
#pragma unroll
            for (int c = 0; c < 8; ++c) win[r][c] = win[r + 1][c];
        unpack8(rows[i + 3], win[3]);
        float u[8];
        if (raw) {
#pragma unroll
            for (int c = 0; c < 8; ++c) u[c] = win[3][c];
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) u[c] = bias[c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r < 4 - K) continue;  // not a tap
#pragma unroll
                for (int c = 0; c < 8; ++c) u[c] = fmaf(w[r][c], win[r][c], u[c]);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) u[c] = silu_fast(u[c]);
        }
        emit(i, u);
    }
}

__global__ void __launch_bounds__(kPtThreads, 2) k_prologue_tc(const __grid_constant__ PrefillArgs A) {
    using L = Act<__nv_bfloat16>;
    constexpr int D = 128, C = 64;
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv, K = g.K, Cch = g.C_ch;
    const int unit = blockIdx.x;
    const int64_t cs = (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
    if (cs >= A.ncs) return;
    const int sq = slot_seq(J, cs);
    int64_t start, end;
    seq_bounds(J, sq, start, end);
    const int64_t t0 = (cs - (start / C + sq)) * C + start;
    if (t0 < start || t0 >= end) return;  // a slot between two sequences' chunks
    const int n = (int)((end - t0) < C ? (end - t0) : C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool raw = g.flags & kFlagRawQKV;
    int slot_ok;
    const void* cin = seq_conv_in(J, g, sq, slot_ok);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    const bool qk = unit < Hk;
    const int cg = qk ? lane : (lane & 15);  // 8-channel group inside the unit's channels
    int ch;
    if (qk) ch = (cg < 16 ? unit * D : (Hk + unit) * D) + (cg & 15) * 8;
    else ch = 2 * Hk * D + (unit - Hk) * D + cg * 8;
    // w[r][c]: weight of window row r (row tau-3+r) for channel c; tap m of the
    // K taps multiplies row tau-(K-1)+m, i.e. window row r = 4-K+m
    float w[4][8], bias[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        bias[c] = (!raw && A.p.conv_b) ? L::ld(A.p.conv_b, ch + c) : 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int m = r - (4 - K);
            w[r][c] = (!raw && m >= 0) ? L::ld(A.p.conv_w, (size_t)(ch + c) * K + m) : 0.f;
        }
    }
    if (qk) {
        // staging: [K^; Q^] [128][128] at 0, K^T [128][64] at 64 KB
        unsigned char* st = sm;
        unsigned char* kt = sm + 65536;
        const int tt0 = warp * 8;
        uint4 rows[11];
        load_window<8>(J, Cch, K, ch, t0 + tt0, start, end, cin, rows);
        const bool is_q = cg < 16;
        const int d0 = (cg & 15) * 8;
        conv_tokens<8>(rows, w, bias, K, raw, [&](int i, float u[8]) {
            const int t = tt0 + i;
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) ss = fmaf(u[c], u[c], ss);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            float scale = is_q ? g.q_scale : 1.f;
            if (!(g.flags & kFlagNoL2)) scale *= rsqrtf(ss + g.l2_eps);
            if (t >= n) scale = 0.f;  // past the sequence end
            const int r = is_q ? C + t : t;
#pragma unroll
            for (int c = 0; c < 8; c += 4)
                tc::st_row4(st, D, r, d0 + c, u[c] * scale, u[c + 1] * scale, u[c + 2] * scale, u[c + 3] * scale);
        });
        __syncthreads();
        {  // K^T from the K^ rows: thread = (d, half of the tokens)
            const int d = tid & 127, th = (tid >> 7) * 32;
#pragma unroll
            for (int t4 = 0; t4 < 32; t4 += 4) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = *reinterpret_cast<const float*>(st + tc::sw_off(D, th + t4 + e, d));
                *reinterpret_cast<float4*>(kt + tc::sw_off(D, d, th + t4)) = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            unsigned char* dst = A.tqk + ((size_t)cs * Hk + unit) * kTileQK;
            for (int p = 0; p < 3; ++p) bulk_s2g(dst + p * 32768, sm + p * 32768, 32768);
            bulk_commit();
            bulk_wait_read_all();
        }
    } else {
        // staging: V rows [64][128] at 0, V^T [128][64] at 32 KB
        const int j = unit - Hk;
        unsigned char* vs = sm;
        unsigned char* vt = sm + 32768;
        const int tt0 = (warp * 2 + (lane >> 4)) * 4;
        uint4 rows[7];
        load_window<4>(J, Cch, K, ch, t0 + tt0, start, end, cin, rows);
        const int d0 = cg * 8;
        conv_tokens<4>(rows, w, bias, K, raw, [&](int i, float u[8]) {
            const int t = tt0 + i;
            const float keep = t < n ? 1.f : 0.f;
#pragma unroll
            for (int c = 0; c < 8; c += 4)
                tc::st_row4(vs, C, t, d0 + c, u[c] * keep, u[c + 1] * keep, u[c + 2] * keep, u[c + 3] * keep);
        });
        if (tid < C) {  // gates of token t
            const bool direct = g.flags & kFlagGatesDirect;
            float gl = 0.f, be = 0.f;
            if (tid < n) {
                const size_t tok = (size_t)(t0 + tid);
                gates(L::ld(J.a, tok * Hv + j), L::ld(J.b, tok * Hv + j), direct ? 0.f : A.p.A_log[j],
                      (!direct && A.p.dt_bias) ? A.p.dt_bias[j] : 0.f, direct, gl, be);
            }
            float* gb = A.tgb + ((size_t)cs * Hv + j) * 128;
            gb[tid] = gl;
            gb[C + tid] = be;
        }
        __syncthreads();
        {  // V^T from the V rows: thread = (dv, half of the tokens)
            const int d = tid & 127, th = (tid >> 7) * 32;
#pragma unroll
            for (int t4 = 0; t4 < 32; t4 += 4) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = *reinterpret_cast<const float*>(vs + tc::sw_off(C, th + t4 + e, d));
                *reinterpret_cast<float4*>(vt + tc::sw_off(D, d, th + t4)) = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g(A.tv + ((size_t)cs * Hv + j) * kTileV, vt, 32768);
            bulk_commit();
            bulk_wait_read_all();
        }
    }
}

// ---------------------------------------------------------------------------
// 2. final conv state of every sequence
// ---------------------------------------------------------------------------
template <typename TA>
__global__ void k_conv_final(const __grid_constant__ PrefillArgs A) {
    using L = Act<TA>;
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int C = g.C_ch, Km1 = g.K - 1;
    const size_t total = (size_t)J.n_seq * C;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int ch = (int)(idx % C), s = (int)(idx / C);
        int64_t start, end;
        seq_bounds(J, s, start, end);
        int slot_ok;
        const void* cin = seq_conv_in(J, g, s, slot_ok);
        if (!slot_ok) continue;
        void* cout = J.cu_seqlens ? static_cast<char*>(J.conv_pool) +
                                        (size_t)J.slot_idx[s] * Km1 * C * (g.act_bf16 ? 2 : 4)
                                  : J.conv_final;
        const int64_t T = end - start;
        float old[3];
#pragma unroll
        for (int m = 0; m < 3; ++m) old[m] = (m < Km1 && cin) ? L::ld(cin, (size_t)m * C + ch) : 0.f;
        float nv[3];
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            if (m >= Km1) break;
            const int64_t p = T + m;  // position in [old (Km1 rows), x rows of the sequence]
            nv[m] = p < Km1 ? old[p] : L::ld(J.x, (size_t)(start + p - Km1) * C + ch);
        }
        for (int m = 0; m < Km1; ++m) L::st(cout, (size_t)m * C + ch, nv[m]);
    }
}

// conv states of the prefix snapshots: the d_conv-1 raw inputs before each
// snapshot boundary (thread = channel; grid z strides over the snapshots)
template <typename TA>
__global__ void k_conv_ckpt(const __grid_constant__ PrefillArgs A) {
    using L = Act<TA>;
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Cch = g.C_ch, Km1 = g.K - 1;
    const int ch = blockIdx.x * blockDim.x + threadIdx.x, s = blockIdx.y;
    if (ch >= Cch) return;
    int64_t start, end;
    seq_bounds(J, s, start, end);
    const size_t elt = g.act_bf16 ? 2 : 4;
    for (int64_t done = (int64_t)(blockIdx.z + 1) * J.ckpt_every; done <= end - start;
         done += (int64_t)gridDim.z * J.ckpt_every) {
        const int ck = ckpt_slot(J, s, done / J.ckpt_every - 1);
        if (ck < 0) continue;
        void* dst = static_cast<char*>(J.conv_pool) + (size_t)ck * Km1 * Cch * elt;
        for (int m = 0; m < Km1; ++m)  // (done >= chunk > d_conv - 1: all rows inside the sequence)
            L::st(dst, (size_t)m * Cch + ch, L::ld(J.x, (size_t)(start + done - Km1 + m) * Cch + ch));
    }
}


// ---------------------------------------------------------------------------
// 3. chunk kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float c[4], const uint32_t a[4], const uint32_t b[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// One warp computes 16x8 output tiles of C = A B, tile by tile.
// A(m,k) = Ap[m*am + k*ak], B(k,n) = Bp[k*bk + n*bn]; M % 16 == 0, N % 8 == 0,
// K % 8 == 0.  epi(m, n, value) receives every output element exactly once.
template <bool PRECISE, typename Epi>
__device__ __forceinline__ void warp_gemm(int M, int N, int K, const float* Ap, int am, int ak, const float* Bp,
                                          int bk, int bn, int warp, int nwarp, int lane, Epi epi) {
    const int gq = lane >> 2, t4 = lane & 3;
    const int tn = N / 8, ntile = (M / 16) * tn;
    for (int tile = warp; tile < ntile; tile += nwarp) {
        const int m0 = (tile / tn) * 16, n0 = (tile % tn) * 8;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const float* a_r0 = Ap + (size_t)(m0 + gq) * am;
        const float* a_r1 = Ap + (size_t)(m0 + gq + 8) * am;
        const float* b_c = Bp + (size_t)(n0 + gq) * bn;
        for (int k0 = 0; k0 < K; k0 += 8) {
            const float fa[4] = {a_r0[(k0 + t4) * ak], a_r1[(k0 + t4) * ak], a_r0[(k0 + t4 + 4) * ak],
                                 a_r1[(k0 + t4 + 4) * ak]};
            const float fb[2] = {b_c[(k0 + t4) * bk], b_c[(k0 + t4 + 4) * bk]};
            uint32_t ah[4], bh[2];
#pragma unroll
            for (int e = 0; e < 4; ++e) ah[e] = to_tf32(fa[e]);
#pragma unroll
            for (int e = 0; e < 2; ++e) bh[e] = to_tf32(fb[e]);
            if (PRECISE) {
                uint32_t al[4], bl[2];
#pragma unroll
                for (int e = 0; e < 4; ++e) al[e] = to_tf32(fa[e] - __uint_as_float(ah[e]));
#pragma unroll
                for (int e = 0; e < 2; ++e) bl[e] = to_tf32(fb[e] - __uint_as_float(bh[e]));
                mma_tf32(c, al, bh);
                mma_tf32(c, ah, bl);
            }
            mma_tf32(c, ah, bh);
        }
        epi(m0 + gq, n0 + 2 * t4, c[0]);
        epi(m0 + gq, n0 + 2 * t4 + 1, c[1]);
        epi(m0 + gq + 8, n0 + 2 * t4, c[2]);
        epi(m0 + gq + 8, n0 + 2 * t4 + 1, c[3]);
    }
}

constexpr int kChunkThreads = 256;

struct ChunkSmem {  // float offsets into dynamic shared memory
    int ks, qs, vs, ss, am, tm, pm, ws, us, gam, beta, eg, ssq, total;
    int ldk, ldv, ldc;
};

__host__ __device__ inline ChunkSmem chunk_smem(int C, int D, int DV) {
    ChunkSmem s;
    s.ldk = D + 4;
    s.ldv = DV + 4;
    s.ldc = C + 4;
    int o = 0;
    s.ks = o; o += C * s.ldk;   // K^ of the chunk            [C][D]
    s.qs = o; o += C * s.ldk;   // Q^                          [C][D]
    s.vs = o; o += C * s.ldv;   // beta V (this slice)         [C][DV]
    s.ss = o; o += DV * s.ldk;  // state slice S               [DV][D]
    s.am = o; o += C * s.ldc;   // A, then T diag(beta e^g)    [C][C]
    s.tm = o; o += C * s.ldc;   // T = (I + A)^-1              [C][C]
    s.pm = o; o += C * s.ldc;   // Q K^T o Gamma (incl. diag)  [C][C]
    s.ws = o; o += C * s.ldk;   // W, later O                  [C][D]
    s.us = o; o += C * s.ldv;   // U~ -> U -> U diag(e^(gC-g)) [C][DV]
    s.gam = o; o += C;
    s.beta = o; o += C;
    s.eg = o; o += C;
    s.ssq = o; o += 2 * C;      // per-token partial sum of O^2, double-buffered
    s.total = o;
    return s;
}

template <int D, bool PRECISE, typename TA>
__global__ void __launch_bounds__(kChunkThreads, 1) k_chunk(const __grid_constant__ PrefillArgs A) {
    using L = Act<TA>;
    cg::cluster_group cluster = cg::this_cluster();
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int NS = A.NS, DV = D / NS, C = g.chunk, Hk = g.Hk, Hv = g.Hv;
    const int s_idx = blockIdx.x, j = blockIdx.y, seq = blockIdx.z, h = j / g.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = kChunkThreads / 32;
    const ChunkSmem lay = chunk_smem(C, D, DV);
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    float *Ks = sm + lay.ks, *Qs = sm + lay.qs, *Vs = sm + lay.vs, *Ss = sm + lay.ss;
    float *Am = sm + lay.am, *Tm = sm + lay.tm, *Pm = sm + lay.pm, *Ws = sm + lay.ws, *Us = sm + lay.us;
    float *gam = sm + lay.gam, *bet = sm + lay.beta, *eg = sm + lay.eg, *ssq = sm + lay.ssq;
    const int ldk = lay.ldk, ldv = lay.ldv, ldc = lay.ldc;

    int64_t start, end;
    seq_bounds(J, seq, start, end);
    // state in / out
    const float* Sin = nullptr;
    float* Sout = nullptr;
    if (!J.cu_seqlens) {
        Sin = J.s0 ? J.s0 + (size_t)j * D * D : nullptr;
        Sout = J.s_final + (size_t)j * D * D;
    } else {
        const int slot = J.slot_idx[seq];
        if (slot >= 0 && slot < J.n_slots) {
            Sout = J.state_pool + ((size_t)slot * Hv + j) * D * D;
            if (J.has_init && J.has_init[seq]) Sin = Sout;
        }
    }
    for (int i = tid; i < DV * D; i += kChunkThreads) {
        const int r = i / D, c = i % D;
        Ss[r * ldk + c] = Sin ? Sin[(size_t)(s_idx * DV + r) * D + c] : 0.f;
    }

    const int64_t T = end - start;
    const int n_chunks = (int)((T + C - 1) / C);
    const bool outnorm = !(g.flags & kFlagNoOutNorm);
    for (int ci = 0; ci < n_chunks; ++ci) {
        const int64_t t0 = start + (int64_t)ci * C;
        const int n = (int)((end - t0) < C ? (end - t0) : C);
        __syncthreads();  // previous chunk done with every buffer
        // ---- load the chunk (rows >= n are zero: exact no-op padding) ----------
        for (int i = tid; i < C * (D / 4); i += kChunkThreads) {
            const int r = i / (D / 4), c4 = i % (D / 4);
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), qv = kv;
            if (r < n) {
                const size_t tok = (size_t)(t0 + r);
                kv = *reinterpret_cast<const float4*>(A.qk + (tok * 2 * Hk + Hk + h) * D + c4 * 4);
                qv = *reinterpret_cast<const float4*>(A.qk + (tok * 2 * Hk + h) * D + c4 * 4);
            }
            *reinterpret_cast<float4*>(Ks + r * ldk + c4 * 4) = kv;
            *reinterpret_cast<float4*>(Qs + r * ldk + c4 * 4) = qv;
        }
        for (int i = tid; i < C; i += kChunkThreads) {
            float gv = 0.f, bv = 0.f;
            if (i < n) {
                gv = A.gl[(size_t)(t0 + i) * Hv + j];
                bv = A.beta[(size_t)(t0 + i) * Hv + j];
            }
            gam[i] = gv;
            bet[i] = bv;
        }
        for (int i = tid; i < C * (DV / 4); i += kChunkThreads) {
            const int r = i / (DV / 4), c4 = i % (DV / 4);
            float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < n) vv = *reinterpret_cast<const float4*>(A.v + ((size_t)(t0 + r) * Hv + j) * D + s_idx * DV + c4 * 4);
            *reinterpret_cast<float4*>(Vs + r * ldv + c4 * 4) = vv;
        }
        __syncthreads();
        // ---- gamma = cumsum(g) (one warp), beta V; KK^T and QK^T -----------------
        if (warp == 0) {
            float run = 0.f;
            for (int base = 0; base < C; base += 32) {
                float v = (base + lane < C) ? gam[base + lane] : 0.f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, v, off);
                    if (lane >= off) v += o;
                }
                v += run;
                if (base + lane < C) {
                    gam[base + lane] = v;
                    eg[base + lane] = expf(v);
                }
                run = __shfl_sync(0xffffffffu, v, 31);
            }
        }
        for (int i = tid; i < C * DV; i += kChunkThreads) {
            const int r = i / DV, c = i % DV;
            Vs[r * ldv + c] *= bet[r];
        }
        warp_gemm<PRECISE>(C, C, D, Ks, ldk, 1, Ks, 1, ldk, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Am[m * ldc + nn] = v; });
        warp_gemm<PRECISE>(C, C, D, Qs, ldk, 1, Ks, 1, ldk, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Pm[m * ldc + nn] = v; });
        __syncthreads();
        // ---- decay masks --------------------------------------------------------
        for (int i = tid; i < C * C; i += kChunkThreads) {
            const int t = i / C, c = i % C;
            const float dec = c <= t ? expf(gam[t] - gam[c]) : 0.f;  // exponent <= 0 only
            Am[t * ldc + c] = c < t ? bet[t] * dec * Am[t * ldc + c] : 0.f;
            Pm[t * ldc + c] = dec * Pm[t * ldc + c];
        }
        __syncthreads();
        // ---- T = (I + A)^-1: 16x16 diagonal blocks by forward substitution -------
        const int nb = C / 16;
        if (warp < nb) {
            const int b0 = warp * 16;
            for (int i = 0; i < 16; ++i) {
                float arow[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) arow[k] = Am[(b0 + i) * ldc + b0 + k];
                __syncwarp();
                if (lane < 16) {
                    float x = (lane == i) ? 1.f : 0.f;
                    for (int k = lane; k < i; ++k) x -= arow[k] * Tm[(b0 + k) * ldc + b0 + lane];
                    Tm[(b0 + i) * ldc + b0 + lane] = (lane <= i) ? x : 0.f;
                }
                __syncwarp();
            }
        }
        // zero the strictly upper off-diagonal blocks
        for (int i = tid; i < C * C; i += kChunkThreads) {
            const int t = i / C, c = i % C;
            if ((c >> 4) > (t >> 4)) Tm[t * ldc + c] = 0.f;
        }
        __syncthreads();
        // off-diagonal blocks by distance: X_ab = -X_aa sum_{c=b}^{a-1} A_ac X_cb
        for (int d = 1; d < nb; ++d) {
            for (int bb = warp; bb < nb - d; bb += nwarp) {
                const int a0 = (bb + d) * 16, c0b = bb * 16;
                // Y = sum_c A_ac X_cb : 16x16, 8 elements per lane
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int idx = lane + 32 * e, r = idx >> 4, c = idx & 15;
                    float acc = 0.f;
                    for (int k = c0b; k < a0; ++k) acc = fmaf(Am[(a0 + r) * ldc + k], Tm[k * ldc + c0b + c], acc);
                    y[e] = acc;
                }
                // stage Y into the (still zero) target block, then X_ab = -X_aa Y
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int idx = lane + 32 * e, r = idx >> 4, c = idx & 15;
                    Tm[(a0 + r) * ldc + c0b + c] = y[e];
                }
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int idx = lane + 32 * e, r = idx >> 4, c = idx & 15;
                    float acc = 0.f;
                    for (int k = 0; k < 16; ++k)
                        acc = fmaf(Tm[(a0 + r) * ldc + a0 + k], Tm[(a0 + k) * ldc + c0b + c], acc);
                    y[e] = -acc;
                }
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int idx = lane + 32 * e, r = idx >> 4, c = idx & 15;
                    Tm[(a0 + r) * ldc + c0b + c] = y[e];
                }
            }
            __syncthreads();
        }
        // ---- Am <- T diag(beta e^gamma); U~ = T (beta V); W = Am K ----------------
        for (int i = tid; i < C * C; i += kChunkThreads) {
            const int t = i / C, c = i % C;
            Am[t * ldc + c] = Tm[t * ldc + c] * bet[c] * eg[c];
        }
        __syncthreads();
        warp_gemm<PRECISE>(C, DV, C, Tm, ldc, 1, Vs, ldv, 1, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Us[m * ldv + nn] = v; });
        warp_gemm<PRECISE>(C, D, C, Am, ldc, 1, Ks, ldk, 1, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Ws[m * ldk + nn] = v; });
        __syncthreads();
        // ---- U = U~ - W S^T ---------------------------------------------------------
        warp_gemm<PRECISE>(C, DV, D, Ws, ldk, 1, Ss, 1, ldk, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Us[m * ldv + nn] -= v; });
        __syncthreads();
        // ---- O = diag(e^gamma) Q S^T + P U  (O stored over W) ---------------------
        float* Os = Ws;
        const int ldo = ldk;
        warp_gemm<PRECISE>(C, DV, D, Qs, ldk, 1, Ss, 1, ldk, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Os[m * ldo + nn] = eg[m] * v; });
        __syncthreads();
        warp_gemm<PRECISE>(C, DV, C, Pm, ldc, 1, Us, ldv, 1, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Os[m * ldo + nn] += v; });
        __syncthreads();
        // ---- U rows *= e^(gamma_C - gamma_t); per-token partial sum of O^2 ---------
        const float gC = gam[C - 1];
        for (int i = tid; i < C * DV; i += kChunkThreads) {
            const int r = i / DV, c = i % DV;
            Us[r * ldv + c] *= expf(gC - gam[r]);
        }
        float* ssq_cur = ssq + (ci & 1) * C;
        for (int t = warp; t < C; t += nwarp) {
            float acc = 0.f;
            for (int c = lane; c < DV; c += 32) {
                const float o = Os[t * ldo + c];
                acc = fmaf(o, o, acc);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) ssq_cur[t] = acc;
        }
        cluster.sync();  // (also a CTA barrier) partial sums visible to the slices
        // ---- S <- e^gamma_C S + U^T K' ---------------------------------------------
        const float egC = eg[C - 1];
        warp_gemm<PRECISE>(DV, D, C, Us, 1, ldv, Ks, ldk, 1, warp, nwarp, lane,
                           [&](int m, int nn, float v) { Ss[m * ldk + nn] = fmaf(egC, Ss[m * ldk + nn], v); });
        // ---- y = gated RMSNorm(O) ---------------------------------------------------
        for (int i = tid; i < n * DV; i += kChunkThreads) {
            const int t = i / DV, c = i % DV;
            const size_t tok = (size_t)(t0 + t);
            const int dv = s_idx * DV + c;
            float yv = Os[t * ldo + c];
            if (outnorm) {
                float tot = 0.f;
                for (int s2 = 0; s2 < NS; ++s2) tot += *cluster.map_shared_rank(&ssq_cur[t], s2);
                const float zz = L::ld(J.z, tok * (size_t)Hv * D + (size_t)j * D + dv);
                yv = yv * rsqrtf(tot / (float)D + g.norm_eps) * L::ld(A.p.norm_w, dv) * siluf_(zz);
            }
            L::st(J.y, tok * (size_t)Hv * D + (size_t)j * D + dv, yv);
        }
        const int ck = ckpt_after(J, seq, (int64_t)(ci + 1) * C, T);  // (uniform over the CTA)
        if (ck >= 0) {
            __syncthreads();  // the state update is complete
            float* dst = J.state_pool + ((size_t)ck * Hv + j) * D * D;
            for (int i = tid; i < DV * D; i += kChunkThreads) {
                const int r = i / D, c = i % D;
                dst[(size_t)(s_idx * DV + r) * D + c] = Ss[r * ldk + c];
            }
        }
    }
    __syncthreads();
    if (Sout) {
        for (int i = tid; i < DV * D; i += kChunkThreads) {
            const int r = i / D, c = i % D;
            Sout[(size_t)(s_idx * DV + r) * D + c] = Ss[r * ldk + c];
        }
    }
    cluster.sync();  // peers may still read this CTA's partial sums
}

// ---------------------------------------------------------------------------
// 3b. tcgen05 path (d = 128, C = 64, bf16): two prep kernels + chain kernel
// ---------------------------------------------------------------------------
// The chunk form splits into work that does not depend on the state and a
// short sequential chain that does.  With U~ = T diag(beta) V,
// W = T diag(beta e^gamma) K and P = (QK^T o decay, lower incl.),
//   U = U~ - W S^T,  O = diag(e^gamma) Q S^T + P U = Q' S^T + X,
//   Q' = diag(e^gamma) Q - P W,  X = P U~,
//   S^T <- e^gamma_C S^T + K^T diag(e^(gamma_C - gamma)) U,
// so only one product with the state gives both U and O, and the second
// updates the state.
//
// k_chunk_prep (per chunk slot, v-head; all chunks in parallel): gamma =
//   cumsum(g), KK^T and QK^T (tcgen05), A = strict-lower(beta_t
//   e^(gamma_t - gamma_i) KK^T), P, T = (I + A)^-1 (16x16 blocks, fp32) and
//   T diag(beta) -> record.
// k_chunk_prep2 (same grid): W^T = (K^T diag(e^gamma)) (T diag(beta))^T and
//   U~^T = V^T (T diag(beta))^T, then (P W)^T = W^T P^T and X^T = U~^T P^T
//   (tcgen05, M = 128) -> record: the stacked operand [-W; Q'] and, per slice
//   of 32 state rows, U~ and X in fp32.
// k_chunk_tc<NSL> (per sequence, v-head, slice; the NSL = 4 or 2 slices a
//   cluster): the fp32 state slice lives in TMEM as S^T (lane = d_k index,
//   128 / NSL columns = the slice's d_v rows); per chunk
//     Ra  D = [-W; Q'] S^T                    (M = 128, K = 128)
//         U = U~ + D[0:64],  O = X + D[64:128]
//     Rb  S^T <- e^gamma_C S^T + K^T (diag(e^(gamma_C - gamma)) U)
//   and y = gated RMSNorm(O) of chunk c is computed while Ra of chunk c+1 runs.
//   The tensor core takes about one MMA instruction per 140 cycles whatever
//   its M and N, so the chain's cost is its 24 instructions per chunk (16 for
//   Ra with K = 128, 8 for Rb with K = 64); everything else is arranged around
//   them.
// TF32 operands are rounded to nearest; accumulation is fp32 in TMEM.

// One warp: the 16x8 tile C = A(16 x K) B(K x 8) with A(m,k) = Ap[m*lda + k] and
// B(k,n) = Bp[k*ldb + n], K a multiple of 8, fp32-accurate through the 3xTF32
// split (hi*hi + hi*lo + lo*hi).  Lane layout of c: (g, 2t), (g, 2t+1),
// (g+8, 2t), (g+8, 2t+1) with g = lane / 4, t = lane % 4.
__device__ __forceinline__ void warp_tile16x8_precise(const float* Ap, int lda, const float* Bp, int ldb, int K,
                                                      int lane, float c[4]) {
    const int gq = lane >> 2, t4 = lane & 3;
    c[0] = c[1] = c[2] = c[3] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 8) {
        const float fa[4] = {Ap[gq * lda + k0 + t4], Ap[(gq + 8) * lda + k0 + t4], Ap[gq * lda + k0 + t4 + 4],
                             Ap[(gq + 8) * lda + k0 + t4 + 4]};
        const float fb[2] = {Bp[(k0 + t4) * ldb + gq], Bp[(k0 + t4 + 4) * ldb + gq]};
        uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ah[e] = to_tf32(fa[e]);
            al[e] = to_tf32(fa[e] - __uint_as_float(ah[e]));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            bh[e] = to_tf32(fb[e]);
            bl[e] = to_tf32(fb[e] - __uint_as_float(bh[e]));
        }
        mma_tf32(c, al, bh);
        mma_tf32(c, ah, bl);
        mma_tf32(c, ah, bh);
    }
}

// byte offset of (t, v) in a [64][32] fp32 block of U~ or X: 16-byte chunks
// XOR-swizzled by t % 8, so that a warp reading one row per lane is
// conflict-free
__device__ __forceinline__ uint32_t ux_off(int t, int v) {
    return (uint32_t)(t * 128 + ((((v >> 2) ^ (t & 7))) << 4) + ((v & 3) << 2));
}

namespace tcp {
constexpr int C = 64, D = 128, THREADS = 256, LDA = 68;
// k_chunk_prep shared memory
constexpr int PR_R0 = 0;                       // [K^; Q^] tile (64 KB), then P | T diag(b) staging at 32 KB
constexpr int PR_R1 = 32768;
constexpr int PR_AM = 65536;                   // fp32 A [64][68]
constexpr int PR_TM = PR_AM + C * LDA * 4;     // fp32 T [64][68]
constexpr int PR_SMALL = PR_TM + C * LDA * 4;  // gam, bet, e^g, e^(gC-g)
constexpr int PR_SMEM = PR_SMALL + 4 * C * 4 + 64;
constexpr int PR_SMEM_ALLOC = PR_SMEM + 1024;
constexpr int PR_TMEM_COLS = 64;  // [KK^T; QK^T] (M = 128, N = 64)
// k_chunk_prep2 shared memory
constexpr int P2_KT = 0;           // K^T tile, then W^T  [128][64]
constexpr int P2_VT = 32768;       // V^T tile, then U~^T [128][64]
constexpr int P2_TB = 65536;       // T diag(b) [64][64]
constexpr int P2_P = 81920;        // P         [64][64]
constexpr int P2_G = 98304;        // e^g [64]
constexpr int P2_SMEM = P2_G + C * 4 + 64;
constexpr int P2_SMEM_ALLOC = P2_SMEM + 1024;
constexpr int P2_TMEM_COLS = 128;  // two M=128 x N=64 accumulators
constexpr int kIssuers = 4;  // warps issuing the K-steps of a chain state product (one accumulator each)
}  // namespace tcp

__global__ void __launch_bounds__(tcp::THREADS, 2) k_chunk_prep(const __grid_constant__ PrefillArgs A) {
    using namespace tcp;
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv;
    const int j = blockIdx.x, h = j / g.G;
    const int64_t cs = (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
    if (cs >= A.ncs) return;
    int64_t t0;
    int n;
    if (!slot_chunk(J, cs, t0, n)) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hf = warp >> 2;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    unsigned char *R0 = sm + PR_R0, *R1 = sm + PR_R1;
    unsigned char *Ps = R1, *TBs = R1 + 16384;
    float* Am = reinterpret_cast<float*>(sm + PR_AM);
    float* Tm = reinterpret_cast<float*>(sm + PR_TM);
    float* gam = reinterpret_cast<float*>(sm + PR_SMALL);
    float* bet = gam + C;
    float* eg = bet + C;
    float* erev = eg + C;  // e^g and e^(gC-g) contiguous: one bulk store
    uint64_t* mbar = reinterpret_cast<uint64_t*>(erev + C);
    uint64_t* barQK = mbar + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 2);
    const unsigned char* tile = A.tqk + ((size_t)cs * Hk + h) * kTileQK;
    unsigned char* rec = A.trec + ((size_t)cs * Hv + j) * kTileRec;

    if (warp == 0) tc::alloc(tslot, PR_TMEM_COLS);
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(barQK, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(barQK, 65536);
        bulk_g2s(R0, tile, 32768, barQK);
        bulk_g2s(R1, tile + 32768, 32768, barQK);
    }
    if (tid < C) {  // (zero past the sequence end)
        const float* gb = A.tgb + ((size_t)cs * Hv + j) * 128;
        gam[tid] = gb[tid];
        bet[tid] = gb[C + tid];
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;
    bool ok = true;

    // ---- gamma = cumsum(g), e^gamma, e^(gamma_C - gamma) ----------------------------
    if (warp == 0) {
        float run = 0.f;
        for (int base = 0; base < C; base += 32) {
            float v = gam[base + lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += o;
            }
            v += run;
            gam[base + lane] = v;
            eg[base + lane] = expf(v);
            run = __shfl_sync(0xffffffffu, v, 31);
        }
        __syncwarp();
        for (int t = lane; t < C; t += 32) erev[t] = expf(gam[C - 1] - gam[t]);
    }
    {
        bool w = true;
        if (warp == 0) {
            w = mbar_wait(barQK, 0);
            if (!w) w = mbar_wait(barQK, 0);
        }
        ok = __syncthreads_and(w);
    }
    // ---- [KK^T; QK^T] = [K^; Q^] K^T: one M = 128 product (B = the K^ rows of
    // the stacked tile, whose atoms are 128 rows apart) --------------------------------
    tc::fence_before();
    __syncthreads();
    if (tid == 0) {
        if (ok) {
            tc::fence_after();
            tc::mma_tf32(tm, R0, 2 * C, R0, 2 * C, D, tc::idesc_tf32(2 * C, C), false);
        }
        tc::commit(mbar);
    }
    {
        bool w = true;
        if (ok && warp == 0) {
            w = mbar_wait(mbar, 0);
            if (!w) w = mbar_wait(mbar, 0);
        }
        ok = __syncthreads_and(ok && w);
        tc::fence_after();
    }
    // ---- decay masks: A (strictly lower, beta_t) from the KK^T rows (lanes 0..63),
    // P (lower incl.) from the QK^T rows (lanes 64..127), over the stacked tile -----------
    {
        const bool arow = q4 < 2;
        const int t = 32 * (q4 & 1) + lane;
        const float gt = gam[t], bt = bet[t];
        float v[32];
        tc::ld16x2(tc::taddr(tm, 32 * q4, hf * 32), v, tc::taddr(tm, 32 * q4, hf * 32 + 16), v + 16);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            float o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = hf * 32 + c + e;
                const float dec = i <= t ? __expf(gt - gam[i]) : 0.f;  // exponent <= 0 only
                o4[e] = arow ? (i < t ? bt * dec * v[c + e] : 0.f) : dec * v[c + e];
            }
            if (arow) *reinterpret_cast<float4*>(Am + t * LDA + hf * 32 + c) = make_float4(o4[0], o4[1], o4[2], o4[3]);
            else tc::st_row4(Ps, C, t, hf * 32 + c, o4[0], o4[1], o4[2], o4[3]);
        }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(rec + kRecP, Ps, 16384);
        bulk_s2g(rec + kRecG, eg, 2 * C * 4);
        bulk_commit();
    }
    // ---- T = (I + A)^-1: 16x16 diagonal blocks, then block merges ------------------
    // diagonal blocks: a lane owns column j of a block (x[i] = X_ij) and
    // column j of A; right-looking substitution: once x_k is final, every
    // later row takes -A_ik x_k (A_ik from lane k by shuffle), so the
    // dependent chain is 16 FMAs long
    if (warp < 2) {
        const int b0 = (warp * 2 + (lane >> 4)) * 16, jc = lane & 15, lb = lane & 16;
        float acol[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acol[i] = Am[(b0 + i) * LDA + b0 + jc];
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == jc) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < 15; ++k) {
#pragma unroll
            for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-__shfl_sync(0xffffffffu, acol[i], lb + k), x[k], x[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tm[(b0 + i) * LDA + b0 + jc] = x[i];
    }
    for (int f = tid; f < C * C; f += THREADS) {
        const int t = f >> 6, c = f & 63;
        if ((c >> 4) > (t >> 4)) Tm[t * LDA + c] = 0.f;
    }
    __syncthreads();
    // off-diagonal blocks by distance: X_ab = -X_aa sum_{c=b}^{a-1} A_ac X_cb;
    // the 16x16 block products run on warp-level mma.sync (3xTF32), one
    // 16x8 half block per warp
    for (int dd = 1; dd < 4; ++dd) {
        const int ntile = (4 - dd) * 2;
        for (int tl = warp; tl < ntile; tl += THREADS / 32) {  // Y = A_a[b..a) X_[b..a)b
            const int bb = tl >> 1, nt = tl & 1;
            const int a0 = (bb + dd) * 16, c0b = bb * 16;
            float cc[4];
            warp_tile16x8_precise(Am + a0 * LDA + c0b, LDA, Tm + c0b * LDA + c0b + 8 * nt, LDA, a0 - c0b, lane, cc);
            const int gq = lane >> 2, t4 = lane & 3;
            float* y0 = Tm + a0 * LDA + c0b + 8 * nt;
            y0[gq * LDA + 2 * t4] = cc[0];
            y0[gq * LDA + 2 * t4 + 1] = cc[1];
            y0[(gq + 8) * LDA + 2 * t4] = cc[2];
            y0[(gq + 8) * LDA + 2 * t4 + 1] = cc[3];
        }
        __syncthreads();
        for (int tl = warp; tl < ntile; tl += THREADS / 32) {  // X_ab = -X_aa Y
            const int bb = tl >> 1, nt = tl & 1;
            const int a0 = (bb + dd) * 16, c0b = bb * 16;
            float cc[4];
            warp_tile16x8_precise(Tm + a0 * LDA + a0, LDA, Tm + a0 * LDA + c0b + 8 * nt, LDA, 16, lane, cc);
            const int gq = lane >> 2, t4 = lane & 3;
            float* x0 = Tm + a0 * LDA + c0b + 8 * nt;
            x0[gq * LDA + 2 * t4] = -cc[0];
            x0[gq * LDA + 2 * t4 + 1] = -cc[1];
            x0[(gq + 8) * LDA + 2 * t4] = -cc[2];
            x0[(gq + 8) * LDA + 2 * t4 + 1] = -cc[3];
        }
        __syncthreads();
    }
    // ---- T diag(beta) -> record -----------------------------------------------------------
    for (int f = tid; f < C * 16; f += THREADS) {
        const int t = f >> 4, i = (f & 15) * 4;
        const float4 tv = *reinterpret_cast<const float4*>(Tm + t * LDA + i);
        tc::st_row4(TBs, C, t, i, tv.x * bet[i], tv.y * bet[i + 1], tv.z * bet[i + 2], tv.w * bet[i + 3]);
    }
    fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(rec + kRecTB, TBs, 16384);
        bulk_commit();
        bulk_wait_read_all();  // shared memory stays valid until the stores have read it
    }
    if (!ok && tid == 0) report_device_status(kDevWaitTimeout);
    if (warp == 0) tc::dealloc(tm, PR_TMEM_COLS);
}

__global__ void __launch_bounds__(tcp::THREADS, 2) k_chunk_prep2(const __grid_constant__ PrefillArgs A) {
    using namespace tcp;
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv;
    const int j = blockIdx.x, h = j / g.G;
    const int64_t cs = (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
    if (cs >= A.ncs) return;
    int64_t t0;
    int n;
    if (!slot_chunk(J, cs, t0, n)) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hf = warp >> 2;
    const int row = 32 * q4 + lane;  // the accumulator row (M = 128) this thread reads

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    unsigned char *KTs = sm + P2_KT, *VTs = sm + P2_VT, *TBs = sm + P2_TB, *Ps = sm + P2_P;
    float* eg = reinterpret_cast<float*>(sm + P2_G);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(eg + C);
    uint64_t* barIn = mbar + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 2);
    const unsigned char* tile = A.tqk + ((size_t)cs * Hk + h) * kTileQK;
    unsigned char* rec = A.trec + ((size_t)cs * Hv + j) * kTileRec;

    if (warp == 0) tc::alloc(tslot, P2_TMEM_COLS);
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(barIn, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(barIn, 32768 + 32768 + 16384 + 16384 + C * 4);
        bulk_g2s(KTs, tile + 65536, 32768, barIn);
        bulk_g2s(VTs, A.tv + ((size_t)cs * Hv + j) * kTileV, 32768, barIn);
        bulk_g2s(TBs, rec + kRecTB, 16384, barIn);
        bulk_g2s(Ps, rec + kRecP, 16384, barIn);
        bulk_g2s(eg, rec + kRecG, C * 4, barIn);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;
    bool ok = true;
    uint32_t phase = 0;
    auto wait_mma = [&]() {
        bool w = true;
        if (ok && warp == 0) {
            w = mbar_wait(mbar, phase);
            if (!w) w = mbar_wait(mbar, phase);
        }
        phase ^= 1u;
        ok = __syncthreads_and(ok && w);
        tc::fence_after();
    };
    {
        bool w = true;
        if (warp == 0) {
            w = mbar_wait(barIn, 0);
            if (!w) w = mbar_wait(barIn, 0);
        }
        ok = __syncthreads_and(w);
    }
    // K^T <- K^T diag(e^gamma), so that (K^T diag(e^gamma)) (T diag(beta))^T = W^T
    for (int f = tid; f < D * 16; f += THREADS) {
        const int d = f >> 4, t = (f & 15) * 4;
        float4* kp = reinterpret_cast<float4*>(KTs + tc::sw_off(D, d, t));
        const float4 kv = *kp;
        *kp = make_float4(tc::to_tf32_rn(kv.x * eg[t]), tc::to_tf32_rn(kv.y * eg[t + 1]),
                          tc::to_tf32_rn(kv.z * eg[t + 2]), tc::to_tf32_rn(kv.w * eg[t + 3]));
    }
    // ---- W^T = K'^T TB^T, U~^T = V^T TB^T (M = 128, N = 64, K = 64) ------------------------
    tc::fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        if (ok) {
            tc::fence_after();
            tc::mma_tf32(tm + 0, KTs, D, TBs, C, C, tc::idesc_tf32(D, C), false);
            tc::mma_tf32(tm + 64, VTs, D, TBs, C, C, tc::idesc_tf32(D, C), false);
        }
        tc::commit(mbar);
    }
    wait_mma();
    // -W -> rows 0..63 of the stacked operand; W^T and U~^T -> operand tiles
    // over K^T and V^T; U~ -> the slice blocks of the record
    unsigned char* ra = rec + kRecA;
    unsigned char* ux = rec + kRecUX + (size_t)q4 * 16384;  // slice q4 holds v = 32 q4 .. 32 q4 + 31
    for (int cb = 0; cb < 2; ++cb) {
        const int i0 = hf * 32 + cb * 16;
        float w16[16], u16[16];
        tc::ld16x2(tc::taddr(tm, 32 * q4, i0), w16, tc::taddr(tm, 32 * q4, 64 + i0), u16);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            *reinterpret_cast<float*>(ra + tc::sw_off(D, i0 + c, row)) = -tc::to_tf32_rn(w16[c]);
            *reinterpret_cast<float*>(ux + ux_off(i0 + c, lane)) = u16[c];
        }
#pragma unroll
        for (int c = 0; c < 16; c += 4) {
            tc::st_row4(KTs, D, row, i0 + c, w16[c], w16[c + 1], w16[c + 2], w16[c + 3]);
            tc::st_row4(VTs, D, row, i0 + c, u16[c], u16[c + 1], u16[c + 2], u16[c + 3]);
        }
    }
    // Q^ values of this thread's d (its column of Q) for the Q' epilogue, loaded
    // while the next products run
    const float* qtile = reinterpret_cast<const float*>(tile);  // [K^; Q^] tile (TF32 values)
    float qv[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) qv[c] = qtile[tc::sw_off(2 * C, C + hf * 32 + c, row) >> 2];
    // ---- (P W)^T = W^T P^T, X^T = U~^T P^T -------------------------------------------------
    tc::fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        if (ok) {
            tc::fence_after();
            tc::mma_tf32(tm + 0, KTs, D, Ps, C, C, tc::idesc_tf32(D, C), false);
            tc::mma_tf32(tm + 64, VTs, D, Ps, C, C, tc::idesc_tf32(D, C), false);
        }
        tc::commit(mbar);
    }
    wait_mma();
    // Q' = diag(e^gamma) Q - P W -> rows 64..127 of the stacked operand; X -> record
    for (int cb = 0; cb < 2; ++cb) {
        const int t0c = hf * 32 + cb * 16;
        float pw[16], x16[16];
        tc::ld16x2(tc::taddr(tm, 32 * q4, t0c), pw, tc::taddr(tm, 32 * q4, 64 + t0c), x16);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int t = t0c + c;
            const float qp = t < n ? fmaf(eg[t], qv[cb * 16 + c], -pw[c]) : 0.f;
            *reinterpret_cast<float*>(ra + tc::sw_off(D, C + t, row)) = tc::to_tf32_rn(qp);
            *reinterpret_cast<float*>(ux + 8192 + ux_off(t, lane)) = x16[c];
        }
    }
    if (!ok && tid == 0) report_device_status(kDevWaitTimeout);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tm, P2_TMEM_COLS);
}

// chain kernel shared memory and TMEM for NSL slices of DV = 128 / NSL state rows
template <int NSL>
struct ChainLay {
    static constexpr int DV = tcp::D / NSL;
    static constexpr int OFF_A = 0;                             // [-W; Q']   [128][128]
    static constexpr int OFF_KT = OFF_A + 65536;                // K^T        [128][64]
    static constexpr int OFF_UX = OFF_KT + 32768;               // U~ | X of the CTA's 32-row slices, 16 KB each
    static constexpr int OFF_UP = OFF_UX + (DV / 32) * 16384;   // (diag(e^(gC-g)) U)^T [DV][64]
    static constexpr int OFF_S0 = OFF_UP + DV * 64 * 4;         // S   [DV][128] (this CTA's rows)
    static constexpr int OFF_G = OFF_S0 + DV * 128 * 4;         // e^g [64] | e^(gC-g) [64]
    static constexpr int OFF_SMALL = OFF_G + 512;               // ssq [2][NSL][64], ored [2][64], norm_w [DV]
    static constexpr int SMALL_FLOATS = 2 * NSL * tcp::C + 2 * tcp::C + DV;
    static constexpr int SMEM = OFF_SMALL + SMALL_FLOATS * 4 + 64;  // + 6 mbarriers and the TMEM address
    static constexpr int SMEM_ALLOC = SMEM + 1024;                  // room to align the base to 1024 bytes
    // Ra: kIssuers partial accumulators of D, DV columns apart; Rb: S^T and kIssuers - 1 partials
    static constexpr int cD = 0, cS = DV * tcp::kIssuers, TMEM_COLS = 2 * DV * tcp::kIssuers;
};

template <int NSL>
__global__ void __launch_bounds__(tcp::THREADS, 1) k_chunk_tc(const __grid_constant__ PrefillArgs A) {
    using namespace tcp;
    using Lay = ChainLay<NSL>;
    constexpr int DV = Lay::DV;
    constexpr int HC = DV / 2;   // columns of a thread (its half of the slice)
    constexpr int NB = HC / 16;  // 16-column blocks of a thread
    constexpr int cD = Lay::cD, cS = Lay::cS;
    cg::cluster_group cluster = cg::this_cluster();
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv;
    const int s_idx = blockIdx.x, j = blockIdx.y, seq = blockIdx.z, h = j / g.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    unsigned char *As = sm + Lay::OFF_A, *KTs = sm + Lay::OFF_KT, *UXs = sm + Lay::OFF_UX;
    unsigned char *UPs = sm + Lay::OFF_UP, *S0s = sm + Lay::OFF_S0;
    float* Gs = reinterpret_cast<float*>(sm + Lay::OFF_G);     // e^g [64] | e^(gC-g) [64]
    float* ssq = reinterpret_cast<float*>(sm + Lay::OFF_SMALL);  // [2][NSL][C] row sums of squares per slice
    float* ored = ssq + 2 * NSL * C;                             // [2][C] half-row sums of squares
    float* nwsl = ored + 2 * C;                                  // norm_w of this slice
    uint64_t* mbar = reinterpret_cast<uint64_t*>(nwsl + DV);  // MMA rounds
    uint64_t* barA = mbar + 1;    // [-W; Q'] of a chunk
    uint64_t* barB = mbar + 2;    // K^T of a chunk
    uint64_t* barC = mbar + 3;    // U~, X, gates of a chunk
    uint64_t* barSq = mbar + 4;   // [2]: the peers' sums of squares of a chunk (by parity)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 6);

    if (warp == 0) tc::alloc(tslot, Lay::TMEM_COLS);
    const bool outnorm = !(g.flags & kFlagNoOutNorm);
    constexpr uint32_t kSqBytes = (NSL - 1) * C * 4;  // the peers' row sums of one chunk
    if (tid == 0) {
        mbar_init(mbar, kIssuers);  // one commit per issuing warp
        mbar_init(barA, 1);
        mbar_init(barB, 1);
        mbar_init(barC, 1);
        mbar_init(barSq, 1);
        mbar_init(barSq + 1, 1);
        fence_mbar_init();
        if (outnorm) {  // chunks 0 and 1
            mbar_arrive_expect_tx(barSq, kSqBytes);
            mbar_arrive_expect_tx(barSq + 1, kSqBytes);
        }
    }
    tc::fence_before();
    cluster.sync();  // every CTA's barriers are initialised before a peer stores into them
    tc::fence_after();
    const uint32_t tm = *tslot;
    uint32_t phase = 0;
    bool ok = true;
    const uint32_t my_rank = cluster.block_rank();

    int64_t start, end;
    seq_bounds(J, seq, start, end);
    const float* Sin = nullptr;
    float* Sout = nullptr;
    if (!J.cu_seqlens) {
        Sin = J.s0 ? J.s0 + (size_t)j * D * D : nullptr;
        Sout = J.s_final + (size_t)j * D * D;
    } else {
        const int slot = J.slot_idx[seq];
        if (slot >= 0 && slot < J.n_slots) {
            Sout = J.state_pool + ((size_t)slot * Hv + j) * D * D;
            if (J.has_init && J.has_init[seq]) Sin = Sout;
        }
    }
    const int dS = 32 * q4 + lane;  // the d_k index this thread owns in S^T
    const int col0 = hf * HC;       // this thread's first column (state row) inside the slice
    if (tid < DV) nwsl[tid] = outnorm ? Act<__nv_bfloat16>::ld(A.p.norm_w, s_idx * DV + tid) : 1.f;

    // every thread polls a barrier itself (no CTA-wide barrier needed to learn
    // that an MMA round or a copy has completed)
    auto poll = [&](uint64_t* b, uint32_t par) {
        bool w = mbar_wait(b, par);
        if (!w) w = mbar_wait(b, par);
        ok = ok && w;
    };
    auto wait_mma = [&]() {
        poll(mbar, phase);
        phase ^= 1u;
        tc::fence_after();
    };
    // the K-steps of each state product are issued by lane 0 of warps 0..3 into
    // 4 accumulators (parts) DV columns apart: the tensor core accepts
    // instructions from several warps faster than from one
    const bool issuer = lane == 0 && warp < kIssuers;

    const int64_t T = end - start;
    const int n_chunks = (int)((T + C - 1) / C);
    const bool urow = q4 < 2;                  // rows 0..63 of D: U; rows 64..127: O
    const int trow = 32 * (q4 & 1) + lane;     // the chunk row of this thread's D row
    auto rows_of = [&](int c) -> int {
        const int64_t left = end - (start + (int64_t)c * C);
        return (int)(left < C ? left : C);
    };
    // U~ (or X, +8 KB) of column c of the CTA: 32-row slice c / 32 of the record, 16 KB each
    auto ux = [&](int c, int t) -> const unsigned char* { return UXs + (c >> 5) * 16384 + ux_off(t, c & 31); };
    // operand tiles come ready-made (prologue and prep kernels): bulk copies
    // issued for chunk c+1 as soon as chunk c's last use of the buffer is done
    auto cslot = [&](int c) -> size_t { return (size_t)(start / C + seq + c); };
    auto issue_a = [&](int c) {
        mbar_arrive_expect_tx(barA, 65536);
        bulk_g2s(As, A.trec + (cslot(c) * Hv + j) * kTileRec + kRecA, 65536, barA);
    };
    auto issue_b = [&](int c) {
        mbar_arrive_expect_tx(barB, 32768);
        bulk_g2s(KTs, A.tqk + (cslot(c) * Hk + h) * kTileQK + 65536, 32768, barB);
    };
    auto issue_c = [&](int c) {
        const unsigned char* rc = A.trec + (cslot(c) * Hv + j) * kTileRec;
        mbar_arrive_expect_tx(barC, (DV / 32) * 16384 + 2 * C * 4);
        bulk_g2s(UXs, rc + kRecUX + (size_t)s_idx * (DV / 32) * 16384, (DV / 32) * 16384, barC);
        bulk_g2s(Gs, rc + kRecG, 2 * C * 4, barC);
    };
    // Ra of chunk c: D = [-W; Q'] S^T with S0s holding the state entering c
    auto issue_ra = [&](int c) {
        tc::fence_before();
        fence_proxy_async_smem();
        ok = __syncthreads_and(ok);  // S0s complete
        if (issuer) {
            poll(barA, (uint32_t)(c & 1));
            if (ok) {
                tc::fence_after();
                tc::mma_tf32_part(tm + cD, As, D, S0s, DV, D, tc::idesc_tf32(D, DV), warp, kIssuers, DV, false);
            }
            tc::commit(mbar);
        }
    };

    // initial state: S0s <- S (TF32), TMEM S^T <- e^gamma_C S for the first chunk
    float sv[HC];  // this thread's part of the state (d_k = dS, columns col0 ..)
#pragma unroll
    for (int c = 0; c < HC; ++c) {
        sv[c] = Sin ? Sin[(size_t)(s_idx * DV + col0 + c) * D + dS] : 0.f;
        tc::st_elem(S0s, DV, col0 + c, dS, sv[c]);
    }
    if (n_chunks > 0) {
        if (tid == 0) {
            issue_a(0);
            issue_b(0);
            issue_c(0);
        }
        poll(barC, 0);
        const float egC = Gs[C - 1];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = sv[b * 16 + c] * egC;
            tc::st16(tc::taddr(tm, 32 * q4, cS + col0 + b * 16), v);
        }
        issue_ra(0);
    }
    for (int ci = 0; ci < n_chunks; ++ci) {
        const int64_t t0 = start + (int64_t)ci * C;
        const int n = rows_of(ci);
        const uint32_t par = (uint32_t)(ci & 1);
        wait_mma();                                          // Ra of this chunk
        if (tid == 0 && ci + 1 < n_chunks) issue_a(ci + 1);  // [-W; Q'] is free
        // ---- U = U~ + D[0:64] -> (diag(e^(gC - g)) U)^T tile (warps 0,1,4,5); O = X +
        // D[64:128] and its sums of squares (warps 2,3,6,7); HC columns per thread -------
        float* ssq_cur = ssq + (ci & 1) * NSL * C;  // [NSL][C]
        uint64_t* bar_sq = barSq + (ci & 1);
        float ov[HC];
        if (urow) {
            const float er = Gs[C + trow];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float d16[16];
                tc::ld16_sum4(tc::taddr(tm, 32 * q4, cD + col0 + b * 16), DV, d16);
#pragma unroll
                for (int c4 = 0; c4 < 16; c4 += 4) {
                    const int c = col0 + b * 16 + c4;
                    const float4 a = *reinterpret_cast<const float4*>(ux(c, trow));
                    tc::st_elem(UPs, DV, c, trow, (a.x + d16[c4]) * er);
                    tc::st_elem(UPs, DV, c + 1, trow, (a.y + d16[c4 + 1]) * er);
                    tc::st_elem(UPs, DV, c + 2, trow, (a.z + d16[c4 + 2]) * er);
                    tc::st_elem(UPs, DV, c + 3, trow, (a.w + d16[c4 + 3]) * er);
                }
            }
            fence_proxy_async_smem();  // U' is read by the tensor core
        } else {
            float part = 0.f;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float d16[16];
                tc::ld16_sum4(tc::taddr(tm, 32 * q4, cD + col0 + b * 16), DV, d16);
#pragma unroll
                for (int c4 = 0; c4 < 16; c4 += 4) {
                    const float4 a = *reinterpret_cast<const float4*>(ux(col0 + b * 16 + c4, trow) + 8192);
                    float* o = ov + b * 16 + c4;
                    o[0] = a.x + d16[c4];
                    o[1] = a.y + d16[c4 + 1];
                    o[2] = a.z + d16[c4 + 2];
                    o[3] = a.w + d16[c4 + 3];
#pragma unroll
                    for (int e = 0; e < 4; ++e) part = fmaf(o[e], o[e], part);
                }
            }
            ored[hf * C + trow] = part;
            named_bar_sync(1, 128);  // warps 2,3,6,7
            if (hf == 0 && outnorm) {  // this slice's row sum -> every CTA of the cluster
                const float sq = ored[trow] + ored[C + trow];
                float* mine = ssq_cur + my_rank * C + trow;
                *mine = sq;
#pragma unroll
                for (int r = 0; r < NSL; ++r)
                    if (r != (int)my_rank)
                        st_async_f32(mapa_shared(tc::smem_addr(mine), r), sq, mapa_shared(tc::smem_addr(bar_sq), r));
            }
        }
        // ---- Rb: S^T += K^T U' --------------------------------------------------------------
        // warps 0..5: the U' writers (0, 1, 4, 5) and the issuers (0..3); the O warps 6, 7
        // have passed barrier 1 with warps 2, 3, so every read of U~, X and the gates is done
        if (warp < 6) {
            tc::fence_before();
            named_bar_sync(2, 192);
        }
        if (issuer) {
            poll(barB, par);
            if (ok) {
                tc::fence_after();
                tc::mma_tf32_part(tm + cS, KTs, D, UPs, DV, C, tc::idesc_tf32(D, DV), warp, kIssuers, DV, true);
            }
            tc::commit(mbar);
        }
        if (tid == 0 && ci + 1 < n_chunks) issue_c(ci + 1);  // U~, X and the gates have been read
        uint4 zr[HC / 8];  // z of this thread's output row
        if (!urow && outnorm && trow < n) {
            const uint4* zp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(J.z) +
                                                             (size_t)(t0 + trow) * Hv * D + (size_t)j * D +
                                                             s_idx * DV + col0);
#pragma unroll
            for (int q = 0; q < HC / 8; ++q) zr[q] = zp[q];
        }
        wait_mma();                                          // Rb
        if (tid == 0 && ci + 1 < n_chunks) issue_b(ci + 1);  // K^T is free
        // ---- S^T -> S operand tile for the next chunk ----------------------------------------
#pragma unroll
        for (int b = 0; b < NB; ++b) tc::ld16_sum4(tc::taddr(tm, 32 * q4, cS + col0 + b * 16), DV, sv + b * 16);
#pragma unroll
        for (int c = 0; c < HC; ++c) tc::st_elem(S0s, DV, col0 + c, dS, sv[c]);
        const int ck = ckpt_after(J, seq, (int64_t)(ci + 1) * C, T);
        if (ck >= 0) {  // a prefix snapshot ends with this chunk
            float* dst = J.state_pool + ((size_t)ck * Hv + j) * D * D;
#pragma unroll
            for (int c = 0; c < HC; ++c) dst[(size_t)(s_idx * DV + col0 + c) * D + dS] = sv[c];
        }
        if (ci + 1 < n_chunks) {
            issue_ra(ci + 1);
            poll(barC, par ^ 1u);  // gates of the next chunk: S^T <- e^gamma_C S^T (the sum) in TMEM
            const float egC = Gs[C - 1];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float v[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) v[c] = sv[b * 16 + c] * egC;
                tc::st16(tc::taddr(tm, 32 * q4, cS + col0 + b * 16), v);
            }
        }
        // ---- y = gated RMSNorm(O) of this chunk (while Ra of the next chunk runs) ---------
        if (!urow) {
            float rstd = 1.f;
            if (outnorm) {  // the peers' row sums of this chunk have landed
                const uint32_t sq_par = (uint32_t)((ci >> 1) & 1);
                bool w = mbar_wait(bar_sq, sq_par);
                if (!w) w = mbar_wait(bar_sq, sq_par);
                ok = ok && w;
                if (tid == 64) mbar_arrive_expect_tx(bar_sq, kSqBytes);  // for chunk ci + 2
                float tot = 0.f;
#pragma unroll
                for (int r = 0; r < NSL; ++r) tot += ssq_cur[r * C + trow];
                rstd = rsqrtf(tot / (float)D + g.norm_eps);
            }
            if (trow < n) {
                const __nv_bfloat162* zh = reinterpret_cast<const __nv_bfloat162*>(zr);
                uint4 pk[HC / 8];
                __nv_bfloat162* hp = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
                for (int c = 0; c < HC / 2; ++c) {
                    float y0 = ov[2 * c], y1 = ov[2 * c + 1];
                    if (outnorm) {
                        const float2 zz = __bfloat1622float2(zh[c]);
                        y0 = y0 * rstd * nwsl[col0 + 2 * c] * silu_fast(zz.x);
                        y1 = y1 * rstd * nwsl[col0 + 2 * c + 1] * silu_fast(zz.y);
                    }
                    hp[c] = __floats2bfloat162_rn(y0, y1);
                }
                uint4* yp = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(J.y) + (size_t)(t0 + trow) * Hv * D +
                                                     (size_t)j * D + s_idx * DV + col0);
#pragma unroll
                for (int q = 0; q < HC / 8; ++q) yp[q] = pk[q];
            }
        }
    }
    // ---- final state (the S operand registers hold the state after the last chunk) ---------
    if (Sout) {
#pragma unroll
        for (int c = 0; c < HC; ++c) Sout[(size_t)(s_idx * DV + col0 + c) * D + dS] = sv[c];
    }
    tc::fence_before();
    ok = __syncthreads_and(ok);
    if (!ok && tid == 0) report_device_status(kDevWaitTimeout);
    if (warp == 0) tc::dealloc(tm, Lay::TMEM_COLS);
    cluster.sync();  // every st.async into this CTA's shared memory has landed
}

// Slices of the chain per (sequence, v-head): 4 CTAs of 32 state rows finish a
// long sequence soonest; when the chain CTAs fill the GPU more than once over,
// 2 CTAs of 64 rows do the same work in half the instructions (an MMA costs
// about the same at N = 64 as at N = 32), so the waves drain sooner.
int chain_slices(const PrefillArgs& A) {
    if (const char* e = std::getenv("GDN_CHAIN_SLICES")) {
        const int v = std::atoi(e);
        if (v == 2 || v == 4) return v;
    }
    return (int64_t)A.J.n_seq * A.g.Hv * 4 > (int64_t)sm_count() ? 2 : 4;
}

template <int NSL>
cudaError_t launch_chain(const PrefillArgs& A, cudaStream_t st) {
    static std::atomic<uint64_t> smem_set{0};
    {
        const cudaError_t e = raise_smem_limit(k_chunk_tc<NSL>, ChainLay<NSL>::SMEM_ALLOC, smem_set);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(NSL, A.g.Hv, A.J.n_seq);
    cfg.blockDim = dim3(tcp::THREADS);
    cfg.dynamicSmemBytes = ChainLay<NSL>::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = NSL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_chunk_tc<NSL>, A);
}

cudaError_t launch_chunk_tc(const PrefillArgs& A, int64_t n_slots, cudaStream_t st) {
    static std::atomic<uint64_t> attr1{0}, attr2{0};
    {
        cudaError_t e = raise_smem_limit(k_chunk_prep, tcp::PR_SMEM_ALLOC, attr1);
        if (e != cudaSuccess) return e;
        e = raise_smem_limit(k_chunk_prep2, tcp::P2_SMEM_ALLOC, attr2);
        if (e != cudaSuccess) return e;
    }
    if (n_slots > 0) {
        const int64_t ny = n_slots < 32768 ? n_slots : 32768;
        const dim3 grid((unsigned)A.g.Hv, (unsigned)ny, (unsigned)((n_slots + ny - 1) / ny));
        k_chunk_prep<<<grid, tcp::THREADS, tcp::PR_SMEM_ALLOC, st>>>(A);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        k_chunk_prep2<<<grid, tcp::THREADS, tcp::P2_SMEM_ALLOC, st>>>(A);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return chain_slices(A) == 2 ? launch_chain<2>(A, st) : launch_chain<4>(A, st);
}

int prefill_slices(int D) {
    if (const char* e = std::getenv("GDN_PREFILL_SLICES")) {
        const int v = std::atoi(e);
        if ((v == 1 || v == 2 || v == 4 || v == 8) && D / v >= 16) return v;
    }
    return D >= 128 ? 4 : (D >= 64 ? 2 : 1);
}

template <int D, typename TA>
cudaError_t launch_prefill_t(const Geom& g, const LayerParams& p, const PrefillJob& J, cudaStream_t st) {
    const WsLayout wl = ws_layout(g, J.n_tokens);
    char* ws = static_cast<char*>(J.workspace);
    PrefillArgs A;
    A.g = g;
    A.p = p;
    A.J = J;
    A.qk = reinterpret_cast<float*>(ws + wl.qk);
    A.v = reinterpret_cast<float*>(ws + wl.v);
    A.gl = reinterpret_cast<float*>(ws + wl.g);
    A.beta = reinterpret_cast<float*>(ws + wl.beta);
    A.NS = prefill_slices(D);
    A.tiles = (D == 128 && g.chunk == 64 && g.act_bf16 && std::getenv("GDN_PREFILL_PRECISE") == nullptr &&
               std::getenv("GDN_PREFILL_MMA_SYNC") == nullptr)
                  ? 1
                  : 0;
    if (A.tiles) {
        const TileWs tl = tile_ws(g, J.n_tokens, J.n_seq);
        A.tqk = reinterpret_cast<unsigned char*>(ws + tl.qk);
        A.tv = reinterpret_cast<unsigned char*>(ws + tl.v);
        A.tgb = reinterpret_cast<float*>(ws + tl.gb);
        A.trec = reinterpret_cast<unsigned char*>(ws + tl.rec);
        A.ncs = tl.ncs;
    }
    if (A.tiles) {
        static std::atomic<uint64_t> smem_set{0};
        {
            const cudaError_t e = raise_smem_limit(k_prologue_tc, kPtSmemAlloc, smem_set);
            if (e != cudaSuccess) return e;
        }
        const int64_t ny = A.ncs < 32768 ? A.ncs : 32768;
        const dim3 grid((unsigned)(g.Hk + g.Hv), (unsigned)ny, (unsigned)((A.ncs + ny - 1) / ny));
        k_prologue_tc<<<grid, kPtThreads, kPtSmemAlloc, st>>>(A);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else if (J.n_tokens > 0) {
        constexpr int VEC = 16 / (int)sizeof(TA);
        const dim3 blocks((unsigned)((J.n_tokens + kProTok - 1) / kProTok),
                          (unsigned)((g.C_ch / VEC + kProThreads - 1) / kProThreads));
        k_prologue<D, TA><<<blocks, kProThreads, 0, st>>>(A);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const size_t total = (size_t)J.n_seq * g.C_ch;
        const int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 8);
        k_conv_final<TA><<<blocks, 256, 0, st>>>(A);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (J.ckpt_every > 0 && J.n_tokens > 0) {
        k_conv_ckpt<TA><<<dim3((unsigned)((g.C_ch + 255) / 256), (unsigned)J.n_seq, 16u), 256, 0, st>>>(A);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (A.tiles) return launch_chunk_tc(A, A.ncs, st);
    const int DV = D / A.NS;
    const ChunkSmem lay = chunk_smem(g.chunk, D, DV);
    const size_t smem = (size_t)lay.total * sizeof(float);
    const bool precise = !g.act_bf16 || std::getenv("GDN_PREFILL_PRECISE") != nullptr;
    auto kern = precise ? k_chunk<D, true, TA> : k_chunk<D, false, TA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(A.NS, g.Hv, J.n_seq);
    cfg.blockDim = dim3(kChunkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = A.NS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, A);
}

}  // namespace

cudaError_t take_device_status_prefill(unsigned* out) { return take_device_status_tu(out); }

size_t prefill_workspace_bytes(const Geom& g, int64_t n_tokens, int n_seq) {
    if (n_tokens <= 0) return 0;
    size_t bytes = ws_layout(g, n_tokens).total;
    if (g.D == 128 && g.chunk == 64 && g.act_bf16) bytes = std::max(bytes, tile_ws(g, n_tokens, n_seq).total);
    return bytes;
}

cudaError_t launch_prefill(const Geom& g, const LayerParams& p, const PrefillJob& J, cudaStream_t st) {
    if (J.n_seq == 0) return cudaSuccess;
    if (g.act_bf16) {
        switch (g.D) {
            case 32: return launch_prefill_t<32, __nv_bfloat16>(g, p, J, st);
            case 64: return launch_prefill_t<64, __nv_bfloat16>(g, p, J, st);
            case 128: return launch_prefill_t<128, __nv_bfloat16>(g, p, J, st);
        }
    } else {
        switch (g.D) {
            case 32: return launch_prefill_t<32, float>(g, p, J, st);
            case 64: return launch_prefill_t<64, float>(g, p, J, st);
            case 128: return launch_prefill_t<128, float>(g, p, J, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
