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

// 16-byte global -> shared copy; src_bytes = 0 fills the 16 bytes with zeros
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst_smem)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

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
//   per (slot, k-head): Q^ [64][128] | K^ [64][128] | K^T [128][64]   (3 x 32 KB)
//   per (slot, v-head, slice): V^T [32][64]                           (8 KB)
//   per (slot, v-head): g [64], beta [64]                              (512 B)
//   per (slot, v-head): chain record written by the prep kernel       (65 KB)
//     W [64][128] | T diag(beta) [64][64] | P [64][64] | e^gamma [64], e^(gamma_C - gamma) [64]
constexpr size_t kTileQK = 3 * 32768, kTileV = 4 * 8192, kTileGB = 2 * 64 * 4;
constexpr size_t kRecW = 0, kRecTB = 32768, kRecP = 49152, kRecG = 65536, kTileRec = 66560;

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

// chunk slot and row of token n of sequence s (start = its first token)
__device__ __forceinline__ void chunk_slot(int64_t n, int64_t start, int s, int64_t& cs, int& r) {
    const int64_t rel = n - start;
    cs = start / 64 + s + rel / 64;
    r = (int)(rel % 64);
}

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
            if (A.tiles) {
                const int sq = find_seq(J, n);
                int64_t st_, en_, cs;
                int r;
                seq_bounds(J, sq, st_, en_);
                chunk_slot(n, st_, sq, cs, r);
                float* gb = A.tgb + ((size_t)cs * Hv + j) * 128;
                gb[r] = gl;
                gb[64 + r] = be;
            } else {
                A.gl[(size_t)n * Hv + j] = gl;
                A.beta[(size_t)n * Hv + j] = be;
            }
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
    // tile mode: K^T and V^T tile rows are t-contiguous; 4 consecutive tokens of
    // the same chunk slot go out as one 16-byte store per channel
    float tb[VEC][4];
    int64_t tb_cs = -1;
    int tb_r0 = 0, tb_n = 0;
    unsigned char* tb_base = nullptr;
    int tb_rows = 0, tb_row0 = 0;  // tile rows (128 for K^T, 32 for V^T) and this thread's first row
    auto tb_flush = [&]() {
        if (tb_n == 0) return;
        if (tb_n == 4 && (tb_r0 & 3) == 0) {
#pragma unroll
            for (int c = 0; c < VEC; ++c)
                *reinterpret_cast<float4*>(tb_base + tc::sw_off(tb_rows, tb_row0 + c, tb_r0)) =
                    make_float4(tb[c][0], tb[c][1], tb[c][2], tb[c][3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < tb_n) {
#pragma unroll
                    for (int c = 0; c < VEC; ++c)
                        *reinterpret_cast<float*>(tb_base + tc::sw_off(tb_rows, tb_row0 + c, tb_r0 + e)) = tb[c][e];
                }
        }
        tb_n = 0;
    };
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
            if (A.tiles && D == 128) {
                if (active) {
                    int64_t cs;
                    int r;
                    chunk_slot(n, start, s, cs, r);
                    const int hq = ch0 / D, d0 = ch0 % D;
                    const int hh = hq < Hk ? hq : hq - Hk;
                    unsigned char* tile = A.tqk + ((size_t)cs * Hk + hh) * kTileQK + (hq < Hk ? 0 : 32768);
#pragma unroll
                    for (int c = 0; c < VEC; c += 4)
                        *reinterpret_cast<float4*>(tile + tc::sw_off(64, r, d0 + c)) =
                            make_float4(tc::to_tf32_rn(u[c] * scale), tc::to_tf32_rn(u[c + 1] * scale),
                                        tc::to_tf32_rn(u[c + 2] * scale), tc::to_tf32_rn(u[c + 3] * scale));
                    if (hq >= Hk) {  // K^T tile: element (d, t), buffered over 4 tokens
                        if (tb_n > 0 && (cs != tb_cs || r != tb_r0 + tb_n || tb_n == 4)) tb_flush();
                        if (tb_n == 0) {
                            tb_cs = cs;
                            tb_r0 = r;
                            tb_base = A.tqk + ((size_t)cs * Hk + hh) * kTileQK + 65536;
                            tb_rows = 128;
                            tb_row0 = d0;
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (e == tb_n) {
#pragma unroll
                                for (int c = 0; c < VEC; ++c) tb[c][e] = tc::to_tf32_rn(u[c] * scale);
                            }
                        ++tb_n;
                    }
                }
            } else if (active) {
                float4* dst = reinterpret_cast<float4*>(A.qk + (size_t)n * 2 * Hk * D + ch0);
#pragma unroll
                for (int c = 0; c < VEC; c += 4)
                    dst[c / 4] = make_float4(u[c] * scale, u[c + 1] * scale, u[c + 2] * scale, u[c + 3] * scale);
            }
        } else if (active && A.tiles && D == 128) {
            int64_t cs;
            int r;
            chunk_slot(n, start, s, cs, r);
            const int c0 = ch0 - 2 * Hk * D, jj = c0 / D, dv0 = c0 % D, sl = dv0 / 32;
            if (tb_n > 0 && (cs != tb_cs || r != tb_r0 + tb_n || tb_n == 4)) tb_flush();
            if (tb_n == 0) {
                tb_cs = cs;
                tb_r0 = r;
                tb_base = A.tv + (((size_t)cs * Hv + jj) * 4 + sl) * 8192;
                tb_rows = 32;
                tb_row0 = dv0 % 32;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e == tb_n) {
#pragma unroll
                    for (int c = 0; c < VEC; ++c) tb[c][e] = tc::to_tf32_rn(u[c]);
                }
            ++tb_n;
        } else if (active) {
            float4* dst = reinterpret_cast<float4*>(A.v + (size_t)n * Hv * D + (ch0 - 2 * Hk * D));
#pragma unroll
            for (int c = 0; c < VEC; c += 4) dst[c / 4] = make_float4(u[c], u[c + 1], u[c + 2], u[c + 3]);
        }
    }
    if (A.tiles && D == 128) tb_flush();
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
// 3b. tcgen05 path (d = 128, C = 64, bf16): prep kernel + chain kernel
// ---------------------------------------------------------------------------
// The chunk form splits into work that does not depend on the state and the
// short sequential chain that does.
//
// k_chunk_prep, one CTA per (chunk slot, v-head j), all chunks in parallel:
//   gamma = cumsum(g), KK^T and QK^T (tcgen05), the decay masks
//   A = strict-lower(beta_t e^(gamma_t - gamma_i) KK^T) and
//   P = lower-incl(e^(gamma_t - gamma_i) QK^T), T = (I + A)^-1 (16x16 blocks,
//   fp32), T diag(beta), and W = T diag(beta e^gamma) K (tcgen05); W, T
//   diag(beta), P as TF32 operand tiles and e^gamma, e^(gamma_C - gamma) go
//   to the chain record of the chunk.
// k_chunk_tc, one CTA per (sequence, v-head j, slice of 32 of the 128 state
// rows), the 4 slices of a v-head a cluster: the fp32 state slice lives in
// TMEM as S^T (lane = d_k index, 32 columns = this slice's d_v rows) for the
// whole sequence, and per chunk two rounds of tcgen05.mma
//   Ra  U = T diag(beta) V - W S^T,  O1 = Q S^T
//   Rb  O2 = P U,  S^T <- e^gamma_C S^T + K^T (diag(e^(gamma_C - gamma)) U)
// with y = gated RMSNorm(diag(e^gamma) O1 + O2) of chunk c written while Ra
// of chunk c+1 runs.  TF32 operands are rounded to nearest; accumulation is
// fp32 in TMEM.

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

namespace tcp {
constexpr int C = 64, D = 128, DV = 32, NS = 4, THREADS = 256, LDA = 68;
// prep kernel shared memory
constexpr int PR_R0 = 0;                       // Q^, then K^T, then W staging   (32 KB)
constexpr int PR_R1 = 32768;                   // K^, then P | T diag(b) staging (32 KB)
constexpr int PR_AM = 65536;                   // fp32 A [64][68], then the T diag(b e^g) tile
constexpr int PR_TM = PR_AM + C * LDA * 4;     // fp32 T [64][68]
constexpr int PR_SMALL = PR_TM + C * LDA * 4;  // gam, bet, e^g, e^(gC-g)
constexpr int PR_SMEM = PR_SMALL + 4 * C * 4 + 64;
constexpr int PR_SMEM_ALLOC = PR_SMEM + 1024;
constexpr int pKK = 0, pQK = 64, pW = 128, PR_TMEM_COLS = 256;
// chain kernel shared memory
constexpr int OFF_Q = 0;                   // Q^  [64][128]
constexpr int OFF_W = OFF_Q + 32768;       // W   [64][128]
constexpr int OFF_KT = OFF_W + 32768;      // K^T [128][64]
constexpr int OFF_TB = OFF_KT + 32768;     // T diag(b) [64][64]
constexpr int OFF_P = OFF_TB + 16384;      // P   [64][64]
constexpr int OFF_VT = OFF_P + 16384;      // V^T of this slice [32][64]
constexpr int OFF_UP = OFF_VT + 8192;      // (diag(e^(gC-g)) U)^T [32][64]
constexpr int OFF_UT = OFF_UP + 8192;      // U^T [32][64]
constexpr int OFF_S0 = OFF_UT + 8192;      // S   [32][128] (this slice's rows)
constexpr int OFF_G = OFF_S0 + 16384;      // e^g [64] | e^(gC-g) [64]
constexpr int OFF_SMALL = OFF_G + 512;     // ssq [2][64], ored [2][64], norm_w slice [32]
constexpr int SMALL_FLOATS = 4 * C + DV;
constexpr int SMEM = OFF_SMALL + SMALL_FLOATS * 4 + 64;  // + 3 mbarriers and the TMEM address
constexpr int SMEM_ALLOC = SMEM + 1024;                  // room to align the base to 1024 bytes
constexpr int cU = 0, cO1 = 32, cO2 = 64, cS = 96, TMEM_COLS = 128;
}  // namespace tcp

__global__ void __launch_bounds__(tcp::THREADS, 2) k_chunk_prep(const __grid_constant__ PrefillArgs A) {
    using namespace tcp;
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv;
    const int j = blockIdx.x, h = j / g.G;
    const int64_t cs = (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
    if (cs >= A.ncs) return;
    const int sq = slot_seq(J, cs);
    int64_t start, end;
    seq_bounds(J, sq, start, end);
    const int64_t t0 = (cs - (start / C + sq)) * C + start;
    if (t0 < start || t0 >= end) return;  // a slot between two sequences' chunks
    const int n = (int)((end - t0) < C ? (end - t0) : C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hf = warp >> 2;
    const int trow = 16 * q4 + (lane & 15);  // the chunk row this thread reads from M=64 accumulators
    const bool rowok = lane < 16;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    unsigned char *R0 = sm + PR_R0, *R1 = sm + PR_R1;
    unsigned char *Ps = R1, *TBs = R1 + 16384, *TWs = sm + PR_AM;
    float* Am = reinterpret_cast<float*>(sm + PR_AM);
    float* Tm = reinterpret_cast<float*>(sm + PR_TM);
    float* gam = reinterpret_cast<float*>(sm + PR_SMALL);
    float* bet = gam + C;
    float* eg = bet + C;
    float* erev = eg + C;  // e^g and e^(gC-g) contiguous: one bulk store
    uint64_t* mbar = reinterpret_cast<uint64_t*>(erev + C);
    uint64_t* barQK = mbar + 1;
    uint64_t* barKT = mbar + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 3);
    const unsigned char* tile = A.tqk + ((size_t)cs * Hk + h) * kTileQK;
    unsigned char* rec = A.trec + ((size_t)cs * Hv + j) * kTileRec;

    if (warp == 0) tc::alloc(tslot, PR_TMEM_COLS);
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(barQK, 1);
        mbar_init(barKT, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(barQK, 65536);
        bulk_g2s(R0, tile, 32768, barQK);
        bulk_g2s(R1, tile + 32768, 32768, barQK);
    }
    if (tid < C) {
        const float* gb = A.tgb + ((size_t)cs * Hv + j) * 128;
        gam[tid] = tid < n ? gb[tid] : 0.f;
        bet[tid] = tid < n ? gb[C + tid] : 0.f;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;
    uint32_t phase = 0;
    bool ok = true;
    auto wait_bar = [&](uint64_t* b, uint32_t par) {  // one warp polls, then everyone
        bool w = true;
        if (ok && warp == 0) {
            w = mbar_wait(b, par);
            if (!w) w = mbar_wait(b, par);
        }
        ok = __syncthreads_and(ok && w);
    };
    auto mma_round_begin = [&]() {
        tc::fence_before();
        fence_proxy_async_smem();
        __syncthreads();
    };
    auto mma_round_end = [&]() {
        if (tid == 0) tc::commit(mbar);
        bool w = true;
        if (ok && warp == 0) {
            w = mbar_wait(mbar, phase);
            if (!w) w = mbar_wait(mbar, phase);
        }
        phase ^= 1u;
        ok = __syncthreads_and(ok && w);
        tc::fence_after();
    };

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
    wait_bar(barQK, 0);
    if (n < C) {  // rows past the sequence end were never written: zero them
        for (int f = tid; f < (C - n) * 32; f += THREADS) {
            const int r = n + (f >> 5), c4 = (f & 31) * 4;
            *reinterpret_cast<float4*>(R0 + tc::sw_off(C, r, c4)) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(R1 + tc::sw_off(C, r, c4)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // ---- KK^T, QK^T ----------------------------------------------------------------------
    mma_round_begin();
    if (tid == 0 && ok) {
        tc::fence_after();
        tc::mma_tf32(tm + pKK, R1, C, R1, C, D, tc::idesc_tf32(C, C), false);
        tc::mma_tf32(tm + pQK, R0, C, R1, C, D, tc::idesc_tf32(C, C), false);
    }
    mma_round_end();
    if (tid == 0) {  // Q^ is no longer read: K^T into its place
        mbar_arrive_expect_tx(barKT, 32768);
        bulk_g2s(R0, tile + 65536, 32768, barKT);
    }
    // ---- decay masks: A (strictly lower, beta_t), P (lower incl.) -----------------------
    for (int cb = 0; cb < 2; ++cb) {
        const int i0 = hf * 32 + cb * 16;
        float kk[16], qk[16];
        tc::ld16x2(tc::taddr(tm, 32 * q4, pKK + i0), kk, tc::taddr(tm, 32 * q4, pQK + i0), qk);
        if (rowok) {
            const int t = trow;
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
                float a4[4], p4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = i0 + c + e;
                    const float dec = i <= t ? __expf(gam[t] - gam[i]) : 0.f;  // exponent <= 0 only
                    a4[e] = i < t ? bet[t] * dec * kk[c + e] : 0.f;
                    p4[e] = dec * qk[c + e];
                }
                *reinterpret_cast<float4*>(Am + t * LDA + i0 + c) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                tc::st_row4(Ps, C, t, i0 + c, p4[0], p4[1], p4[2], p4[3]);
            }
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
    // ---- T diag(beta) (to the record) and T diag(beta e^gamma) (over A) -------------------
    for (int f = tid; f < C * 16; f += THREADS) {
        const int t = f >> 4, i = (f & 15) * 4;
        const float4 tv = *reinterpret_cast<const float4*>(Tm + t * LDA + i);
        tc::st_row4(TBs, C, t, i, tv.x * bet[i], tv.y * bet[i + 1], tv.z * bet[i + 2], tv.w * bet[i + 3]);
        tc::st_row4(TWs, C, t, i, tv.x * bet[i] * eg[i], tv.y * bet[i + 1] * eg[i + 1],
                    tv.z * bet[i + 2] * eg[i + 2], tv.w * bet[i + 3] * eg[i + 3]);
    }
    fence_proxy_async_smem();
    wait_bar(barKT, 0);
    if (tid == 0) {
        bulk_s2g(rec + kRecTB, TBs, 16384);
        bulk_commit();
    }
    if (n < C) {  // tail columns (t >= n) of K^T
        for (int f = tid; f < D * (C - n); f += THREADS) {
            const int row = f / (C - n), t = n + f % (C - n);
            *reinterpret_cast<float*>(R0 + tc::sw_off(D, row, t)) = 0.f;
        }
    }
    // ---- W = T diag(beta e^gamma) K --------------------------------------------------------
    mma_round_begin();
    if (tid == 0 && ok) {
        tc::fence_after();
        tc::mma_tf32(tm + pW, TWs, C, R0, D, C, tc::idesc_tf32(C, D), false);
    }
    mma_round_end();
    for (int cb = 0; cb < 4; ++cb) {  // W -> operand tile over K^T (no longer read)
        const int d0 = hf * 64 + cb * 16;
        float w16[16];
        tc::ld16(tc::taddr(tm, 32 * q4, pW + d0), w16);
        if (rowok) {
#pragma unroll
            for (int c = 0; c < 16; c += 4) tc::st_row4(R0, C, trow, d0 + c, w16[c], w16[c + 1], w16[c + 2], w16[c + 3]);
        }
    }
    fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(rec + kRecW, R0, 32768);
        bulk_commit();
        bulk_wait_all();  // shared memory stays valid until the stores have completed
    }
    if (!ok && tid == 0) report_device_status(kDevWaitTimeout);
    if (warp == 0) tc::dealloc(tm, PR_TMEM_COLS);
}

__global__ void __launch_bounds__(tcp::THREADS, 1) k_chunk_tc(const __grid_constant__ PrefillArgs A) {
    using namespace tcp;
    cg::cluster_group cluster = cg::this_cluster();
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
    const int Hk = g.Hk, Hv = g.Hv;
    const int s_idx = blockIdx.x, j = blockIdx.y, seq = blockIdx.z, h = j / g.G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half

    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (tc::smem_addr(smem_raw) & 1023)) & 1023);
    unsigned char *Qs = sm + OFF_Q, *Ws = sm + OFF_W, *KTs = sm + OFF_KT, *TBs = sm + OFF_TB, *Ps = sm + OFF_P;
    unsigned char *VTs = sm + OFF_VT, *UPs = sm + OFF_UP, *UTs = sm + OFF_UT, *S0s = sm + OFF_S0;
    float* Gs = reinterpret_cast<float*>(sm + OFF_G);  // e^g [64] | e^(gC-g) [64]
    float* ssq = reinterpret_cast<float*>(sm + OFF_SMALL);  // [2][C]
    float* ored = ssq + 2 * C;                               // [2][C]
    float* nwsl = ored + 2 * C;                              // norm_w of this slice
    uint64_t* mbar = reinterpret_cast<uint64_t*>(nwsl + DV);  // MMA rounds
    uint64_t* barA = mbar + 1;  // Q^, W, T diag(b), V^T of a chunk
    uint64_t* barB = mbar + 2;  // K^T, P, gates of a chunk
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 3);

    if (warp == 0) tc::alloc(tslot, TMEM_COLS);
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init(barA, 1);
        mbar_init(barB, 1);
        fence_mbar_init();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;
    uint32_t phase = 0;
    bool ok = true;

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
    if (tid < DV) nwsl[tid] = (g.flags & kFlagNoOutNorm) ? 1.f : Act<__nv_bfloat16>::ld(A.p.norm_w, s_idx * DV + tid);
    {
        float v[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int dv = hf * 16 + c;
            v[c] = Sin ? Sin[(size_t)(s_idx * DV + dv) * D + dS] : 0.f;
            tc::st_elem(S0s, DV, dv, dS, v[c]);
        }
        tc::st16(tc::taddr(tm, 32 * q4, cS + hf * 16), v);
    }

    auto mma_round_begin = [&]() {
        tc::fence_before();
        fence_proxy_async_smem();
        __syncthreads();
    };
    auto wait_mma = [&]() {
        bool w = true;
        if (ok && warp == 0) {  // one warp polls, the others sleep in bar.sync
            w = mbar_wait(mbar, phase);
            if (!w) w = mbar_wait(mbar, phase);
        }
        phase ^= 1u;
        ok = __syncthreads_and(ok && w);
        tc::fence_after();
    };
    auto wait_bar = [&](uint64_t* b, uint32_t par) {
        bool w = true;
        if (ok && warp == 0) {
            w = mbar_wait(b, par);
            if (!w) w = mbar_wait(b, par);
        }
        ok = __syncthreads_and(ok && w);
    };

    const int64_t T = end - start;
    const int n_chunks = (int)((T + C - 1) / C);
    const bool outnorm = !(g.flags & kFlagNoOutNorm);
    const int trow = 16 * q4 + (lane & 15);  // the chunk row this thread reads from M=64 accumulators
    const bool rowok = lane < 16;
    auto rows_of = [&](int c) -> int {
        const int64_t left = end - (start + (int64_t)c * C);
        return (int)(left < C ? left : C);
    };
    // operand tiles come ready-made (prologue and prep kernel): bulk copies
    // issued for chunk c+1 as soon as chunk c's last use of the buffer is done
    auto cslot = [&](int c) -> size_t { return (size_t)(start / C + seq + c); };
    auto issue_a = [&](int c) {
        const unsigned char* tq = A.tqk + (cslot(c) * Hk + h) * kTileQK;
        const unsigned char* rc = A.trec + (cslot(c) * Hv + j) * kTileRec;
        mbar_arrive_expect_tx(barA, 32768 + 32768 + 16384 + 8192);
        bulk_g2s(Qs, tq, 32768, barA);
        bulk_g2s(Ws, rc + kRecW, 32768, barA);
        bulk_g2s(TBs, rc + kRecTB, 16384, barA);
        bulk_g2s(VTs, A.tv + ((cslot(c) * Hv + j) * 4 + s_idx) * 8192, 8192, barA);
    };
    auto issue_b = [&](int c) {
        const unsigned char* tq = A.tqk + (cslot(c) * Hk + h) * kTileQK;
        const unsigned char* rc = A.trec + (cslot(c) * Hv + j) * kTileRec;
        mbar_arrive_expect_tx(barB, 32768 + 16384 + 2 * C * 4);
        bulk_g2s(KTs, tq + 65536, 32768, barB);
        bulk_g2s(Ps, rc + kRecP, 16384, barB);
        bulk_g2s(Gs, rc + kRecG, 2 * C * 4, barB);
    };
    // Ra of chunk c: U = T diag(b) V - W S^T, O1 = Q S^T (S0s holds the state
    // entering chunk c); committed, not waited for
    auto issue_ra = [&](int c) {
        wait_bar(barA, (uint32_t)(c & 1));
        const int nc = rows_of(c);
        if (nc < C) {  // tokens past the sequence end were never written: zero Q^ rows, V^T columns
            for (int f = tid; f < (C - nc) * 32; f += THREADS) {
                const int r = nc + (f >> 5), c4 = (f & 31) * 4;
                *reinterpret_cast<float4*>(Qs + tc::sw_off(C, r, c4)) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int f = tid; f < DV * (C - nc); f += THREADS) {
                const int row = f / (C - nc), t = nc + f % (C - nc);
                *reinterpret_cast<float*>(VTs + tc::sw_off(DV, row, t)) = 0.f;
            }
        }
        mma_round_begin();
        if (tid == 0) {
            if (ok) {
                tc::fence_after();
                tc::mma_tf32(tm + cU, TBs, C, VTs, DV, C, tc::idesc_tf32(C, DV), false);
                tc::mma_tf32(tm + cU, Ws, C, S0s, DV, D, tc::idesc_tf32(C, DV, true), true);
                tc::mma_tf32(tm + cO1, Qs, C, S0s, DV, D, tc::idesc_tf32(C, DV), false);
            }
            tc::commit(mbar);
        }
    };

    if (tid == 0 && n_chunks > 0) {
        issue_a(0);
        issue_b(0);
    }
    if (n_chunks > 0) issue_ra(0);
    for (int ci = 0; ci < n_chunks; ++ci) {
        const int64_t t0 = start + (int64_t)ci * C;
        const int n = rows_of(ci);
        const uint32_t par = (uint32_t)(ci & 1);
        wait_mma();                                          // Ra of this chunk
        if (tid == 0 && ci + 1 < n_chunks) issue_a(ci + 1);  // Q^, W, T diag(b), V^T are free
        wait_bar(barB, par);
        if (n < C) {  // tail columns (t >= n) of K^T
            for (int f = tid; f < D * (C - n); f += THREADS) {
                const int row = f / (C - n), t = n + f % (C - n);
                *reinterpret_cast<float*>(KTs + tc::sw_off(D, row, t)) = 0.f;
            }
        }
        // ---- U -> U^T and (diag(e^(gC - g)) U)^T tiles; S^T *= e^gC in TMEM -----------------
        float egt = 0.f;  // e^gamma of this thread's output row
        {
            float u16[16];
            tc::ld16(tc::taddr(tm, 32 * q4, cU + hf * 16), u16);
            if (rowok) {
                const float er = Gs[C + trow];
                egt = Gs[trow];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    tc::st_elem(UTs, DV, hf * 16 + c, trow, u16[c]);
                    tc::st_elem(UPs, DV, hf * 16 + c, trow, u16[c] * er);
                }
            }
            float s16[16];
            tc::ld16(tc::taddr(tm, 32 * q4, cS + hf * 16), s16);
            const float egC = Gs[C - 1];
#pragma unroll
            for (int c = 0; c < 16; ++c) s16[c] *= egC;
            tc::st16(tc::taddr(tm, 32 * q4, cS + hf * 16), s16);
        }
        // ---- Rb: O2 = P U, S^T += K^T U' ---------------------------------------------------
        mma_round_begin();
        if (tid == 0) {
            if (ok) {
                tc::fence_after();
                tc::mma_tf32(tm + cO2, Ps, C, UTs, DV, C, tc::idesc_tf32(C, DV), false);
                tc::mma_tf32(tm + cS, KTs, D, UPs, DV, C, tc::idesc_tf32(D, DV), true);
            }
            tc::commit(mbar);
        }
        float zpre[16];  // z of this thread's output row (loaded while Rb runs)
        if (outnorm && rowok && trow < n) {
            const uint4* zp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(J.z) +
                                                             (size_t)(t0 + trow) * Hv * D + (size_t)j * D +
                                                             s_idx * DV + hf * 16);
            const uint4 z0 = zp[0], z1 = zp[1];
            const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&z0);
            const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&z1);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 a = __bfloat1622float2(h0[c]), b = __bfloat1622float2(h1[c]);
                zpre[2 * c] = a.x; zpre[2 * c + 1] = a.y; zpre[8 + 2 * c] = b.x; zpre[8 + 2 * c + 1] = b.y;
            }
        }
        wait_mma();
        if (tid == 0 && ci + 1 < n_chunks) issue_b(ci + 1);  // K^T, P, gates are read
        // ---- O = diag(e^g) O1 + O2; S^T -> S operand tile for the next chunk ----------------
        float o16[16];
        {
            float a16[16];
            tc::ld16x2(tc::taddr(tm, 32 * q4, cO1 + hf * 16), a16, tc::taddr(tm, 32 * q4, cO2 + hf * 16), o16);
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                o16[c] = fmaf(egt, a16[c], o16[c]);
                part = fmaf(o16[c], o16[c], part);
            }
            if (rowok) ored[hf * C + trow] = part;
            float s16[16];
            tc::ld16(tc::taddr(tm, 32 * q4, cS + hf * 16), s16);
#pragma unroll
            for (int c = 0; c < 16; ++c) tc::st_elem(S0s, DV, hf * 16 + c, dS, s16[c]);
        }
        __syncthreads();
        float* ssq_cur = ssq + (ci & 1) * C;
        if (tid < C) ssq_cur[tid] = ored[tid] + ored[C + tid];
        cluster_arrive_release();
        if (ci + 1 < n_chunks) issue_ra(ci + 1);  // runs while this chunk's output is normalised
        cluster_wait_acquire();
        if (rowok && trow < n) {
            const size_t tok = (size_t)(t0 + trow);
            float rstd = 1.f;
            if (outnorm) {
                float tot = 0.f;
                for (int s2 = 0; s2 < NS; ++s2) tot += *cluster.map_shared_rank(&ssq_cur[trow], s2);
                rstd = rsqrtf(tot / (float)D + g.norm_eps);
            }
            float yv[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) yv[c] = outnorm ? o16[c] * rstd * nwsl[hf * 16 + c] * siluf_(zpre[c]) : o16[c];
            uint4 pk[2];
            __nv_bfloat162* hp = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int c = 0; c < 8; ++c) hp[c] = __floats2bfloat162_rn(yv[2 * c], yv[2 * c + 1]);
            uint4* yp = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(J.y) + tok * (size_t)Hv * D +
                                                 (size_t)j * D + s_idx * DV + hf * 16);
            yp[0] = pk[0];
            yp[1] = pk[1];
        }
    }
    // ---- final state ------------------------------------------------------------------------
    {
        float s16[16];
        tc::ld16(tc::taddr(tm, 32 * q4, cS + hf * 16), s16);
        if (Sout) {
#pragma unroll
            for (int c = 0; c < 16; ++c) Sout[(size_t)(s_idx * DV + hf * 16 + c) * D + dS] = s16[c];
        }
    }
    if (!ok && tid == 0) report_device_status(kDevWaitTimeout);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tm, TMEM_COLS);
    cluster.sync();  // peers may still read this CTA's partial sums
}

cudaError_t launch_chunk_tc(const PrefillArgs& A, int64_t n_slots, cudaStream_t st) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_chunk_prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             tcp::PR_SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_chunk_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, tcp::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    if (n_slots > 0) {
        const int64_t ny = n_slots < 32768 ? n_slots : 32768;
        const dim3 grid((unsigned)A.g.Hv, (unsigned)ny, (unsigned)((n_slots + ny - 1) / ny));
        k_chunk_prep<<<grid, tcp::THREADS, tcp::PR_SMEM_ALLOC, st>>>(A);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tcp::NS, A.g.Hv, A.J.n_seq);
    cfg.blockDim = dim3(tcp::THREADS);
    cfg.dynamicSmemBytes = tcp::SMEM_ALLOC;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = tcp::NS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_chunk_tc, A);
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
    if (J.n_tokens > 0) {
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
