// gdn_prefill.cu -- chunkwise (WY / UT-transform) prefill, single sequence and
// packed variable-length: the path for every geometry, and the dispatch.
//
// d_k = d_v = 128 with chunk 64 and bf16 activations runs the tcgen05 path of
// gdn_chunk16.cu.  Every other geometry (d in {32, 64, 128}, chunks 16/32/64,
// fp32 or bf16 activations) runs three launches on the caller's stream:
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
// prefill kernel with deterministic reduction).  Prefix snapshots of the conv
// state (k_conv_ckpt) and the final conv states serve both paths.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstdlib>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_prefill_common.cuh"

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


struct PrefillArgs {
    Geom g;
    LayerParams p;
    PrefillJob J;
    float* qk;    // [N][2*Hk][D]  q^ (scaled) heads then k^ heads
    float* v;     // [N][Hv][D]
    float* gl;    // [N][Hv]       g = log(alpha)
    float* beta;  // [N][Hv]
    int NS;
};

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

int prefill_slices(int D) {
    if (const char* e = std::getenv("GDN_PREFILL_SLICES")) {
        const int v = std::atoi(e);
        if ((v == 1 || v == 2 || v == 4 || v == 8) && D / v >= 16) return v;
    }
    return D >= 128 ? 4 : (D >= 64 ? 2 : 1);
}

template <typename TA>
cudaError_t launch_conv_tail_t(const PrefillArgs& A, cudaStream_t st) {
    const Geom& g = A.g;
    const PrefillJob& J = A.J;
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
    return cudaSuccess;
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
    if (J.n_tokens > 0) {
        constexpr int VEC = 16 / (int)sizeof(TA);
        const dim3 blocks((unsigned)((J.n_tokens + kProTok - 1) / kProTok),
                          (unsigned)((g.C_ch / VEC + kProThreads - 1) / kProThreads));
        k_prologue<D, TA><<<blocks, kProThreads, 0, st>>>(A);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const cudaError_t e = launch_conv_tail_t<TA>(A, st);
        if (e != cudaSuccess) return e;
    }
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
    if (chunk16_applies(g)) return chunk16_workspace_bytes(g, n_tokens, n_seq);
    return ws_layout(g, n_tokens).total;
}

cudaError_t launch_prefill(const Geom& g, const LayerParams& p, const PrefillJob& J, cudaStream_t st) {
    if (J.n_seq == 0) return cudaSuccess;
    if (chunk16_applies(g)) {
        // the state chain, then the conv states: both kernels of the chain path read
        // the conv states the sequences start from
        cudaError_t e = chunk16_launch(g, p, J, st);
        if (e != cudaSuccess) return e;
        PrefillArgs A = {};
        A.g = g;
        A.p = p;
        A.J = J;
        return launch_conv_tail_t<__nv_bfloat16>(A, st);
    }
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
