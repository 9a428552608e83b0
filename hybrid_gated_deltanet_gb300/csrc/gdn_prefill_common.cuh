// gdn_prefill_common.cuh -- device helpers shared by the two chunked-prefill
// paths (gdn_prefill.cu: any geometry, warp-level MMA; gdn_chunk16.cu: d = 128,
// chunk 64, bf16 activations, tcgen05 with fp16 operands).
//
// Sequences are packed back to back by cu_seqlens (none: one sequence of
// n_tokens).  Chunks restart at each sequence start; the tile workspaces give
// sequence s's chunk c the "chunk slot" floor(start_s / 64) + s + c, so two
// sequences never share a slot.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

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

// chunk of slot cs: its sequence, first token t0 and row count n; false for a
// slot between two sequences' chunks
__device__ __forceinline__ bool slot_chunk(const PrefillJob& J, int64_t cs, int& sq, int64_t& start, int64_t& end,
                                           int64_t& t0, int& n) {
    sq = slot_seq(J, cs);
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

// conv state a sequence starts from (NULL: zeros); slot_ok = 0 when its pool
// slot is out of range (the sequence then reads and writes no pool entry)
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

// ---- conv + SiLU of bf16 rows held in registers ----------------------------
// conv window of one thread: rows tau0-3 .. tau0+NT-1 of its 8 channels
// (taps before the sequence start from its conv state), packed bf16
template <int NT>
__device__ __forceinline__ void load_window(const PrefillJob& J, int Cch, int K, int ch, int64_t tau0, int64_t start,
                                            int64_t end, const void* cin, uint4 rows[NT + 3]) {
    // every load is issued (rows outside both sources read row 0 of x and are
    // zeroed after), so that the NT + 3 loads are in flight together
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(J.x);
    const __nv_bfloat16* cs = static_cast<const __nv_bfloat16*>(cin);
    bool live[NT + 3];
#pragma unroll
    for (int r = 0; r < NT + 3; ++r) {
        const int64_t tau = tau0 - 3 + r;
        const bool in_x = tau >= start && tau < end;
        const bool in_c = !in_x && tau < start && cs && tau - start >= -(K - 1);
        live[r] = in_x || in_c;
        const __nv_bfloat16* p = in_x ? x + (size_t)tau * Cch + ch
                                      : (in_c ? cs + (size_t)((K - 1) + (tau - start)) * Cch + ch : x + ch);
        rows[r] = __ldg(reinterpret_cast<const uint4*>(p));
    }
#pragma unroll
    for (int r = 0; r < NT + 3; ++r)
        if (!live[r]) rows[r] = make_uint4(0, 0, 0, 0);
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

// SiLU through one hardware tanh: x sigma(x) = h + h tanh(h), h = x / 2.  One
// special-function operation instead of two; the error (tanh to about 2^-11
// relative, i.e. at most about 2.5e-4 of |x|) is below the fp16 rounding that the
// tensor-core operands built from it receive.
__device__ __forceinline__ float silu_tanh(float x) {
    const float h = 0.5f * x;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// conv + SiLU of the NT tokens of one thread's window (rows i .. i+3 are the
// taps of token i), through a sliding window of 4 unpacked rows; emit(i, u)
// receives token i's 8 channels.  w[r][c]: weight of window row r for
// channel c (rows before the first live tap are zero weights when d_conv < 4).
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
            for (int c = 0; c < 8; ++c) u[c] = silu_tanh(u[c]);
        }
        emit(i, u);
    }
}

// conv weights and bias of 8 consecutive channels (ch a multiple of 8) as
// window-row weights: w[r][c] multiplies row tau-3+r; tap m of the K taps
// multiplies row tau-(K-1)+m, i.e. window row r = 4-K+m.  The 8 K weights are
// contiguous ([C_ch][K] bf16, 16-byte aligned): K vector loads.
__device__ __forceinline__ void conv_weights8(const LayerParams& p, int K, bool raw, int ch, float w[4][8],
                                              float bias[8]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        bias[c] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) w[r][c] = 0.f;
    }
    if (raw) return;
    if (p.conv_b) unpack8(*reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.conv_b) + ch), bias);
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.conv_w) + (size_t)ch * K);
    // element e = c KK + m of the 8 KK values is channel c's tap m (register indices
    // resolved at compile time for each d_conv)
    auto unpack_taps = [&](auto kk) {
        constexpr int KK = decltype(kk)::value;
        float f[8 * KK];
#pragma unroll
        for (int v = 0; v < KK; ++v) unpack8(src[v], f + 8 * v);
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int m = 0; m < KK; ++m) w[4 - KK + m][c] = f[c * KK + m];
    };
    if (K == 4) unpack_taps(std::integral_constant<int, 4>{});
    else if (K == 3) unpack_taps(std::integral_constant<int, 3>{});
    else unpack_taps(std::integral_constant<int, 2>{});
}

// ---- the UT transform: T = (I + A)^-1 of a strictly lower 64 x 64 A ----------
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma16x8x8_tf32(float c[4], const uint32_t a[4], const uint32_t b[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

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
            ah[e] = tf32_bits(fa[e]);
            al[e] = tf32_bits(fa[e] - __uint_as_float(ah[e]));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            bh[e] = tf32_bits(fb[e]);
            bl[e] = tf32_bits(fb[e] - __uint_as_float(bh[e]));
        }
        mma16x8x8_tf32(c, al, bh);
        mma16x8x8_tf32(c, ah, bl);
        mma16x8x8_tf32(c, ah, bh);
    }
}

constexpr int kUtLd = 68;  // row stride (floats) of the 64 x 64 matrices of ut_inverse64

// Tm = (I + Am)^-1 for a strictly lower 64 x 64 Am (row stride kUtLd), by the
// whole CTA of nthreads (a multiple of 32, at least 64) threads; ends with a
// CTA barrier.  16x16 diagonal blocks by register-resident right-looking
// substitution: a lane owns column j of a block and column j of A; once x_k
// is final, every later row takes -A_ik x_k (A_ik from lane k by shuffle), so
// the dependent chain is 16 FMAs long.  The off-diagonal blocks follow by
// distance, X_ab = -X_aa sum_{c=b}^{a-1} A_ac X_cb, on warp-level MMAs in the
// fp32-accurate 3xTF32 split.
__device__ __forceinline__ void ut_inverse64(const float* Am, float* Tm, int tid, int nthreads) {
    constexpr int LD = kUtLd;
    const int lane = tid & 31, warp = tid >> 5, nwarp = nthreads >> 5;
    if (warp < 2) {
        const int b0 = (warp * 2 + (lane >> 4)) * 16, jc = lane & 15, lb = lane & 16;
        float acol[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acol[i] = Am[(b0 + i) * LD + b0 + jc];
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == jc) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < 15; ++k) {
#pragma unroll
            for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-__shfl_sync(0xffffffffu, acol[i], lb + k), x[k], x[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tm[(b0 + i) * LD + b0 + jc] = x[i];
    }
    for (int f = tid; f < 64 * 64; f += nthreads) {
        const int t = f >> 6, c = f & 63;
        if ((c >> 4) > (t >> 4)) Tm[t * LD + c] = 0.f;
    }
    __syncthreads();
    for (int dd = 1; dd < 4; ++dd) {
        const int ntile = (4 - dd) * 2;
        for (int tl = warp; tl < ntile; tl += nwarp) {  // Y = A_a[b..a) X_[b..a)b
            const int bb = tl >> 1, nt = tl & 1;
            const int a0 = (bb + dd) * 16, c0b = bb * 16;
            float cc[4];
            warp_tile16x8_precise(Am + a0 * LD + c0b, LD, Tm + c0b * LD + c0b + 8 * nt, LD, a0 - c0b, lane, cc);
            const int gq = lane >> 2, t4 = lane & 3;
            float* y0 = Tm + a0 * LD + c0b + 8 * nt;
            y0[gq * LD + 2 * t4] = cc[0];
            y0[gq * LD + 2 * t4 + 1] = cc[1];
            y0[(gq + 8) * LD + 2 * t4] = cc[2];
            y0[(gq + 8) * LD + 2 * t4 + 1] = cc[3];
        }
        __syncthreads();
        for (int tl = warp; tl < ntile; tl += nwarp) {  // X_ab = -X_aa Y
            const int bb = tl >> 1, nt = tl & 1;
            const int a0 = (bb + dd) * 16, c0b = bb * 16;
            float cc[4];
            warp_tile16x8_precise(Tm + a0 * LD + a0, LD, Tm + a0 * LD + c0b + 8 * nt, LD, 16, lane, cc);
            const int gq = lane >> 2, t4 = lane & 3;
            float* x0 = Tm + a0 * LD + c0b + 8 * nt;
            x0[gq * LD + 2 * t4] = -cc[0];
            x0[gq * LD + 2 * t4 + 1] = -cc[1];
            x0[(gq + 8) * LD + 2 * t4] = -cc[2];
            x0[(gq + 8) * LD + 2 * t4 + 1] = -cc[3];
        }
        __syncthreads();
    }
}

}  // namespace gdn
