// gdn_decode.cu -- decode step and verify rows: one pass over each slot's
// fp32 state, everything else of the layer fused around it.
//
// Work decomposition (sm_103a):
//   grid    = (G * NS, H_k, B), one thread-block cluster per (slot, k-head h)
//   cluster = the G v-heads of k-head h x NS row slices of each v-head's state
//   CTA     = (slot, v-head j, row slice s): D/NS state rows, 8 rows per warp,
//             each row read as D/4 lanes x one 128-bit load (fully coalesced)
// Rows of S evolve independently given (q^, k^, v_i, alpha, beta), so a CTA
// keeps its rows in registers for all r rows of a verify and touches HBM
// exactly once for the read and once per written state.  Every CTA recomputes
// the conv + SiLU + L2 norm of its k-head's q/k (2*D channels, a few KB from
// L2) instead of exchanging them.  The output RMSNorm needs the sum of o^2
// over all D rows of a v-head: the NS slices exchange partial sums through
// distributed shared memory after a cluster barrier.  The same barrier orders
// every conv-state read of the cluster before the conv-state writes, which is
// what makes the in-place conv-state update race-free within one launch (all
// readers of a k-head group's conv channels live in one cluster).
//
// State update per row i (S_i the row, k^, q^ the normalised key/query):
//   dk = S_i . k^,  dq = S_i . q^          (old state)
//   e  = v_i - alpha dk
//   S_i <- alpha S_i + beta e k^
//   o_i = alpha dq + beta e (k^ . q^)       (= S_i_new . q^)
// which is S_t = alpha S (I - beta k k^T) + beta v k^T, o = S_t q of the
// gated delta rule ("Hybrid transformers under load ...", braintools.ru,
// section 3), in a single read and a single write of the state.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstdlib>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tma.cuh"

namespace cg = cooperative_groups;

namespace gdn {
namespace {

struct RowsArgs {
    Geom g;
    LayerParams p;
    RowsJob job;
    int NS;
};

// barrier over the 256 threads of one consumer group only (named barrier 1 + group),
// AND of a predicate
__device__ __forceinline__ bool __syncthreads_and_consumers(bool pred, int group) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n bar.red.and.pred q, %2, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(1 + group)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Shared-memory layout of one k_rows CTA (byte offsets, 16-byte aligned runs).
struct RowsSmem {
    int bar, S, x, c, w, z, nw, ab, qs, ks, vs, red, tsc, obuf, ssp, total;
};

__host__ __device__ inline RowsSmem rows_smem(int D, int RPC, int r, int K, int E) {
    auto up = [](int v) { return (v + 15) & ~15; };
    const int NCH = 2 * D + RPC;
    RowsSmem s;
    int o = 0;
    s.bar = o; o += 16;                   // two mbarriers
    s.S = o; o += RPC * D * 4;            // the CTA's state rows, fp32
    s.x = o; o = up(o + r * NCH * E);     // x of the CTA's channels, per row
    s.c = o; o = up(o + (K - 1) * NCH * E);  // conv state of those channels
    s.w = o; o = up(o + NCH * K * E);     // conv weights of those channels
    s.z = o; o = up(o + r * RPC * E);     // z of the CTA's rows
    s.nw = o; o = up(o + RPC * E);        // norm weight of the CTA's rows
    s.ab = o; o = up(o + 2 * r * 4);      // a, b per row
    s.qs = o; o += r * D * 4;             // q of every token (before the norm)
    s.ks = o; o += r * D * 4;             // k of every token
    s.vs = o; o = up(o + r * RPC * 4);    // v of every token (the CTA's rows)
    s.red = o; o += r * 32 * 4;           // per-warp partial sums, per token
    s.tsc = o; o += r * 8 * 4;            // per-token alpha, beta, scales, q^.k^
    s.obuf = o; o = up(o + r * RPC * 4);
    s.ssp = o; o = up(o + r * 4);
    s.total = o;
    return s;
}

constexpr int kRowsThreads = 256;

template <int D, typename TA>
__global__ void __launch_bounds__(kRowsThreads) k_rows(const __grid_constant__ RowsArgs A) {
    constexpr int LPR = D / 4;     // lanes per state row (4 floats per lane)
    constexpr int RPI = 32 / LPR;  // rows per warp-wide 128-bit access
    constexpr int E = sizeof(TA);
    using L = Act<TA>;
    cg::cluster_group cluster = cg::this_cluster();
    const Geom& g = A.g;
    const RowsJob& J = A.job;
    const int NS = A.NS, G = g.G, Hk = g.Hk, Hv = g.Hv, K = g.K, C = g.C_ch, Km1 = g.K - 1;
    const int CS = G * NS;
    const int gi = blockIdx.x / NS, s = blockIdx.x % NS;
    const int h = blockIdx.y, j = h * G + gi, bb = blockIdx.z;
    const int RPC = D / NS, NCH = 2 * D + RPC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int nthr = kRowsThreads, nwarp = kRowsThreads / 32;
    const int r = J.r;
    const int crank = (int)cluster.block_rank();
    const bool raw = g.flags & kFlagRawQKV;
    const int mode = J.mode;
    const bool outnorm = !(g.flags & kFlagNoOutNorm) && mode != 2;  // (a commit writes no y)
    const bool direct = g.flags & kFlagGatesDirect;
    // One slice per v-head: the output norm is local and the only cluster
    // barrier orders the conv-state reads of the k-head group before its
    // writes, so it can arrive early and wait late.  With NS > 1 the slices
    // also exchange partial sums of o^2 through distributed shared memory.
    const bool whole_head = NS == 1;

    extern __shared__ __align__(128) unsigned char smem[];
    const RowsSmem lay = rows_smem(D, RPC, r, K, E);
    uint64_t* bar_in = reinterpret_cast<uint64_t*>(smem + lay.bar);  // small inputs
    uint64_t* bar_s = bar_in + 1;                                     // the state slice
    float* Sb = reinterpret_cast<float*>(smem + lay.S);
    TA* xs = reinterpret_cast<TA*>(smem + lay.x);
    TA* cs = reinterpret_cast<TA*>(smem + lay.c);
    TA* wsm = reinterpret_cast<TA*>(smem + lay.w);
    TA* zs = reinterpret_cast<TA*>(smem + lay.z);
    TA* nw = reinterpret_cast<TA*>(smem + lay.nw);
    float* ab = reinterpret_cast<float*>(smem + lay.ab);
    float* qs = reinterpret_cast<float*>(smem + lay.qs);
    float* ks = reinterpret_cast<float*>(smem + lay.ks);
    float* vs = reinterpret_cast<float*>(smem + lay.vs);
    float* red = reinterpret_cast<float*>(smem + lay.red);
    float* tsc = reinterpret_cast<float*>(smem + lay.tsc);
    float* obuf = reinterpret_cast<float*>(smem + lay.obuf);
    float* ssp = reinterpret_cast<float*>(smem + lay.ssp);

    // programmatic dependent launch: this grid may be resident before the previous
    // kernel of the stream ends; every read below waits for it (and its memory)
    griddep_wait();
    griddep_launch_dependents();
    const int slot = J.slot_idx[bb];
    if (slot < 0 || slot >= J.n_slots) return;  // the whole cluster shares bb
    // rows to run: all r, or for a commit by recompute the accepted ones
    int nr = r;
    if (mode == 2) {
        const int acc = J.accepted[bb];
        nr = acc < 0 ? 0 : (acc > r ? r : acc);
        if (nr == 0) return;  // nothing accepted: the slot keeps its state (whole cluster)
    }

    // the CTA's channels: q and k of k-head h, the slice of v of v-head j
    const int ch_q = h * D, ch_k = Hk * D + h * D, ch_v = 2 * Hk * D + j * D + s * RPC;
    float* Sg = J.state_pool + (((size_t)slot * Hv + j) * D + (size_t)s * RPC) * D;

    // ---- stage everything with bulk async copies (one thread issues) ----------
    if (tid == 0) {
        mbar_init(bar_in, 1);
        mbar_init(bar_s, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_s, RPC * D * 4);
        bulk_g2s(Sb, Sg, RPC * D * 4, bar_s);
        const bool conv_w = !raw && A.p.conv_w;
        const uint32_t bytes = (r + Km1) * NCH * E + (conv_w ? NCH * K * E : 0) + (outnorm ? (r + 1) * RPC * E : 0);
        mbar_arrive_expect_tx(bar_in, bytes);
        const char* cg_ = static_cast<const char*>(J.conv_pool);
        for (int m = 0; m < Km1; ++m) {
            const char* row = cg_ + ((size_t)slot * Km1 + m) * C * E;
            bulk_g2s(cs + m * NCH, row + (size_t)ch_q * E, D * E, bar_in);
            bulk_g2s(cs + m * NCH + D, row + (size_t)ch_k * E, D * E, bar_in);
            bulk_g2s(cs + m * NCH + 2 * D, row + (size_t)ch_v * E, RPC * E, bar_in);
        }
        const char* xg = static_cast<const char*>(J.x);
        for (int t = 0; t < r; ++t) {
            const char* row = xg + ((size_t)bb * r + t) * C * E;
            bulk_g2s(xs + t * NCH, row + (size_t)ch_q * E, D * E, bar_in);
            bulk_g2s(xs + t * NCH + D, row + (size_t)ch_k * E, D * E, bar_in);
            bulk_g2s(xs + t * NCH + 2 * D, row + (size_t)ch_v * E, RPC * E, bar_in);
        }
        if (conv_w) {
            const char* w = static_cast<const char*>(A.p.conv_w);
            bulk_g2s(wsm, w + (size_t)ch_q * K * E, D * K * E, bar_in);
            bulk_g2s(wsm + D * K, w + (size_t)ch_k * K * E, D * K * E, bar_in);
            bulk_g2s(wsm + 2 * D * K, w + (size_t)ch_v * K * E, RPC * K * E, bar_in);
        }
        if (outnorm) {
            const char* zg = static_cast<const char*>(J.z);
            for (int t = 0; t < r; ++t)
                bulk_g2s(zs + t * RPC, zg + (((size_t)bb * r + t) * Hv * D + (size_t)j * D + s * RPC) * E, RPC * E,
                         bar_in);
            bulk_g2s(nw, static_cast<const char*>(A.p.norm_w) + (size_t)s * RPC * E, RPC * E, bar_in);
        }
    }
    for (int i = tid; i < 2 * r; i += nthr) {
        const size_t rowx = (size_t)bb * r + (i >> 1);
        ab[i] = L::ld((i & 1) ? J.b : J.a, rowx * Hv + j);
    }
    const float A_log_j = direct ? 0.0f : A.p.A_log[j];
    const float dt_j = (!direct && A.p.dt_bias) ? A.p.dt_bias[j] : 0.0f;
    __syncthreads();  // barriers initialised, a/b staged
    // one warp polls the barrier, the others sleep in bar.sync
    bool ok = true;
    if (warp == 0) {
        ok = mbar_wait(bar_in, 0);
        if (!ok) mbar_wait(bar_in, 0);  // bounded again: let the copies in flight land
    }
    ok = __syncthreads_and(ok);
    if (whole_head) cluster_arrive_release();  // this CTA's conv-state reads are done (in shared memory)

    // ---- prologue of every row (conv, norms, gates) from shared memory --------
    // A state row's update over the r tokens involves no other state row, so
    // the q, k, v and gates of all r tokens are prepared first (in parallel
    // over tokens and channels) and each warp then carries its state rows
    // through all tokens without a CTA barrier between tokens.
    auto conv = [&](int lc, int t) -> float {
        if (raw) return L::ld(xs, (size_t)t * NCH + lc);
        const int ch = lc < D ? ch_q + lc : (lc < 2 * D ? ch_k + lc - D : ch_v + lc - 2 * D);
        float c = A.p.conv_b ? L::ld(A.p.conv_b, ch) : 0.0f;
        for (int m = 0; m < K; ++m) {
            const int tau = t - Km1 + m;
            const float xv = tau >= 0 ? L::ld(xs, (size_t)tau * NCH + lc) : L::ld(cs, (size_t)(Km1 + tau) * NCH + lc);
            c = fmaf(L::ld(wsm, (size_t)lc * K + m), xv, c);
        }
        return siluf_(c);
    };
    const int col4 = lane % LPR, rsub = lane / LPR;
    if (ok) {
        for (int t = 0; t < nr; ++t) {
            float sq = 0.f, sk = 0.f, sqk = 0.f;
            // work item w < D: channel w of q and k; D <= w < D + RPC: channel w - D of v
            for (int w = tid; w < D + RPC; w += nthr) {
                if (w < D) {
                    const float qv = conv(w, t), kv = conv(D + w, t);
                    qs[t * D + w] = qv;
                    ks[t * D + w] = kv;
                    sq = fmaf(qv, qv, sq);
                    sk = fmaf(kv, kv, sk);
                    sqk = fmaf(qv, kv, sqk);
                } else {
                    vs[t * RPC + (w - D)] = conv(2 * D + (w - D), t);
                }
            }
            sq = warp_sum(sq);
            sk = warp_sum(sk);
            sqk = warp_sum(sqk);
            if (lane == 0) {
                red[(t * nwarp + warp) * 4 + 0] = sq;
                red[(t * nwarp + warp) * 4 + 1] = sk;
                red[(t * nwarp + warp) * 4 + 2] = sqk;
            }
        }
    }
    {
        bool s_ok = true;
        if (warp == 0) {
            s_ok = mbar_wait(bar_s, 0);
            if (!s_ok) mbar_wait(bar_s, 0);  // bounded again: let the state copy land
        }
        ok = __syncthreads_and(ok && s_ok);  // one verdict for the whole CTA; red complete
        if (!ok && tid == 0) report_device_status(kDevWaitTimeout);
    }
    // per-token scalars: alpha, beta, the q and k scales, q^.k^
    for (int t = tid; t < nr; t += nthr) {
        float sq = 0.f, sk = 0.f, sqk = 0.f;
        for (int w = 0; w < nwarp; ++w) {
            sq += red[(t * nwarp + w) * 4 + 0];
            sk += red[(t * nwarp + w) * 4 + 1];
            sqk += red[(t * nwarp + w) * 4 + 2];
        }
        float rq, rk;
        if (g.flags & kFlagNoL2) {
            rq = g.q_scale;
            rk = 1.0f;
        } else {
            rq = g.q_scale * rsqrtf(sq + g.l2_eps);
            rk = rsqrtf(sk + g.l2_eps);
        }
        float gl, beta;
        gates(ab[2 * t], ab[2 * t + 1], A_log_j, dt_j, direct, gl, beta);
        tsc[t * 8 + 0] = expf(gl);
        tsc[t * 8 + 1] = beta;
        tsc[t * 8 + 2] = rq;
        tsc[t * 8 + 3] = rk;
        tsc[t * 8 + 4] = sqk * rq * rk;
    }
    __syncthreads();
    if (ok) {
        auto snap_rows = [&](int t) -> float* {  // verify snapshot of token t, or nullptr
            const int dst = (mode == 0 && J.snap_idx) ? J.snap_idx[(size_t)bb * r + t] : -1;
            return (dst >= 0 && dst < J.n_slots) ? J.state_pool + (((size_t)dst * Hv + j) * D + (size_t)s * RPC) * D
                                                 : nullptr;
        };
        if constexpr (D == 128) {
            // 8 rows per warp group; the 16 partial dot products (S.k, S.q of the
            // 8 rows) are reduced across the 32 lanes with a transposing butterfly
            // (16 shuffles instead of 80): lane l ends with the sum of value l >> 1.
            for (int rb = warp * 8; rb < RPC; rb += nwarp * 8) {
                float4 sv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) sv[i] = *reinterpret_cast<const float4*>(Sb + (rb + i) * D + lane * 4);
                for (int t = 0; t < nr; ++t) {
                    const float alpha = tsc[t * 8 + 0], beta = tsc[t * 8 + 1], rq = tsc[t * 8 + 2],
                                rk = tsc[t * 8 + 3], kq = tsc[t * 8 + 4];
                    float kr[4], qr[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kr[e] = ks[t * D + col4 * 4 + e] * rk;
                        qr[e] = qs[t * D + col4 * 4 + e] * rq;
                    }
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float dk = sv[i].x * kr[0];
                        dk = fmaf(sv[i].y, kr[1], dk);
                        dk = fmaf(sv[i].z, kr[2], dk);
                        v[i] = fmaf(sv[i].w, kr[3], dk);
                        float dq = sv[i].x * qr[0];
                        dq = fmaf(sv[i].y, qr[1], dq);
                        dq = fmaf(sv[i].z, qr[2], dq);
                        v[8 + i] = fmaf(sv[i].w, qr[3], dq);
                    }
#pragma unroll
                    for (int n = 8, off = 16; n >= 1; n >>= 1, off >>= 1) {
                        const bool upper = lane & off;
#pragma unroll
                        for (int i = 0; i < n; ++i) {
                            const float send = upper ? v[i] : v[i + n];
                            const float keep = upper ? v[i + n] : v[i];
                            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                        }
                    }
                    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
                    const int idx = lane >> 1;  // 0..7: S.k of row rb+idx; 8..15: S.q of row rb+idx-8
                    const float e_mine = idx < 8 ? vs[t * RPC + rb + idx] - alpha * v[0] : 0.f;
                    float ei[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) ei[i] = __shfl_sync(0xffffffffu, e_mine, 2 * i);
                    const float e_for_q = __shfl_sync(0xffffffffu, e_mine, ((idx - 8) & 7) * 2);
                    if (idx >= 8 && !(lane & 1)) obuf[t * RPC + rb + idx - 8] = fmaf(alpha, v[0], beta * e_for_q * kq);
                    float* Sd = snap_rows(t);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float be = beta * ei[i];
                        sv[i].x = fmaf(alpha, sv[i].x, be * kr[0]);
                        sv[i].y = fmaf(alpha, sv[i].y, be * kr[1]);
                        sv[i].z = fmaf(alpha, sv[i].z, be * kr[2]);
                        sv[i].w = fmaf(alpha, sv[i].w, be * kr[3]);
                        if (Sd) *reinterpret_cast<float4*>(Sd + (rb + i) * D + lane * 4) = sv[i];  // verify snapshot
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) *reinterpret_cast<float4*>(Sb + (rb + i) * D + lane * 4) = sv[i];
            }
        } else {
#pragma unroll 4
            for (int rb = warp * RPI; rb < RPC; rb += nwarp * RPI) {
                const int rl = rb + rsub;  // row within the slice
                float4* sp = reinterpret_cast<float4*>(Sb + rl * D + col4 * 4);
                float4 sv = *sp;
                for (int t = 0; t < nr; ++t) {
                    const float alpha = tsc[t * 8 + 0], beta = tsc[t * 8 + 1], rq = tsc[t * 8 + 2],
                                rk = tsc[t * 8 + 3], kq = tsc[t * 8 + 4];
                    float kr[4], qr[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kr[e] = ks[t * D + col4 * 4 + e] * rk;
                        qr[e] = qs[t * D + col4 * 4 + e] * rq;
                    }
                    float dk = sv.x * kr[0];
                    dk = fmaf(sv.y, kr[1], dk);
                    dk = fmaf(sv.z, kr[2], dk);
                    dk = fmaf(sv.w, kr[3], dk);
                    float dq = sv.x * qr[0];
                    dq = fmaf(sv.y, qr[1], dq);
                    dq = fmaf(sv.z, qr[2], dq);
                    dq = fmaf(sv.w, qr[3], dq);
#pragma unroll
                    for (int off = LPR / 2; off > 0; off >>= 1) {
                        dk += __shfl_xor_sync(0xffffffffu, dk, off);
                        dq += __shfl_xor_sync(0xffffffffu, dq, off);
                    }
                    const float e = vs[t * RPC + rl] - alpha * dk;
                    const float be = beta * e;
                    sv.x = fmaf(alpha, sv.x, be * kr[0]);
                    sv.y = fmaf(alpha, sv.y, be * kr[1]);
                    sv.z = fmaf(alpha, sv.z, be * kr[2]);
                    sv.w = fmaf(alpha, sv.w, be * kr[3]);
                    float* Sd = snap_rows(t);
                    if (Sd) *reinterpret_cast<float4*>(Sd + rl * D + col4 * 4) = sv;  // verify snapshot
                    if (col4 == 0) obuf[t * RPC + rl] = fmaf(alpha, dq, be * kq);
                }
                *sp = sv;
            }
        }
    }
    __syncthreads();  // obuf complete, the state rows back in shared memory

    // ---- state back (decode: in place, one bulk store) and the output ---------
    fence_proxy_async_smem();
    for (int t = warp; t < nr; t += nwarp) {
        float ss = 0.f;
        for (int rr = lane; rr < RPC; rr += 32) {
            const float o = obuf[t * RPC + rr];
            ss = fmaf(o, o, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) ssp[t] = ss;
    }
    __syncthreads();
    if (!whole_head) cluster_arrive_release();  // partial sums and conv-state reads are done
    if (tid == 0 && ok && !J.snap_idx && mode != 1) {  // decode, commit: the state in place
        bulk_s2g(Sg, Sb, RPC * D * 4);
        bulk_commit();
    }
    if (!whole_head) cluster_wait_acquire();

    if (ok && mode != 2) {
        for (int idx = tid; idx < r * RPC; idx += nthr) {
            const int t = idx / RPC, rr = idx % RPC;
            const size_t rowx = (size_t)bb * r + t;
            const int dv = s * RPC + rr;
            const float o = obuf[idx];
            float yv = o;
            if (outnorm) {
                float tot = ssp[t];
                if (!whole_head) {
                    tot = 0.f;
                    for (int s2 = 0; s2 < NS; ++s2) tot += *cluster.map_shared_rank(&ssp[t], gi * NS + s2);
                }
                yv = o * rsqrtf(tot / (float)D + g.norm_eps) * L::ld(nw, rr) * siluf_(L::ld(zs, idx));
            }
            L::st(J.y, rowx * (size_t)Hv * D + (size_t)j * D + dv, yv);
        }
    }
    if (whole_head) cluster_wait_acquire();  // every CTA of the group has read its conv state
    if (ok && mode != 1) {
        // conv state: the last K-1 raw inputs, copied bit for bit
        TA* cpool = static_cast<TA*>(J.conv_pool);
        auto roll = [&](int lc, int ch) {
            auto val = [&](int p) -> TA { return p < Km1 ? cs[p * NCH + lc] : xs[(p - Km1) * NCH + lc]; };
            if (!J.snap_idx) {
                for (int m = 0; m < Km1; ++m) cpool[((size_t)slot * Km1 + m) * C + ch] = val(nr + m);
            } else {
                for (int t = 0; t < r; ++t) {
                    const int dst = J.snap_idx[(size_t)bb * r + t];
                    if (dst < 0 || dst >= J.n_slots) continue;
                    for (int m = 0; m < Km1; ++m) cpool[((size_t)dst * Km1 + m) * C + ch] = val(t + 1 + m);
                }
            }
        };
        for (int c = crank + CS * tid; c < 2 * D; c += CS * nthr) roll(c, c < D ? ch_q + c : ch_k + c - D);
        for (int c = tid; c < RPC; c += nthr) roll(2 * D + c, ch_v + c);
    }
    if (!whole_head) {
        cluster_arrive_relaxed();  // peers are done reading this CTA's partial sums
        cluster_wait_acquire();
    }
    if (tid == 0) bulk_wait_read_all();  // the state store has read its shared-memory source
}

// ---- persistent, pipelined decode (d = 128, one token per slot) ---------------
// One CTA per SM walks a strided list of (slot, k-head) units, each the G
// (slot, v-head) items of that k-head.  Warp 16 is the producer: it reads an
// item's slot index and gates, issues the bulk copies of its 64 KB state tile
// and small inputs into one of 3 shared-memory stages (up to 3 items ahead),
// and once the consumers are done with an item writes its state back with one
// bulk store, and the rolled conv rows of its v channels (and, after the
// unit's last item, of the k-head's q and k channels) from the stage.  Only
// this CTA reads those conv rows, and it retires items in order, so every
// read of the old rows has landed before they are overwritten: no second
// launch and no wait between CTAs.  Two consumer groups of 8 warps (warps
// 0..7, 8..15) take the CTA's items in turn, so that one group's serial
// phases (conv + SiLU + L2 norm + gates from shared memory, the row update
// with the transposing butterfly, the gated RMSNorm and y, with a group
// barrier between them) overlap the other's.
namespace pd {
constexpr int D = 128, NCH = 3 * D, STAGES = 3, GROUPS = 2, CONSUMERS = 256;
constexpr int THREADS = GROUPS * CONSUMERS + 32;
constexpr int SCRATCH = 3 * D + 64 + D + 16;  // floats per consumer group: q, k, v, partial sums, o, sum of o^2
template <typename TA>
struct Stage {
    static constexpr int E = sizeof(TA);
    static constexpr int S = 0;                                // fp32 [128][128]
    static constexpr int X = S + D * D * 4;                    // act [NCH]
    static constexpr int CV = X + NCH * E;                     // act [3][NCH] (d_conv - 1 <= 3)
    static constexpr int W = CV + 3 * NCH * E;                 // act [NCH][4]
    static constexpr int Z = W + NCH * 4 * E;                  // act [D]
    static constexpr int NW = Z + D * E;                       // act [D]
    static constexpr int HDR = NW + D * E;                     // a, b, slot, flags
    static constexpr int BYTES = ((HDR + 16) + 127) & ~127;
};
template <typename TA>
constexpr int smem_bytes() {
    return STAGES * Stage<TA>::BYTES + 4 * STAGES * 8 /*mbarriers*/ + GROUPS * SCRATCH * 4 + 128;
}
}  // namespace pd

template <typename TA>
__global__ void __launch_bounds__(pd::THREADS, 1) k_decode_persist(const __grid_constant__ RowsArgs A) {
    using namespace pd;
    using L = Act<TA>;
    using St = Stage<TA>;
    constexpr int E = sizeof(TA);
    const Geom& g = A.g;
    const RowsJob& J = A.job;
    const int Hk = g.Hk, Hv = g.Hv, G = g.G, K = g.K, Km1 = g.K - 1, C = g.C_ch;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool raw = g.flags & kFlagRawQKV;
    const bool outnorm = !(g.flags & kFlagNoOutNorm);
    const bool direct = g.flags & kFlagGatesDirect;
    // Work units (sequence b, k-head h), strided over the CTAs; a unit is the G items
    // (b, v-head h G + g), taken in turn.  A CTA owns every reader of the unit's q and k
    // conv rows, so it rolls them itself once the unit's last item is done.
    const int n_units = J.B * Hk;
    const int my_units = (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int n_local = my_units * G;  // this CTA's items, k = 0 .. n_local - 1
    auto item_of = [&](int kk, int& bb, int& jj) {
        const int unit = (int)blockIdx.x + (kk / G) * (int)gridDim.x;
        bb = unit / Hk;
        jj = (unit % Hk) * G + kk % G;
    };

    // programmatic dependent launch: this grid may be resident before the previous
    // kernel of the stream ends; every read below waits for it (and its memory)
    griddep_wait();
    griddep_launch_dependents();

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * St::BYTES);
    uint64_t* fullS = full + STAGES;     // the state tile of the stage
    uint64_t* done = fullS + STAGES;     // consumers finished the stage's item
    const int group = warp / (CONSUMERS / 32) < GROUPS ? warp / (CONSUMERS / 32) : 0;
    float* qs = reinterpret_cast<float*>(done + STAGES + STAGES) + group * SCRATCH;  // this group's scratch
    float* ks = qs + D;
    float* vs = ks + D;
    float* red = vs + D;
    float* obuf = red + 64;
    float* ssp = obuf + D;

    if (tid == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&fullS[st], 1);
            mbar_init(&done[st], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == GROUPS * CONSUMERS / 32) {
        // ---------------- producer ----------------
        if (lane == 0) {
            // the conv state: rows m = 0 .. K-2 become rows 1 .. K-2 and the new x (from the stage)
            char* cpool = static_cast<char*>(J.conv_pool);
            auto roll_part = [&](const unsigned char* sb, int slot, int part, int ch0) {
                for (int m = 0; m < Km1; ++m) {
                    const int src_row = m + 1;  // row of the window that becomes row m
                    const unsigned char* src = src_row < Km1 ? sb + St::CV + (size_t)(src_row * NCH + part * D) * E
                                                             : sb + St::X + (size_t)(part * D) * E;
                    bulk_s2g(cpool + (((size_t)slot * Km1 + m) * C + ch0) * E, src, D * E);
                }
            };
            for (int k = 0; k < n_local + STAGES; ++k) {
                const int st = k % STAGES;
                const int pk = k - STAGES;  // the item that used this stage before
                if (pk >= 0 && pk < n_local) {  // retire it
                    if (!mbar_wait(&done[st], ((k / STAGES) - 1) & 1)) report_device_status(kDevWaitTimeout);
                    unsigned char* sb = smem + st * St::BYTES;
                    const int* hdr = reinterpret_cast<const int*>(sb + St::HDR);
                    if (hdr[2] >= 0) {  // state back in place, conv rows rolled
                        int pb, pj;
                        item_of(pk, pb, pj);
                        const int ph = pj / G;
                        bulk_s2g(J.state_pool + ((size_t)hdr[2] * Hv + pj) * D * D, sb + St::S, D * D * 4);
                        roll_part(sb, hdr[2], 2, 2 * Hk * D + pj * D);  // the item's own v channels
                        if (pk % G == G - 1) {  // the unit's last item: every reader of its q, k rows is done
                            roll_part(sb, hdr[2], 0, ph * D);
                            roll_part(sb, hdr[2], 1, Hk * D + ph * D);
                        }
                        bulk_commit();
                    }
                    bulk_wait_read_all();  // the stage may be refilled
                }
                if (k >= n_local) continue;
                unsigned char* sb = smem + st * St::BYTES;
                int bb, j;
                item_of(k, bb, j);
                const int h = j / G;
                const int slot = J.slot_idx[bb];
                const bool valid = slot >= 0 && slot < J.n_slots;
                int* hdr = reinterpret_cast<int*>(sb + St::HDR);
                float* hf = reinterpret_cast<float*>(sb + St::HDR);
                hf[0] = L::ld(J.a, (size_t)bb * Hv + j);
                hf[1] = L::ld(J.b, (size_t)bb * Hv + j);
                hdr[2] = valid ? slot : -1;
                if (!valid) {
                    mbar_arrive_expect_tx(&fullS[st], 0);
                    mbar_arrive_expect_tx(&full[st], 0);
                    continue;
                }
                const int ch_q = h * D, ch_k = Hk * D + h * D, ch_v = 2 * Hk * D + j * D;
                mbar_arrive_expect_tx(&fullS[st], D * D * 4);
                bulk_g2s(sb + St::S, J.state_pool + ((size_t)slot * Hv + j) * D * D, D * D * 4, &fullS[st]);
                const bool conv_w = !raw && A.p.conv_w;
                const uint32_t bytes =
                    NCH * E + Km1 * NCH * E + (conv_w ? NCH * K * E : 0) + (outnorm ? 2 * D * E : 0);
                mbar_arrive_expect_tx(&full[st], bytes);  // releases the header writes too
                const char* xrow = static_cast<const char*>(J.x) + (size_t)bb * C * E;
                bulk_g2s(sb + St::X, xrow + (size_t)ch_q * E, D * E, &full[st]);
                bulk_g2s(sb + St::X + D * E, xrow + (size_t)ch_k * E, D * E, &full[st]);
                bulk_g2s(sb + St::X + 2 * D * E, xrow + (size_t)ch_v * E, D * E, &full[st]);
                const char* cg_ = static_cast<const char*>(J.conv_pool);
                for (int m = 0; m < Km1; ++m) {
                    const char* row = cg_ + ((size_t)slot * Km1 + m) * C * E;
                    bulk_g2s(sb + St::CV + m * NCH * E, row + (size_t)ch_q * E, D * E, &full[st]);
                    bulk_g2s(sb + St::CV + (m * NCH + D) * E, row + (size_t)ch_k * E, D * E, &full[st]);
                    bulk_g2s(sb + St::CV + (m * NCH + 2 * D) * E, row + (size_t)ch_v * E, D * E, &full[st]);
                }
                if (conv_w) {
                    const char* w = static_cast<const char*>(A.p.conv_w);
                    bulk_g2s(sb + St::W, w + (size_t)ch_q * K * E, D * K * E, &full[st]);
                    bulk_g2s(sb + St::W + D * K * E, w + (size_t)ch_k * K * E, D * K * E, &full[st]);
                    bulk_g2s(sb + St::W + 2 * D * K * E, w + (size_t)ch_v * K * E, D * K * E, &full[st]);
                }
                if (outnorm) {
                    bulk_g2s(sb + St::Z, static_cast<const char*>(J.z) + ((size_t)bb * Hv + j) * D * E, D * E,
                             &full[st]);
                    bulk_g2s(sb + St::NW, A.p.norm_w, D * E, &full[st]);
                }
            }
            bulk_wait_read_all();
        }
        return;
    }

    // ---------------- consumers (group g: warps 8g .. 8g + 7, items k = g, g + 2, ...) ----------------
    const int col4 = lane;  // D = 128: a warp covers one row, 4 floats per lane
    const int gtid = tid - group * CONSUMERS, gwarp = gtid >> 5;
    for (int k = group; k < n_local; k += GROUPS) {
        const int st = k % STAGES;
        const uint32_t par = (k / STAGES) & 1;
        unsigned char* sb = smem + st * St::BYTES;
        const TA* xs = reinterpret_cast<const TA*>(sb + St::X);
        const TA* cs = reinterpret_cast<const TA*>(sb + St::CV);
        const TA* wsm = reinterpret_cast<const TA*>(sb + St::W);
        const TA* zs = reinterpret_cast<const TA*>(sb + St::Z);
        const TA* nw = reinterpret_cast<const TA*>(sb + St::NW);
        float* Sb = reinterpret_cast<float*>(sb + St::S);
        int bb, j;
        item_of(k, bb, j);
        const int h = j / G;
        bool ok = true;
        if (gwarp == 0) {
            ok = mbar_wait(&full[st], par);
            if (!ok) mbar_wait(&full[st], par);
        }
        ok = __syncthreads_and_consumers(ok, group);
        const int* hdr = reinterpret_cast<const int*>(sb + St::HDR);
        const float* hfl = reinterpret_cast<const float*>(sb + St::HDR);
        const bool valid = hdr[2] >= 0;
        const int ch_q = h * D, ch_k = Hk * D + h * D, ch_v = 2 * Hk * D + j * D;
        auto conv = [&](int lc) -> float {
            if (raw) return L::ld(xs, lc);
            const int ch = lc < D ? ch_q + lc : (lc < 2 * D ? ch_k + lc - D : ch_v + lc - 2 * D);
            float c = A.p.conv_b ? L::ld(A.p.conv_b, ch) : 0.0f;
            for (int m = 0; m < K; ++m) {
                const int tau = m - Km1;  // taps before the current token come from the conv state
                const float xv = tau >= 0 ? L::ld(xs, lc) : L::ld(cs, (size_t)(Km1 + tau) * NCH + lc);
                c = fmaf(L::ld(wsm, (size_t)lc * K + m), xv, c);
            }
            return siluf_(c);
        };
        float sq = 0.f, sk = 0.f, sqk = 0.f;
        if (ok && valid) {  // threads 0..127: channel c of q and k; 128..255: channel c of v
            const int c = gtid & (D - 1);
            if (gtid < D) {
                const float qv = conv(c), kv = conv(D + c);
                qs[c] = qv;
                ks[c] = kv;
                sq = fmaf(qv, qv, sq);
                sk = fmaf(kv, kv, sk);
                sqk = fmaf(qv, kv, sqk);
            } else {
                vs[c] = conv(2 * D + c);
            }
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        sqk = warp_sum(sqk);
        if (lane == 0) {
            red[gwarp * 4 + 0] = sq;
            red[gwarp * 4 + 1] = sk;
            red[gwarp * 4 + 2] = sqk;
        }
        bool s_ok = true;
        if (gwarp == 0 && ok) {
            s_ok = mbar_wait(&fullS[st], par);
            if (!s_ok) mbar_wait(&fullS[st], par);
        }
        ok = __syncthreads_and_consumers(ok && s_ok, group);
        if (ok && valid) {
            sq = sk = sqk = 0.f;
            for (int w = 0; w < CONSUMERS / 32; ++w) {
                sq += red[w * 4 + 0];
                sk += red[w * 4 + 1];
                sqk += red[w * 4 + 2];
            }
            float rq, rk;
            if (g.flags & kFlagNoL2) {
                rq = g.q_scale;
                rk = 1.0f;
            } else {
                rq = g.q_scale * rsqrtf(sq + g.l2_eps);
                rk = rsqrtf(sk + g.l2_eps);
            }
            const float kq = sqk * rq * rk;
            float gl, beta;
            gates(hfl[0], hfl[1], direct ? 0.f : A.p.A_log[j], (!direct && A.p.dt_bias) ? A.p.dt_bias[j] : 0.f,
                  direct, gl, beta);
            const float alpha = expf(gl);
            float kr[4], qr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kr[e] = ks[col4 * 4 + e] * rk;
                qr[e] = qs[col4 * 4 + e] * rq;
            }
            for (int rb = gwarp * 8; rb < D; rb += 8 * (CONSUMERS / 32)) {
                float4 sv[8];
                float v[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    sv[i] = *reinterpret_cast<const float4*>(Sb + (rb + i) * D + lane * 4);
                    float dk = sv[i].x * kr[0];
                    dk = fmaf(sv[i].y, kr[1], dk);
                    dk = fmaf(sv[i].z, kr[2], dk);
                    v[i] = fmaf(sv[i].w, kr[3], dk);
                    float dq = sv[i].x * qr[0];
                    dq = fmaf(sv[i].y, qr[1], dq);
                    dq = fmaf(sv[i].z, qr[2], dq);
                    v[8 + i] = fmaf(sv[i].w, qr[3], dq);
                }
#pragma unroll
                for (int n = 8, off = 16; n >= 1; n >>= 1, off >>= 1) {
                    const bool upper = lane & off;
#pragma unroll
                    for (int i = 0; i < n; ++i) {
                        const float send = upper ? v[i] : v[i + n];
                        const float keep = upper ? v[i + n] : v[i];
                        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
                const int idx = lane >> 1;
                const float e_mine = idx < 8 ? vs[rb + idx] - alpha * v[0] : 0.f;
                float ei[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) ei[i] = __shfl_sync(0xffffffffu, e_mine, 2 * i);
                const float e_for_q = __shfl_sync(0xffffffffu, e_mine, ((idx - 8) & 7) * 2);
                if (idx >= 8 && !(lane & 1)) obuf[rb + idx - 8] = fmaf(alpha, v[0], beta * e_for_q * kq);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float be = beta * ei[i];
                    sv[i].x = fmaf(alpha, sv[i].x, be * kr[0]);
                    sv[i].y = fmaf(alpha, sv[i].y, be * kr[1]);
                    sv[i].z = fmaf(alpha, sv[i].z, be * kr[2]);
                    sv[i].w = fmaf(alpha, sv[i].w, be * kr[3]);
                    *reinterpret_cast<float4*>(Sb + (rb + i) * D + lane * 4) = sv[i];
                }
            }
        }
        fence_proxy_async_smem();  // the state tile goes out through the async proxy
        __syncthreads_and_consumers(true, group);
        if (ok && valid) {
            // output gated RMSNorm over the whole v-head
            if (gwarp == 0) {
                float ss = 0.f;
                for (int rr = lane; rr < D; rr += 32) ss = fmaf(obuf[rr], obuf[rr], ss);
                ss = warp_sum(ss);
                if (lane == 0) ssp[0] = ss;
            }
            __syncthreads_and_consumers(true, group);
            for (int rr = gtid; rr < D; rr += CONSUMERS) {
                float yv = obuf[rr];
                if (outnorm) yv = yv * rsqrtf(ssp[0] / (float)D + g.norm_eps) * L::ld(nw, rr) * siluf_(L::ld(zs, rr));
                L::st(J.y, ((size_t)bb * Hv + j) * D + rr, yv);
            }
        }
        if (!ok && gtid == 0) report_device_status(kDevWaitTimeout);
        __syncthreads_and_consumers(true, group);  // qs/ks/vs/obuf/red reused by the next item; stage fully read
        if (gtid == 0) mbar_arrive(&done[st]);  // the producer may store and refill the stage
    }
}

int choose_slices(const Geom& g, int B) {
    const int max_ns = std::min(8 / g.G, g.D / 8);
    if (const char* e = std::getenv("GDN_DECODE_SLICES")) {
        int v = std::atoi(e);
        if (v >= 1 && v <= max_ns && (v & (v - 1)) == 0) return v;
    }
    // One CTA per v-head (whole 128x128 state in shared memory, local output
    // norm) measured best or equal at every batch from 1 to 256 on GB300;
    // slicing the rows (NS > 1) stays available for experiments and tests.
    return 1;
}

template <int D, typename TA>
cudaError_t launch_rows_t(const Geom& g, const LayerParams& p, const RowsJob& job, cudaStream_t st) {
    const int NS = choose_slices(g, job.B);
    RowsArgs A{g, p, job, NS};
    const RowsSmem lay = rows_smem(D, D / NS, job.r, g.K, (int)sizeof(TA));
    static std::atomic<uint64_t> smem_set{0};  // allow up to 200 KB
    {
        const cudaError_t e = raise_smem_limit(k_rows<D, TA>, 200 * 1024, smem_set);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.G * NS, g.Hk, job.B);
    cfg.blockDim = dim3(kRowsThreads);
    cfg.dynamicSmemBytes = (size_t)lay.total;
    cfg.stream = st;
    // a cluster per k-head group; programmatic stream serialization lets the grid be
    // scheduled while its predecessor finishes (it waits in griddep_wait)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = g.G * NS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_rows<D, TA>, A);
}

// ---- standalone conv state update ---------------------------------------------
template <typename TA>
__global__ void k_conv_silu(const Geom g, const LayerParams p, const ConvJob J) {
    using L = Act<TA>;
    const int C = g.C_ch, K = g.K;
    const size_t total = (size_t)J.n_seq * J.n_tok * C;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int ch = (int)(idx % C);
        const size_t row = idx / C;
        const int sq = (int)(row / J.n_tok), t = (int)(row % J.n_tok);
        const int slot = J.slot_idx[sq];
        if (slot < 0 || slot >= J.n_slots) continue;
        float c = p.conv_b ? L::ld(p.conv_b, ch) : 0.0f;
        for (int m = 0; m < K; ++m) {
            const int tau = t - (K - 1) + m;
            const float xv = tau >= 0 ? L::ld(J.x, ((size_t)sq * J.n_tok + tau) * C + ch)
                                      : L::ld(J.conv_pool, ((size_t)slot * (K - 1) + (K - 1 + tau)) * C + ch);
            c = fmaf(L::ld(p.conv_w, (size_t)ch * K + m), xv, c);
        }
        L::st(J.u_out, idx, siluf_(c));
    }
}

template <typename TA>
__global__ void k_conv_roll(const Geom g, const ConvJob J) {
    using L = Act<TA>;
    const int C = g.C_ch, Km1 = g.K - 1;
    const size_t total = (size_t)J.n_seq * C;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int ch = (int)(idx % C), sq = (int)(idx / C);
        const int slot = J.slot_idx[sq];
        if (slot < 0 || slot >= J.n_slots) continue;
        float old[3];
#pragma unroll
        for (int m = 0; m < 3; ++m) old[m] = m < Km1 ? L::ld(J.conv_pool, ((size_t)slot * Km1 + m) * C + ch) : 0.f;
        for (int m = 0; m < Km1; ++m) {
            const int pidx = J.n_tok + m;
            const float v = pidx < Km1 ? old[pidx] : L::ld(J.x, ((size_t)sq * J.n_tok + (pidx - Km1)) * C + ch);
            L::st(J.conv_pool, ((size_t)slot * Km1 + m) * C + ch, v);
        }
    }
}


// ---- commit by copy -----------------------------------------------------------
__global__ void k_commit(const Geom g, const CommitJob J, int elt_bytes) {
    const int b = blockIdx.y;
    const int a = J.accepted[b];
    if (a < 1 || a > J.r) return;
    const int src = J.snap_idx[(size_t)b * J.r + (a - 1)], dst = J.slot_idx[b];
    if (src < 0 || src >= J.n_slots || dst < 0 || dst >= J.n_slots || src == dst) return;
    const size_t n4 = (size_t)g.Hv * g.D * g.D / 4;
    const float4* S = reinterpret_cast<const float4*>(J.state_pool + (size_t)src * g.Hv * g.D * g.D);
    float4* Dd = reinterpret_cast<float4*>(J.state_pool + (size_t)dst * g.Hv * g.D * g.D);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        Dd[i] = S[i];
    const size_t cbytes = (size_t)(g.K - 1) * g.C_ch * elt_bytes;  // a multiple of 16
    const float4* cs = reinterpret_cast<const float4*>(static_cast<const char*>(J.conv_pool) + (size_t)src * cbytes);
    float4* cd = reinterpret_cast<float4*>(static_cast<char*>(J.conv_pool) + (size_t)dst * cbytes);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < cbytes / 16; i += (size_t)gridDim.x * blockDim.x)
        cd[i] = cs[i];
}

}  // namespace

template <typename TA>
cudaError_t launch_decode_persist(const Geom& g, const LayerParams& p, const RowsJob& job, cudaStream_t st) {
    constexpr int smem = pd::smem_bytes<TA>();
    static_assert(smem <= 227 * 1024, "persistent decode: shared memory");
    static std::atomic<uint64_t> smem_set{0};
    {
        const cudaError_t e = raise_smem_limit(k_decode_persist<TA>, smem, smem_set);
        if (e != cudaSuccess) return e;
    }
    const int sms = sm_count();
    const int units = job.B * g.Hk;
    RowsArgs A{g, p, job, 1};
    // programmatic stream serialization: the grid may be scheduled while its
    // predecessor finishes and waits for it (griddep_wait) before its first access
    // to memory, which hides the launch gap
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(units, sms));
    cfg.blockDim = dim3(pd::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_decode_persist<TA>, A);
}

// CTAs of k_rows<128, TA> resident per SM in a decode step (cached per device)
template <typename TA>
int rows_ctas_per_sm(const Geom& g) {
    static std::atomic<int> cache[64];  // static storage: zero, i.e. not yet queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::atomic<int>& c = cache[dev & 63];
    int n = c.load(std::memory_order_relaxed);
    if (n > 0) return n;
    static std::atomic<uint64_t> smem_set{0};
    if (raise_smem_limit(k_rows<128, TA>, 200 * 1024, smem_set) != cudaSuccess) return 1;
    const RowsSmem lay = rows_smem(128, 128, 1, g.K, (int)sizeof(TA));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_rows<128, TA>, kRowsThreads, (size_t)lay.total) !=
            cudaSuccess ||
        n <= 0)
        n = 1;
    c.store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_rows(const Geom& g, const LayerParams& p, const RowsJob& job, cudaStream_t st) {
    if (job.B == 0) return cudaSuccess;
    // A decode step runs on the persistent kernel (three stages in shared memory: bf16
    // inputs only) or on k_rows (one CTA per item).  Measured at the 4B geometry,
    // us per layer call, k_rows / persistent: B = 1: 7.4 / 9.3; 4: 8.9 / 10.6;
    // 6: 11.3 / 11.0; 8: 13.9 / 11.9; 10: 14.9 / 16.1; 12: 15.5 / 16.5;
    // 16: 22.4 / 17.2; 64: - / 47.7.  The persistent kernel costs about one item's
    // chain per (slot, k-head) unit a CTA holds; k_rows about one chain per wave.  So:
    // k_rows for about one item per SM or fewer, the persistent kernel while a CTA
    // holds one unit, k_rows while its CTAs fit in one wave, the persistent kernel
    // beyond.
    if (g.D == 128 && g.act_bf16 && job.r == 1 && !job.snap_idx && job.mode == 0 &&
        std::getenv("GDN_DECODE_CLUSTERED") == nullptr && std::getenv("GDN_DECODE_SLICES") == nullptr) {
        const long items = (long)job.B * g.Hv, units = (long)job.B * g.Hk, sms = sm_count();
        bool persist;
        if (items * 4 <= sms * 5) persist = false;
        else if (units <= sms) persist = true;
        else persist = items > (long)rows_ctas_per_sm<__nv_bfloat16>(g) * sms;
        if (persist) return launch_decode_persist<__nv_bfloat16>(g, p, job, st);
    }
    if (g.act_bf16) {
        switch (g.D) {
            case 32: return launch_rows_t<32, __nv_bfloat16>(g, p, job, st);
            case 64: return launch_rows_t<64, __nv_bfloat16>(g, p, job, st);
            case 128: return launch_rows_t<128, __nv_bfloat16>(g, p, job, st);
        }
    } else {
        switch (g.D) {
            case 32: return launch_rows_t<32, float>(g, p, job, st);
            case 64: return launch_rows_t<64, float>(g, p, job, st);
            case 128: return launch_rows_t<128, float>(g, p, job, st);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_conv_update(const Geom& g, const LayerParams& p, const ConvJob& job, cudaStream_t st) {
    if (job.n_seq == 0) return cudaSuccess;
    const int threads = 256;
    if (job.u_out && job.n_tok > 0) {
        const size_t total = (size_t)job.n_seq * job.n_tok * g.C_ch;
        const int blocks = (int)std::min<size_t>((total + threads - 1) / threads, 152 * 16);
        if (g.act_bf16) k_conv_silu<__nv_bfloat16><<<blocks, threads, 0, st>>>(g, p, job);
        else k_conv_silu<float><<<blocks, threads, 0, st>>>(g, p, job);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (job.n_tok > 0) {
        const size_t total = (size_t)job.n_seq * g.C_ch;
        const int blocks = (int)std::min<size_t>((total + threads - 1) / threads, 152 * 16);
        if (g.act_bf16) k_conv_roll<__nv_bfloat16><<<blocks, threads, 0, st>>>(g, job);
        else k_conv_roll<float><<<blocks, threads, 0, st>>>(g, job);
    }
    return cudaGetLastError();
}

// ---- debug check of slot indices (GDN_DEBUG) -------------------------------
// result: [0] first position holding an index outside [0, n_slots) (INT32_MAX: none),
// [1..2] first pair (i, j), i < j, holding the same index (packed i * 2^32 + j;
// ~0: none).  Positions run over the concatenation of idx_a [na] and idx_b [nb].
namespace {
__device__ unsigned long long g_slot_check[2];

__global__ void k_check_slots(const int32_t* idx_a, int na, const int32_t* idx_b, int nb, int n_slots) {
    // one thread per position i compares it with every later position: quadratic,
    // which is fine for a debugging aid at the batch sizes the calls take
    const int n = na + nb;
    auto at = [&](int k) { return k < na ? __ldg(idx_a + k) : __ldg(idx_b + (k - na)); };
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int v = at(i);
    bool bad = false;
    if (v < 0 || v >= n_slots) {
        atomicMin(&g_slot_check[0], (unsigned long long)i);
        bad = true;
    }
    for (int j = i + 1; j < n; ++j) {
        if (at(j) == v) {
            atomicMin(&g_slot_check[1], ((unsigned long long)i << 32) | (unsigned long long)j);
            bad = true;
            break;
        }
    }
    if (bad) report_device_status(kDevBadSlot);
}

__global__ void k_check_reset() { g_slot_check[0] = g_slot_check[1] = ~0ull; }
}  // namespace

cudaError_t check_slots(const int32_t* idx_a, int na, const int32_t* idx_b, int nb, int n_slots, cudaStream_t st,
                        bool wait, long long* bad_range, long long* dup_i, long long* dup_j, int32_t* value) {
    // a reset kernel rather than a host copy keeps the check capturable
    k_check_reset<<<1, 1, 0, st>>>();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int n = na + nb;
    k_check_slots<<<(n + 255) / 256, 256, 0, st>>>(idx_a, na, idx_b, nb, n_slots);
    e = cudaGetLastError();
    if (e != cudaSuccess || !wait) return e;
    unsigned long long got[2];
    e = cudaMemcpyFromSymbolAsync(got, g_slot_check, sizeof got, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    *bad_range = got[0] == ~0ull ? -1 : (long long)got[0];
    *dup_i = got[1] == ~0ull ? -1 : (long long)(got[1] >> 32);
    *dup_j = got[1] == ~0ull ? -1 : (long long)(got[1] & 0xffffffffull);
    // the offending value, read back for the message
    *value = 0;
    const long long k = *bad_range >= 0 ? *bad_range : *dup_i;
    if (k >= 0) {
        const int32_t* src = k < na ? idx_a + k : idx_b + (k - na);
        e = cudaMemcpyAsync(value, src, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    return e;
}

cudaError_t take_device_status_decode(unsigned* out) { return take_device_status_tu(out); }

cudaError_t launch_commit(const Geom& g, const CommitJob& job, cudaStream_t st) {
    if (job.B == 0) return cudaSuccess;
    dim3 grid(64, job.B);
    k_commit<<<grid, 256, 0, st>>>(g, job, g.act_bf16 ? 2 : 4);
    return cudaGetLastError();
}

}  // namespace gdn
