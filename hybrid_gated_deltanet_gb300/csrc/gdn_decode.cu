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

namespace cg = cooperative_groups;

namespace gdn {
namespace {

constexpr int kMaxRows = 16;

struct RowsArgs {
    Geom g;
    LayerParams p;
    RowsJob job;
    int NS;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// silu(conv) (or the raw value) of channel ch for verify row t of batch entry bb
template <typename TA>
__device__ __forceinline__ float conv_at(const RowsArgs& A, int ch, int t, int bb, int slot) {
    using L = Act<TA>;
    const Geom& g = A.g;
    const RowsJob& J = A.job;
    const int C = g.C_ch, K = g.K;
    if (g.flags & kFlagRawQKV) return L::ld(J.x, ((size_t)bb * J.r + t) * C + ch);
    float c = A.p.conv_b ? L::ld(A.p.conv_b, ch) : 0.0f;
    for (int m = 0; m < K; ++m) {
        const int tau = t - (K - 1) + m;
        const float xv = tau >= 0 ? L::ld(J.x, ((size_t)bb * J.r + tau) * C + ch)
                                  : L::ld(J.conv_pool, ((size_t)slot * (K - 1) + (K - 1 + tau)) * C + ch);
        c = fmaf(L::ld(A.p.conv_w, (size_t)ch * K + m), xv, c);
    }
    return siluf_(c);
}

template <int D, typename TA>
__global__ void __launch_bounds__(512) k_rows(const __grid_constant__ RowsArgs A) {
    constexpr int LPR = D / 4;     // lanes per state row (4 floats per lane)
    constexpr int RPI = 32 / LPR;  // rows per warp-wide 128-bit access
    constexpr int NV = D / 16;     // float4 per lane: 8 rows per warp
    using L = Act<TA>;
    cg::cluster_group cluster = cg::this_cluster();
    const Geom& g = A.g;
    const RowsJob& J = A.job;
    const int NS = A.NS, G = g.G, Hk = g.Hk, Hv = g.Hv, K = g.K, C = g.C_ch;
    const int CS = G * NS;
    const int gi = blockIdx.x / NS, s = blockIdx.x % NS;
    const int h = blockIdx.y, j = h * G + gi, bb = blockIdx.z;
    const int RPC = D / NS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = blockDim.x, nwarp = nthr >> 5;
    const int r = J.r;
    const int crank = (int)cluster.block_rank();

    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    float* qs = sm;                    // [D]   conv+SiLU output of q (this row)
    float* ks = qs + D;                // [D]   ... of k
    float* vs = ks + D;                // [RPC] ... of this slice's v
    float* red = vs + D;               // [16 warps][4]
    float* obuf = red + 64;            // [kMaxRows][RPC] o of every row
    float* ssp = obuf + kMaxRows * D;  // [kMaxRows] partial sum of o^2

    const int slot = J.slot_idx[bb];
    if (slot < 0 || slot >= J.n_slots) return;  // the whole cluster shares bb

    // ---- issue the state loads first: they overlap the prologue --------------
    const int row0 = s * RPC + warp * 8;
    const int col4 = lane % LPR, rsub = lane / LPR;
    float4 sreg[NV];
    {
        const float* Sb = J.state_pool + ((size_t)slot * Hv + j) * D * D;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            sreg[i] = *reinterpret_cast<const float4*>(Sb + (size_t)(row0 + i * RPI + rsub) * D + col4 * 4);
    }

    const bool direct = g.flags & kFlagGatesDirect;
    const float A_log_j = direct ? 0.0f : A.p.A_log[j];
    const float dt_j = (!direct && A.p.dt_bias) ? A.p.dt_bias[j] : 0.0f;

    for (int t = 0; t < r; ++t) {
        const size_t rowx = (size_t)bb * r + t;
        __syncthreads();  // readers of qs/ks/vs/red from the previous row are done
        float sq = 0.f, sk = 0.f, sqk = 0.f;
        for (int c = tid; c < D; c += nthr) {
            const float qv = conv_at<TA>(A, h * D + c, t, bb, slot);
            const float kv = conv_at<TA>(A, Hk * D + h * D + c, t, bb, slot);
            qs[c] = qv;
            ks[c] = kv;
            sq = fmaf(qv, qv, sq);
            sk = fmaf(kv, kv, sk);
            sqk = fmaf(qv, kv, sqk);
        }
        for (int c = tid; c < RPC; c += nthr) vs[c] = conv_at<TA>(A, 2 * Hk * D + j * D + s * RPC + c, t, bb, slot);
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        sqk = warp_sum(sqk);
        if (lane == 0) {
            red[warp * 4 + 0] = sq;
            red[warp * 4 + 1] = sk;
            red[warp * 4 + 2] = sqk;
        }
        __syncthreads();
        sq = sk = sqk = 0.f;
        for (int w = 0; w < nwarp; ++w) {
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
        gates(L::ld(J.a, rowx * Hv + j), L::ld(J.b, rowx * Hv + j), A_log_j, dt_j, direct, gl, beta);
        const float alpha = expf(gl);
        float kr[4], qr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            kr[e] = ks[col4 * 4 + e] * rk;
            qr[e] = qs[col4 * 4 + e] * rq;
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float dk = sreg[i].x * kr[0];
            dk = fmaf(sreg[i].y, kr[1], dk);
            dk = fmaf(sreg[i].z, kr[2], dk);
            dk = fmaf(sreg[i].w, kr[3], dk);
            float dq = sreg[i].x * qr[0];
            dq = fmaf(sreg[i].y, qr[1], dq);
            dq = fmaf(sreg[i].z, qr[2], dq);
            dq = fmaf(sreg[i].w, qr[3], dq);
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) {
                dk += __shfl_xor_sync(0xffffffffu, dk, off);
                dq += __shfl_xor_sync(0xffffffffu, dq, off);
            }
            const int rl = warp * 8 + i * RPI + rsub;  // row within the slice
            const float e = vs[rl] - alpha * dk;
            const float be = beta * e;
            sreg[i].x = fmaf(alpha, sreg[i].x, be * kr[0]);
            sreg[i].y = fmaf(alpha, sreg[i].y, be * kr[1]);
            sreg[i].z = fmaf(alpha, sreg[i].z, be * kr[2]);
            sreg[i].w = fmaf(alpha, sreg[i].w, be * kr[3]);
            if (col4 == 0) obuf[t * RPC + rl] = fmaf(alpha, dq, be * kq);
        }
        if (J.snap_idx) {  // verify: the state after row t goes to its snapshot slot
            const int dst = J.snap_idx[rowx];
            if (dst >= 0 && dst < J.n_slots) {
                float* Sd = J.state_pool + ((size_t)dst * Hv + j) * D * D;
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    *reinterpret_cast<float4*>(Sd + (size_t)(row0 + i * RPI + rsub) * D + col4 * 4) = sreg[i];
            }
        }
    }
    if (!J.snap_idx) {  // decode: in place
        float* Sd = J.state_pool + ((size_t)slot * Hv + j) * D * D;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            *reinterpret_cast<float4*>(Sd + (size_t)(row0 + i * RPI + rsub) * D + col4 * 4) = sreg[i];
    }

    // ---- output gated RMSNorm: sum of o^2 over the head's D rows --------------
    __syncthreads();
    for (int t = warp; t < r; t += nwarp) {
        float ss = 0.f;
        for (int rr = lane; rr < RPC; rr += 32) {
            const float o = obuf[t * RPC + rr];
            ss = fmaf(o, o, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) ssp[t] = ss;
    }
    cluster.sync();  // partials visible; every conv-state read in this cluster is done

    const bool outnorm = !(g.flags & kFlagNoOutNorm);
    for (int idx = tid; idx < r * RPC; idx += nthr) {
        const int t = idx / RPC, rr = idx % RPC;
        const size_t rowx = (size_t)bb * r + t;
        const int dv = s * RPC + rr;
        const float o = obuf[idx];
        float yv = o;
        if (outnorm) {
            float tot = 0.f;
            for (int s2 = 0; s2 < NS; ++s2) tot += *cluster.map_shared_rank(&ssp[t], gi * NS + s2);
            const float zz = L::ld(J.z, rowx * (size_t)Hv * D + (size_t)j * D + dv);
            yv = o * rsqrtf(tot / (float)D + g.norm_eps) * L::ld(A.p.norm_w, dv) * siluf_(zz);
        }
        L::st(J.y, rowx * (size_t)Hv * D + (size_t)j * D + dv, yv);
    }

    // ---- conv state: last K-1 raw inputs, after the barrier --------------------
    const int Km1 = K - 1;
    auto roll = [&](int ch) {
        float old[3];
#pragma unroll
        for (int m = 0; m < 3; ++m)
            old[m] = m < Km1 ? L::ld(J.conv_pool, ((size_t)slot * Km1 + m) * C + ch) : 0.0f;
        auto val = [&](int p) -> float {
            return p < Km1 ? old[p] : L::ld(J.x, ((size_t)bb * r + (p - Km1)) * C + ch);
        };
        if (!J.snap_idx) {
            for (int m = 0; m < Km1; ++m) L::st(J.conv_pool, ((size_t)slot * Km1 + m) * C + ch, val(r + m));
        } else {
            for (int t = 0; t < r; ++t) {
                const int dst = J.snap_idx[(size_t)bb * r + t];
                if (dst < 0 || dst >= J.n_slots) continue;
                for (int m = 0; m < Km1; ++m)
                    L::st(J.conv_pool, ((size_t)dst * Km1 + m) * C + ch, val(t + 1 + m));
            }
        }
    };
    for (int c = crank + CS * tid; c < 2 * D; c += CS * nthr) roll(c < D ? h * D + c : Hk * D + h * D + (c - D));
    for (int c = tid; c < RPC; c += nthr) roll(2 * Hk * D + j * D + s * RPC + c);

    cluster.sync();  // peers may still read this CTA's partial sums
}

int choose_slices(const Geom& g, int B) {
    const int max_ns = std::min(8 / g.G, g.D / 8);
    if (const char* e = std::getenv("GDN_DECODE_SLICES")) {
        int v = std::atoi(e);
        if (v >= 1 && v <= max_ns && (v & (v - 1)) == 0) return v;
    }
    // enough CTAs to cover 152 SMs a few times over, fewest slices otherwise
    int ns = 1;
    while (ns < max_ns && (long)B * g.Hv * ns < 4L * 152) ns *= 2;
    if (g.D == 128 && ns < 2 && max_ns >= 2) ns = 2;  // 256-thread CTAs for the 128x128 state
    return ns;
}

template <int D, typename TA>
cudaError_t launch_rows_t(const Geom& g, const LayerParams& p, const RowsJob& job, cudaStream_t st) {
    const int NS = choose_slices(g, job.B);
    RowsArgs A{g, p, job, NS};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.G * NS, g.Hk, job.B);
    cfg.blockDim = dim3((D / NS) * 4);  // D/NS rows, 8 rows per warp
    cfg.dynamicSmemBytes = (size_t)(3 * D + 64 + kMaxRows * D + kMaxRows) * sizeof(float);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = g.G * NS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
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

cudaError_t launch_rows(const Geom& g, const LayerParams& p, const RowsJob& job, cudaStream_t st) {
    if (job.B == 0) return cudaSuccess;
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

cudaError_t launch_commit(const Geom& g, const CommitJob& job, cudaStream_t st) {
    if (job.B == 0) return cudaSuccess;
    dim3 grid(64, job.B);
    k_commit<<<grid, 256, 0, st>>>(g, job, g.act_bf16 ? 2 : 4);
    return cudaGetLastError();
}

}  // namespace gdn
