// gdn_common.cuh -- device helpers shared by the libgdn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// ---- activation dtype access ------------------------------------------------
template <typename T>
struct Act;

template <>
struct Act<float> {
    static __device__ __forceinline__ float ld(const void* p, size_t i) {
        return static_cast<const float*>(p)[i];
    }
    static __device__ __forceinline__ void st(void* p, size_t i, float v) {
        static_cast<float*>(p)[i] = v;
    }
};

template <>
struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const void* p, size_t i) {
        return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    }
    static __device__ __forceinline__ void st(void* p, size_t i, float v) {
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    }
};

// ---- scalar math (CUDA's own expf/log1pf; nothing re-implemented) ----------
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplusf_(float x) {
    // log(1 + e^x) without overflow: max(x, 0) + log1p(e^-|x|)
    return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}

// gate of one (token, v-head): g = log(alpha), beta
__device__ __forceinline__ void gates(float a, float b, float A_log, float dt, bool direct,
                                      float& g, float& beta) {
    if (direct) {
        g = a;
        beta = b;
    } else {
        g = -expf(A_log) * softplusf_(a + dt);
        beta = sigmoidf_(b);
    }
}

constexpr uint32_t kFlagRawQKV = 1u, kFlagNoL2 = 2u, kFlagGatesDirect = 4u, kFlagNoOutNorm = 8u;

// ---- device status word ------------------------------------------------------
// A kernel whose bounded wait gives up ORs a code into this word instead of
// spinning forever; gdn_device_status() reads and clears it.  The kernels are
// compiled without relocatable device code, so every translation unit that
// includes this header has its own word and its own reader below.
constexpr unsigned kDevWaitTimeout = 1u;
constexpr unsigned kDevBadSlot = 2u;  // GDN_DEBUG: a slot index out of range or repeated

static __device__ unsigned int g_device_status = 0;

__device__ __forceinline__ void report_device_status(unsigned code) { atomicOr(&g_device_status, code); }

static inline cudaError_t take_device_status_tu(unsigned* out) {
    unsigned v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    *out = v;
    return e;
}

}  // namespace gdn
