// gdn_noalloc.cu -- chunked prefill for callers that cannot allocate device
// memory: the prefill workspace lives in a fixed static device array of this
// library instead of a caller-provided buffer.
//
// Why: some callers cannot call cudaMalloc when they need a prefill.  A host
// runtime may own the whole device memory budget through its own allocator
// and give a plugin no way to reach it; code may run while its stream is
// being captured into a CUDA graph, where cudaMalloc/cudaFree are not
// allowed; a latency-critical path may not afford the device-wide
// synchronisation that cudaFree implies.  Such callers still own and pass
// their inputs, outputs and states; only the scratch moves here.
//
// Contract:
// - The scratch is kNoAllocScratchBytes (64 MiB).  A device holds it from the
//   moment the library's module is loaded there (at the first use of the library
//   on that device under CUDA's lazy loading) until the process exits.
// - Each call looks up the array's device address for the current device and
//   context with cudaGetSymbolAddress the first time that context is seen, and
//   caches it under the context's unique id; a device reset or a new primary
//   context makes the next call look it up again.  Make the first call in a
//   context before any stream capture.
// - All calls share the one array, which keeps the previous call's contents.
//   Nothing in it needs to start at zero: the prefill writes every workspace
//   entry it reads.  Calls that overlap on the GPU (different streams, or
//   different host threads without ordering) race on the array and give
//   undefined results.
// - This file calls no cudaMalloc, cudaFree or allocating library routine.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
int report_error(int status, const char* message);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side stand-in;
// kernels receive the address obtained from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
// per device: the context id the address was looked up in, and the address
unsigned long long g_ctx_id[kMaxDevices] = {};
void* g_scratch_ptr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, unsigned version) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// unique id of the current context (0 if it cannot be read: the address is then
// looked up on every call)
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_ctx || !get_id || get_ctx(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

gdn_status scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "gdn_chunk_prefill_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
        return (gdn_status)gdn::report_error(GDN_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices) {
        char msg[256];
        snprintf(msg, sizeof msg, "device: found ordinal %d, required 0..%d", dev, kMaxDevices - 1);
        return (gdn_status)gdn::report_error(GDN_ERR_UNSUPPORTED, msg);
    }
    // id 0: no current context yet (cudaGetSymbolAddress below makes the primary one
    // current) or the driver entry points are missing: look the address up this time
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev] || id == 0 || g_ctx_id[dev] != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "gdn_chunk_prefill_noalloc: cudaGetSymbolAddress of the static scratch "
                     "failed on device %d: %s", dev, cudaGetErrorString(e));
            return (gdn_status)gdn::report_error(GDN_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
        g_ctx_id[dev] = id;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_chunk_prefill_noalloc(const gdn_config* cfg, const gdn_params* prm, const void* x,
                                                const void* z, const void* a, const void* b, int64_t T,
                                                const float* s0, const void* conv0, float* s_final,
                                                void* conv_final, void* y, void* stream) {
    // an invalid config gives need = 0 here and is reported by gdn_chunk_prefill below
    const size_t need = gdn_workspace_size(cfg, GDN_OP_CHUNK_PREFILL, T, 1);
    if (need > kNoAllocScratchBytes) {
        char msg[320];
        snprintf(msg, sizeof msg, "T: found %lld tokens needing %zu bytes of workspace, required at most the "
                 "%zu bytes of the static scratch of gdn_chunk_prefill_noalloc (use gdn_chunk_prefill with a "
                 "caller-owned workspace)", (long long)T, need, kNoAllocScratchBytes);
        return (gdn_status)gdn::report_error(GDN_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    if (need > 0) {
        gdn_status st = scratch_for_current_device(&scratch);
        if (st != GDN_OK) return st;
    }
    return gdn_chunk_prefill(cfg, prm, x, z, a, b, T, s0, conv0, s_final, conv_final, y, scratch,
                             need > 0 ? kNoAllocScratchBytes : 0, stream);
}
