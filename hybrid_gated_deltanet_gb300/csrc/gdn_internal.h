// gdn_internal.h -- launcher interface between the C-ABI layer (gdn_api.cu)
// and the kernel files.  Host-only types; nothing here is exported.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace gdn {

// A kernel's dynamic shared-memory limit belongs to its instance on one device,
// so it is raised once per device: bit d of `done` records device d (devices
// 0..63).  Two threads racing through the first call both raise it, which is
// harmless.
template <typename... KArgs>
cudaError_t raise_smem_limit(void (*kernel)(KArgs...), int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// SMs of the current device, queried once per device (1 if the query fails).
int sm_count();

// Launch with programmatic stream serialization: the kernel may become resident
// while the previous kernel of the stream finishes; it calls griddep_wait()
// before touching memory, so the stream order of memory effects is unchanged.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Geometry + options after validation (all derived fields filled in).
struct Geom {
    int Hk, Hv, D, K, G, C_ch, chunk;
    int act_bf16;  // 1: bf16 activations, 0: fp32
    float q_scale, l2_eps, norm_eps;
    uint32_t flags;
};

struct LayerParams {
    const void* conv_w;
    const void* conv_b;
    const float* A_log;
    const float* dt_bias;
    const void* norm_w;
};

// decode (r = 1, snap_idx = NULL: in place) and verify (snap_idx [B][r])
struct RowsJob {
    const void *x, *z, *a, *b;
    void* conv_pool;
    float* state_pool;
    const int32_t* slot_idx;
    const int32_t* snap_idx;
    void* y;
    int B, r, n_slots;
    // 0: decode (state in place) or verify with snapshots; 1: verify that
    // writes y only; 2: commit by recompute -- the first accepted[b] rows
    // applied in place, no y
    int mode = 0;
    const int32_t* accepted = nullptr;
};
cudaError_t launch_rows(const Geom& g, const LayerParams& prm, const RowsJob& job, cudaStream_t st);

// conv + SiLU over all channels, then roll each sequence's conv state
struct ConvJob {
    const void* x;
    void* conv_pool;
    const int32_t* slot_idx;
    void* u_out;
    int n_seq, n_tok, n_slots;
};
cudaError_t launch_conv_update(const Geom& g, const LayerParams& prm, const ConvJob& job,
                               cudaStream_t st);

struct CommitJob {
    void* conv_pool;
    float* state_pool;
    const int32_t *slot_idx, *snap_idx, *accepted;
    int B, r, n_slots;
};
cudaError_t launch_commit(const Geom& g, const CommitJob& job, cudaStream_t st);

// prefill: single sequence (cu_seqlens == NULL) or packed varlen
struct PrefillJob {
    const void *x, *z, *a, *b;
    void* y;
    int64_t n_tokens;
    int n_seq;
    const int32_t* cu_seqlens;  // NULL: one sequence [0, n_tokens)
    // varlen: pools + slots
    const int32_t* slot_idx;
    const uint8_t* has_init;
    float* state_pool;
    void* conv_pool;
    int n_slots;
    // single sequence: direct pointers
    const float* s0;
    float* s_final;
    const void* conv0;
    void* conv_final;
    void* workspace;
    size_t ws_bytes;
    // varlen snapshots every ckpt_every tokens (0: none) into pool slots
    // ckpt_slots[ckpt_offset[s] + k]
    int32_t ckpt_every;
    const int32_t* ckpt_offset;
    const int32_t* ckpt_slots;
};
size_t prefill_workspace_bytes(const Geom& g, int64_t n_tokens, int n_seq);
// the tcgen05 path for d = 128, chunk 64, bf16 activations (gdn_chunk16.cu):
// the state chain only; the caller launches the conv-state tail after it
bool chunk16_applies(const Geom& g);
size_t chunk16_workspace_bytes(const Geom& g, int64_t n_tokens, int n_seq);
cudaError_t chunk16_launch(const Geom& g, const LayerParams& prm, const PrefillJob& job, cudaStream_t st);
cudaError_t launch_prefill(const Geom& g, const LayerParams& prm, const PrefillJob& job,
                           cudaStream_t st);

// out[t][n] = sum_k act[t][k] w[n][k] (bf16, fp32 accumulation); weight rows
// [seg.n0, seg.n1) land in columns [0, n1 - n0) of seg.out (row stride seg.ld)
struct ProjOut {
    void* out;
    int64_t ld;
    int32_t n0, n1;
};
struct ProjJob {
    const void* w;    // bf16 [n_out][k]
    const void* act;  // bf16 [n_tok][k]
    int32_t n_out, k;
    int64_t n_tok;
    int nseg;
    ProjOut seg[4];
    void* ws;  // fp32 partial sums when K is split (proj_plan().ws_bytes)
    size_t ws_bytes;
};
struct ProjPlan {
    int bt;           // tokens per tile
    int64_t n_tiles;  // (128-row weight block, token block) tiles
    int ks;           // CTAs per tile splitting K (1: none)
    size_t ws_bytes;  // workspace for the split's partial sums
};
ProjPlan proj_plan(int32_t n_out, int32_t k, int64_t n_tok);
cudaError_t launch_proj(const ProjJob& job, cudaStream_t st);

// decode attention over a paged KV cache (bf16), GQA with G = Hq / Hkv in
// {1, 2, 4, 8, 12, 16}; D in {128, 256}
struct AttnJob {
    const void *q, *k_new, *v_new;
    void *k_pool, *v_pool;
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* o;
    void* ws;
    int B, Hq, Hkv, D, page, max_pages, n_pages, max_seq_len;
    float scale;
};
struct AttnPlan {
    int n_split, span;
};
AttnPlan attn_plan(int B, int Hq, int Hkv, int max_seq_len);
size_t attn_workspace_bytes(int B, int Hq, int Hkv, int D, int max_seq_len);
cudaError_t launch_attn_decode(const AttnJob& job, cudaStream_t st);

// prefill attention: new tokens cu_seqlens[s] .. cu_seqlens[s+1] of sequence s at
// positions ctx_lens[s] + i, appended to the pages, then causal attention
struct AttnPfJob {
    const void *q, *k_new, *v_new;
    void *k_pool, *v_pool;
    const int32_t* block_table;
    const int32_t* cu_seqlens;
    const int32_t* ctx_lens;
    void* o;
    int n_seq, Hq, Hkv, D, page, max_pages, n_pages;
    int64_t n_tokens;
    float scale;
};
cudaError_t launch_attn_prefill(const AttnPfJob& job, cudaStream_t st);

// GDN_DEBUG: device-side check that the na + nb indices of idx_a then idx_b lie in
// [0, n_slots) and are distinct.  A violation ORs kDevBadSlot into the device status
// word.  With wait, the stream is synchronised and the first bad position (or -1)
// and the first repeated pair (or -1, -1) are returned, with the value found at
// the first of them.
cudaError_t check_slots(const int32_t* idx_a, int na, const int32_t* idx_b, int nb, int n_slots, cudaStream_t st,
                        bool wait, long long* bad_range, long long* dup_i, long long* dup_j, int32_t* value);

// read and clear the device status word of each kernel file (synchronous)
cudaError_t take_device_status_decode(unsigned* out);
cudaError_t take_device_status_prefill(unsigned* out);
cudaError_t take_device_status_chunk16(unsigned* out);
cudaError_t take_device_status_proj(unsigned* out);

}  // namespace gdn
