/*
 * gdn.h -- C ABI of libgdn, a GB300 (sm_103a) implementation of the Gated
 * DeltaNet linear-attention layer of hybrid Qwen3.5/3.6-style models.
 *
 * The layer, per token and per v-head j (k-head h = floor(j / G), G = H_v/H_k):
 *   u   = silu(causal depthwise conv1d over the [q|k|v] channels)
 *   q^  = q_scale q / sqrt(|q|^2 + l2_eps),   k^ = k / sqrt(|k|^2 + l2_eps)
 *   g   = -exp(A_log_j) softplus(a_j + dt_bias_j),  alpha = exp(g),  beta = sigmoid(b_j)
 *   S   = alpha S (I - beta k^ k^T) + beta v k^T,   o = S q^
 *   y   = norm_w * o / sqrt(mean(o^2) + norm_eps) * silu(z)
 * The pages describe this layer in words: a fixed-size state that a gate
 * partly erases and a delta-rule write corrects ("Hybrid transformers under
 * load: where Gated DeltaNet loses to full attention", braintools.ru,
 * section 3), with the per-layer state stated in bytes in its section 4.1
 * (32 x 128 x 128 fp32 = 2,097,152 B plus a 49,152 B conv part for
 * Qwen3.5-4B) and the wide geometry in "Chapter 6: engine start-up and memory
 * plan" (Strata), section 6.2 (16 k-heads, 48 v-heads, d_conv 4, 10240 conv
 * channels = 2*128*16 + 128*48).
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Every array argument is a DEVICE pointer, except the two structs, which
 *   are read on the host during the call.  The caller owns every buffer,
 *   including the state pools and the workspace; the library keeps no pointer
 *   after the call returns and allocates no memory (Strata chapter 6,
 *   section 6.10: the token path allocates nothing).
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream) and never synchronise.  A failed launch returns
 *   GDN_ERR_CUDA.
 * - Arguments are checked on the host before any launch; on failure nothing is
 *   launched, the status is returned and gdn_last_error() names the argument,
 *   the value found and the value required (Strata chapter 6, sections 6.2
 *   and 6.5: report the tensor, the shape found and the shape required;
 *   refuse with both numbers).
 * - Alignment (GDN_ERR_ALIGN otherwise): 16 bytes for the state pools, s0,
 *   s_final, the conv pools, conv_w, norm_w, the workspace, x and z, and
 *   the y of the prefill calls (these move with bulk or 128-bit copies);
 *   the element size (2 for bf16, 4 for fp32) for a, b, conv_b, dt_bias,
 *   A_log and the y of decode/verify; 4 bytes for int32 arrays.
 * - Layouts are row-major and dense.  "act" means the activation dtype of the
 *   config (bf16 or fp32).  Channel order of x is [q | k | v], head-major:
 *   q of k-head h at h*d_k, k at H_k*d_k + h*d_k, v of v-head j at
 *   2*H_k*d_k + j*d_v.  C_ch = 2*H_k*d_k + H_v*d_v.
 * - State pool: float [n_slots][H_v][d_v][d_k], one fp32 state per slot,
 *   updated in place.  Conv pool: act [n_slots][d_conv-1][C_ch], the last
 *   d_conv-1 raw (pre-conv) inputs of the slot, oldest first.
 * - Slot indices are read on the device.  An index outside [0, n_slots) is
 *   skipped by the kernels (nothing is read or written for that entry; its y
 *   rows are left as they were).  Duplicate slots within one call race and
 *   give undefined results.
 * - Debug mode: with the environment variable GDN_DEBUG set (and not "0"),
 *   gdn_decode_step, gdn_verify_rows(_nosnap), gdn_commit_rows(_recompute) and
 *   gdn_varlen_prefill(_ckpt) first check their slot indices on the device
 *   (slot_idx, and snap_idx where the call takes one, together): every index
 *   in [0, n_slots) and no index twice.  Unless the stream is being captured,
 *   the call waits for the check and returns GDN_ERR_RANGE naming the first
 *   offending position and value (the refusal convention above, Strata
 *   chapter 6, sections 6.2 and 6.5).  Under stream capture it cannot wait:
 *   the check then only sets GDN_DEV_BAD_SLOT in the device status.  The
 *   check never traps.  It costs one extra small launch and a host wait per
 *   call, so it is off by default.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL = -1,        /* a required pointer is NULL */
    GDN_ERR_SHAPE = -2,       /* a size or geometry field is invalid */
    GDN_ERR_DTYPE = -3,       /* unknown act_dtype */
    GDN_ERR_ALIGN = -4,       /* a pointer is misaligned for its use */
    GDN_ERR_RANGE = -5,       /* a host-side count or index is out of range */
    GDN_ERR_WORKSPACE = -6,   /* workspace too small (both sizes in gdn_last_error) */
    GDN_ERR_UNSUPPORTED = -7, /* valid but not implemented (e.g. d_k != d_v) */
    GDN_ERR_CUDA = -8         /* a CUDA call failed (message in gdn_last_error) */
} gdn_status;

/* activation dtype of x, z, a, b, y, conv weights/bias, norm weight, conv states */
enum { GDN_DTYPE_BF16 = 0, GDN_DTYPE_F32 = 1 };

/* flags: switch steps off so that closed forms can be checked on the GPU */
enum {
    GDN_FLAG_RAW_QKV = 1u,      /* x already holds [q|k|v]: no conv, no SiLU */
    GDN_FLAG_NO_L2NORM = 2u,    /* q^ = q_scale q, k^ = k */
    GDN_FLAG_GATES_DIRECT = 4u, /* a holds g = log(alpha) <= 0, b holds beta */
    GDN_FLAG_NO_OUTNORM = 8u    /* y = o */
};

/* op codes for gdn_workspace_size */
enum {
    GDN_OP_CONV_STATE_UPDATE = 0,
    GDN_OP_DECODE_STEP = 1,
    GDN_OP_VERIFY_ROWS = 2,
    GDN_OP_CHUNK_PREFILL = 3,
    GDN_OP_VARLEN_PREFILL = 4,
    GDN_OP_LAYER_DECODE = 5,         /* gdn_layer_workspace_size only: gdn_layer_decode, n_tokens = B */
    GDN_OP_LAYER_VARLEN_PREFILL = 6  /* gdn_layer_workspace_size only: gdn_layer_varlen_prefill */
};

/* Layer geometry and options.  Requirements (GDN_ERR_SHAPE otherwise):
 * n_k_heads >= 1, n_v_heads % n_k_heads == 0, G = n_v_heads/n_k_heads <= 8
 * (G > 8: GDN_ERR_UNSUPPORTED), n_v_heads <= 4096 (GDN_ERR_UNSUPPORTED otherwise:
 * it keeps every channel count and grid dimension in range),
 * d_k = d_v in {32, 64, 128} (d_k != d_v: GDN_ERR_UNSUPPORTED),
 * 2 <= d_conv <= 4, chunk in {16, 32, 64} (prefill only). */
typedef struct gdn_config {
    int32_t n_k_heads, n_v_heads, d_k, d_v, d_conv, chunk;
    int32_t act_dtype;                 /* GDN_DTYPE_* */
    float q_scale, l2_eps, norm_eps;   /* 1.0, 1e-6, 1e-6 are the defaults */
    uint32_t flags;                    /* GDN_FLAG_* */
} gdn_config;

/* Per-layer parameters (device pointers). */
typedef struct gdn_params {
    const void* conv_w;   /* act [C_ch][d_conv]; tap d_conv-1 multiplies the current token */
    const void* conv_b;   /* act [C_ch] or NULL (no bias) */
    const float* A_log;   /* [H_v] */
    const float* dt_bias; /* [H_v] or NULL (zero) */
    const void* norm_w;   /* act [d_v], shared by all v-heads */
} gdn_params;

/* Causal conv1d + SiLU over all C_ch channels for n_seq sequences of n_tok
 * tokens each, continuing from and updating each sequence's conv state.
 *   x       act [n_seq*n_tok][C_ch]  (sequence-major)
 *   u_out   act [n_seq*n_tok][C_ch]  silu(conv(x)); may be NULL to only roll the state
 *   conv_pool act [n_slots][d_conv-1][C_ch], read and written in place
 *   slot_idx int32 [n_seq]
 * The conv part of the layer state is "the conv part" of section 4.1 of the
 * braintools.ru page (3 raw rows of 8192 bf16 channels = 49,152 B). */
gdn_status gdn_conv_state_update(const gdn_config* cfg, const gdn_params* prm, const void* x,
                                 void* conv_pool, const int32_t* slot_idx, int32_t n_seq,
                                 int32_t n_tok, int32_t n_slots, void* u_out, void* stream);

/* One decode step: one token for each of B slots, state read once and written
 * back in place (one pass over the state: "Forge: how I wrote my own inference
 * engine", entry of 25-26 August, the single-pass DeltaNet decode kernel).
 *   x act [B][C_ch], z act [B][H_v*d_v], a, b act [B][H_v], y act [B][H_v*d_v]
 *   slot_idx int32 [B]; state_pool and conv_pool updated in place. */
gdn_status gdn_decode_step(const gdn_config* cfg, const gdn_params* prm, const void* x,
                           const void* z, const void* a, const void* b, void* conv_pool,
                           float* state_pool, const int32_t* slot_idx, int32_t B,
                           int32_t n_slots, void* y, void* stream);

/* Speculative-decoding verify: r rows (draft tokens) per slot, processed in
 * sequence with the state kept on chip; the state and conv state after row i
 * are written to pool slot snap_idx[b][i] ("Forge ...", entry of 27 August:
 * verify of k tokens is a k-row chunk, DeltaNet runs through sequential rows,
 * with shadow snapshots between rows so that rollback is a copy).  The slot
 * slot_idx[b] itself is read, not written (unless it appears in snap_idx).
 * Accepting a rows selects snap_idx[b][a-1] (a = 0 keeps slot_idx[b]): remap
 * the slot table on the host, or copy with gdn_commit_rows.
 *   x act [B][r][C_ch], z act [B][r][H_v*d_v], a, b act [B][r][H_v],
 *   y act [B][r][H_v*d_v], slot_idx int32 [B], snap_idx int32 [B][r], 1 <= r <= 16. */
gdn_status gdn_verify_rows(const gdn_config* cfg, const gdn_params* prm, const void* x,
                           const void* z, const void* a, const void* b, void* conv_pool,
                           float* state_pool, const int32_t* slot_idx, const int32_t* snap_idx,
                           int32_t B, int32_t r, int32_t n_slots, void* y, void* stream);

/* Rollback/commit by copy: for each b with accepted[b] >= 1 copies the state
 * and conv state of snap_idx[b][accepted[b]-1] into slot_idx[b]; accepted[b]
 * = 0 leaves slot_idx[b] as it was before the verify.  accepted int32 [B]
 * (device), values outside [0, r] are treated as 0. */
gdn_status gdn_commit_rows(const gdn_config* cfg, void* conv_pool, float* state_pool,
                           const int32_t* slot_idx, const int32_t* snap_idx,
                           const int32_t* accepted, int32_t B, int32_t r, int32_t n_slots,
                           void* stream);

/* Verify without snapshots: the same r rows per slot as gdn_verify_rows and
 * the same y, but no state is written anywhere -- the slot keeps its
 * pre-verify state and conv state.  Paired with gdn_commit_rows_recompute it
 * replaces the r snapshot writes of gdn_verify_rows + gdn_commit_rows by one
 * more read and write of the state: 3 state volumes per slot and verify
 * instead of 1 + r (+2 for the commit copy).  "Forge: how I wrote my own
 * inference engine", 27 August, verifies rows in sequence and rolls back by
 * copying a snapshot; this is the variant that recomputes instead.
 * Arguments as gdn_verify_rows without snap_idx. */
gdn_status gdn_verify_rows_nosnap(const gdn_config* cfg, const gdn_params* prm, const void* x,
                                  const void* z, const void* a, const void* b, void* conv_pool,
                                  float* state_pool, const int32_t* slot_idx, int32_t B, int32_t r,
                                  int32_t n_slots, void* y, void* stream);

/* Commit by recompute: applies the first accepted[b] of the r verified rows
 * of entry b (x, a, b: the inputs given to gdn_verify_rows_nosnap, [B][r]...)
 * to the state and conv state of slot_idx[b], in place; accepted[b] = 0 (or
 * outside [0, r]: clamped) leaves the slot as it is.  The arithmetic and its
 * order are those of the verify, so the committed state equals bit for bit
 * the snapshot gdn_verify_rows would have written after row accepted[b].
 * No y is produced; z is not read.  accepted int32 [B] (device). */
gdn_status gdn_commit_rows_recompute(const gdn_config* cfg, const gdn_params* prm, const void* x,
                                     const void* a, const void* b, void* conv_pool, float* state_pool,
                                     const int32_t* slot_idx, const int32_t* accepted, int32_t B,
                                     int32_t r, int32_t n_slots, void* stream);

/* Chunkwise (WY / UT-transform) prefill of one sequence of T tokens
 * ("Forge ...", entry of 25-26 August: a chunked DeltaNet prefill kernel with
 * deterministic reduction).  Results equal the token-by-token evaluation
 * (Strata chapter 6, section 6.9: prefill is the decode path one token at a
 * time) up to rounding; the reduction order is fixed, so results are
 * bitwise reproducible.
 *   x act [T][C_ch], z act [T][H_v*d_v], a, b act [T][H_v], y act [T][H_v*d_v]
 *   s0 float [H_v][d_v][d_k] or NULL (zeros); s_final float [H_v][d_v][d_k]
 *   (may equal s0); conv0 act [d_conv-1][C_ch] or NULL (zeros); conv_final
 *   act [d_conv-1][C_ch] (may equal conv0).
 *   workspace: at least gdn_workspace_size(cfg, GDN_OP_CHUNK_PREFILL, T, 1) bytes. */
gdn_status gdn_chunk_prefill(const gdn_config* cfg, const gdn_params* prm, const void* x,
                             const void* z, const void* a, const void* b, int64_t T,
                             const float* s0, const void* conv0, float* s_final, void* conv_final,
                             void* y, void* workspace, size_t ws_bytes, void* stream);

/* Packed variable-length prefill: n_seq sequences back to back, sequence s
 * covering tokens [cu_seqlens[s], cu_seqlens[s+1]).  Chunks restart at each
 * sequence start; sequence s reads its initial state and conv state from pool
 * slot slot_idx[s] when has_init[s] != 0 (zeros otherwise, or always when
 * has_init is NULL) and writes its final ones there.
 *   x act [n_tokens][C_ch], z, y act [n_tokens][H_v*d_v], a, b act [n_tokens][H_v]
 *   cu_seqlens int32 [n_seq+1] (device; 0 = cu_seqlens[0] <= ... <= cu_seqlens[n_seq]
 *   = n_tokens; out-of-range entries are clamped into [0, n_tokens])
 *   slot_idx int32 [n_seq], has_init uint8 [n_seq] or NULL.
 *   workspace: gdn_workspace_size(cfg, GDN_OP_VARLEN_PREFILL, n_tokens, n_seq) bytes. */
gdn_status gdn_varlen_prefill(const gdn_config* cfg, const gdn_params* prm, const void* x,
                              const void* z, const void* a, const void* b,
                              const int32_t* cu_seqlens, int32_t n_seq, int64_t n_tokens,
                              const int32_t* slot_idx, const uint8_t* has_init, void* conv_pool,
                              float* state_pool, int32_t n_slots, void* y, void* workspace,
                              size_t ws_bytes, void* stream);

/* gdn_varlen_prefill that also leaves snapshots of the recurrent state every
 * ckpt_every tokens of each sequence, for prefix reuse ("Hybrid transformers
 * under load ...", braintools.ru, section 3: a request that shares a prefix
 * with an earlier one resumes from a copy of the state saved at the prefix
 * end, since the live state has moved on; section 4.2: a snapshot at every
 * block boundary, state and conv state of every layer).
 *   Snapshot k (k = 0, 1, ...) of sequence s is the state after its first
 *   (k+1)*ckpt_every tokens (an initial state read from the pool counts as the
 *   state before token 0).  It goes to pool slot ckpt_slots[ckpt_offset[s] + k]
 *   for k < ckpt_offset[s+1] - ckpt_offset[s] and k < floor(L_s / ckpt_every);
 *   later boundaries are not written.  The slot receives what a slot holds
 *   after a prefill ending there -- the fp32 state of every v-head and the conv
 *   state (the d_conv-1 raw inputs before the boundary) -- so a decode, verify
 *   or prefill can resume from it.
 *   ckpt_every: a positive multiple of cfg->chunk, else GDN_ERR_RANGE.
 *   ckpt_offset int32 [n_seq+1] (device, non-decreasing), ckpt_slots int32
 *   [ckpt_offset[n_seq]] (device).  Snapshot slots must differ from one another
 *   and from every slot_idx[s] (the sequences' own slots are read while the
 *   snapshots are written); indices outside [0, n_slots) are skipped.
 *   All other arguments, the workspace and the errors are gdn_varlen_prefill's. */
gdn_status gdn_varlen_prefill_ckpt(const gdn_config* cfg, const gdn_params* prm, const void* x,
                                   const void* z, const void* a, const void* b,
                                   const int32_t* cu_seqlens, int32_t n_seq, int64_t n_tokens,
                                   const int32_t* slot_idx, const uint8_t* has_init,
                                   void* conv_pool, float* state_pool, int32_t n_slots, void* y,
                                   int32_t ckpt_every, const int32_t* ckpt_offset,
                                   const int32_t* ckpt_slots, void* workspace, size_t ws_bytes,
                                   void* stream);

/* Chunked prefill for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point: it exists for callers that cannot
 * call cudaMalloc when they run a prefill -- a host runtime that owns the
 * whole device memory budget through its own allocator, code running while
 * its stream is captured into a CUDA graph (cudaMalloc/cudaFree are not
 * allowed there), or a latency-critical path that cannot pay for the
 * device-wide synchronisation of cudaFree.
 * Same arguments and results as gdn_chunk_prefill, minus the workspace: the
 * workspace is a static device array of 64 MiB inside libgdn, held on each
 * device where the library has been used (its module loaded there) until the
 * process exits.  T is limited to what fits:
 * gdn_workspace_size(cfg, GDN_OP_CHUNK_PREFILL, T, 1) <= 64 MiB (1727 tokens
 * at the Qwen3.5-4B geometry); larger T returns GDN_ERR_WORKSPACE with
 * both sizes in gdn_last_error().
 * A call looks up the array's device address (cudaGetSymbolAddress, with the
 * device current) the first time it runs in a CUDA context and caches it under
 * that context's unique id, so a device reset or a new primary context makes the
 * next call look it up again: make the first call in a context before any stream
 * capture.  All calls share the array and it keeps the previous call's contents
 * (nothing in it needs to start at zero); calls that overlap on the GPU race on
 * it.  Nothing here allocates. */
gdn_status gdn_chunk_prefill_noalloc(const gdn_config* cfg, const gdn_params* prm, const void* x,
                                     const void* z, const void* a, const void* b, int64_t T,
                                     const float* s0, const void* conv0, float* s_final,
                                     void* conv_final, void* y, void* stream);

/* ---- The projections either side of the layer -------------------------------
 * The layer's inputs [x | z | a | b] come from one in-projection of the
 * model's hidden states h, and its output y goes back to the model width
 * through one out-projection.  "Forge: how I wrote my own inference engine and
 * overtook llama.cpp" (24 August) measures the matrix projections at 59% of its
 * hybrid prefill, and its opening formulas bound decode by the weight bytes
 * read per token over the memory bandwidth.  These calls run them on the
 * tensor cores (tcgen05, bf16 operands, fp32 accumulation, the bf16 result
 * rounded to nearest even) and chain them with the layer. */

/* out[t][n] = sum_k act[t][k] * w[n][k] for t < n_tok, n < n_out (w in the
 * nn.Linear layout [n_out][k]).
 *   act bf16 [n_tok][k] and w bf16 [n_out][k], dense, 16-byte aligned;
 *   out bf16 with rows of ld_out >= n_out elements, 2-byte aligned.
 *   k: a positive multiple of 8 (rows start on 16-byte boundaries);
 *   n_out >= 1; 0 <= n_tok < 2^31 (0: nothing to do).
 *   workspace: gdn_proj_workspace_size(n_tok, n_out, k) bytes, 16-byte
 *   aligned (NULL when that is 0).  With few tokens (up to 256) and few
 *   128-row blocks of w, K is split over several CTAs per block whose fp32
 *   partial sums meet in the workspace; the sums are added in a fixed order,
 *   so results do not change from call to call. */
gdn_status gdn_proj_gemm(const void* act, const void* w, void* out, int64_t n_tok, int32_t n_out,
                         int32_t k, int64_t ld_out, void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes of gdn_proj_gemm for these sizes (0: none needed or invalid
 * sizes).  Depends on the sizes only. */
size_t gdn_proj_workspace_size(int64_t n_tok, int32_t n_out, int32_t k);

/* Projection weights of one layer (device pointers, bf16, row-major). */
typedef struct gdn_proj {
    const void* w_in;   /* [C_ch + 2*H_v + H_v*d_v][hidden]: the rows of x (C_ch), then
                           z (H_v*d_v), then a (H_v), then b (H_v) */
    const void* w_out;  /* [hidden][H_v*d_v] */
    int32_t hidden;     /* model width: a positive multiple of 8 */
} gdn_proj;

/* One decode step of the whole layer for B slots: [x|z|a|b] = h w_in^T, the
 * step of gdn_decode_step on them, out = y w_out^T.
 *   h, out bf16 [B][hidden]; conv_pool, state_pool, slot_idx, B, n_slots as in
 *   gdn_decode_step.  act_dtype must be GDN_DTYPE_BF16 (else
 *   GDN_ERR_UNSUPPORTED).
 *   workspace: gdn_layer_workspace_size(cfg, GDN_OP_LAYER_DECODE, B, 1,
 *   proj->hidden) bytes; it holds x, z, a, b and y of the B tokens (bf16)
 *   between the three steps and the projections' partial sums. */
gdn_status gdn_layer_decode(const gdn_config* cfg, const gdn_params* prm, const gdn_proj* proj,
                            const void* h, void* conv_pool, float* state_pool,
                            const int32_t* slot_idx, int32_t B, int32_t n_slots, void* out,
                            void* workspace, size_t ws_bytes, void* stream);

/* The whole layer over packed sequences: in-projection, gdn_varlen_prefill,
 * out-projection.  h, out bf16 [n_tokens][hidden]; the other arguments as in
 * gdn_varlen_prefill; act_dtype must be GDN_DTYPE_BF16.
 *   workspace: gdn_layer_workspace_size(cfg, GDN_OP_LAYER_VARLEN_PREFILL,
 *   n_tokens, n_seq, proj->hidden) bytes: x, z, a, b, y of the tokens, the
 *   projections' partial sums and the prefill's own workspace. */
gdn_status gdn_layer_varlen_prefill(const gdn_config* cfg, const gdn_params* prm,
                                    const gdn_proj* proj, const void* h,
                                    const int32_t* cu_seqlens, int32_t n_seq, int64_t n_tokens,
                                    const int32_t* slot_idx, const uint8_t* has_init,
                                    void* conv_pool, float* state_pool, int32_t n_slots, void* out,
                                    void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes an op needs for n_tokens tokens in n_seq sequences (0 for
 * the ops that need none).  Returns 0 and sets gdn_last_error on an invalid
 * config. */
size_t gdn_workspace_size(const gdn_config* cfg, int32_t op, int64_t n_tokens, int32_t n_seq);

/* ---- Decode attention of the hybrid's full-attention layers ------------------
 * The hybrid's other layers are ordinary grouped-query attention over a KV
 * cache ("Forge: how I wrote my own inference engine and overtook llama.cpp",
 * its architecture section: 16 of 64 layers GQA attention, 4 kv-heads of 256
 * dims; its 25-26 August entry: split-KV decode, the query heads of a kv-head
 * packed together so that each kv-head is read once).  The cache is paged: a
 * page holds the K and V of page_size tokens of one layer ("Hybrid
 * transformers under load ...", braintools.ru, section 4.1: 4 kv-heads x 256
 * bf16 values per token for Qwen3.5-4B).  Query head h reads kv-head
 * floor(h / G), G = n_q_heads / n_kv_heads. */
typedef struct gdn_attn_config {
    int32_t n_q_heads, n_kv_heads; /* G = n_q_heads / n_kv_heads in {1, 2} or a multiple of 4 up to 32 */
    int32_t head_dim;              /* 128 or 256 */
    int32_t page_size;             /* tokens per page: a multiple of 8, 8 .. 4096 */
    float scale;                   /* softmax scale; 0 means 1 / sqrt(head_dim) */
} gdn_attn_config;

/* One decode step for B sequences: sequence b holds seq_lens[b] tokens in the
 * cache; its new token (q, k_new, v_new) is appended at position seq_lens[b]
 * and attends to all seq_lens[b] + 1 tokens:
 *   o[b][h] = softmax_t(scale q[b][h] . K[b][t][kvh]) V[b][t][kvh], kvh = floor(h / G).
 *   q, o bf16 [B][n_q_heads][head_dim]; k_new, v_new bf16 [B][n_kv_heads][head_dim]
 *   k_pool, v_pool bf16 [n_pages][n_kv_heads][page_size][head_dim]: token t of
 *   sequence b sits on page block_table[b][t / page_size] at row t % page_size.
 *   block_table int32 [B][max_pages]; seq_lens int32 [B] (device).
 *   max_seq_len: host bound on every seq_lens[b] + 1 (tokens past it are left out).
 *   A token whose page index is outside [0, n_pages) is left out of the
 *   softmax; a sequence with seq_lens[b] < 0 or seq_lens[b] >= max_pages *
 *   page_size is skipped (nothing read or written, its o rows left as they
 *   were).  The page receiving a new token must belong to that sequence alone
 *   (pages shared between sequences are read only).
 *   workspace: gdn_attn_workspace_size(cfg, B, max_seq_len) bytes (the
 *   partial results of the context splits; NULL when 0).
 *   All pointers 16-byte aligned.  bf16 in, fp32 softmax and accumulation,
 *   bf16 out.  With G = 8, 12 or 16 the two products run on the tensor cores:
 *   q scale is rounded to bf16 before Q K^T and the softmax weights to bf16
 *   before P V (fp32 accumulation in both). */
gdn_status gdn_attn_decode(const gdn_attn_config* cfg, const void* q, const void* k_new,
                           const void* v_new, void* k_pool, void* v_pool,
                           const int32_t* block_table, const int32_t* seq_lens, int32_t B,
                           int32_t max_pages, int32_t n_pages, int32_t max_seq_len, void* o,
                           void* workspace, size_t ws_bytes, void* stream);

/* Prefill (chunk) attention: sequence s brings n_s = cu_seqlens[s+1] -
 * cu_seqlens[s] new tokens at positions ctx_lens[s] .. ctx_lens[s] + n_s - 1.
 * Their K and V are appended to the pages, and new token i attends causally to
 * the sequence's positions 0 .. ctx_lens[s] + i (forge, 27 August: a chunk of k
 * tokens is a prefill with the mask aligned at the bottom right, row i sees
 * 0 .. kv0 + i).
 *   q, o bf16 [n_tokens][n_q_heads][head_dim]; k_new, v_new bf16
 *   [n_tokens][n_kv_heads][head_dim]; pools and block_table as in
 *   gdn_attn_decode (block_table [n_seq][max_pages]); cu_seqlens int32
 *   [n_seq+1] (device; 0 = cu_seqlens[0] <= ... = n_tokens); ctx_lens int32
 *   [n_seq] (device).  A sequence whose pages would run past max_pages, or
 *   with ctx_lens[s] < 0, is skipped; tokens on pages outside [0, n_pages) are
 *   left out of the softmax.  Same alignment and precision as gdn_attn_decode;
 *   S = Q K^T and O = P V run on the tensor cores (bf16 operands, fp32
 *   accumulation), P is rounded to bf16.  No workspace. */
gdn_status gdn_attn_prefill(const gdn_attn_config* cfg, const void* q, const void* k_new,
                            const void* v_new, void* k_pool, void* v_pool,
                            const int32_t* block_table, const int32_t* cu_seqlens,
                            const int32_t* ctx_lens, int32_t n_seq, int64_t n_tokens,
                            int32_t max_pages, int32_t n_pages, void* o, void* stream);

/* Workspace bytes of gdn_attn_decode (depends on the sizes only; 0 on invalid
 * arguments, with gdn_last_error set). */
size_t gdn_attn_workspace_size(const gdn_attn_config* cfg, int32_t B, int32_t max_seq_len);

/* Workspace bytes of gdn_layer_decode (op GDN_OP_LAYER_DECODE, n_tokens = B)
 * or gdn_layer_varlen_prefill (op GDN_OP_LAYER_VARLEN_PREFILL) for a model
 * width `hidden`.  Returns 0 and sets gdn_last_error on invalid arguments. */
size_t gdn_layer_workspace_size(const gdn_config* cfg, int32_t op, int64_t n_tokens, int32_t n_seq,
                                int32_t hidden);

/* Message of the last failed call on this host thread ("" if none).  The
 * string stays valid until the next call on this thread. */
const char* gdn_last_error(void);

/* Device-side status: every wait inside the kernels is bounded (about one
 * second); a kernel whose wait gives up skips its remaining work, leaves its
 * outputs incomplete and ORs a code into a status word on the device instead
 * of hanging.  This call reads and clears that word for the current device
 * (*status = 0: nothing reported; bit GDN_DEV_WAIT_TIMEOUT: a wait gave up;
 * bit GDN_DEV_BAD_SLOT: a GDN_DEBUG slot check found a bad or repeated index).
 * It synchronises the current device. */
enum { GDN_DEV_WAIT_TIMEOUT = 1u, GDN_DEV_BAD_SLOT = 2u };
gdn_status gdn_device_status(uint32_t* status);

/* Library version string. */
const char* gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
