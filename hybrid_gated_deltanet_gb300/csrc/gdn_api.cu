// gdn_api.cu -- the exported C ABI of libgdn (see include/gdn.h).
//
// Every entry point validates its arguments on the host, then launches on the
// caller's stream.  Nothing here allocates device memory or synchronises.
// Error messages follow the Strata convention (chapter 6, sections 6.2 and
// 6.5): name the argument, the value found and the value required.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

thread_local std::string g_last_error;

gdn_status fail(gdn_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

gdn_status ok() {
    g_last_error.clear();
    return GDN_OK;
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1u)) == 0; }

// State buffers and the workspace are moved with 128-bit accesses (16-byte
// alignment); activation arrays, parameters and index arrays need their
// element alignment (`al` below: 2 for bf16, 4 otherwise).
#define GDN_PTR_ALIGN(p, name, al)                                                           \
    do {                                                                                     \
        if (!aligned((p), (al)))                                                             \
            return fail(GDN_ERR_ALIGN, "%s: found address %p, required %u-byte alignment", name, \
                        (const void*)(p), (unsigned)(al));                                   \
    } while (0)

#define GDN_REQUIRE_PTR_A(p, name, al)                                                        \
    do {                                                                                     \
        if (!(p)) return fail(GDN_ERR_NULL, "%s: found NULL, required a device pointer", name); \
        GDN_PTR_ALIGN(p, name, al);                                                          \
    } while (0)

#define GDN_OPTIONAL_PTR_A(p, name, al)                                                       \
    do {                                                                                     \
        if (p) GDN_PTR_ALIGN(p, name, al);                                                   \
    } while (0)

#define GDN_REQUIRE_PTR(p, name) GDN_REQUIRE_PTR_A(p, name, 16u)
#define GDN_OPTIONAL_PTR(p, name) GDN_OPTIONAL_PTR_A(p, name, 16u)

gdn_status make_geom(const gdn_config* cfg, bool need_chunk, gdn::Geom* g) {
    if (!cfg) return fail(GDN_ERR_NULL, "cfg: found NULL, required a gdn_config");
    if (cfg->act_dtype != GDN_DTYPE_BF16 && cfg->act_dtype != GDN_DTYPE_F32)
        return fail(GDN_ERR_DTYPE, "cfg.act_dtype: found %d, required GDN_DTYPE_BF16 (0) or GDN_DTYPE_F32 (1)",
                    cfg->act_dtype);
    if (cfg->n_k_heads < 1 || cfg->n_v_heads < 1)
        return fail(GDN_ERR_SHAPE, "cfg.n_k_heads/n_v_heads: found %d/%d, required >= 1", cfg->n_k_heads,
                    cfg->n_v_heads);
    if (cfg->n_v_heads % cfg->n_k_heads != 0)
        return fail(GDN_ERR_SHAPE, "cfg.n_v_heads: found %d, required a multiple of n_k_heads = %d",
                    cfg->n_v_heads, cfg->n_k_heads);
    if (cfg->n_v_heads > 4096)
        return fail(GDN_ERR_UNSUPPORTED, "cfg.n_v_heads: found %d, required <= 4096", cfg->n_v_heads);
    const int G = cfg->n_v_heads / cfg->n_k_heads;
    if (G > 8) return fail(GDN_ERR_UNSUPPORTED, "cfg.n_v_heads/n_k_heads: found %d, required <= 8", G);
    if (cfg->d_k != 32 && cfg->d_k != 64 && cfg->d_k != 128)
        return fail(GDN_ERR_SHAPE, "cfg.d_k: found %d, required 32, 64 or 128", cfg->d_k);
    if (cfg->d_v != 32 && cfg->d_v != 64 && cfg->d_v != 128)
        return fail(GDN_ERR_SHAPE, "cfg.d_v: found %d, required 32, 64 or 128", cfg->d_v);
    if (cfg->d_k != cfg->d_v)
        return fail(GDN_ERR_UNSUPPORTED, "cfg.d_v: found %d, required d_v == d_k = %d", cfg->d_v, cfg->d_k);
    if (cfg->d_conv < 2 || cfg->d_conv > 4)
        return fail(GDN_ERR_SHAPE, "cfg.d_conv: found %d, required 2..4", cfg->d_conv);
    if (need_chunk && cfg->chunk != 16 && cfg->chunk != 32 && cfg->chunk != 64)
        return fail(GDN_ERR_SHAPE, "cfg.chunk: found %d, required 16, 32 or 64", cfg->chunk);
    if (!(cfg->l2_eps >= 0.f) || !(cfg->norm_eps >= 0.f))
        return fail(GDN_ERR_SHAPE, "cfg.l2_eps/norm_eps: found %g/%g, required >= 0", (double)cfg->l2_eps,
                    (double)cfg->norm_eps);
    if (cfg->flags & ~15u) return fail(GDN_ERR_SHAPE, "cfg.flags: found 0x%x, required a subset of 0xf", cfg->flags);
    g->Hk = cfg->n_k_heads;
    g->Hv = cfg->n_v_heads;
    g->D = cfg->d_k;
    g->K = cfg->d_conv;
    g->G = G;
    g->C_ch = 2 * cfg->n_k_heads * cfg->d_k + cfg->n_v_heads * cfg->d_v;
    g->chunk = cfg->chunk;
    g->act_bf16 = cfg->act_dtype == GDN_DTYPE_BF16;
    g->q_scale = cfg->q_scale;
    g->l2_eps = cfg->l2_eps;
    g->norm_eps = cfg->norm_eps;
    g->flags = cfg->flags;
    return GDN_OK;
}

gdn_status make_params(const gdn_params* prm, const gdn::Geom& g, bool need_all, gdn::LayerParams* p) {
    if (!prm) return fail(GDN_ERR_NULL, "prm: found NULL, required a gdn_params");
    const bool conv = !(g.flags & GDN_FLAG_RAW_QKV);
    const bool gates = !(g.flags & GDN_FLAG_GATES_DIRECT);
    const bool norm = !(g.flags & GDN_FLAG_NO_OUTNORM);
    const unsigned ae = g.act_bf16 ? 2u : 4u;
    if (conv || !need_all) GDN_REQUIRE_PTR(prm->conv_w, "prm.conv_w");
    else GDN_OPTIONAL_PTR(prm->conv_w, "prm.conv_w");
    GDN_OPTIONAL_PTR_A(prm->conv_b, "prm.conv_b", ae);
    if (need_all && gates) GDN_REQUIRE_PTR_A(prm->A_log, "prm.A_log", 4u);
    else GDN_OPTIONAL_PTR_A(prm->A_log, "prm.A_log", 4u);
    GDN_OPTIONAL_PTR_A(prm->dt_bias, "prm.dt_bias", 4u);
    if (need_all && norm) GDN_REQUIRE_PTR(prm->norm_w, "prm.norm_w");
    else GDN_OPTIONAL_PTR(prm->norm_w, "prm.norm_w");
    p->conv_w = prm->conv_w;
    p->conv_b = prm->conv_b;
    p->A_log = prm->A_log;
    p->dt_bias = prm->dt_bias;
    p->norm_w = prm->norm_w;
    return GDN_OK;
}

gdn_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(GDN_ERR_CUDA, "%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
}

}  // namespace

namespace gdn {
// Lets another translation unit of the library report a failure through
// gdn_last_error (same thread-local message as the entry points here).
int report_error(int status, const char* message) {
    g_last_error = message;
    return status;
}

int sm_count() {
    static std::atomic<int> cache[64];  // static storage: zero, i.e. not yet queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::atomic<int>& c = cache[dev & 63];
    int n = c.load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
        c.store(n, std::memory_order_relaxed);
    }
    return n;
}
}  // namespace gdn

extern "C" {

const char* gdn_last_error(void) { return g_last_error.c_str(); }

const char* gdn_version(void) { return "libgdn 0.1 (sm_103a)"; }

gdn_status gdn_device_status(uint32_t* status) {
    if (!status) return fail(GDN_ERR_NULL, "status: found NULL, required a host pointer");
    unsigned a = 0, b = 0;
    unsigned c = 0, d = 0;
    cudaError_t e = gdn::take_device_status_decode(&a);
    if (e == cudaSuccess) e = gdn::take_device_status_prefill(&b);
    if (e == cudaSuccess) e = gdn::take_device_status_proj(&c);
    if (e == cudaSuccess) e = gdn::take_device_status_chunk16(&d);
    *status = a | b | c | d;
    return cuda_status(e, "gdn_device_status");
}

// the in-projection's outputs and y of n tokens (bf16) and the projections'
// split-K partial sums, each on a 256-byte boundary; a layer prefill's own
// workspace follows at `rest`
struct LayerWs {
    size_t x, z, a, b, y, part, rest;
};
static LayerWs layer_ws(const gdn::Geom& g, int64_t n, int32_t hidden) {
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t t = (size_t)(n > 0 ? n : 0);
    LayerWs L;
    size_t o = 0;
    L.x = o; o += al(t * g.C_ch * 2);
    L.z = o; o += al(t * g.Hv * g.D * 2);
    L.a = o; o += al(t * g.Hv * 2);
    L.b = o; o += al(t * g.Hv * 2);
    L.y = o; o += al(t * g.Hv * g.D * 2);
    // split-K partial sums of either projection (they run one after the other)
    const size_t p_in = gdn::proj_plan(g.C_ch + g.Hv * g.D + 2 * g.Hv, hidden, n).ws_bytes;
    const size_t p_out = gdn::proj_plan(hidden, g.Hv * g.D, n).ws_bytes;
    L.part = o; o += al(p_in > p_out ? p_in : p_out);
    L.rest = o;
    return L;
}

size_t gdn_proj_workspace_size(int64_t n_tok, int32_t n_out, int32_t k) {
    if (n_tok < 0 || n_out < 1 || k < 1) return 0;
    return gdn::proj_plan(n_out, k, n_tok).ws_bytes;
}

size_t gdn_layer_workspace_size(const gdn_config* cfg, int32_t op, int64_t n_tokens, int32_t n_seq, int32_t hidden) {
    gdn::Geom g;
    const bool prefill = op == GDN_OP_LAYER_VARLEN_PREFILL;
    if (op != GDN_OP_LAYER_DECODE && !prefill) {
        fail(GDN_ERR_RANGE, "op: found %d, required GDN_OP_LAYER_DECODE (5) or GDN_OP_LAYER_VARLEN_PREFILL (6)", op);
        return 0;
    }
    if (make_geom(cfg, prefill, &g) != GDN_OK) return 0;
    if (n_tokens < 0 || n_seq < 0 || hidden < 8 || hidden % 8 != 0) {
        fail(GDN_ERR_RANGE, "n_tokens/n_seq/hidden: found %lld/%d/%d, required >= 0/>= 0/a positive multiple of 8",
             (long long)n_tokens, n_seq, hidden);
        return 0;
    }
    ok();
    const size_t base = layer_ws(g, n_tokens, hidden).rest;
    return prefill ? base + gdn::prefill_workspace_bytes(g, n_tokens, n_seq) : base;
}

size_t gdn_workspace_size(const gdn_config* cfg, int32_t op, int64_t n_tokens, int32_t n_seq) {
    gdn::Geom g;
    const bool prefill = op == GDN_OP_CHUNK_PREFILL || op == GDN_OP_VARLEN_PREFILL;
    if (make_geom(cfg, prefill, &g) != GDN_OK) return 0;
    if (n_tokens < 0 || n_seq < 0) {
        fail(GDN_ERR_RANGE, "n_tokens/n_seq: found %lld/%d, required >= 0", (long long)n_tokens, n_seq);
        return 0;
    }
    ok();
    if (!prefill) return 0;
    return gdn::prefill_workspace_bytes(g, n_tokens, op == GDN_OP_CHUNK_PREFILL ? 1 : n_seq);
}

gdn_status gdn_conv_state_update(const gdn_config* cfg, const gdn_params* prm, const void* x, void* conv_pool,
                                 const int32_t* slot_idx, int32_t n_seq, int32_t n_tok, int32_t n_slots,
                                 void* u_out, void* stream) {
    gdn::Geom g;
    gdn::LayerParams p;
    gdn_status st = make_geom(cfg, false, &g);
    if (st) return st;
    if (n_seq < 0 || n_tok < 0 || n_slots < 1)
        return fail(GDN_ERR_RANGE, "n_seq/n_tok/n_slots: found %d/%d/%d, required >= 0/>= 0/>= 1", n_seq, n_tok,
                    n_slots);
    if (n_seq > 0 && n_tok > 0) {
        if ((st = make_params(prm, g, false, &p))) return st;
        GDN_REQUIRE_PTR_A(x, "x", g.act_bf16 ? 2u : 4u);
        GDN_REQUIRE_PTR(conv_pool, "conv_pool");
        GDN_REQUIRE_PTR_A(slot_idx, "slot_idx", 4u);
        GDN_OPTIONAL_PTR_A(u_out, "u_out", g.act_bf16 ? 2u : 4u);
    } else {
        return ok();
    }
    gdn::ConvJob job{x, conv_pool, slot_idx, u_out, n_seq, n_tok, n_slots};
    return cuda_status(gdn::launch_conv_update(g, p, job, (cudaStream_t)stream), "gdn_conv_state_update");
}

// GDN_DEBUG set (and not "0"): slot indices are checked on the device before the
// call's kernels; unless the stream is being captured, the call then waits for the
// check and refuses bad indices with GDN_ERR_RANGE (the capture case only sets the
// status bit GDN_DEV_BAD_SLOT for gdn_device_status)
static bool debug_on() {
    const char* e = std::getenv("GDN_DEBUG");
    return e && e[0] && !(e[0] == '0' && e[1] == 0);
}

static gdn_status debug_check_slots(const char* name_a, const int32_t* idx_a, int na, const char* name_b,
                                    const int32_t* idx_b, int nb, int n_slots, void* stream) {
    if (!debug_on() || na + nb == 0) return GDN_OK;
    cudaStream_t st = (cudaStream_t)stream;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cap);
    if (e != cudaSuccess) return cuda_status(e, "GDN_DEBUG slot check");
    long long bad = -1, di = -1, dj = -1;
    int32_t v = 0;
    e = gdn::check_slots(idx_a, na, idx_b, nb, n_slots, st, cap == cudaStreamCaptureStatusNone, &bad, &di, &dj, &v);
    if (e != cudaSuccess) return cuda_status(e, "GDN_DEBUG slot check");
    auto name = [&](long long k) { return k < na ? name_a : name_b; };
    auto pos = [&](long long k) { return k < na ? k : k - na; };
    if (bad >= 0)
        return fail(GDN_ERR_RANGE, "%s[%lld]: found slot %d, required 0..%d (GDN_DEBUG)", name(bad), pos(bad), v,
                    n_slots - 1);
    if (di >= 0)
        return fail(GDN_ERR_RANGE, "%s[%lld] and %s[%lld]: found slot %d twice, required distinct slots (GDN_DEBUG)",
                    name(di), pos(di), name(dj), pos(dj), v);
    return GDN_OK;
}

static gdn_status rows_check(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z,
                             const void* a, const void* b, void* conv_pool, float* state_pool,
                             const int32_t* slot_idx, int32_t B, int32_t r, int32_t n_slots, void* y, int mode,
                             const int32_t* accepted, gdn::Geom* g, gdn::LayerParams* p) {
    gdn_status st = make_geom(cfg, false, g);
    if (st) return st;
    if (B < 0 || B > 65535) return fail(GDN_ERR_RANGE, "B: found %d, required 0..65535", B);
    if (r < 1 || r > 16) return fail(GDN_ERR_RANGE, "r: found %d, required 1..16", r);
    if (n_slots < 1) return fail(GDN_ERR_RANGE, "n_slots: found %d, required >= 1", n_slots);
    if (B == 0) return GDN_OK;
    if ((st = make_params(prm, *g, true, p))) return st;
    GDN_REQUIRE_PTR(x, "x");  // x and z are staged with bulk copies: 16-byte aligned
    if (!(g->flags & GDN_FLAG_NO_OUTNORM) && mode != 2) GDN_REQUIRE_PTR(z, "z");
    GDN_REQUIRE_PTR_A(a, "a", g->act_bf16 ? 2u : 4u);
    GDN_REQUIRE_PTR_A(b, "b", g->act_bf16 ? 2u : 4u);
    GDN_REQUIRE_PTR(conv_pool, "conv_pool");
    GDN_REQUIRE_PTR(state_pool, "state_pool");
    GDN_REQUIRE_PTR_A(slot_idx, "slot_idx", 4u);
    if (mode != 2) GDN_REQUIRE_PTR_A(y, "y", g->act_bf16 ? 2u : 4u);
    else GDN_REQUIRE_PTR_A(accepted, "accepted", 4u);
    return GDN_OK;
}

static gdn_status rows_common(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z,
                              const void* a, const void* b, void* conv_pool, float* state_pool,
                              const int32_t* slot_idx, const int32_t* snap_idx, int32_t B, int32_t r,
                              int32_t n_slots, void* y, void* stream, const char* who, int mode = 0,
                              const int32_t* accepted = nullptr) {
    gdn::Geom g;
    gdn::LayerParams p;
    gdn_status st = rows_check(cfg, prm, x, z, a, b, conv_pool, state_pool, slot_idx, B, r, n_slots, y, mode,
                               accepted, &g, &p);
    if (st) return st;
    if (B == 0) return ok();
    if ((st = debug_check_slots("slot_idx", slot_idx, B, "snap_idx", snap_idx, snap_idx ? B * r : 0, n_slots,
                                stream)))
        return st;
    gdn::RowsJob job{x, z, a, b, conv_pool, state_pool, slot_idx, snap_idx, y, B, r, n_slots};
    job.mode = mode;
    job.accepted = accepted;
    return cuda_status(gdn::launch_rows(g, p, job, (cudaStream_t)stream), who);
}

gdn_status gdn_decode_step(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z, const void* a,
                           const void* b, void* conv_pool, float* state_pool, const int32_t* slot_idx, int32_t B,
                           int32_t n_slots, void* y, void* stream) {
    return rows_common(cfg, prm, x, z, a, b, conv_pool, state_pool, slot_idx, nullptr, B, 1, n_slots, y, stream,
                       "gdn_decode_step");
}

gdn_status gdn_verify_rows(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z, const void* a,
                           const void* b, void* conv_pool, float* state_pool, const int32_t* slot_idx,
                           const int32_t* snap_idx, int32_t B, int32_t r, int32_t n_slots, void* y, void* stream) {
    if (B > 0) GDN_REQUIRE_PTR_A(snap_idx, "snap_idx", 4u);
    return rows_common(cfg, prm, x, z, a, b, conv_pool, state_pool, slot_idx, snap_idx, B, r, n_slots, y, stream,
                       "gdn_verify_rows");
}

gdn_status gdn_verify_rows_nosnap(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z,
                                  const void* a, const void* b, void* conv_pool, float* state_pool,
                                  const int32_t* slot_idx, int32_t B, int32_t r, int32_t n_slots, void* y,
                                  void* stream) {
    return rows_common(cfg, prm, x, z, a, b, conv_pool, state_pool, slot_idx, nullptr, B, r, n_slots, y, stream,
                       "gdn_verify_rows_nosnap", 1);
}

gdn_status gdn_commit_rows_recompute(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* a,
                                     const void* b, void* conv_pool, float* state_pool, const int32_t* slot_idx,
                                     const int32_t* accepted, int32_t B, int32_t r, int32_t n_slots, void* stream) {
    return rows_common(cfg, prm, x, nullptr, a, b, conv_pool, state_pool, slot_idx, nullptr, B, r, n_slots, nullptr,
                       stream, "gdn_commit_rows_recompute", 2, accepted);
}

gdn_status gdn_commit_rows(const gdn_config* cfg, void* conv_pool, float* state_pool, const int32_t* slot_idx,
                           const int32_t* snap_idx, const int32_t* accepted, int32_t B, int32_t r, int32_t n_slots,
                           void* stream) {
    gdn::Geom g;
    gdn_status st = make_geom(cfg, false, &g);
    if (st) return st;
    if (B < 0 || B > 65535) return fail(GDN_ERR_RANGE, "B: found %d, required 0..65535", B);
    if (r < 1 || r > 16) return fail(GDN_ERR_RANGE, "r: found %d, required 1..16", r);
    if (n_slots < 1) return fail(GDN_ERR_RANGE, "n_slots: found %d, required >= 1", n_slots);
    if (B == 0) return ok();
    GDN_REQUIRE_PTR(conv_pool, "conv_pool");
    GDN_REQUIRE_PTR(state_pool, "state_pool");
    GDN_REQUIRE_PTR_A(slot_idx, "slot_idx", 4u);
    GDN_REQUIRE_PTR_A(snap_idx, "snap_idx", 4u);
    GDN_REQUIRE_PTR_A(accepted, "accepted", 4u);
    if ((st = debug_check_slots("slot_idx", slot_idx, B, "snap_idx", snap_idx, B * r, n_slots, stream))) return st;
    gdn::CommitJob job{conv_pool, state_pool, slot_idx, snap_idx, accepted, B, r, n_slots};
    return cuda_status(gdn::launch_commit(g, job, (cudaStream_t)stream), "gdn_commit_rows");
}

static gdn_status prefill_check(const gdn_config* cfg, const gdn_params* prm, const gdn::PrefillJob& job,
                                gdn::Geom* g, gdn::LayerParams* p) {
    gdn_status st = make_geom(cfg, true, g);
    if (st) return st;
    if (job.n_tokens < 0 || job.n_tokens > (int64_t)1 << 31)
        return fail(GDN_ERR_RANGE, "n_tokens: found %lld, required 0..2^31", (long long)job.n_tokens);
    if ((st = make_params(prm, *g, true, p))) return st;
    if (job.n_tokens > 0) {
        GDN_REQUIRE_PTR(job.x, "x");  // x, z, y move in 16-byte vectors
        if (!(g->flags & GDN_FLAG_NO_OUTNORM)) GDN_REQUIRE_PTR(job.z, "z");
        GDN_REQUIRE_PTR_A(job.a, "a", g->act_bf16 ? 2u : 4u);
        GDN_REQUIRE_PTR_A(job.b, "b", g->act_bf16 ? 2u : 4u);
        GDN_REQUIRE_PTR(job.y, "y");
    }
    const size_t need = gdn::prefill_workspace_bytes(*g, job.n_tokens, job.cu_seqlens ? job.n_seq : 1);
    if (need > 0) GDN_REQUIRE_PTR(job.workspace, "workspace");
    if (job.ws_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace: found %zu bytes, required %zu bytes", job.ws_bytes, need);
    return GDN_OK;
}

static gdn_status prefill_common(const gdn_config* cfg, const gdn_params* prm, gdn::PrefillJob& job, void* stream,
                                 const char* who) {
    gdn::Geom g;
    gdn::LayerParams p;
    gdn_status st = prefill_check(cfg, prm, job, &g, &p);
    if (st) return st;
    if (job.slot_idx &&
        (st = debug_check_slots("slot_idx", job.slot_idx, (int)job.n_seq, "", nullptr, 0, job.n_slots, stream)))
        return st;
    return cuda_status(gdn::launch_prefill(g, p, job, (cudaStream_t)stream), who);
}

gdn_status gdn_chunk_prefill(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z, const void* a,
                             const void* b, int64_t T, const float* s0, const void* conv0, float* s_final,
                             void* conv_final, void* y, void* workspace, size_t ws_bytes, void* stream) {
    GDN_OPTIONAL_PTR(s0, "s0");
    GDN_OPTIONAL_PTR(conv0, "conv0");
    GDN_REQUIRE_PTR(s_final, "s_final");
    GDN_REQUIRE_PTR(conv_final, "conv_final");
    GDN_OPTIONAL_PTR(workspace, "workspace");
    gdn::PrefillJob job = {};
    job.x = x; job.z = z; job.a = a; job.b = b; job.y = y;
    job.n_tokens = T;
    job.n_seq = 1;
    job.s0 = s0; job.s_final = s_final; job.conv0 = conv0; job.conv_final = conv_final;
    job.workspace = workspace; job.ws_bytes = ws_bytes;
    return prefill_common(cfg, prm, job, stream, "gdn_chunk_prefill");
}

gdn_status gdn_varlen_prefill(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z, const void* a,
                              const void* b, const int32_t* cu_seqlens, int32_t n_seq, int64_t n_tokens,
                              const int32_t* slot_idx, const uint8_t* has_init, void* conv_pool, float* state_pool,
                              int32_t n_slots, void* y, void* workspace, size_t ws_bytes, void* stream) {
    if (n_seq < 0 || n_seq > 65535) return fail(GDN_ERR_RANGE, "n_seq: found %d, required 0..65535", n_seq);
    if (n_slots < 1) return fail(GDN_ERR_RANGE, "n_slots: found %d, required >= 1", n_slots);
    if (n_seq == 0) {
        if (n_tokens != 0)
            return fail(GDN_ERR_RANGE, "n_tokens: found %lld with n_seq = 0, required 0", (long long)n_tokens);
        gdn::Geom g;
        gdn_status st = make_geom(cfg, true, &g);
        return st ? st : ok();
    }
    GDN_REQUIRE_PTR_A(cu_seqlens, "cu_seqlens", 4u);
    GDN_REQUIRE_PTR_A(slot_idx, "slot_idx", 4u);
    GDN_OPTIONAL_PTR_A(has_init, "has_init", 1u);
    GDN_REQUIRE_PTR(conv_pool, "conv_pool");
    GDN_REQUIRE_PTR(state_pool, "state_pool");
    GDN_OPTIONAL_PTR(workspace, "workspace");
    gdn::PrefillJob job = {};
    job.x = x; job.z = z; job.a = a; job.b = b; job.y = y;
    job.n_tokens = n_tokens;
    job.n_seq = n_seq;
    job.cu_seqlens = cu_seqlens;
    job.slot_idx = slot_idx; job.has_init = has_init;
    job.state_pool = state_pool; job.conv_pool = conv_pool; job.n_slots = n_slots;
    job.workspace = workspace; job.ws_bytes = ws_bytes;
    return prefill_common(cfg, prm, job, stream, "gdn_varlen_prefill");
}

gdn_status gdn_varlen_prefill_ckpt(const gdn_config* cfg, const gdn_params* prm, const void* x, const void* z,
                                   const void* a, const void* b, const int32_t* cu_seqlens, int32_t n_seq,
                                   int64_t n_tokens, const int32_t* slot_idx, const uint8_t* has_init,
                                   void* conv_pool, float* state_pool, int32_t n_slots, void* y, int32_t ckpt_every,
                                   const int32_t* ckpt_offset, const int32_t* ckpt_slots, void* workspace,
                                   size_t ws_bytes, void* stream) {
    if (n_seq < 0 || n_seq > 65535) return fail(GDN_ERR_RANGE, "n_seq: found %d, required 0..65535", n_seq);
    if (n_slots < 1) return fail(GDN_ERR_RANGE, "n_slots: found %d, required >= 1", n_slots);
    {
        gdn::Geom g;
        gdn_status st = make_geom(cfg, true, &g);
        if (st) return st;
        if (ckpt_every <= 0 || ckpt_every % cfg->chunk != 0)
            return fail(GDN_ERR_RANGE, "ckpt_every: found %d, required a positive multiple of chunk = %d", ckpt_every,
                        cfg->chunk);
    }
    if (n_seq == 0) {
        if (n_tokens != 0)
            return fail(GDN_ERR_RANGE, "n_tokens: found %lld with n_seq = 0, required 0", (long long)n_tokens);
        return ok();
    }
    GDN_REQUIRE_PTR_A(cu_seqlens, "cu_seqlens", 4u);
    GDN_REQUIRE_PTR_A(slot_idx, "slot_idx", 4u);
    GDN_OPTIONAL_PTR_A(has_init, "has_init", 1u);
    GDN_REQUIRE_PTR(conv_pool, "conv_pool");
    GDN_REQUIRE_PTR(state_pool, "state_pool");
    GDN_REQUIRE_PTR_A(ckpt_offset, "ckpt_offset", 4u);
    GDN_REQUIRE_PTR_A(ckpt_slots, "ckpt_slots", 4u);
    GDN_OPTIONAL_PTR(workspace, "workspace");
    gdn::PrefillJob job = {};
    job.x = x; job.z = z; job.a = a; job.b = b; job.y = y;
    job.n_tokens = n_tokens;
    job.n_seq = n_seq;
    job.cu_seqlens = cu_seqlens;
    job.slot_idx = slot_idx; job.has_init = has_init;
    job.state_pool = state_pool; job.conv_pool = conv_pool; job.n_slots = n_slots;
    job.ckpt_every = ckpt_every; job.ckpt_offset = ckpt_offset; job.ckpt_slots = ckpt_slots;
    job.workspace = workspace; job.ws_bytes = ws_bytes;
    return prefill_common(cfg, prm, job, stream, "gdn_varlen_prefill_ckpt");
}

gdn_status gdn_proj_gemm(const void* act, const void* w, void* out, int64_t n_tok, int32_t n_out, int32_t k,
                         int64_t ld_out, void* workspace, size_t ws_bytes, void* stream) {
    if (n_tok < 0 || n_tok >= ((int64_t)1 << 31))
        return fail(GDN_ERR_RANGE, "n_tok: found %lld, required 0..2^31-1", (long long)n_tok);
    if (n_out < 1) return fail(GDN_ERR_SHAPE, "n_out: found %d, required >= 1", n_out);
    if (k < 8 || k % 8 != 0) return fail(GDN_ERR_SHAPE, "k: found %d, required a positive multiple of 8", k);
    if (ld_out < n_out)
        return fail(GDN_ERR_SHAPE, "ld_out: found %lld, required >= n_out = %d", (long long)ld_out, n_out);
    if (n_tok == 0) return ok();
    GDN_REQUIRE_PTR(act, "act");
    GDN_REQUIRE_PTR(w, "w");
    GDN_REQUIRE_PTR_A(out, "out", 2u);
    const size_t need = gdn::proj_plan(n_out, k, n_tok).ws_bytes;
    if (need > 0) GDN_REQUIRE_PTR(workspace, "workspace");
    if (ws_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace: found %zu bytes, required %zu bytes", ws_bytes, need);
    gdn::ProjJob job = {};
    job.w = w; job.act = act; job.n_out = n_out; job.k = k; job.n_tok = n_tok;
    job.ws = workspace; job.ws_bytes = ws_bytes;
    job.nseg = 1;
    job.seg[0] = gdn::ProjOut{out, ld_out, 0, n_out};
    return cuda_status(gdn::launch_proj(job, (cudaStream_t)stream), "gdn_proj_gemm");
}

static gdn_status proj_check(const gdn::Geom& g, const gdn_proj* proj) {
    if (!g.act_bf16)
        return fail(GDN_ERR_UNSUPPORTED, "cfg.act_dtype: found 1 (GDN_DTYPE_F32), required GDN_DTYPE_BF16 (0) "
                                         "with the projections");
    if (!proj) return fail(GDN_ERR_NULL, "proj: found NULL, required a gdn_proj");
    if (proj->hidden < 8 || proj->hidden % 8 != 0)
        return fail(GDN_ERR_SHAPE, "proj.hidden: found %d, required a positive multiple of 8", proj->hidden);
    GDN_REQUIRE_PTR(proj->w_in, "proj.w_in");
    GDN_REQUIRE_PTR(proj->w_out, "proj.w_out");
    return GDN_OK;
}

// [x | z | a | b] = h w_in^T into the workspace
static cudaError_t launch_in_proj(const gdn::Geom& g, const gdn_proj* proj, const void* h, int64_t n,
                                  unsigned char* ws, const LayerWs& L, cudaStream_t st) {
    const int32_t vd = g.Hv * g.D;
    gdn::ProjJob j = {};
    j.w = proj->w_in; j.act = h; j.k = proj->hidden; j.n_tok = n;
    j.n_out = g.C_ch + vd + 2 * g.Hv;
    j.nseg = 4;
    j.seg[0] = gdn::ProjOut{ws + L.x, g.C_ch, 0, g.C_ch};
    j.seg[1] = gdn::ProjOut{ws + L.z, vd, g.C_ch, g.C_ch + vd};
    j.seg[2] = gdn::ProjOut{ws + L.a, g.Hv, g.C_ch + vd, g.C_ch + vd + g.Hv};
    j.seg[3] = gdn::ProjOut{ws + L.b, g.Hv, g.C_ch + vd + g.Hv, g.C_ch + vd + 2 * g.Hv};
    j.ws = ws + L.part;
    j.ws_bytes = L.rest - L.part;
    return gdn::launch_proj(j, st);
}

// out = y w_out^T
static cudaError_t launch_out_proj(const gdn::Geom& g, const gdn_proj* proj, const void* y, int64_t n, void* out,
                                   unsigned char* ws, const LayerWs& L, cudaStream_t st) {
    gdn::ProjJob j = {};
    j.w = proj->w_out; j.act = y; j.k = g.Hv * g.D; j.n_tok = n;
    j.n_out = proj->hidden;
    j.nseg = 1;
    j.seg[0] = gdn::ProjOut{out, proj->hidden, 0, proj->hidden};
    j.ws = ws + L.part;
    j.ws_bytes = L.rest - L.part;
    return gdn::launch_proj(j, st);
}

gdn_status gdn_layer_decode(const gdn_config* cfg, const gdn_params* prm, const gdn_proj* proj, const void* h,
                            void* conv_pool, float* state_pool, const int32_t* slot_idx, int32_t B, int32_t n_slots,
                            void* out, void* workspace, size_t ws_bytes, void* stream) {
    gdn::Geom g;
    gdn::LayerParams p;
    gdn_status st = make_geom(cfg, false, &g);
    if (st) return st;
    if ((st = proj_check(g, proj))) return st;
    if (B < 0 || B > 65535) return fail(GDN_ERR_RANGE, "B: found %d, required 0..65535", B);
    if (B == 0) return n_slots < 1 ? fail(GDN_ERR_RANGE, "n_slots: found %d, required >= 1", n_slots) : ok();
    GDN_REQUIRE_PTR(h, "h");
    GDN_REQUIRE_PTR_A(out, "out", 2u);
    const LayerWs L = layer_ws(g, B, proj->hidden);
    GDN_REQUIRE_PTR(workspace, "workspace");
    if (ws_bytes < L.rest)
        return fail(GDN_ERR_WORKSPACE, "workspace: found %zu bytes, required %zu bytes", ws_bytes, L.rest);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    // every check of the decode step before the first launch
    if ((st = rows_check(cfg, prm, ws + L.x, ws + L.z, ws + L.a, ws + L.b, conv_pool, state_pool, slot_idx, B, 1,
                         n_slots, ws + L.y, 0, nullptr, &g, &p)))
        return st;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_in_proj(g, proj, h, B, ws, L, s);
    if (e != cudaSuccess) return cuda_status(e, "gdn_layer_decode (in-projection)");
    gdn::RowsJob job{ws + L.x, ws + L.z, ws + L.a, ws + L.b, conv_pool, state_pool, slot_idx, nullptr, ws + L.y,
                     B, 1, n_slots};
    e = gdn::launch_rows(g, p, job, s);
    if (e != cudaSuccess) return cuda_status(e, "gdn_layer_decode (decode step)");
    return cuda_status(launch_out_proj(g, proj, ws + L.y, B, out, ws, L, s), "gdn_layer_decode (out-projection)");
}

gdn_status gdn_layer_varlen_prefill(const gdn_config* cfg, const gdn_params* prm, const gdn_proj* proj, const void* h,
                                    const int32_t* cu_seqlens, int32_t n_seq, int64_t n_tokens,
                                    const int32_t* slot_idx, const uint8_t* has_init, void* conv_pool,
                                    float* state_pool, int32_t n_slots, void* out, void* workspace, size_t ws_bytes,
                                    void* stream) {
    gdn::Geom g;
    gdn::LayerParams p;
    gdn_status st = make_geom(cfg, true, &g);
    if (st) return st;
    if ((st = proj_check(g, proj))) return st;
    if (n_seq < 0 || n_seq > 65535) return fail(GDN_ERR_RANGE, "n_seq: found %d, required 0..65535", n_seq);
    if (n_slots < 1) return fail(GDN_ERR_RANGE, "n_slots: found %d, required >= 1", n_slots);
    if (n_seq == 0) {
        if (n_tokens != 0)
            return fail(GDN_ERR_RANGE, "n_tokens: found %lld with n_seq = 0, required 0", (long long)n_tokens);
        return ok();
    }
    if (n_tokens < 0 || n_tokens > (int64_t)1 << 31)
        return fail(GDN_ERR_RANGE, "n_tokens: found %lld, required 0..2^31", (long long)n_tokens);
    GDN_REQUIRE_PTR_A(cu_seqlens, "cu_seqlens", 4u);
    GDN_REQUIRE_PTR_A(slot_idx, "slot_idx", 4u);
    GDN_OPTIONAL_PTR_A(has_init, "has_init", 1u);
    GDN_REQUIRE_PTR(conv_pool, "conv_pool");
    GDN_REQUIRE_PTR(state_pool, "state_pool");
    if (n_tokens > 0) {
        GDN_REQUIRE_PTR(h, "h");
        GDN_REQUIRE_PTR_A(out, "out", 2u);
    }
    const LayerWs L = layer_ws(g, n_tokens, proj->hidden);
    const size_t need = L.rest + gdn::prefill_workspace_bytes(g, n_tokens, n_seq);
    GDN_REQUIRE_PTR(workspace, "workspace");
    if (ws_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace: found %zu bytes, required %zu bytes", ws_bytes, need);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    gdn::PrefillJob job = {};
    job.x = ws + L.x; job.z = ws + L.z; job.a = ws + L.a; job.b = ws + L.b; job.y = ws + L.y;
    job.n_tokens = n_tokens;
    job.n_seq = n_seq;
    job.cu_seqlens = cu_seqlens;
    job.slot_idx = slot_idx; job.has_init = has_init;
    job.state_pool = state_pool; job.conv_pool = conv_pool; job.n_slots = n_slots;
    job.workspace = ws + L.rest; job.ws_bytes = ws_bytes - L.rest;
    if ((st = prefill_check(cfg, prm, job, &g, &p))) return st;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_in_proj(g, proj, h, n_tokens, ws, L, s);
    if (e != cudaSuccess) return cuda_status(e, "gdn_layer_varlen_prefill (in-projection)");
    e = gdn::launch_prefill(g, p, job, s);
    if (e != cudaSuccess) return cuda_status(e, "gdn_layer_varlen_prefill (prefill)");
    return cuda_status(launch_out_proj(g, proj, ws + L.y, n_tokens, out, ws, L, s),
                       "gdn_layer_varlen_prefill (out-projection)");
}

static gdn_status attn_check(const gdn_attn_config* cfg) {
    if (!cfg) return fail(GDN_ERR_NULL, "cfg: found NULL, required a gdn_attn_config");
    if (cfg->n_kv_heads < 1 || cfg->n_q_heads < 1 || cfg->n_q_heads % cfg->n_kv_heads != 0)
        return fail(GDN_ERR_SHAPE, "cfg.n_q_heads/n_kv_heads: found %d/%d, required a positive multiple",
                    cfg->n_q_heads, cfg->n_kv_heads);
    const int G = cfg->n_q_heads / cfg->n_kv_heads;
    if (!(G == 1 || G == 2 || (G % 4 == 0 && G <= 32)))
        return fail(GDN_ERR_UNSUPPORTED, "cfg: G = n_q_heads / n_kv_heads = %d, required 1, 2 or a multiple of 4 "
                                         "up to 32", G);
    if (cfg->head_dim != 128 && cfg->head_dim != 256)
        return fail(GDN_ERR_SHAPE, "cfg.head_dim: found %d, required 128 or 256", cfg->head_dim);
    if (cfg->page_size < 8 || cfg->page_size > 4096 || cfg->page_size % 8 != 0)
        return fail(GDN_ERR_SHAPE, "cfg.page_size: found %d, required a multiple of 8 in 8..4096", cfg->page_size);
    if (!(cfg->scale >= 0.f)) return fail(GDN_ERR_SHAPE, "cfg.scale: found %g, required >= 0", (double)cfg->scale);
    return GDN_OK;
}

size_t gdn_attn_workspace_size(const gdn_attn_config* cfg, int32_t B, int32_t max_seq_len) {
    if (attn_check(cfg) != GDN_OK) return 0;
    if (B < 0 || max_seq_len < 1) {
        fail(GDN_ERR_RANGE, "B/max_seq_len: found %d/%d, required >= 0/>= 1", B, max_seq_len);
        return 0;
    }
    ok();
    return gdn::attn_workspace_bytes(B, cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim, max_seq_len);
}

gdn_status gdn_attn_decode(const gdn_attn_config* cfg, const void* q, const void* k_new, const void* v_new,
                           void* k_pool, void* v_pool, const int32_t* block_table, const int32_t* seq_lens, int32_t B,
                           int32_t max_pages, int32_t n_pages, int32_t max_seq_len, void* o, void* workspace,
                           size_t ws_bytes, void* stream) {
    gdn_status st = attn_check(cfg);
    if (st) return st;
    if (B < 0 || B > 65535) return fail(GDN_ERR_RANGE, "B: found %d, required 0..65535", B);
    if (max_pages < 1 || n_pages < 1 || max_seq_len < 1)
        return fail(GDN_ERR_RANGE, "max_pages/n_pages/max_seq_len: found %d/%d/%d, required >= 1", max_pages, n_pages,
                    max_seq_len);
    if (B == 0) return ok();
    GDN_REQUIRE_PTR(q, "q");
    GDN_REQUIRE_PTR(k_new, "k_new");
    GDN_REQUIRE_PTR(v_new, "v_new");
    GDN_REQUIRE_PTR(k_pool, "k_pool");
    GDN_REQUIRE_PTR(v_pool, "v_pool");
    GDN_REQUIRE_PTR_A(block_table, "block_table", 4u);
    GDN_REQUIRE_PTR_A(seq_lens, "seq_lens", 4u);
    GDN_REQUIRE_PTR(o, "o");
    const size_t need = gdn::attn_workspace_bytes(B, cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim, max_seq_len);
    if (need > 0) GDN_REQUIRE_PTR(workspace, "workspace");
    if (ws_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace: found %zu bytes, required %zu bytes", ws_bytes, need);
    gdn::AttnJob j;
    j.q = q; j.k_new = k_new; j.v_new = v_new; j.k_pool = k_pool; j.v_pool = v_pool;
    j.block_table = block_table; j.seq_lens = seq_lens; j.o = o; j.ws = workspace;
    j.B = B; j.Hq = cfg->n_q_heads; j.Hkv = cfg->n_kv_heads; j.D = cfg->head_dim; j.page = cfg->page_size;
    j.max_pages = max_pages; j.n_pages = n_pages; j.max_seq_len = max_seq_len;
    j.scale = cfg->scale > 0.f ? cfg->scale : 1.0f / sqrtf((float)cfg->head_dim);
    return cuda_status(gdn::launch_attn_decode(j, (cudaStream_t)stream), "gdn_attn_decode");
}

gdn_status gdn_attn_prefill(const gdn_attn_config* cfg, const void* q, const void* k_new, const void* v_new,
                            void* k_pool, void* v_pool, const int32_t* block_table, const int32_t* cu_seqlens,
                            const int32_t* ctx_lens, int32_t n_seq, int64_t n_tokens, int32_t max_pages,
                            int32_t n_pages, void* o, void* stream) {
    gdn_status st = attn_check(cfg);
    if (st) return st;
    if (n_seq < 0 || n_seq > 65535) return fail(GDN_ERR_RANGE, "n_seq: found %d, required 0..65535", n_seq);
    if (n_tokens < 0 || n_tokens > (int64_t)1 << 30)
        return fail(GDN_ERR_RANGE, "n_tokens: found %lld, required 0..2^30", (long long)n_tokens);
    if (max_pages < 1 || n_pages < 1)
        return fail(GDN_ERR_RANGE, "max_pages/n_pages: found %d/%d, required >= 1", max_pages, n_pages);
    if (n_seq == 0 || n_tokens == 0) return ok();
    GDN_REQUIRE_PTR(q, "q");
    GDN_REQUIRE_PTR(k_new, "k_new");
    GDN_REQUIRE_PTR(v_new, "v_new");
    GDN_REQUIRE_PTR(k_pool, "k_pool");
    GDN_REQUIRE_PTR(v_pool, "v_pool");
    GDN_REQUIRE_PTR_A(block_table, "block_table", 4u);
    GDN_REQUIRE_PTR_A(cu_seqlens, "cu_seqlens", 4u);
    GDN_REQUIRE_PTR_A(ctx_lens, "ctx_lens", 4u);
    GDN_REQUIRE_PTR(o, "o");
    gdn::AttnPfJob j;
    j.q = q; j.k_new = k_new; j.v_new = v_new; j.k_pool = k_pool; j.v_pool = v_pool;
    j.block_table = block_table; j.cu_seqlens = cu_seqlens; j.ctx_lens = ctx_lens; j.o = o;
    j.n_seq = n_seq; j.Hq = cfg->n_q_heads; j.Hkv = cfg->n_kv_heads; j.D = cfg->head_dim; j.page = cfg->page_size;
    j.max_pages = max_pages; j.n_pages = n_pages; j.n_tokens = n_tokens;
    j.scale = cfg->scale > 0.f ? cfg->scale : 1.0f / sqrtf((float)cfg->head_dim);
    return cuda_status(gdn::launch_attn_prefill(j, (cudaStream_t)stream), "gdn_attn_prefill");
}

}  // extern "C"
