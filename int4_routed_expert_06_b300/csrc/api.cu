// C ABI of the routed int4 MoE layer: argument checks, blob layout,
// workspace carving and kernel dispatch.  Every entry point returns a
// moe_status; messages are kept per thread.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "internal.h"

namespace moe {

static thread_local char t_msg[512] = "";
static thread_local int g_kernel_path = 0;

int kernel_path() { return g_kernel_path; }

moe_status fail(moe_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
    va_end(ap);
    return st;
}

moe_status cuda_check(cudaError_t e, const char *what)
{
    if (e == cudaSuccess)
        return MOE_OK;
    cudaGetLastError(); // a rejected launch also sets the last-error state; leave it clear for the caller
    return fail(e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
static int scale_bytes(int dt) { return dt == MOE_F16 ? 2 : 4; }

moe_status check_config(const moe_config *c, Shape *s)
{
    if (!c)
        return fail(MOE_ERR_INVALID_ARG, "config is NULL");
    if (c->hidden <= 0 || c->hidden % 32)
        return fail(MOE_ERR_INVALID_ARG, "hidden %d must be a positive multiple of 32", c->hidden);
    if (c->n_experts <= 0 || c->n_experts > 1024)
        return fail(MOE_ERR_INVALID_ARG, "n_experts %d must be in [1, 1024]", c->n_experts);
    if (c->top_k <= 0 || c->top_k > 16 || c->top_k > c->n_experts)
        return fail(MOE_ERR_INVALID_ARG, "top_k %d must be in [1, min(16, n_experts)]", c->top_k);
    if (c->group_size != 32 && c->group_size != 64 && c->group_size != 128)
        return fail(MOE_ERR_UNSUPPORTED, "group_size %d: 32, 64 or 128 supported", c->group_size);
    if (c->inter <= 0 || c->inter % 32 || c->inter % c->group_size)
        return fail(MOE_ERR_INVALID_ARG, "inter %d must be a positive multiple of 32 and of the group", c->inter);
    if (c->shared_inter < 0 || c->shared_inter % 32 || c->shared_inter % c->group_size)
        return fail(MOE_ERR_INVALID_ARG, "shared_inter %d must be 0 or a multiple of 32 and of the group",
                    c->shared_inter);
    if (c->hidden % c->group_size)
        return fail(MOE_ERR_INVALID_ARG, "hidden %d must be a multiple of group_size %d", c->hidden, c->group_size);
    if (c->inter > 4096 || c->shared_inter > 4096 || c->hidden > 16384)
        return fail(MOE_ERR_UNSUPPORTED, "inter/shared_inter <= 4096 and hidden <= 16384 supported");
    if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16)
        return fail(MOE_ERR_UNSUPPORTED, "act_dtype must be MOE_F32 or MOE_BF16");
    if (c->router_dtype != MOE_F32 && c->router_dtype != MOE_BF16)
        return fail(MOE_ERR_UNSUPPORTED, "router_dtype must be MOE_F32 or MOE_BF16");
    if (c->qscale_dtype != MOE_F32 && c->qscale_dtype != MOE_F16)
        return fail(MOE_ERR_UNSUPPORTED, "qscale_dtype must be MOE_F32 or MOE_F16");
    if (c->bits != 0 && c->bits != 4 && c->bits != 8)
        return fail(MOE_ERR_UNSUPPORTED, "bits %d: 4 or 8 supported (0 means 4)", c->bits);
    if (s) {
        s->H = c->hidden;
        s->E = c->n_experts;
        s->k = c->top_k;
        s->I = c->inter;
        s->Is = c->shared_inter;
        s->G = c->group_size;
        s->act = c->act_dtype;
        s->router = c->router_dtype;
        s->qscale = c->qscale_dtype;
        s->bits = c->bits == 8 ? 8 : 4;
    }
    return MOE_OK;
}

// Workspace carving, 256-byte aligned pieces.
struct Ws {
    size_t logits, sg, idx, w, a, tok, hist, pre, total;
};

static int imax_of(const Shape &s) { return s.I > s.Is ? s.I : s.Is; }

// 2 <= T <= kTokLoopTokens on the default kernel path: the single-token
// kernels run once a token (each token's output depends on that token
// alone).  On the 80B-shaped layer a token then costs about 13.4 us, against
// 64 us for two tokens and 166 us for eight on the generic kernels; at 16
// tokens the two are level.
constexpr int kTokLoopTokens = 12;
static bool tok_loop(const Shape &s, int T)
{
    return T >= 2 && T <= kTokLoopTokens && kernel_path() == 0 && tok::eligible(s);
}

static Ws layer_ws(const Shape &s, int T)
{
    Ws w{};
    size_t o = 0;
    w.logits = o; o += align256(sizeof(float) * (size_t)T * s.E);
    w.sg = o;     o += align256(sizeof(float) * (size_t)T);
    w.idx = o;    o += align256(sizeof(int32_t) * (size_t)T * s.k);
    w.w = o;      o += align256(sizeof(float) * (size_t)T * s.k);
    w.a = o;      o += align256(sizeof(float) * (size_t)T * (s.k + 1) * imax_of(s));
    w.tok = o;    o += (T == 1 || tok_loop(s, T)) ? align256(tok::bufs_bytes(s)) : 0;
    w.hist = o;   o += align256(sizeof(int32_t) * (size_t)bucket_chunks(T * s.k) * s.E);
    w.pre = o;
    if (prefill::wanted(s, T))
        o += align256(prefill::layout(s, T).total);
    w.total = o;
    return w;
}

static void fill_offsets(const moe_blob_layout &l, size_t off[9])
{
    off[M_QG] = l.q_gate; off[M_QU] = l.q_up; off[M_QD] = l.q_down;
    off[M_SG] = l.s_gate; off[M_BG] = l.b_gate; off[M_SU] = l.s_up;
    off[M_BU] = l.b_up; off[M_SD] = l.s_down; off[M_BD] = l.b_down;
}

} // namespace moe

using namespace moe;

extern "C" {

const char *moe_last_error_message(void) { return t_msg; }

const char *moe_version(void) { return "moe_int4 0.2 (sm_103a)"; }

moe_status moe_set_kernel_path(int32_t path)
{
    if (path < 0 || path > 2)
        return fail(MOE_ERR_INVALID_ARG, "moe_set_kernel_path: path %d must be 0, 1 or 2", path);
    g_kernel_path = path;
    return MOE_OK;
}

moe_status moe_blob_layout_get(const moe_config *cfg, int32_t inter, moe_blob_layout *out)
{
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (!out)
        return fail(MOE_ERR_INVALID_ARG, "moe_blob_layout_get: out is NULL");
    if (inter <= 0 || inter % 32 || inter % s.G)
        return fail(MOE_ERR_INVALID_ARG, "moe_blob_layout_get: inter %d", inter);
    const size_t sb = scale_bytes(s.qscale);
    const size_t qgu = (size_t)inter * s.H * s.bits / 8, qd = (size_t)s.H * inter * s.bits / 8;
    const size_t sgu = (size_t)inter * (s.H / s.G) * sb, sd = (size_t)s.H * (inter / s.G) * sb;
    size_t o = 0;
    out->q_gate = o; o = align256(o + qgu);
    out->q_up = o;   o = align256(o + qgu);
    out->q_down = o; o = align256(o + qd);
    out->s_gate = o; o = align256(o + sgu);
    out->b_gate = o; o = align256(o + sgu);
    out->s_up = o;   o = align256(o + sgu);
    out->b_up = o;   o = align256(o + sgu);
    out->s_down = o; o = align256(o + sd);
    out->b_down = o; o = align256(o + sd);
    out->bytes = o;
    return MOE_OK;
}

moe_status moe_pack_expert(const moe_config *cfg, int32_t inter, const moe_expert *src, void *dst)
{
    moe_blob_layout l;
    moe_status st = moe_blob_layout_get(cfg, inter, &l);
    if (st != MOE_OK)
        return st;
    if (!src || !dst)
        return fail(MOE_ERR_INVALID_ARG, "moe_pack_expert: NULL argument");
    const moe_qmat *m[3] = {&src->gate, &src->up, &src->down};
    for (int j = 0; j < 3; ++j)
        if (!m[j]->q || !m[j]->scale || !m[j]->bias)
            return fail(MOE_ERR_INVALID_ARG, "moe_pack_expert: NULL array in matrix %d", j);
    const size_t sb = scale_bytes(cfg->qscale_dtype);
    const int bits = cfg->bits == 8 ? 8 : 4;
    const size_t qgu = (size_t)inter * cfg->hidden * bits / 8, qd = (size_t)cfg->hidden * inter * bits / 8;
    const size_t sgu = (size_t)inter * (cfg->hidden / cfg->group_size) * sb;
    const size_t sd = (size_t)cfg->hidden * (inter / cfg->group_size) * sb;
    char *d = static_cast<char *>(dst);
    memset(d, 0, l.bytes);
    memcpy(d + l.q_gate, src->gate.q, qgu);
    memcpy(d + l.q_up, src->up.q, qgu);
    memcpy(d + l.q_down, src->down.q, qd);
    memcpy(d + l.s_gate, src->gate.scale, sgu);
    memcpy(d + l.b_gate, src->gate.bias, sgu);
    memcpy(d + l.s_up, src->up.scale, sgu);
    memcpy(d + l.b_up, src->up.bias, sgu);
    memcpy(d + l.s_down, src->down.scale, sd);
    memcpy(d + l.b_down, src->down.bias, sd);
    return MOE_OK;
}

size_t moe_route_workspace_bytes(const moe_config *cfg, int32_t T)
{
    Shape s;
    if (check_config(cfg, &s) != MOE_OK || T < 0)
        return 0;
    return layer_ws(s, T).total;
}
size_t moe_bucket_workspace_bytes(const moe_config *cfg, int32_t T)
{
    Shape s;
    if (check_config(cfg, &s) != MOE_OK || T < 0)
        return 0;
    return align256(sizeof(int32_t) * (size_t)bucket_chunks(T * s.k) * s.E) + 256;
}
size_t moe_expert_workspace_bytes(const moe_config *cfg, int32_t T)
{
    Shape s;
    if (check_config(cfg, &s) != MOE_OK || T < 0)
        return 0;
    return layer_ws(s, T).total;
}
size_t moe_layer_workspace_bytes(const moe_config *cfg, int32_t T)
{
    Shape s;
    if (check_config(cfg, &s) != MOE_OK || T < 0)
        return 0;
    return layer_ws(s, T).total;
}

moe_status moe_route(const moe_config *cfg, const void *x, int32_t T, const void *w_router,
                     const float *router_bias, const void *w_shared_gate, int32_t *topk_idx,
                     float *topk_w, float *shared_gate_logit, float *logits_out, void *workspace,
                     size_t ws_bytes, cudaStream_t stream)
{
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (T < 0 || T > (1 << 20))
        return fail(MOE_ERR_INVALID_ARG, "moe_route: T %d out of range", T);
    if (T == 0)
        return MOE_OK;
    if (!x || !w_router || !topk_idx || !topk_w)
        return fail(MOE_ERR_INVALID_ARG, "moe_route: NULL x, w_router, topk_idx or topk_w");
    if (!aligned(x, 16) || !aligned(w_router, 16) || (w_shared_gate && !aligned(w_shared_gate, 16)))
        return fail(MOE_ERR_INVALID_ARG, "moe_route: x, w_router and w_shared_gate must be 16-byte aligned");
    if ((s.Is > 0) != (w_shared_gate != nullptr) || (s.Is > 0) != (shared_gate_logit != nullptr))
        return fail(MOE_ERR_INVALID_ARG, "moe_route: w_shared_gate and shared_gate_logit are required iff shared_inter > 0");
    float *logits = logits_out;
    if (!logits) {
        Ws w = layer_ws(s, T);
        if (!workspace || !aligned(workspace, 256) || ws_bytes < w.total)
            return fail(MOE_ERR_OOM, "moe_route: workspace needs %zu bytes (256-byte aligned), got %zu", w.total, ws_bytes);
        logits = reinterpret_cast<float *>(static_cast<char *>(workspace) + w.logits);
    }
    cudaError_t e;
    if (T == 1 && tok::eligible(s))
        e = tok::launch_router(s, x, w_router, router_bias, w_shared_gate, logits, 0, 1, shared_gate_logit,
                               nullptr, 0, stream);
    else
        e = launch_router(s, x, T, w_router, router_bias, s.Is > 0 ? w_shared_gate : nullptr, logits,
                          shared_gate_logit, stream);
    if (e != cudaSuccess)
        return cuda_check(e, "moe_route: router");
    e = launch_topk(s, logits, T, topk_idx, topk_w, stream);
    return cuda_check(e, "moe_route: top-k");
}

moe_status moe_bucket(const moe_config *cfg, const int32_t *topk_idx, int32_t T, int32_t *counts,
                      int32_t *offsets, int32_t *perm_tok, int32_t *perm_rank, void *workspace,
                      size_t ws_bytes, cudaStream_t stream)
{
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (T < 0 || (int64_t)T * s.k > (1 << 26))
        return fail(MOE_ERR_INVALID_ARG, "moe_bucket: T %d out of range", T);
    if (!counts || !offsets || (T > 0 && (!topk_idx || !perm_tok || !perm_rank)))
        return fail(MOE_ERR_INVALID_ARG, "moe_bucket: NULL argument");
    const size_t need = moe_bucket_workspace_bytes(cfg, T);
    if (T > 0 && (!workspace || !aligned(workspace, 256) || ws_bytes < need))
        return fail(MOE_ERR_OOM, "moe_bucket: workspace needs %zu bytes (256-byte aligned), got %zu", need, ws_bytes);
    cudaError_t e = launch_bucket(s, topk_idx, T, counts, offsets, perm_tok, perm_rank,
                                  static_cast<int32_t *>(workspace), stream);
    return cuda_check(e, "moe_bucket");
}

static moe_status check_qmat(const moe_qmat &m, const char *name)
{
    if (!m.q || !m.scale || !m.bias)
        return fail(MOE_ERR_INVALID_ARG, "moe_expert_forward: NULL array in %s", name);
    if (!aligned(m.q, 16))
        return fail(MOE_ERR_INVALID_ARG, "moe_expert_forward: %s.q must be 16-byte aligned", name);
    return MOE_OK;
}

moe_status moe_expert_forward(const moe_config *cfg, const moe_expert *ex, int32_t inter, const void *x,
                              int32_t T, void *y, float *y_f32, void *workspace, size_t ws_bytes,
                              cudaStream_t stream)
{
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (T < 0 || T > 65535)
        return fail(MOE_ERR_INVALID_ARG, "moe_expert_forward: T %d out of range [0, 65535]", T);
    if (T == 0)
        return MOE_OK;
    if (!ex || !x || !y)
        return fail(MOE_ERR_INVALID_ARG, "moe_expert_forward: NULL expert, x or y");
    if (inter <= 0 || inter % 32 || inter % s.G || inter > 4096)
        return fail(MOE_ERR_INVALID_ARG, "moe_expert_forward: inter %d", inter);
    if ((st = check_qmat(ex->gate, "gate")) != MOE_OK || (st = check_qmat(ex->up, "up")) != MOE_OK ||
        (st = check_qmat(ex->down, "down")) != MOE_OK)
        return st;
    if (!aligned(x, 16))
        return fail(MOE_ERR_INVALID_ARG, "moe_expert_forward: x must be 16-byte aligned");
    Shape s1 = s;
    s1.I = inter;
    s1.Is = inter;
    const size_t need = align256(sizeof(float) * (size_t)T * inter);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < need)
        return fail(MOE_ERR_OOM, "moe_expert_forward: workspace needs %zu bytes (256-byte aligned), got %zu", need,
                    ws_bytes);
    ExpertSrc src{};
    src.explicit_mode = 1;
    src.ptr[M_QG] = ex->gate.q; src.ptr[M_SG] = ex->gate.scale; src.ptr[M_BG] = ex->gate.bias;
    src.ptr[M_QU] = ex->up.q;   src.ptr[M_SU] = ex->up.scale;   src.ptr[M_BU] = ex->up.bias;
    src.ptr[M_QD] = ex->down.q; src.ptr[M_SD] = ex->down.scale; src.ptr[M_BD] = ex->down.bias;
    float *a = static_cast<float *>(workspace);
    cudaError_t e = launch_gateup(s1, x, T, 0, 1, nullptr, src, a, inter, stream);
    if (e != cudaSuccess)
        return cuda_check(e, "moe_expert_forward: gate/up");
    e = launch_down(s1, a, T, 0, 1, inter, nullptr, nullptr, nullptr, src, y, y_f32, stream);
    return cuda_check(e, "moe_expert_forward: down");
}

static moe_status make_src(const moe_config *cfg, const Shape &s, const moe_layer *L, ExpertSrc *src,
                           const char *who)
{
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "%s: layer is NULL", who);
    if (!L->pool || !aligned(L->pool, 256) || !L->slot_table || L->n_slots <= 0)
        return fail(MOE_ERR_INVALID_ARG, "%s: pool (256-byte aligned), slot_table and n_slots > 0 are required", who);
    moe_blob_layout lr, ls{};
    moe_blob_layout_get(cfg, s.I, &lr);
    if (L->expert_stride < lr.bytes || (L->expert_stride & 255))
        return fail(MOE_ERR_INVALID_ARG, "%s: expert_stride %zu must be a multiple of 256 and >= %zu", who,
                    L->expert_stride, lr.bytes);
    if (s.Is > 0) {
        if (!L->shared_blob || !aligned(L->shared_blob, 256))
            return fail(MOE_ERR_INVALID_ARG, "%s: shared_blob (256-byte aligned) is required when shared_inter > 0", who);
        moe_blob_layout_get(cfg, s.Is, &ls);
    }
    *src = ExpertSrc{};
    src->pool = static_cast<const char *>(L->pool);
    src->stride = L->expert_stride;
    src->table = L->slot_table;
    src->n_slots = L->n_slots;
    src->n_experts = s.E;
    src->shared = static_cast<const char *>(L->shared_blob);
    fill_offsets(lr, src->off);
    if (s.Is > 0)
        fill_offsets(ls, src->off_sh);
    return MOE_OK;
}

moe_status moe_experts_forward(const moe_config *cfg, const moe_layer *L, const void *x, int32_t T,
                               const int32_t *topk_idx, const float *topk_w, const float *shared_gate_logit,
                               void *y, float *y_f32, void *workspace, size_t ws_bytes, cudaStream_t stream)
{
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (T < 0 || T > 65535)
        return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: T %d out of range [0, 65535]", T);
    if (T == 0)
        return MOE_OK;
    if (!x || !y || !topk_idx || !topk_w)
        return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: NULL x, y, topk_idx or topk_w");
    if ((s.Is > 0) != (shared_gate_logit != nullptr))
        return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: shared_gate_logit is required iff shared_inter > 0");
    if (!aligned(x, 16))
        return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: x must be 16-byte aligned");
    ExpertSrc src;
    if ((st = make_src(cfg, s, L, &src, "moe_experts_forward")) != MOE_OK)
        return st;
    Ws w = layer_ws(s, T);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < w.total)
        return fail(MOE_ERR_OOM, "moe_experts_forward: workspace needs %zu bytes (256-byte aligned), got %zu",
                    w.total, ws_bytes);
    float *a = reinterpret_cast<float *>(static_cast<char *>(workspace) + w.a);
    if (prefill::eligible(s, T) && w.total > w.pre)
        return cuda_check(prefill::experts_forward(s, src, x, T, topk_idx, topk_w, shared_gate_logit, y, y_f32,
                                                   static_cast<char *>(workspace) + w.pre, stream),
                          "moe_experts_forward: grouped GEMM");
    if (T == 1 && tok::eligible(s)) {
        const tok::Bufs b = tok::bufs_carve(s, static_cast<char *>(workspace) + w.tok);
        cudaError_t e = tok::launch_router(s, x, nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, b.xrec, b.xrs,
                                           stream);
        if (e != cudaSuccess)
            return cuda_check(e, "moe_experts_forward: x records");
        tok::Routing R{nullptr, 0, topk_idx, topk_w, nullptr, nullptr, shared_gate_logit};
        return cuda_check(tok::launch_experts(s, b, src, R, y, y_f32, stream), "moe_experts_forward");
    }
    const int n_act = s.k + (s.Is > 0 ? 1 : 0);
    cudaError_t e = launch_gateup(s, x, T, s.k, n_act, topk_idx, src, a, imax_of(s), stream);
    if (e != cudaSuccess)
        return cuda_check(e, "moe_experts_forward: gate/up");
    e = launch_down(s, a, T, s.k, n_act, imax_of(s), topk_idx, topk_w, s.Is > 0 ? shared_gate_logit : nullptr,
                    src, y, y_f32, stream);
    return cuda_check(e, "moe_experts_forward: down");
}

moe_status moe_layer_forward(const moe_config *cfg, const moe_layer *L, const void *x, int32_t T, void *y,
                             float *y_f32, int32_t *topk_idx_out, float *topk_w_out, void *workspace,
                             size_t ws_bytes, cudaStream_t stream)
{
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (T < 0 || T > 65535)
        return fail(MOE_ERR_INVALID_ARG, "moe_layer_forward: T %d out of range [0, 65535]", T);
    if (T == 0)
        return MOE_OK;
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "moe_layer_forward: layer is NULL");
    Ws w = layer_ws(s, T);
    if (!workspace || !aligned(workspace, 256) || ws_bytes < w.total)
        return fail(MOE_ERR_OOM, "moe_layer_forward: workspace needs %zu bytes (256-byte aligned), got %zu",
                    w.total, ws_bytes);
    char *ws = static_cast<char *>(workspace);
    int32_t *idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t *>(ws + w.idx);
    float *tw = topk_w_out ? topk_w_out : reinterpret_cast<float *>(ws + w.w);
    float *sg = s.Is > 0 ? reinterpret_cast<float *>(ws + w.sg) : nullptr;
    if ((T == 1 && tok::eligible(s)) || tok_loop(s, T)) {
        if (!aligned(x, 16) || !L->w_router || !aligned(L->w_router, 16) || !L->w_shared_gate ||
            !aligned(L->w_shared_gate, 16) || !y)
            return fail(MOE_ERR_INVALID_ARG, "moe_layer_forward: x, y, w_router and w_shared_gate must be non-NULL "
                                             "and 16-byte aligned");
        ExpertSrc src;
        if ((st = make_src(cfg, s, L, &src, "moe_layer_forward")) != MOE_OK)
            return st;
        // one token at a time through the same buffers: each call's kernels
        // wait (PDL) for the previous call's before touching them
        const tok::Bufs b = tok::bufs_carve(s, ws + w.tok);
        const size_t row = sizeof(__nv_bfloat16) * (size_t)s.H; // x and y rows (bf16)
        for (int t = 0; t < T; ++t) {
            const char *xt = static_cast<const char *>(x) + t * row;
            cudaError_t e = tok::launch_router(s, xt, L->w_router, L->router_bias, L->w_shared_gate, b.lg, b.lgs,
                                               tok::kRep, nullptr, b.xrec, b.xrs, stream);
            if (e != cudaSuccess)
                return cuda_check(e, "moe_layer_forward: router");
            tok::Routing R{b.lg, b.lgs, nullptr, nullptr, idx + (size_t)t * s.k, tw + (size_t)t * s.k, nullptr};
            e = tok::launch_experts(s, b, src, R, static_cast<char *>(y) + t * row,
                                    y_f32 ? y_f32 + (size_t)t * s.H : nullptr, stream);
            if (e != cudaSuccess)
                return cuda_check(e, "moe_layer_forward: experts");
        }
        return MOE_OK;
    }
    st = moe_route(cfg, x, T, L->w_router, L->router_bias, s.Is > 0 ? L->w_shared_gate : nullptr, idx, tw, sg,
                   reinterpret_cast<float *>(ws + w.logits), nullptr, 0, stream);
    if (st != MOE_OK)
        return st;
    return moe_experts_forward(cfg, L, x, T, idx, tw, sg, y, y_f32, workspace, ws_bytes, stream);
}

moe_status moe_get_device_error(cudaStream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return cuda_check(e, "moe_get_device_error: stream");
    int code = 0;
    e = cudaMemcpyFromSymbol(&code, g_device_error, sizeof(int));
    if (e != cudaSuccess)
        return cuda_check(e, "moe_get_device_error: read");
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (e != cudaSuccess)
        return cuda_check(e, "moe_get_device_error: clear");
    if (code != 0)
        return fail(static_cast<moe_status>(code), "a kernel recorded device error %d", code);
    return MOE_OK;
}

} // extern "C"
