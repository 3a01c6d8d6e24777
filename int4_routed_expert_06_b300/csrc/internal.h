// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"
#include "moe_int4.h"

namespace moe {

struct Shape {
    int H, E, k, I, Is, G;
    int act, router, qscale; // moe_dtype values
    int bits;                // code width: 4 or 8
};

// Record a thread-local message and return `st`.
moe_status fail(moe_status st, const char *fmt, ...);
moe_status cuda_check(cudaError_t e, const char *what);
// Validate a config and copy it into `s` (may be NULL).
moe_status check_config(const moe_config *c, Shape *s);

// Router logits [T, E] and shared-gate logit [T].
cudaError_t launch_router(const Shape &s, const void *x, int T, const void *w_router,
                          const float *bias, const void *w_sg, float *logits, float *sg_logit,
                          cudaStream_t st);
// Calls with at least this many tokens compute the router logits (and the
// shared-gate logit) as one bf16 tensor-core GEMM with fp32 accumulation.
constexpr int kRouterGemmMinTokens = 16;
bool router_gemm_eligible(const Shape &s, int T);
cudaError_t launch_router_gemm(const Shape &s, const void *x, int T, const void *w_router, const float *bias,
                               const void *w_sg, float *logits, float *sg_logit, cudaStream_t st);
// Top-k + renormalised softmax from logits [T, E].
cudaError_t launch_topk(const Shape &s, const float *logits, int T, int32_t *idx, float *w,
                        cudaStream_t st);
// a[t, i, :] = silu(W_g x) * (W_u x) for the n_act active experts of each token.
cudaError_t launch_gateup(const Shape &s, const void *x, int T, int k_eff, int n_act,
                          const int32_t *topk_idx, const ExpertSrc &src, float *a, int Imax,
                          cudaStream_t st);
// y[t] = sum_i weight_i * W_d,i a[t, i, :].
cudaError_t launch_down(const Shape &s, const float *a, int T, int k_eff, int n_act, int Imax,
                        const int32_t *topk_idx, const float *topk_w, const float *gate_logit,
                        const ExpertSrc &src, void *y, float *y32, cudaStream_t st);
// Stable counting sort of (token, rank) pairs by expert.
cudaError_t launch_bucket(const Shape &s, const int32_t *idx, int T, int32_t *counts,
                          int32_t *offsets, int32_t *perm_tok, int32_t *perm_rank,
                          int32_t *chunk_hist, cudaStream_t st);
int bucket_chunks(int pairs);

// 0 = use the single-token kernels where eligible, 1 = generic kernels only.
int kernel_path();

namespace tok {
// Small per-call buffers that every CTA of a kernel reads are written in
// kRep copies; CTA c reads copy c % kRep, which spreads the reads of 148
// SMs over more L2 lines.
constexpr int kRep = 8;
// Per-call scratch of the single-token path, carved from the workspace.
struct Bufs {
    float *lg;           // [kRep][lgs]: the E logits, then the shared-gate logit at [E]
    int lgs;             // floats per logits copy
    unsigned char *xrec; // [kRep][xrs]: fixed-point records of x
    size_t xrs;          // bytes per x copy
    unsigned char *arec; // [kRep][ars]: activation records of the 32-row chunks of a
    size_t ars;          // bytes per record copy
};
size_t bufs_bytes(const Shape &s);
Bufs bufs_carve(const Shape &s, char *base);
// Routing of one token for the single-token expert kernels: either top-k
// from logits (every CTA recomputes it) or given idx / w.
struct Routing {
    const float *logits;     // copy 0 of the logits (+ shared-gate logit at [E]), or NULL when idx/w are given
    int lgs;                 // floats between logits copies
    const int32_t *idx;      // [k] given, or NULL
    const float *w;          // [k] given, or NULL
    int32_t *idx_out;        // [k] written by CTA 0 of gate/up (logits mode), or NULL
    float *w_out;            // [k]
    const float *sg_logit;   // [1] shared-gate logit when logits == NULL
};
// Shapes the single-token kernels handle (bf16 activations and router,
// H in {1024, 2048}, a shared expert, 16-byte scale rows, per-CTA shares that
// fit shared memory).
bool eligible(const Shape &s);
// Router logits (rows skipped when w_router is NULL) into `lg` (lgs floats
// apart, nrep copies; the shared-gate logit goes to lg[E] of each copy when
// lgs > 0 and to *sg when sg is non-NULL) and, when xrec is non-NULL, the
// fixed-point records of x into kRep copies xrs bytes apart.
cudaError_t launch_router(const Shape &s, const void *x, const void *w_router, const float *bias,
                          const void *w_sg, float *lg, int lgs, int nrep, float *sg, unsigned char *xrec,
                          size_t xrs, cudaStream_t st);
// gate/up SwiGLU, then down + weighted combine: two PDL-chained kernels.
cudaError_t launch_experts(const Shape &s, const Bufs &b, const ExpertSrc &src, const Routing &R, void *y,
                           float *y32, cudaStream_t st);
} // namespace tok

namespace prefill {
// Calls with at least this many tokens take the grouped-GEMM path (kernel
// path 0); kernel path 2 takes it from 2 tokens up.
constexpr int kMinTokens = 64;
int min_tokens();
// Byte offsets of the prefill buffers inside a workspace region.
struct Layout {
    size_t counts, offsets, perm_tok, perm_rank, hist, inv, wpair, units_gu, units_dn, n_units, xs, act, pout,
        total;
};
Layout layout(const Shape &s, int T);
// The shape and token count take the grouped GEMMs under the calling
// thread's kernel path: bf16 activations, 4-bit codes, H a multiple of 128,
// I and I_s multiples of 128, a shared expert, T >= min_tokens().
bool wanted(const Shape &s, int T);
// wanted() on a Blackwell (sm_10x) device with the tensor-map encoder.
bool eligible(const Shape &s, int T);
cudaError_t experts_forward(const Shape &s, const ExpertSrc &src, const void *x, int T, const int32_t *idx,
                            const float *topk_w, const float *sg, void *y, float *y32, char *ws, cudaStream_t st);
} // namespace prefill

} // namespace moe
