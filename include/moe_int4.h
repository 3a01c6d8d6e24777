/*
 * moe_int4.h -- C ABI of the routed int4 MoE layer for NVIDIA B300 (sm_103a).
 *
 * The layer is the sparse MoE block of the Qwen3-Next / Qwen3.5-3.6 hybrid
 * models that the Swiftlet project pages describe: each token is routed to
 * top_k of n_experts SwiGLU experts (10 of 512 for the 80B model, 8 of 256
 * for 35B; the Swiftlet README "How it works"), a shared expert stays resident beside the
 * router (same section), weights use MLX affine 4-bit group quantisation
 * (Swiftlet README "Relation to TurboFieldfare"), routed experts are packed as
 * fixed-stride blobs so that one expert is one copy, and a bounded pool
 * caches hot experts with LFU-plus-recency eviction (Swiftlet README "How it works").
 * "Swiftlet README" is the project README as reposted under the title
 * "Swiftlet：在 Mac 上运行 80B 版 Qwen（内存 4.3 GB），在 iPhone 上运行 35B 版";
 * section names are given in English.
 *
 * Conventions for every call:
 *   - Pointers named *_dev / device are CUDA device pointers; *_host are host
 *     pointers.  The caller allocates and owns every buffer it passes; the
 *     library only owns the slot_pool object and the device table inside it.
 *   - Device work is enqueued on the given stream and returns without
 *     waiting; argument errors are reported synchronously by the return value
 *     and moe_last_error_message().  No call aborts, exits or throws.
 *   - Faults that kernels detect (a slot table entry that is not resident, a
 *     wait that timed out) are recorded in a per-device error word that
 *     moe_get_device_error() reads and clears; the kernel skips the bad access
 *     and keeps the context usable.
 *   - Counts and ids are int32; byte sizes and offsets are size_t (64-bit
 *     offsets, as the pages' kernels use for multi-GB shards).
 */
#ifndef MOE_INT4_H
#define MOE_INT4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,     /* bad pointer, size, alignment or config */
    MOE_ERR_UNSUPPORTED = 2,     /* valid but not implemented (e.g. group 16) */
    MOE_ERR_CUDA = 3,            /* a CUDA runtime call failed */
    MOE_ERR_OOM = 4,             /* workspace or pool too small, allocation failed */
    MOE_ERR_TIMEOUT = 5,         /* a bounded device wait gave up */
    MOE_ERR_POOL_EXHAUSTED = 6,  /* more distinct experts needed than slots */
    MOE_ERR_NOT_RESIDENT = 7,    /* a routed expert had no slot */
    MOE_ERR_DEVICE_FAULT = 8     /* another fault recorded by a kernel */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_F16 = 2 } moe_dtype;

/* Shape and dtypes of one MoE layer.
 *   hidden (H), n_experts (E), top_k (k <= 16, k <= E), inter (I, routed
 *   expert intermediate), shared_inter (I_s, 0 = no shared expert),
 *   group_size (G: 32, 64 or 128; H and I multiples of G; H, I, I_s
 *   multiples of 32; E <= 1024).
 *   act_dtype: x and y, MOE_F32 or MOE_BF16.
 *   router_dtype: router and shared-gate weights, MOE_F32 or MOE_BF16.
 *   qscale_dtype: per-group scale and bias, MOE_F32 or MOE_F16.
 *   bits: code width of the expert weights, 4 or 8 (MLX affine int4 or
 *   int8 group quantisation, the Swiftlet README "Relation to TurboFieldfare"); 0 means
 *   4, so a zero-initialised field keeps the int4 layout. */
typedef struct {
    int32_t hidden;
    int32_t n_experts;
    int32_t top_k;
    int32_t inter;
    int32_t shared_inter;
    int32_t group_size;
    int32_t act_dtype;
    int32_t router_dtype;
    int32_t qscale_dtype;
    int32_t bits;
} moe_config;

/* One affine matrix W [out, in] (MLX layout) with b-bit codes (b = bits, 4
 * or 8): q is uint32 [out, in*b/32] with column c of row o in word
 * [o, c*b/32] at bits b*(c%(32/b)) .. b*(c%(32/b))+b-1 (lowest column in the
 * lowest bits); scale and bias are [out, in/G] in qscale_dtype;
 * W[o,c] = scale[o,c/G] * q + bias[o,c/G].  q must be 16-byte aligned. */
typedef struct {
    const uint32_t *q;
    const void *scale;
    const void *bias;
} moe_qmat;

/* One SwiGLU expert: gate and up are [inter, H], down is [H, inter]. */
typedef struct {
    moe_qmat gate, up, down;
} moe_expert;

/* Byte offsets of the nine arrays inside one fixed-stride expert blob, and
 * the blob size.  Order: q_gate, q_up, q_down, s_gate, b_gate, s_up, b_up,
 * s_down, b_down, each starting on a 256-byte boundary. */
typedef struct {
    size_t q_gate, q_up, q_down;
    size_t s_gate, b_gate, s_up, b_up, s_down, b_down;
    size_t bytes;
} moe_blob_layout;

/* Layout of an expert blob with intermediate `inter` (I for routed experts,
 * I_s for the shared one).  Pure host computation. */
moe_status moe_blob_layout_get(const moe_config *cfg, int32_t inter, moe_blob_layout *out);

/* Host-side repack: copy the nine arrays of *src (host pointers, MLX layout)
 * into the blob at dst_host (moe_blob_layout_get(...).bytes bytes, any
 * alignment).  The fixed-stride blob is what the slot pool and the layer
 * kernels read; one expert is one contiguous copy. */
moe_status moe_pack_expert(const moe_config *cfg, int32_t inter, const moe_expert *src_host,
                           void *dst_host);

/* Scratch bytes each call needs for T tokens (caller allocates on the device,
 * 256-byte aligned).  The same workspace may be reused by later calls on the
 * same stream. */
size_t moe_route_workspace_bytes(const moe_config *cfg, int32_t T);
size_t moe_bucket_workspace_bytes(const moe_config *cfg, int32_t T);
size_t moe_expert_workspace_bytes(const moe_config *cfg, int32_t T);
size_t moe_layer_workspace_bytes(const moe_config *cfg, int32_t T);

/* Router and top-k (pages: the Swiftlet README "How it works", k of E experts per token;
 * the renormalised softmax follows the Qwen MoE layer).
 *   x [T, H] act_dtype; w_router [E, H] router_dtype; router_bias [E] fp32 or
 *   NULL; w_shared_gate [H] router_dtype or NULL (required iff I_s > 0).
 *   logits[t,e] = w_router[e] . x[t] + bias[e] (fp32 accumulation);
 *   topk_idx [T, k] int32: the k largest logits, ties to the lower expert id,
 *   in descending order; topk_w [T, k] fp32: exp(l_r - l_max) / sum over the
 *   k selected; shared_gate_logit [T] fp32 = w_shared_gate . x[t] (NULL iff no
 *   shared expert); logits_out [T, E] fp32 or NULL.  All device pointers.
 * For T >= 16 with bf16 x and router the logits and the shared-gate logit
 * are one bf16 tensor-core GEMM of the library's own (fp32 accumulation);
 * the library calls no BLAS. */
moe_status moe_route(const moe_config *cfg, const void *x, int32_t T, const void *w_router,
                     const float *router_bias, const void *w_shared_gate, int32_t *topk_idx,
                     float *topk_w, float *shared_gate_logit, float *logits_out,
                     void *workspace, size_t ws_bytes, cudaStream_t stream);

/* Token -> expert bucketing (Swiftlet README "Correctness": sparse MoE routing, each
 * token's k experts; the pages give no bucketing step, this is how the
 * many-token path groups a routed batch by expert for its grouped GEMMs):
 * a stable counting sort of the T*k (token, rank) pairs of topk_idx [T, k]
 * by expert.  counts [E], offsets [E+1] (exclusive
 * prefix sum), perm_tok [T*k] and perm_rank [T*k] list the pairs in
 * (expert, token, rank) order.  Device pointers.  Ids outside [0, E) are
 * recorded as MOE_ERR_DEVICE_FAULT and dropped. */
moe_status moe_bucket(const moe_config *cfg, const int32_t *topk_idx, int32_t T, int32_t *counts,
                      int32_t *offsets, int32_t *perm_tok, int32_t *perm_rank, void *workspace,
                      size_t ws_bytes, cudaStream_t stream);

/* One expert on T tokens, no routing weight (Swiftlet README "How it works": each
 * expert a SwiGLU MLP, gate and up from H to inter, down back to H, weights
 * in MLX affine int4/int8 group quantisation, the Swiftlet README "Relation to
 * TurboFieldfare"): y[t] = W_d (silu(W_g x[t]) * (W_u x[t])) with
 * intermediate `inter`.  e holds device pointers.  y [T, H]
 * act_dtype; y_f32 [T, H] fp32 or NULL (the value before rounding). */
moe_status moe_expert_forward(const moe_config *cfg, const moe_expert *e, int32_t inter,
                              const void *x, int32_t T, void *y, float *y_f32, void *workspace,
                              size_t ws_bytes, cudaStream_t stream);

/* Where a layer's weights live (all device pointers).  Routed experts are
 * fixed-stride blobs in `pool`: expert e is the blob at
 * pool + slot_table[e] * expert_stride (slot_table [E] int32; -1 = not
 * resident).  expert_stride is a multiple of 256 and >= the blob size for
 * `inter`.  The shared expert is one blob (layout for shared_inter). */
typedef struct {
    const void *w_router;        /* [E, H] router_dtype */
    const float *router_bias;    /* [E] fp32 or NULL */
    const void *w_shared_gate;   /* [H] router_dtype; NULL iff shared_inter == 0 */
    const void *shared_blob;     /* NULL iff shared_inter == 0; 256-byte aligned */
    const void *pool;            /* 256-byte aligned */
    size_t expert_stride;
    const int32_t *slot_table;   /* [E] */
    int32_t n_slots;             /* slots addressable from pool (bounds check) */
} moe_layer;

/* Routed experts and combine, given the routing (the part of the layer after
 * moe_route):
 *   y[t] = sum_{r<k} topk_w[t,r] * E_{topk_idx[t,r]}(x[t])
 *          + sigmoid(shared_gate_logit[t]) * E_shared(x[t]),
 * summed in rank order and then the shared term, in fp32.  y [T, H]
 * act_dtype, y_f32 [T, H] fp32 or NULL.  A routed expert whose slot is -1
 * contributes nothing and records MOE_ERR_NOT_RESIDENT. */
moe_status moe_experts_forward(const moe_config *cfg, const moe_layer *layer, const void *x,
                               int32_t T, const int32_t *topk_idx, const float *topk_w,
                               const float *shared_gate_logit, void *y, float *y_f32,
                               void *workspace, size_t ws_bytes, cudaStream_t stream);

/* The whole layer: moe_route then moe_experts_forward.  topk_idx_out [T,k]
 * and topk_w_out [T,k] (device, or NULL) receive the routing.
 * T = 1 (bf16, shapes the single-token kernels take) runs three kernels
 * chained by programmatic dependent launch: router, gate/up (top-k and
 * SwiGLU), down (weighted combine).  No kernel waits on another kernel's
 * CTAs, so the call needs no co-residency and cannot stall behind work on
 * other streams. */
moe_status moe_layer_forward(const moe_config *cfg, const moe_layer *layer, const void *x,
                             int32_t T, void *y, float *y_f32, int32_t *topk_idx_out,
                             float *topk_w_out, void *workspace, size_t ws_bytes,
                             cudaStream_t stream);

/* moe_layer_forward without a caller workspace, for callers that cannot
 * allocate device memory where they run the layer (an engine plugin whose
 * host owns all device memory, a latency-critical loop that must not take
 * cudaMalloc's implicit synchronisation).  The Swiftlet pages have no
 * counterpart; this is an interface convenience.
 * Scratch is a 4 MiB array built into the library's device image, held by
 * every GPU that loads the library until the process exits.  T is limited to
 * what fits: moe_layer_workspace_bytes(cfg, T) <= 4 MiB, which for the 35B-
 * and 80B-shaped layers means T <= 63 (from T = 64 on the grouped-GEMM
 * buffers alone exceed it); larger T returns MOE_ERR_OOM.  Nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library call.  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture.
 * The library as a whole serves one GPU per process (its kernels' attributes
 * are set once per process), so call it from one device only.
 * All calls share the one array and it keeps the last call's contents; calls
 * whose GPU work overlaps race on it, so order them (one stream, or events).
 * Other arguments and behaviour as moe_layer_forward. */
moe_status moe_layer_forward_noalloc(const moe_config *cfg, const moe_layer *layer, const void *x,
                                     int32_t T, void *y, float *y_f32, int32_t *topk_idx_out,
                                     float *topk_w_out, cudaStream_t stream);

/* ------------------------------------------------------------------ pool */

/* A bounded HBM pool of expert slots for n_layers layers, filled on demand
 * from a pinned host backing store (the pages read one fixed-stride expert
 * with one pread into a bounded slot pool; here one cudaMemcpyAsync per
 * expert from pinned host memory).
 *   pool_dev: n_layers * slots_per_layer * expert_stride bytes of device
 *   memory, 256-byte aligned; slot s of layer l is at
 *   pool_dev + (l * slots_per_layer + s) * expert_stride.
 *   backing_host: pinned host memory holding every expert blob, expert e of
 *   layer l at backing_host + (l * E + e) * expert_stride.
 *   side_stream: the stream fills are enqueued on.
 * The pool object owns a device table [n_layers, E] int32 (-1 = absent) and
 * a host mirror of it.  Eviction rule (LFU + recency): a hit adds 1 to the
 * slot's use count and stamps it with the lookup clock (one tick per
 * lookup); a miss takes the lowest empty slot, else evicts, among experts not
 * needed by the same lookup, the smallest count, then the oldest stamp,
 * then the lowest slot id; a filled slot starts at count 1. */
typedef struct slot_pool slot_pool;

typedef struct {
    int64_t lookups, hits, misses, evictions, bytes_filled;
    int64_t exposed_copy_ns; /* time compute streams spent waiting for fills
                                (moe_pooled_layer_forward only) */
} moe_pool_stats;

moe_status slot_pool_create(const moe_config *cfg, int32_t n_layers, int32_t slots_per_layer,
                            void *pool_dev, size_t pool_bytes, const void *backing_host,
                            size_t expert_stride, cudaStream_t side_stream, slot_pool **out);

/* Eviction rules a pool can use (all take empty slots first, lowest id
 * first, and never evict an expert the same lookup needs):
 *   MOE_POOL_LFU_RECENCY  smallest use count, then oldest stamp, then lowest
 *                         slot id (the default; the rule the pages name);
 *   MOE_POOL_LRU          oldest stamp, then lowest slot id;
 *   MOE_POOL_LFU          smallest use count, then lowest slot id.
 * Use counts and stamps are kept the same way under every rule.  The rule
 * may be changed between lookups; it applies to the evictions that follow.
 * Returns MOE_ERR_INVALID_ARG for an unknown rule. */
typedef enum { MOE_POOL_LFU_RECENCY = 0, MOE_POOL_LRU = 1, MOE_POOL_LFU = 2 } moe_pool_policy;
moe_status slot_pool_set_policy(slot_pool *p, int32_t policy);

/* Apply the policy to one lookup of `n` expert ids (host array) of `layer`:
 * hits are stamped, each miss gets a slot (evicting if needed) in the host
 * table.  slots_out [n] (host) receives the slot of every id; miss_ids
 * (host, capacity n) receives the ids that must be filled, *n_miss their
 * number.  MOE_ERR_POOL_EXHAUSTED if the distinct ids exceed the slots. */
moe_status slot_pool_lookup(slot_pool *p, int32_t layer, const int32_t *expert_ids, int32_t n,
                            int32_t *slots_out, int32_t *miss_ids, int32_t *n_miss);

/* Enqueue on the side stream one host->device copy per missed expert into
 * its slot and the matching device-table update, then record `done` (may be
 * NULL).  Work on another stream that reads the layer's slots must wait on
 * `done`.  The copies overwrite the evicted experts' slots: every earlier
 * reader of those slots (kernels on any stream that used the layer's table
 * before this lookup) must have completed before slot_pool_fill is called,
 * or the side stream must be made to wait for them (an event recorded after
 * the last reader, cudaStreamWaitEvent on side_stream).
 * moe_pooled_layer_forward orders this itself.  The miss list is the one the
 * last lookup of this layer returned. */
moe_status slot_pool_fill(slot_pool *p, int32_t layer, const int32_t *miss_ids, int32_t n_miss,
                          cudaEvent_t done);

/* Device table row of `layer` ([E] int32), for moe_layer.slot_table, and the
 * device address of that layer's slot 0, for moe_layer.pool. */
moe_status slot_pool_layer(slot_pool *p, int32_t layer, const int32_t **table_dev,
                           const void **pool_base_dev);

/* Copy of the host table row of `layer` into table_host [E]. */
moe_status slot_pool_table_host(slot_pool *p, int32_t layer, int32_t *table_host);

/* The resident part of one layer: router, optional router bias, shared-gate
 * vector and shared-expert blob (device pointers, as in moe_layer). */
typedef struct {
    const void *w_router;
    const float *router_bias;
    const void *w_shared_gate;
    const void *shared_blob;
} moe_resident_weights;

/* One layer of a pooled stack, end to end: route x on `stream`, read the
 * top-k ids back to the host (the one synchronisation of `stream`), apply the
 * pool policy, fill the misses on the pool's side stream, make `stream` wait
 * for the fills, then run the experts from the pool.  A pool in device mode
 * (slot_pool_enable_device) does the lookup and fills as kernels on `stream`
 * instead, with no synchronisation.  T tokens; their
 * distinct experts must fit the layer's slots (MOE_ERR_POOL_EXHAUSTED
 * otherwise).  x, y, y_f32 (nullable), topk_idx_out (nullable) and workspace
 * (moe_layer_workspace_bytes) are device pointers. */
moe_status moe_pooled_layer_forward(const moe_config *cfg, slot_pool *p, int32_t layer,
                                    const moe_resident_weights *w, const void *x, int32_t T, void *y,
                                    float *y_f32, int32_t *topk_idx_out, void *workspace,
                                    size_t ws_bytes, cudaStream_t stream);

/* Storage tier below host memory: a pool whose backing store is a file of
 * fixed-stride blobs, expert e of layer l at file_offset + (l * E + e) *
 * file_stride (file_stride and file_offset multiples of 4096, file_stride at
 * least the blob rounded up to 4096), as written by the caller (the blob
 * bytes of moe_pack_expert, zero padded).  The file is opened read-only with
 * O_DIRECT where the file system allows it (else buffered).  A fill reads
 * each missing blob with pread, `readers` (1..64) host threads at a time,
 * into one of 16 pinned staging buffers whose previous copy has finished,
 * then copies it to its slot on side_stream: one read and one copy per
 * expert.  The device slots are the blob size rounded up to 256 bytes apart
 * (pool_bytes >= n_layers * slots_per_layer * that).  The policy runs on the
 * host (slot_pool_enable_device is refused).  slot_pool_file_stats: bytes
 * read, nanoseconds spent in the reads, and whether they bypass the page
 * cache (direct = 1). */
moe_status slot_pool_create_file(const moe_config *cfg, int32_t n_layers, int32_t slots_per_layer,
                                 void *pool_dev, size_t pool_bytes, const char *path, size_t file_offset,
                                 size_t file_stride, int32_t readers, cudaStream_t side_stream,
                                 slot_pool **out);
moe_status slot_pool_file_stats(slot_pool *p, int64_t *bytes_read, int64_t *read_ns, int32_t *direct);

/* Device-side policy.  slot_pool_enable_device switches a pool that has
 * served no host lookup to running its rule on the device: the same rule,
 * the same tie breaks and the same clock as slot_pool_lookup, kept in device
 * copies of the use counts, stamps and slot owners.  Its fills are read by a
 * kernel straight from the backing store, which must then be pinned host
 * memory the device can address (MOE_ERR_UNSUPPORTED otherwise); at most
 * 2048 slots per layer.  From then on the host lookup and fill calls are
 * refused, slot_pool_table_host and slot_pool_stats copy from the device
 * (exposed_copy_ns stays 0), and moe_pooled_layer_forward enqueues route,
 * lookup, fills and experts on its stream with no host synchronisation, so
 * a stack of layers can be captured in one CUDA graph.  Device-mode calls on
 * one pool must be ordered (one stream, or events between streams).
 *
 * slot_pool_step_device: one lookup of the n expert ids at ids_dev (device)
 * for `layer`, and the fills it needs, enqueued on `stream`.  Bad ids record
 * MOE_ERR_DEVICE_FAULT, more distinct ids than slots MOE_ERR_POOL_EXHAUSTED,
 * in the device error word (moe_get_device_error); the lookup is then
 * skipped. */
moe_status slot_pool_enable_device(slot_pool *p);
moe_status slot_pool_step_device(slot_pool *p, int32_t layer, const int32_t *ids_dev, int32_t n,
                                 cudaStream_t stream);

moe_status slot_pool_stats(slot_pool *p, moe_pool_stats *out);
void slot_pool_destroy(slot_pool *p);

/* ---------------------------------------------------------------- errors */

/* Read and clear the error word of the current device after the work on
 * `stream` has finished (synchronises the stream).  MOE_OK if no kernel
 * recorded a fault. */
moe_status moe_get_device_error(cudaStream_t stream);

/* Message of the last failing call on this thread ("" if none). */
const char *moe_last_error_message(void);

/* Library version string. */
const char *moe_version(void);

/* Kernel selection for calls made from the calling host thread (the setting
 * is per thread): 0 (default) uses the single-token kernels for T = 1 (and
 * once a token for T = 2 .. 12), the generic kernels up to T = 63 and the
 * tcgen05 grouped GEMMs for T >= 64 where the shape allows; 1 forces the
 * generic kernels everywhere; 2 is 0 with the grouped GEMMs from T = 2 up
 * (small decode batches on the tensor cores).  All compute the same
 * function (the pages' practice of checking fast against scalar kernels);
 * tests compare each against the CPU oracle.  The workspace size a call
 * needs depends on the path: query moe_*_workspace_bytes under the same
 * setting.  MOE_ERR_INVALID_ARG for other values. */
moe_status moe_set_kernel_path(int32_t path);

/* Test hooks, process-wide, for exercising the failure path of bounded
 * device waits without a fault: every wait a kernel of this library makes
 * gives up after wait_ns (default 200,000,000 = 0.2 s) and records
 * MOE_ERR_TIMEOUT; extra_arrivals (default 0, at most 4) is added to the
 * arrivals the single-token down kernel's copy barrier expects, so that with
 * extra_arrivals > 0 that wait always runs out.  After giving up, the kernel
 * supplies those arrivals itself, waits for its copies to land, writes zeros
 * for the affected outputs and returns.  Synchronous (cudaMemcpyToSymbol on
 * the current device); MOE_ERR_INVALID_ARG for wait_ns == 0 or
 * extra_arrivals outside [0, 4].  Not for production use. */
moe_status moe_debug_set_waits(uint64_t wait_ns, int32_t extra_arrivals);

#ifdef __cplusplus
}
#endif
#endif /* MOE_INT4_H */
