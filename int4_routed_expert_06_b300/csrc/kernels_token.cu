// Single-token (batch-1 decode) path of the routed int4 MoE layer on B300.
//
// Three kernels chained with programmatic dependent launch (PDL).  Each kernel
// lets its successor launch as soon as it starts, loads what does not depend
// on its predecessor's output (weights, the slot table) before
// griddepcontrol.wait, and reads its predecessor's outputs and writes its own
// only after the wait, so a successor never races a kernel that still reads
// a buffer it is about to overwrite.
//
//   router_tok  one warp per router row (E experts, then the shared-gate
//               row), the row's bf16 weights held in registers before the
//               wait; after it, x is read and the logits written.  A few
//               extra CTAs convert x into the fixed-point chunk records the
//               expert kernels use.
//   gateup_tok  one CTA per SM.  Before the wait: the CTA's share of the
//               shared expert's gate/up rows is bulk-copied into shared
//               memory and the expert->slot table is staged.  After it: top-k
//               from the logits (one warp per CTA, every CTA), bulk copies of
//               the CTA's share of the routed rows (one lane per copy, so
//               they issue in parallel), then a = silu(W_g x) * (W_u x) row
//               by row as the bytes land.
//   down_tok    one CTA per SM, owning output rows [h0, h1) of every active
//               expert.  Before the wait: top-k again and bulk copies of its
//               rows of every active expert's W_d (they stream while gate/up
//               runs).  After it: a is converted to fixed-point records in
//               shared memory and
//                 y[h] = sum_r w_r (W_d,r a_r)[h] + sigmoid(s) (W_d,sh a_sh)[h]
//               is accumulated in a fixed order.
//
// Code on the critical path is kept small and loop-shaped: these kernels run
// once per token on every SM, and long unrolled stretches stall on
// instruction fetch.
//
// Dot products (the affine int4 format of MLX group quantisation, named on
// the Swiftlet project page, "Relation to TurboFieldfare"): with
// W = s q + b per group,
//   sum_c W_c v_c = s * sum_c q_c v_c + b * sum_c v_c.
// The integer part sum_c q_c v_c runs on dp4a.  The vector v (x, or a) is
// carried per 32-column chunk in 16-bit fixed point, v_c ~ sx * (256 xh_c +
// xl_c) with xh_c a signed and xl_c an unsigned byte and sx = max|v| / 32767
// over the chunk; the step sx is below the bf16 rounding step of the chunk's
// largest element, so this adds less error than storing the chunk in bf16.
// Codes are split into their even and odd nibbles with two LOP3s per word,
// and each 4-column byte group takes one dp4a per fixed-point byte.
// sum_c v_c is taken in fp32 from the unrounded values.
#include <float.h>
#include <math.h>

#include "internal.h"

namespace moe {
namespace tok {

constexpr int kMaxAct = 17;                          // top_k <= 16 plus the shared expert
constexpr int kMaxSeg = 2;                           // gate/up segments per CTA
constexpr int kParts = 1;                            // row parts per segment, one barrier each
constexpr int kMaxE = 1024;                          // experts the staged tables hold
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;   // 0.2 s bound on any barrier wait
constexpr int kRec = 80;                             // bytes per fixed-point chunk record
constexpr int kGuThreads = 256;
constexpr int kDnThreads = 512;

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy completing on `bar`.  Both addresses 16-byte
// aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase 0 of a single-use barrier for at most kWaitNs; false (with
// MOE_ERR_TIMEOUT recorded) if it never completes.
__device__ __noinline__ bool mbar_wait0(uint64_t *bar)
{
    if (mbar_try_wait(bar, 0))
        return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, 0))
            return true;
        if (global_ns() - t0 > kWaitNs) {
            record_error(MOE_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ------------------------------------------------------------ fixed-point chunks

// One 32-column chunk of a vector in the dp4a form.  Word m covers columns
// 8m..8m+7; byte j of he/le holds column 8m+2j (the even nibble j of code
// word m), byte j of ho/lo column 8m+2j+1.  Record in memory: he[4] le[4]
// ho[4] lo[4] (64 B), then sx, X, and 8 bytes of padding (kRec bytes).
struct Chunk {
    uint4 he, le, ho, lo;
    float sx, X;
};

__device__ __forceinline__ Chunk load_chunk(const unsigned char *rec)
{
    Chunk c;
    const uint4 *p = reinterpret_cast<const uint4 *>(rec);
    c.he = p[0];
    c.le = p[1];
    c.ho = p[2];
    c.lo = p[3];
    const float2 f = *reinterpret_cast<const float2 *>(rec + 64);
    c.sx = f.x;
    c.X = f.y;
    return c;
}

// The same from global memory through L2 (written by an earlier kernel).
__device__ __forceinline__ Chunk load_chunk_global(const unsigned char *rec)
{
    Chunk c;
    const uint4 *p = reinterpret_cast<const uint4 *>(rec);
    c.he = __ldcg(p);
    c.le = __ldcg(p + 1);
    c.ho = __ldcg(p + 2);
    c.lo = __ldcg(p + 3);
    const float2 f = __ldcg(reinterpret_cast<const float2 *>(rec + 64));
    c.sx = f.x;
    c.X = f.y;
    return c;
}

// Convert 32 values, 4 consecutive ones per lane in each aligned group of 8
// lanes (lane & 7 = position), into one chunk record, stored at rec and at
// nrep - 1 further copies `stride` bytes apart.  All 32 lanes call it; lanes
// with valid == false (a ragged tail) store nothing.
__device__ __forceinline__ void store_chunk4(const float v[4], unsigned char *rec, int lane, bool valid = true,
                                             int nrep = 1, size_t stride = 0)
{
    const int p = lane & 7;
    float am = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 4));
    float X = (v[0] + v[1]) + (v[2] + v[3]);
    X += __shfl_xor_sync(0xFFFFFFFFu, X, 1);
    X += __shfl_xor_sync(0xFFFFFFFFu, X, 2);
    X += __shfl_xor_sync(0xFFFFFFFFu, X, 4);
    const bool nz = am > 0.f && am < INFINITY;
    const float inv = nz ? 32767.0f / am : 0.f;
    // v * inv + 1.5*2^23: the low 16 bits are rint(v * inv) in two's complement
    uint32_t f[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        f[j] = __float_as_uint(fmaf(v[j], inv, 12582912.0f));
    // [xl(c0), xl(c2), xh(c0), xh(c2)] and the same for c1, c3
    const uint32_t te = __byte_perm(f[0], f[2], 0x5140);
    const uint32_t to = __byte_perm(f[1], f[3], 0x5140);
    if (!valid)
        return;
    const int m = p >> 1, half = p & 1;
    const float2 tail = make_float2(nz ? am / 32767.0f : 0.f, X);
    for (int r = 0; r < nrep; ++r) {
        unsigned char *rr = rec + (size_t)r * stride;
        unsigned short *h = reinterpret_cast<unsigned short *>(rr);
        // he at byte 0, le at 16, ho at 32, lo at 48; this lane fills
        // halfword `half` of word m of each.
        h[2 * m + half] = (unsigned short)(te >> 16);
        h[8 + 2 * m + half] = (unsigned short)(te & 0xFFFFu);
        h[16 + 2 * m + half] = (unsigned short)(to >> 16);
        h[24 + 2 * m + half] = (unsigned short)(to & 0xFFFFu);
        if (p == 0)
            *reinterpret_cast<float2 *>(rr + 64) = tail;
    }
}

// store_chunk4 for U independent groups of values at once (the shuffle
// chains of the U conversions overlap); rec[u] == nullptr stores nothing.
template <int U>
__device__ __forceinline__ void store_chunks4(const float4 (&f)[U], unsigned char *const (&rec)[U], int lane)
{
    float am[U], X[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        am[u] = fmaxf(fmaxf(fabsf(f[u].x), fabsf(f[u].y)), fmaxf(fabsf(f[u].z), fabsf(f[u].w)));
        X[u] = (f[u].x + f[u].y) + (f[u].z + f[u].w);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
        for (int u = 0; u < U; ++u) {
            am[u] = fmaxf(am[u], __shfl_xor_sync(0xFFFFFFFFu, am[u], o));
            X[u] += __shfl_xor_sync(0xFFFFFFFFu, X[u], o);
        }
    const int p = lane & 7, m = p >> 1, half = p & 1;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool nz = am[u] > 0.f && am[u] < INFINITY;
        const float inv = nz ? 32767.0f / am[u] : 0.f;
        const uint32_t f0 = __float_as_uint(fmaf(f[u].x, inv, 12582912.0f));
        const uint32_t f1 = __float_as_uint(fmaf(f[u].y, inv, 12582912.0f));
        const uint32_t f2 = __float_as_uint(fmaf(f[u].z, inv, 12582912.0f));
        const uint32_t f3 = __float_as_uint(fmaf(f[u].w, inv, 12582912.0f));
        const uint32_t te = __byte_perm(f0, f2, 0x5140);
        const uint32_t to = __byte_perm(f1, f3, 0x5140);
        if (rec[u]) {
            unsigned short *h = reinterpret_cast<unsigned short *>(rec[u]);
            h[2 * m + half] = (unsigned short)(te >> 16);
            h[8 + 2 * m + half] = (unsigned short)(te & 0xFFFFu);
            h[16 + 2 * m + half] = (unsigned short)(to >> 16);
            h[24 + 2 * m + half] = (unsigned short)(to & 0xFFFFu);
            if (p == 0)
                *reinterpret_cast<float2 *>(rec[u] + 64) = make_float2(nz ? am[u] / 32767.0f : 0.f, X[u]);
        }
    }
}

// sum_c q_c * (256 xh_c + xl_c) over one chunk of 32 codes (exact integer),
// in four short dp4a chains.
__device__ __forceinline__ int chunk_idot(uint4 q, const Chunk &c)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    const uint32_t he[4] = {c.he.x, c.he.y, c.he.z, c.he.w};
    const uint32_t le[4] = {c.le.x, c.le.y, c.le.z, c.le.w};
    const uint32_t ho[4] = {c.ho.x, c.ho.y, c.ho.z, c.ho.w};
    const uint32_t lo[4] = {c.lo.x, c.lo.y, c.lo.z, c.lo.w};
    int h0 = 0, h1 = 0, l0 = 0, l1 = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t ev = w[m] & 0x0F0F0F0Fu;
        const uint32_t od = (w[m] >> 4) & 0x0F0F0F0Fu;
        h0 = dp4a_us(ev, he[m], h0);
        h1 = dp4a_us(od, ho[m], h1);
        l0 = dp4a_uu(ev, le[m], l0);
        l1 = dp4a_uu(od, lo[m], l1);
    }
    return (h0 + h1) * 256 + (l0 + l1);
}

// s * sum_c q_c v_c + b * sum_c v_c for one chunk.
__device__ __forceinline__ float chunk_term(uint4 q, const Chunk &c, float s, float b)
{
    const float D = (float)chunk_idot(q, c) * c.sx;
    return fmaf(s, D, b * c.X);
}

template <typename TS> __device__ __forceinline__ float ld_sb(const TS *p) { return to_f32(*p); }

// ------------------------------------------------------------ top-k

// Does (va, ea) rank before (vb, eb) under (logit descending, id ascending)?
__device__ __forceinline__ bool ranks_before(float va, int ea, float vb, int eb)
{
    return va > vb || (va == vb && ea < eb);
}

// Routing keys: one 64-bit unsigned integer per logit whose order is the
// routing order (logit descending, then expert id ascending): the logit's bits
// mapped to an unsigned order in the high word (NaN as -inf), the complement
// of the id in the low word.
__device__ __forceinline__ unsigned long long route_key(float f, int e)
{
    uint32_t u = __float_as_uint(isnan(f) ? -INFINITY : f);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)e);
}
__device__ __forceinline__ float key_logit(unsigned long long key)
{
    uint32_t u = (uint32_t)(key >> 32);
    u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(u);
}
__device__ __forceinline__ int key_expert(unsigned long long key) { return (int)(0xFFFFFFFFu - (uint32_t)key); }

// Shared scratch of one warp's top-k.
struct TopkSmem {
    unsigned long long lm[32];   // lane maxima
    unsigned long long cand[32]; // candidates
    unsigned long long sel[16];  // the top k in rank order
};

// Top-k of the E <= 32*PER logits at lg (global, written by an earlier
// kernel) by one warp.  Fills s_idx[r] / s_w[r] for r < k with the r-th
// expert and its renormalised weight exp(l_r - l_0) / sum_{j<k} exp(l_j - l_0)
// (and idx_out / w_out when idx_out is non-NULL).
//
// Lane l holds the keys of experts l + 32 j in registers.  T = the k-th
// largest of the 32 lane maxima: every member of the top k is >= T, since k
// lane maxima are.  The candidates (keys >= T, usually about k of them) are
// ranked by counting over shared-memory broadcast reads.  If a lane holds
// more than two candidates, or there are more than 32, rounds of warp
// arg-max pick the same list instead.
template <int PER>
__device__ __noinline__ void warp_topk(const float *lg, int E, int k, int lane, TopkSmem &S, int *s_idx,
                                       float *s_w, int32_t *idx_out, float *w_out)
{
    unsigned long long kv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        kv[j] = e < E ? route_key(__ldcg(lg + e), e) : 0ull;
    }
    unsigned long long m[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j)
        m[j] = kv[j];
#pragma unroll
    for (int w = PER / 2; w > 0; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j)
            m[j] = max(m[j], m[j + w]);
    S.lm[lane] = m[0];
    __syncwarp();
    int rank = 0;
#pragma unroll
    for (int o = 0; o < 32; o += 2) {
        const ulonglong2 q = *reinterpret_cast<const ulonglong2 *>(&S.lm[o]);
        rank += (q.x > m[0] ? 1 : 0) + (q.y > m[0] ? 1 : 0);
    }
    const unsigned long long T = S.lm[__ffs(__ballot_sync(0xFFFFFFFFu, rank == k - 1)) - 1];
    int cnt = 0;
    unsigned long long c1 = 0, c2 = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const bool ge = kv[j] >= T;
        c2 = (ge && cnt == 1) ? kv[j] : c2;
        c1 = (ge && cnt == 0) ? kv[j] : c1;
        cnt += ge ? 1 : 0;
    }
    const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, cnt >= 1), b2 = __ballot_sync(0xFFFFFFFFu, cnt >= 2);
    const bool many = __any_sync(0xFFFFFFFFu, cnt > 2);
    const int C = __popc(b1) + __popc(b2);
    if (!many && C <= 32) {
        const uint32_t lt = (1u << lane) - 1u;
        const int p1 = __popc(b1 & lt) + __popc(b2 & lt);
        if (cnt >= 1)
            S.cand[p1] = c1;
        if (cnt >= 2)
            S.cand[p1 + 1] = c2;
        __syncwarp();
        const unsigned long long cv = lane < C ? S.cand[lane] : 0ull;
        int r = 0;
        for (int o = 0; o < C; o += 2) {
            const ulonglong2 q = *reinterpret_cast<const ulonglong2 *>(&S.cand[o]);
            r += (q.x > cv ? 1 : 0) + ((o + 1 < C && q.y > cv) ? 1 : 0);
        }
        if (lane < C && r < k)
            S.sel[r] = cv;
    } else {
        unsigned long long prev = ~0ull;
        for (int r = 0; r < k; ++r) {
            unsigned long long best = 0;
#pragma unroll
            for (int j = 0; j < PER; ++j)
                best = (kv[j] < prev && kv[j] > best) ? kv[j] : best;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                best = max(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
            if (lane == 0)
                S.sel[r] = best;
            prev = best;
        }
    }
    __syncwarp();
    const float l0 = key_logit(S.sel[0]);
    float sv = -INFINITY;
    int se = 0;
    if (lane < k) {
        const unsigned long long q = S.sel[lane];
        sv = key_logit(q);
        se = key_expert(q);
    }
    const float ex = lane < k ? expf(sv - l0) : 0.f;
    const float wv = ex / warp_sum(ex);
    if (lane < k) {
        s_idx[lane] = se;
        s_w[lane] = wv;
        if (idx_out) {
            idx_out[lane] = se;
            w_out[lane] = wv;
        }
    }
    __syncwarp();
}

// Routing of this token into s_idx / s_w (shared memory), from logits copy
// `rep` or from the given idx / w.  Warp 0 only.
__device__ __forceinline__ void load_routing(const Routing &R, int rep, int E, int k, int lane, int *s_idx,
                                             float *s_w, TopkSmem &S, bool write_out)
{
    if (R.logits) {
        const float *lg = R.logits + (size_t)rep * R.lgs;
        int32_t *io = write_out ? R.idx_out : nullptr;
        if (E <= 256)
            warp_topk<8>(lg, E, k, lane, S, s_idx, s_w, io, R.w_out);
        else if (E <= 512)
            warp_topk<16>(lg, E, k, lane, S, s_idx, s_w, io, R.w_out);
        else
            warp_topk<32>(lg, E, k, lane, S, s_idx, s_w, io, R.w_out);
    } else {
        if (lane < k) {
            s_idx[lane] = __ldcg(R.idx + lane);
            s_w[lane] = __ldcg(R.w + lane);
        }
        __syncwarp();
    }
}

// Blob address of expert e through a slot table, or nullptr (recorded).
__device__ __forceinline__ const char *routed_base(const ExpertSrc &src, const int *table, int e)
{
    if (e < 0 || e >= src.n_experts) {
        record_error(MOE_ERR_DEVICE_FAULT);
        return nullptr;
    }
    const int slot = table[e];
    if (slot < 0 || slot >= src.n_slots) {
        record_error(MOE_ERR_NOT_RESIDENT);
        return nullptr;
    }
    return src.pool + (size_t)slot * src.stride;
}

// ------------------------------------------------------------ router

// CTAs [0, n_row_ctas): one warp per row (rows 0..E-1 experts, row E the
// shared gate).  CTAs after them: x -> fixed-point records (each warp four
// 32-column chunks), written in kRep copies.  128 threads.  H = 256 * NJ.
template <int NJ>
__global__ void __launch_bounds__(128) router_tok_kernel(const __nv_bfloat16 *__restrict__ x, int E,
                                                        const __nv_bfloat16 *__restrict__ wr,
                                                        const float *__restrict__ bias,
                                                        const __nv_bfloat16 *__restrict__ wsg,
                                                        float *__restrict__ lg, int lgs, int nrep,
                                                        float *__restrict__ sg, unsigned char *__restrict__ xrec,
                                                        size_t xrs, int n_row_ctas)
{
    constexpr int H = 256 * NJ;
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((int)blockIdx.x >= n_row_ctas) {
        // fixed-point records of x: warp v converts chunks 4v .. 4v+3
        const int v = ((int)blockIdx.x - n_row_ctas) * 4 + warp;
        const int q = v * 32 + lane; // 4-column quad of x
        pdl_wait();
        if (v * 128 < H) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(x) + q);
            const float f[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                                __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
            store_chunk4(f, xrec + (size_t)(q >> 3) * kRec, lane, true, kRep, xrs);
        }
        return;
    }
    const int row = blockIdx.x * 4 + warp;
    const int nrows = E + (wsg ? 1 : 0);
    uint4 wv[NJ];
    const bool active = row < nrows;
    if (active) {
        const __nv_bfloat16 *w = row < E ? wr + (size_t)row * H : wsg;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            wv[j] = __ldcs(reinterpret_cast<const uint4 *>(w + (lane + 32 * j) * 8));
    }
    pdl_wait();
    if (!active)
        return;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + (lane + 32 * j) * 8));
        const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t wa[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            acc0 = fmaf(__uint_as_float(wa[m] << 16), __uint_as_float(xa[m] << 16), acc0);
            acc1 = fmaf(__uint_as_float(wa[m] & 0xFFFF0000u), __uint_as_float(xa[m] & 0xFFFF0000u), acc1);
        }
    }
    const float acc = warp_sum(acc0 + acc1);
    if (lane < nrep) {
        if (row < E)
            lg[(size_t)lane * lgs + row] = acc + (bias ? bias[row] : 0.f);
        else if (lgs > 0)
            lg[(size_t)lane * lgs + E] = acc;
    }
    if (lane == 0 && row == E && sg)
        *sg = acc;
}

// ------------------------------------------------------------ gate/up

struct GateUpArgs {
    const unsigned char *xrec; // [kRep][xrs] fixed-point records of x
    size_t xrs;
    ExpertSrc src;
    Routing R;
    float *a;                  // [kRep][as]: [k+1][Imax] each
    size_t as;
    int E, k, I, Is, Imax, log2G;
};

// Rows [o0, o0 + n) of active expert i (i == k: shared) at shared-memory
// byte offset `off`.
struct Seg {
    int i, o0, n;
    uint32_t off;
};

// This CTA's rows of the flat list [shared rows | rank 0 rows | rank 1 ...],
// as at most kMaxSeg segments (the host checks that a share is no longer
// than the shortest expert, so it crosses at most one boundary).
__device__ __forceinline__ int gateup_segments(int c, int n, int k, int I, int Is, uint32_t rowpair, Seg *seg)
{
    const long R = (long)Is + (long)k * I;
    int r = (int)((long)c * R / n);
    const int r1 = (int)((long)(c + 1) * R / n);
    int ns = 0;
    uint32_t off = 0;
    while (r < r1 && ns < kMaxSeg) {
        int i, o, len;
        if (r < Is) {
            i = k;
            o = r;
            len = min(r1, Is) - r;
        } else {
            i = (r - Is) / I;
            o = (r - Is) - i * I;
            len = min(r1 - r, I - o);
        }
        seg[ns++] = Seg{i, o, len, off};
        off += (uint32_t)len * rowpair;
        r += len;
    }
    return ns;
}

// Part p of a segment of n rows: rows [p n / kParts, (p+1) n / kParts); the
// part of row r is floor(((r + 1) kParts - 1) / n).
__device__ __forceinline__ int part_begin(int n, int p) { return p * n / kParts; }
__device__ __forceinline__ int part_of(int n, int r) { return ((r + 1) * kParts - 1) / n; }

// H = 1024 * NXC; TS = scale/bias type.  One CTA per SM.
//
// Shared memory: the segments' rows (codes of gate, codes of up, then the
// four scale/bias arrays, per segment).  Each segment arrives in kParts row
// parts, each completing on its own barrier, so rows are computed while the
// rest of the share streams in.  Lane l takes chunks NXC l .. NXC l + NXC - 1
// of a row; a warp computes two rows per pass.
template <int NXC, typename TS>
__global__ void __launch_bounds__(kGuThreads, 2) gateup_tok_kernel(GateUpArgs A)
{
    constexpr int H = 1024 * NXC;
    constexpr int NW = kGuThreads / 32;
    constexpr int XQ = (H / 32) * kRec / 16; // 16-byte pieces of the x records
    constexpr int XU = (XQ + kGuThreads - 33) / (kGuThreads - 32);
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bars[kMaxSeg][kParts];
    __shared__ int tab[kMaxE];
    __shared__ __align__(16) unsigned char xs[(H / 32) * kRec];
    __shared__ int s_idx[kMaxAct];
    __shared__ float s_w[kMaxAct];
    __shared__ const char *s_base[kMaxSeg];
    __shared__ __align__(16) TopkSmem tks;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = gridDim.x, c = blockIdx.x, rep = c % kRep;
    const int k = A.k;
    const int HG = H >> A.log2G;                     // groups per row
    const uint32_t qrow = H / 2;                     // code bytes per row
    const uint32_t srow = (uint32_t)HG * sizeof(TS); // scale (or bias) bytes per row
    const uint32_t rowpair = 2 * qrow + 4 * srow;

    Seg seg[kMaxSeg];
    const int nseg = gateup_segments(c, n, k, A.I, A.Is, rowpair, seg);

    // Copy m (0..5: gate codes, up codes, gate scales, gate biases, up
    // scales, up biases) of part p of segment s.
    auto issue = [&](int s, int p, int m, const char *base) {
        const Seg &g = seg[s];
        const int r0 = part_begin(g.n, p), nrow = part_begin(g.n, p + 1) - r0;
        if (nrow <= 0)
            return;
        const size_t *offs = (g.i == k) ? A.src.off_sh : A.src.off;
        const uint32_t n_q = (uint32_t)g.n * qrow, n_s = (uint32_t)g.n * srow;
        const int mat = m == 0 ? M_QG : m == 1 ? M_QU : m == 2 ? M_SG : m == 3 ? M_BG : m == 4 ? M_SU : M_BU;
        const uint32_t rb = m < 2 ? qrow : srow;
        const uint32_t doff = (m < 2 ? (uint32_t)m * n_q : 2 * n_q + (uint32_t)(m - 2) * n_s) + (uint32_t)r0 * rb;
        bulk_g2s(smem + g.off + doff, base + offs[mat] + (size_t)(g.o0 + r0) * rb, (uint32_t)nrow * rb, &bars[s][p]);
    };
    auto arm = [&](int s, int p, bool full) {
        const int nrow = part_begin(seg[s].n, p + 1) - part_begin(seg[s].n, p);
        if (nrow > 0)
            mbar_expect_tx(&bars[s][p], full ? (uint32_t)nrow * rowpair : 0u);
    };

    // ---- before the wait: nothing here depends on the router's output
    const bool sh0 = nseg > 0 && seg[0].i == k;
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < kMaxSeg; ++s)
                for (int p = 0; p < kParts; ++p)
                    mbar_init(&bars[s][p], 1);
            fence_mbar_init();
            if (sh0) {
                s_base[0] = A.src.shared;
                for (int p = 0; p < kParts; ++p)
                    arm(0, p, true);
            }
        }
        __syncwarp();
        if (sh0 && lane < 6 * kParts)
            issue(0, lane / 6, lane % 6, A.src.shared);
    }
    for (int e = threadIdx.x; e < A.E; e += kGuThreads)
        tab[e] = __ldg(A.src.table + e);
    __syncthreads();

    // ---- after the wait: warp 0 selects the top k and issues the routed
    // copies, the other warps stage the x records meanwhile
    pdl_wait();
    if (warp == 0) {
        load_routing(A.R, rep, A.E, k, lane, s_idx, s_w, tks, c == 0);
        // lane s kParts + p arms part p of segment s
        const int ls = lane / kParts, lp = lane % kParts;
        const char *b = nullptr;
        if (ls < nseg && seg[ls].i != k) {
            b = routed_base(A.src, tab, s_idx[seg[ls].i]);
            if (lp == 0)
                s_base[ls] = b;
            arm(ls, lp, b != nullptr);
        }
        __syncwarp();
        // copy q = lane + 32 t is copy q % 6 of part (q / 6) % kParts of segment q / (6 kParts)
        for (int q = lane; q < 6 * kParts * nseg; q += 32) {
            const int s = q / (6 * kParts), p = (q / 6) % kParts, m = q % 6;
            if (seg[s].i != k && s_base[s])
                issue(s, p, m, s_base[s]);
        }
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(A.xrec + (size_t)rep * A.xrs);
        uint4 *dst = reinterpret_cast<uint4 *>(xs);
        uint4 v[XU];
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int q = threadIdx.x - 32 + u * (kGuThreads - 32);
            if (q < XQ)
                v[u] = __ldcg(src + q);
        }
#pragma unroll
        for (int u = 0; u < XU; ++u) {
            const int q = threadIdx.x - 32 + u * (kGuThreads - 32);
            if (q < XQ)
                dst[q] = v[u];
        }
    }
    __syncthreads();
    // down may launch now: its prologue (its own top-k and weight copies)
    // would otherwise compete with the routed copies issued above
    pdl_trigger();

    Chunk xv[NXC];
#pragma unroll
    for (int m = 0; m < NXC; ++m)
        xv[m] = load_chunk(xs + (size_t)(NXC * lane + m) * kRec);
    int grp[NXC];
#pragma unroll
    for (int m = 0; m < NXC; ++m)
        grp[m] = ((NXC * lane + m) * 32) >> A.log2G;

    const int total = nseg == 0 ? 0 : (int)(seg[nseg - 1].off / rowpair) + seg[nseg - 1].n;
    uint32_t waited = 0; // bit s * kParts + p: part p of segment s has landed
#pragma unroll 1
    for (int rho0 = warp; rho0 < total; rho0 += 2 * NW) {
        float gacc[2] = {0.f, 0.f}, uacc[2] = {0.f, 0.f};
        float *dst[2] = {nullptr, nullptr};
        bool ok = true;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int rho = rho0 + t * NW;
            if (rho >= total)
                continue;
            int s = 0, r = rho;
            if (nseg > 1 && r >= seg[0].n) {
                r -= seg[0].n;
                s = 1;
            }
            const Seg &g = seg[s];
            const uint32_t bit = 1u << (s * kParts + part_of(g.n, r));
            if (!(waited & bit)) {
                // warp-uniform outcome, so no lane leaves the shuffles below
                if (!__all_sync(0xFFFFFFFFu, mbar_wait0(&bars[s][part_of(g.n, r)]))) {
                    ok = false;
                    continue;
                }
                waited |= bit;
            }
            dst[t] = A.a + (size_t)g.i * A.Imax + g.o0 + r;
            if (s_base[s] == nullptr)
                continue;
            const uint32_t n_q = (uint32_t)g.n * qrow, n_s = (uint32_t)g.n * srow;
            const unsigned char *d = smem + g.off;
            const uint4 *qg = reinterpret_cast<const uint4 *>(d + (size_t)r * qrow);
            const uint4 *qu = reinterpret_cast<const uint4 *>(d + n_q + (size_t)r * qrow);
            const TS *sg = reinterpret_cast<const TS *>(d + 2 * n_q) + (size_t)r * HG;
            const TS *bg = reinterpret_cast<const TS *>(d + 2 * n_q + n_s) + (size_t)r * HG;
            const TS *su = reinterpret_cast<const TS *>(d + 2 * n_q + 2 * n_s) + (size_t)r * HG;
            const TS *bu = reinterpret_cast<const TS *>(d + 2 * n_q + 3 * n_s) + (size_t)r * HG;
#pragma unroll
            for (int m = 0; m < NXC; ++m) {
                const int ch = NXC * lane + m;
                gacc[t] += chunk_term(qg[ch], xv[m], ld_sb(sg + grp[m]), ld_sb(bg + grp[m]));
                uacc[t] += chunk_term(qu[ch], xv[m], ld_sb(su + grp[m]), ld_sb(bu + grp[m]));
            }
        }
        if (!ok)
            return;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            gacc[0] += __shfl_xor_sync(0xFFFFFFFFu, gacc[0], o);
            uacc[0] += __shfl_xor_sync(0xFFFFFFFFu, uacc[0], o);
            gacc[1] += __shfl_xor_sync(0xFFFFFFFFu, gacc[1], o);
            uacc[1] += __shfl_xor_sync(0xFFFFFFFFu, uacc[1], o);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (dst[t] && lane < kRep)
                dst[t][(size_t)lane * A.as] = gacc[t] * sigmoid_f(gacc[t]) * uacc[t];
    }
}

// ------------------------------------------------------------ down + combine

struct DownArgs {
    ExpertSrc src;
    Routing R;
    const float *a;         // [kRep][as]: [k+1][Imax] each
    size_t as;
    __nv_bfloat16 *y;
    float *y32;
    int E, H, k, I, Is, Imax, log2G, n_act;
};

// CTA c owns output rows [h0, h1), nr = h1 - h0 <= 16.  Shared memory: per
// active expert i its rows' codes [nr][I_i/2], scales and biases
// [nr][I_i/G] each; then the fixed-point records of a, [n_act][Imax/32].
//
// Warp w computes output row w: lane l & 15 takes chunks l, l+16, ... of the
// row for the experts of parity l >> 4 (rank order, shared expert last), and
// the warp sums its lanes in a fixed tree, so the order of the sum does not
// depend on where the experts live.
template <typename TS>
__global__ void __launch_bounds__(kDnThreads, 2) down_tok_kernel(DownArgs A)
{
    constexpr int kBatch = 4; // float4 loads of a in flight per thread
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bar;
    __shared__ int s_idx[kMaxAct];
    __shared__ float s_w[kMaxAct + 1];
    __shared__ const char *s_base[kMaxAct];
    __shared__ uint32_t s_eoff[kMaxAct + 1]; // shared-memory offset of expert i's rows
    __shared__ int s_qb[kMaxAct];            // code bytes per row of expert i
    __shared__ int s_ng[kMaxAct];            // groups per row of expert i
    __shared__ __align__(16) TopkSmem tks;

    pdl_trigger(); // the next layer call may start its own weight loads now

    const int n = gridDim.x, c = blockIdx.x, rep = c % kRep;
    const int h0 = (int)((long)c * A.H / n), h1 = (int)((long)(c + 1) * A.H / n);
    const int nr = h1 - h0;
    const int k = A.k, n_act = A.n_act;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sb = sizeof(TS);

    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        uint32_t o = 0;
        for (int i = 0; i < n_act; ++i) {
            const int inter = (i == k) ? A.Is : A.I;
            s_eoff[i] = o;
            s_qb[i] = inter / 2;
            s_ng[i] = inter >> A.log2G;
            o += (uint32_t)nr * ((uint32_t)inter / 2 + 2 * (uint32_t)(inter >> A.log2G) * sb);
        }
        s_eoff[n_act] = o;
        s_w[kMaxAct] = sigmoid_f(__ldcg(A.R.logits ? A.R.logits + (size_t)rep * A.R.lgs + A.E : A.R.sg_logit));
    }
    __syncthreads();
    if (warp == 0) {
        load_routing(A.R, rep, A.E, k, lane, s_idx, s_w, tks, false);
        const char *b = nullptr;
        uint32_t bytes = 0;
        if (lane < n_act) {
            b = lane == k ? A.src.shared : routed_base(A.src, A.src.table, s_idx[lane]);
            s_base[lane] = b;
            if (b)
                bytes = s_eoff[lane + 1] - s_eoff[lane];
        }
        const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, bytes);
        if (lane == 0)
            mbar_expect_tx(&bar, tot);
        __syncwarp();
        if (b) {
            const size_t *offs = (lane == k) ? A.src.off_sh : A.src.off;
            const uint32_t nq = (uint32_t)nr * s_qb[lane], ns = (uint32_t)nr * s_ng[lane] * sb;
            unsigned char *d = smem + s_eoff[lane];
            bulk_g2s(d, b + offs[M_QD] + (size_t)h0 * s_qb[lane], nq, &bar);
            bulk_g2s(d + nq, b + offs[M_SD] + (size_t)h0 * s_ng[lane] * sb, ns, &bar);
            bulk_g2s(d + nq + ns, b + offs[M_BD] + (size_t)h0 * s_ng[lane] * sb, ns, &bar);
        }
    }
    __syncthreads();
    unsigned char *arec = smem + ((s_eoff[n_act] + 15) & ~15u); // [n_act][nchm] records
    const int nchm = A.Imax >> 5;

    pdl_wait();
    // a -> fixed-point records; 8 lanes per 32-value chunk, kBatch loads in
    // flight per thread before any conversion
    {
        const int n4 = n_act * A.Imax / 4;
        const float4 *a4 = reinterpret_cast<const float4 *>(A.a + (size_t)rep * A.as);
#pragma unroll 1
        for (int q0 = 0; q0 < n4; q0 += kBatch * kDnThreads) {
            float4 f[kBatch];
            unsigned char *rec[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int q = q0 + u * kDnThreads + threadIdx.x;
                f[u] = q < n4 ? __ldcg(a4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                // chunk q >> 3 == (i * Imax + col) / 32 == i * nchm + col / 32
                rec[u] = q < n4 ? arec + (size_t)(q >> 3) * kRec : nullptr;
            }
            store_chunks4<kBatch>(f, rec, lane);
        }
    }
    __syncthreads();
    const bool ready = mbar_wait0(&bar);

    const int par = lane >> 4, l16 = lane & 15;
    const int hr = warp;
    float acc = 0.f;
    if (ready && hr < nr) {
        // experts par, par + 2, ... two at a time; every chunk's loads are
        // issued before any of its dot products.  Both half-warps run the
        // same number of passes (the warp-wide vote below needs every lane).
        constexpr int U = 2;
#pragma unroll 1
        for (int i0 = 0; i0 < n_act; i0 += 2 * U) {
            for (int ch0 = 0;; ch0 += 16) {
                uint4 q[U];
                Chunk av[U];
                float sc[U], bc[U], wi[U];
                bool any = false;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = i0 + 2 * u + par;
                    const int ic = min(i, n_act - 1);
                    const int qb = s_qb[ic], ng = s_ng[ic];
                    const int ch = ch0 + l16;
                    const bool live = i < n_act && s_base[ic] != nullptr && ch < (qb >> 4);
                    any |= ch0 < (qb >> 4) && i < n_act;
                    const int chc = live ? ch : 0;
                    const unsigned char *d = smem + s_eoff[ic];
                    const TS *sd = reinterpret_cast<const TS *>(d + nr * qb) + hr * ng;
                    const int g = (chc * 32) >> A.log2G;
                    q[u] = reinterpret_cast<const uint4 *>(d + hr * qb)[chc];
                    av[u] = load_chunk(arec + (size_t)(ic * nchm + chc) * kRec);
                    sc[u] = ld_sb(sd + g);
                    bc[u] = ld_sb(sd + nr * ng + g);
                    wi[u] = live ? ((i < k) ? s_w[i] : s_w[kMaxAct]) : 0.f;
                }
                if (!__any_sync(0xFFFFFFFFu, any))
                    break;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    acc = fmaf(wi[u], chunk_term(q[u], av[u], sc[u], bc[u]), acc);
            }
        }
    }
    acc = warp_sum(acc);
    if (ready && hr < nr && lane == 0) {
        A.y[h0 + hr] = __float2bfloat16_rn(acc);
        if (A.y32)
            A.y32[h0 + hr] = acc;
    }
}

// ------------------------------------------------------------ host side

static int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64)
        return 148;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 148;
    }
    return cached[dev];
}

template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, int grid, int block, size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

static int log2i(int v)
{
    int l = 0;
    while ((1 << l) < v)
        ++l;
    return l;
}

static size_t gateup_smem(const Shape &s, int n)
{
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    const size_t rowpair = (size_t)s.H + 4 * (size_t)(s.H / s.G) * sb;
    const long R = (long)s.Is + (long)s.k * s.I;
    return (size_t)((R + n - 1) / n) * rowpair;
}

static size_t down_smem(const Shape &s, int n)
{
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    const int nr = (s.H + n - 1) / n;
    const int n_act = s.k + 1;
    const int imax = s.I > s.Is ? s.I : s.Is;
    size_t w = 0;
    for (int i = 0; i < n_act; ++i) {
        const int inter = (i == s.k) ? s.Is : s.I;
        w += (size_t)nr * (inter / 2 + 2 * (inter / s.G) * sb);
    }
    w = (w + 15) & ~(size_t)15;
    return w + (size_t)kRec * n_act * (imax / 32);
}

constexpr size_t kSmemBudget = 100 * 1024; // a gate/up and a down CTA share an SM

bool eligible(const Shape &s)
{
    if (kernel_path() != 0)
        return false;
    if (s.act != MOE_BF16 || s.router != MOE_BF16)
        return false;
    if (s.H != 1024 && s.H != 2048)
        return false;
    if (s.Is <= 0 || s.k + 1 > kMaxAct || s.E > kMaxE)
        return false;
    const int sb = s.qscale == MOE_F16 ? 2 : 4;
    if (((s.H / s.G) * sb) % 16 || ((s.I / s.G) * sb) % 16 || ((s.Is / s.G) * sb) % 16)
        return false;
    if (s.I % 32 || s.Is % 32 || s.G < 32)
        return false;
    const int n = sm_count();
    const long R = (long)s.Is + (long)s.k * s.I;
    const long share = (R + n - 1) / n;
    if (share > s.I || share > s.Is) // a CTA's gate/up share crosses at most one expert boundary
        return false;
    if ((s.H + n - 1) / n > kDnThreads / 32) // down: one output row per warp
        return false;
    return gateup_smem(s, n) <= kSmemBudget && down_smem(s, n) <= kSmemBudget;
}

// All three kernels run with the same (maximal) shared-memory carveout: an SM
// whose L1/shared split would have to change between two of them must drain
// first, which would serialise the PDL chain.
template <typename F> static cudaError_t set_carveout(F *kern, bool *done)
{
    if (*done)
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        *done = true;
    return e;
}

static size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t bufs_bytes(const Shape &s)
{
    const int imax = s.I > s.Is ? s.I : s.Is;
    const size_t lg = up256(sizeof(float) * (size_t)(s.E + 1));
    const size_t xr = up256((size_t)kRec * (s.H / 32));
    const size_t a = up256(sizeof(float) * (size_t)(s.k + 1) * imax);
    return kRep * (lg + xr + a);
}

Bufs bufs_carve(const Shape &s, char *base)
{
    const int imax = s.I > s.Is ? s.I : s.Is;
    const size_t lg = up256(sizeof(float) * (size_t)(s.E + 1));
    const size_t xr = up256((size_t)kRec * (s.H / 32));
    const size_t a = up256(sizeof(float) * (size_t)(s.k + 1) * imax);
    Bufs b;
    b.lg = reinterpret_cast<float *>(base);
    b.lgs = (int)(lg / sizeof(float));
    b.xrec = reinterpret_cast<unsigned char *>(base + kRep * lg);
    b.xrs = xr;
    b.a = reinterpret_cast<float *>(base + kRep * (lg + xr));
    b.as = a / sizeof(float);
    return b;
}

cudaError_t launch_router(const Shape &s, const void *x, const void *w_router, const float *bias, const void *w_sg,
                          float *lg, int lgs, int nrep, float *sg, unsigned char *xrec, size_t xrs, cudaStream_t st)
{
    const int rows = w_router ? s.E + (w_sg ? 1 : 0) : 0;
    const int row_ctas = (rows + 3) / 4;
    const int grid = row_ctas + (xrec ? (s.H + 511) / 512 : 0);
    if (grid == 0)
        return cudaSuccess;
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    const __nv_bfloat16 *wr = static_cast<const __nv_bfloat16 *>(w_router);
    const __nv_bfloat16 *ws = static_cast<const __nv_bfloat16 *>(w_sg);
    static bool cv4 = false, cv8 = false;
    cudaError_t e;
    if (s.H == 1024) {
        e = set_carveout(router_tok_kernel<4>, &cv4);
        return e != cudaSuccess ? e
                                : launch_pdl(router_tok_kernel<4>, grid, 128, 0, st, xb, s.E, wr, bias, ws, lg, lgs,
                                             nrep, sg, xrec, xrs, row_ctas);
    }
    e = set_carveout(router_tok_kernel<8>, &cv8);
    return e != cudaSuccess ? e
                            : launch_pdl(router_tok_kernel<8>, grid, 128, 0, st, xb, s.E, wr, bias, ws, lg, lgs, nrep,
                                         sg, xrec, xrs, row_ctas);
}

template <int NXC, typename TS>
static cudaError_t gateup_go(const GateUpArgs &A, int n, size_t smem, cudaStream_t st)
{
    static int cur = 0;
    static bool cv = false;
    cudaError_t e = set_carveout(gateup_tok_kernel<NXC, TS>, &cv);
    if (e == cudaSuccess)
        e = ensure_smem(gateup_tok_kernel<NXC, TS>, smem, &cur);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(gateup_tok_kernel<NXC, TS>, n, kGuThreads, smem, st, A);
}

template <typename TS>
static cudaError_t down_go(const DownArgs &A, int n, size_t smem, cudaStream_t st)
{
    static int cur = 0;
    static bool cv = false;
    cudaError_t e = set_carveout(down_tok_kernel<TS>, &cv);
    if (e == cudaSuccess)
        e = ensure_smem(down_tok_kernel<TS>, smem, &cur);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(down_tok_kernel<TS>, n, kDnThreads, smem, st, A);
}

cudaError_t launch_experts(const Shape &s, const Bufs &b, const ExpertSrc &src, const Routing &R, void *y,
                           float *y32, cudaStream_t st)
{
    const int n = sm_count();
    const int imax = s.I > s.Is ? s.I : s.Is;
    const int lg = log2i(s.G);
    GateUpArgs g{b.xrec, b.xrs, src, R, b.a, b.as, s.E, s.k, s.I, s.Is, imax, lg};
    const size_t gs = gateup_smem(s, n);
    const bool f16 = s.qscale == MOE_F16;
    cudaError_t e;
    if (s.H == 1024)
        e = f16 ? gateup_go<1, __half>(g, n, gs, st) : gateup_go<1, float>(g, n, gs, st);
    else
        e = f16 ? gateup_go<2, __half>(g, n, gs, st) : gateup_go<2, float>(g, n, gs, st);
    if (e != cudaSuccess)
        return e;
    DownArgs d{src, R, b.a, b.as, static_cast<__nv_bfloat16 *>(y), y32, s.E, s.H, s.k, s.I, s.Is, imax, lg,
               s.k + 1};
    d.R.idx_out = nullptr;
    d.R.w_out = nullptr;
    const size_t ds = down_smem(s, n);
    return f16 ? down_go<__half>(d, n, ds, st) : down_go<float>(d, n, ds, st);
}

} // namespace tok
} // namespace moe
