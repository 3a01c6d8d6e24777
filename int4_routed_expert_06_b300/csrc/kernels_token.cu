// Single-token (batch-1 decode) path of the routed int4 MoE layer on B300.
//
// Two kernels chained with programmatic dependent launch (PDL).  Each kernel
// loads what does not depend on its predecessor's output (weights, the slot
// table) before griddepcontrol.wait, and reads its predecessor's outputs and
// writes its own only after the wait, so a successor never races a kernel
// that still reads a buffer it is about to overwrite.
//
//   router_tok   one warp per router row (E experts, then the shared-gate
//                row), the row's bf16 weights held in registers before the
//                wait; after it, x is read and the logits written (in kRep
//                copies).  A few extra CTAs convert x into the fixed-point
//                chunk records the expert kernel uses.
//   experts_tok  one CTA per SM.  Top-k from the logits (one warp per CTA,
//                every CTA), then every weight byte the CTA needs is copied
//                into shared memory at once: its 32-row chunks of the active
//                experts' gate/up rows and its output rows of their W_d.  It
//                computes a = silu(W_g x) * (W_u x) for its chunks and writes
//                each chunk's fixed-point record; after a grid-wide barrier it
//                reads all records and accumulates
//                  y[h] = sum_r w_r (W_d,r a_r)[h] + sigmoid(s) (W_d,sh a_sh)[h]
//                for its output rows in a fixed order.
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
constexpr int kMaxE = 1024;                          // experts the staged tables hold
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;   // 0.2 s bound on any barrier wait
constexpr int kRec = 80;                             // bytes per fixed-point chunk record
constexpr int kExThreads = 512;
constexpr int kMaxSeg = 2;                           // gate/up segments per CTA
constexpr int kMaxUnits = 8;                         // gate/up units (8 row pairs) per CTA
constexpr int kParts = 1;                            // row parts per segment, one barrier each
constexpr int kRowsPerWarp = 4;                      // gate/up row pairs per warp

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

// 16-byte global -> shared copy through L2 (cp.async); both addresses
// 16-byte aligned.  Every thread issues its own pieces, so a CTA stages a
// weight slice without the per-copy setup cost of a bulk copy.
__device__ __forceinline__ void cp16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread has issued so far has
// landed (the barrier's count includes this arrival).
__device__ __forceinline__ void cp_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Copy `bytes` (a multiple of 16) cooperatively: thread t of nt takes the
// 16-byte pieces t, t + nt, ...
__device__ __forceinline__ void cp_slice(void *dst, const void *src, uint32_t bytes, int t, int nt)
{
    for (uint32_t o = (uint32_t)t * 16; o < bytes; o += (uint32_t)nt * 16)
        cp16(static_cast<char *>(dst) + o, static_cast<const char *>(src) + o);
}

// One potentially blocking test of the barrier's phase: the thread sleeps
// until the phase completes or about 1 ms passes (the suspend-time hint), so
// waiting warps leave the issue slots to the other warps of the SM.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
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
// MOE_ERR_TIMEOUT recorded) if it never completes.  Inlined: a call would
// make the caller's loads still in flight land before it.
__device__ __forceinline__ bool mbar_wait0(uint64_t *bar)
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

// The same from global memory through L2 (written by another CTA).
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
                                                        size_t xrs, unsigned int *__restrict__ bar, int n_row_ctas)
{
    constexpr int H = 256 * NJ;
    pdl_trigger();
    // the experts kernel that follows counts its CTAs through its grid
    // barrier from zero (every kernel before this one has completed once the
    // wait returns, so none still uses the counter)
    if (bar && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
        pdl_wait();
        *bar = 0u;
    }
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

// ------------------------------------------------------------ experts

// One kernel computes the experts of the token: gate/up SwiGLU, then (after a
// grid-wide barrier) down + weighted combine.
//
// Gate/up work comes in units of 8 row pairs (gate row o and up row o for 8
// consecutive o), listed as [shared expert's units | rank 0's units | ...];
// CTA c takes the contiguous run [c NU / n, (c + 1) NU / n), at most two
// segments of consecutive rows of one expert.  It computes a = silu(g) u for
// those rows and writes each unit's part of the fixed-point record of a (see
// ARec).  After the barrier every CTA computes output rows [h0, h1) of y from
// its rows of every active expert's W_d, one thread per 32-column chunk of a
// (and half of the rows).
//
// Every code byte the CTA needs is bulk-copied into shared memory right after
// the routing is known (each segment's gate and up code rows, and its rows of
// each active expert's W_d), together with plain loads of the scale and bias
// rows.  Latency-critical reads are kept out of that stream: small reads
// issued while it is in flight wait behind it.
struct ExpertsArgs {
    const unsigned char *xrec; // [kRep][xrs] fixed-point records of x
    size_t xrs;
    ExpertSrc src;
    Routing R;
    unsigned char *arec;       // [kRep][ars]: ARec of each 32-row chunk of a
    size_t ars;
    unsigned int *bar;         // grid barrier counter, zeroed by the router kernel
    __nv_bfloat16 *y;
    float *y32;
    int E, k, I, Is, log2G;
};

// Fixed-point record of 32 consecutive values of a, written a quarter (8
// values) at a time: for quarter m, he[m] le[m] ho[m] lo[m] hold the dp4a
// bytes of its even and odd columns (as in Chunk), sx[m] its step and X[m]
// its sum.  Quarter m occupies bytes 4m of each 16-byte field.
constexpr int kArec = 96;

// Active expert *i of gate/up unit u of the list, and its first row *o0.
__device__ __forceinline__ void unit_of(int u, int k, int I, int Is, int *i, int *o0)
{
    const int ns = Is >> 3;
    if (u < ns) {
        *i = k;
        *o0 = 8 * u;
    } else {
        const int r = (u - ns) / (I >> 3);
        *i = r;
        *o0 = 8 * ((u - ns) - r * (I >> 3));
    }
}

// Index of chunk ch of active expert i in the chunk list [shared | rank 0 | ...].
__device__ __forceinline__ int chunk_index(int i, int ch, int k, int I, int Is)
{
    return i == k ? ch : (Is >> 5) + i * (I >> 5) + ch;
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// s * sum_c q_c a_c + b * sum_c a_c for one 32-code chunk of a W_d row and the
// ARec fields he..lo (uint4 each, word m = quarter m), sx, X (float4).
__device__ __forceinline__ float arec_term(uint4 q, uint4 he, uint4 le, uint4 ho, uint4 lo, float4 sx, float4 X,
                                           float s, float b)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    const uint32_t H_[4] = {he.x, he.y, he.z, he.w}, L_[4] = {le.x, le.y, le.z, le.w};
    const uint32_t HO[4] = {ho.x, ho.y, ho.z, ho.w}, LO[4] = {lo.x, lo.y, lo.z, lo.w};
    const float S[4] = {sx.x, sx.y, sx.z, sx.w};
    float D = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t ev = w[m] & 0x0F0F0F0Fu;
        const uint32_t od = (w[m] >> 4) & 0x0F0F0F0Fu;
        const int h = dp4a_us(od, HO[m], dp4a_us(ev, H_[m], 0));
        const int l = dp4a_uu(od, LO[m], dp4a_uu(ev, L_[m], 0));
        D = fmaf((float)(h * 256 + l), S[m], D);
    }
    return fmaf(s, D, b * ((X.x + X.y) + (X.z + X.w)));
}

// H = 1024 * NXC; TS = scale/bias type.  One CTA of kExThreads per SM.
//
// Shared memory (dynamic): per segment [n gate code rows][n up code rows]
// [n gate scale rows][n gate bias rows][n up scale rows][n up bias rows];
// then per active expert its down rows (codes [nr][I_i/2], scales and biases
// [nr][I_i/G] each); then the partial sums of the down phase.
template <int NXC, typename TS>
__global__ void __maxnreg__(112) experts_tok_kernel(ExpertsArgs A)
{
    constexpr int H = 1024 * NXC;
    constexpr int NW = kExThreads / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t sbar[kMaxSeg][kParts], dbar, xbar;
    __shared__ int tab[kMaxE];
    __shared__ __align__(16) unsigned char xs[(H / 32) * kRec];
    __shared__ int s_idx[kMaxAct];
    __shared__ float s_w[kMaxAct + 1];
    __shared__ const char *s_base[kMaxAct];  // blob of active expert i (i == k: shared), or nullptr
    __shared__ uint32_t s_eoff[kMaxAct + 1]; // offset of expert i's down rows in the down region
    __shared__ int s_qb[kMaxAct];            // down code bytes per row of expert i
    __shared__ int s_ng[kMaxAct];            // down groups per row of expert i
    __shared__ float s_a[8 * kMaxUnits];
    __shared__ __align__(16) TopkSmem tks;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = gridDim.x, c = blockIdx.x, rep = c % kRep;
    const int k = A.k, n_act = k + 1;
    const int HG = H >> A.log2G;                     // groups per gate/up row
    const uint32_t qrow = H / 2;                     // code bytes per gate/up row
    const uint32_t sb = sizeof(TS);
    const uint32_t srow = (uint32_t)HG * sb;         // scale (or bias) bytes per gate/up row
    const uint32_t rowb = 2 * qrow + 4 * srow;       // shared bytes per row pair of a segment
    const int NU = (A.Is >> 3) + k * (A.I >> 3);
    const int NC = (A.Is >> 5) + k * (A.I >> 5);
    const int u0 = (int)((long)c * NU / n), u1 = (int)((long)(c + 1) * NU / n);
    // segments: runs of this CTA's units within one expert
    int nseg = 0, seg_i[kMaxSeg], seg_o0[kMaxSeg], seg_n[kMaxSeg];
    uint32_t seg_off[kMaxSeg];
    {
        uint32_t off = 0;
        for (int u = u0; u < u1 && nseg < kMaxSeg;) {
            int i, o0;
            unit_of(u, k, A.I, A.Is, &i, &o0);
            const int inter = (i == k) ? A.Is : A.I;
            const int len = min(u1 - u, (inter - o0) >> 3);
            seg_i[nseg] = i;
            seg_o0[nseg] = o0;
            seg_n[nseg] = 8 * len;
            seg_off[nseg] = off;
            off += (uint32_t)(8 * len) * rowb;
            ++nseg;
            u += len;
        }
    }
    const int NR = 8 * (u1 - u0); // row pairs of this CTA
    unsigned char *down = smem + (nseg ? seg_off[nseg - 1] + (uint32_t)seg_n[nseg - 1] * rowb : 0u);
    const int h0 = (int)((long)c * (long)H / n), h1 = (int)((long)(c + 1) * (long)H / n);
    const int nr = h1 - h0;

    // The copy warp (the last one; it computes no gate/up rows, since a bulk
    // copy holds its issuing thread until the copy engine takes it) stages
    // part p of segment s (rows [r0, r1) = [p n / kParts, (p + 1) n / kParts))
    // with lanes 6 (s kParts + p) + j: j < 4 copies those rows of the gate
    // scales, gate biases, up scales, up biases (small, so issued first),
    // j = 4 / 5 the gate / up code rows; lane j = 0 arms the part's barrier.
    // Only segments with `pick` set.
    auto stage_rows = [&](bool (*pick)(int, int), const char *const *base) {
        const int q = lane / 6, j = lane - 6 * q, s = q / kParts, p = q - s * kParts;
        const bool valid = q < kMaxSeg * kParts && s < nseg && pick(seg_i[s], k);
        const bool on = valid && base[s] != nullptr;
        uint32_t r0 = 0, nrow = 0;
        if (valid) {
            r0 = (uint32_t)(p * seg_n[s] / kParts);
            nrow = (uint32_t)((p + 1) * seg_n[s] / kParts) - r0;
        }
        if (valid && j == 0 && nrow)
            mbar_expect_tx(&sbar[s][p], on ? nrow * rowb : 0u);
        __syncwarp();
        if (on && nrow) {
            const size_t *offs = (seg_i[s] == k) ? A.src.off_sh : A.src.off;
            const uint32_t nn = (uint32_t)seg_n[s];
            unsigned char *d = smem + seg_off[s];
            const size_t row = (size_t)(seg_o0[s] + (int)r0);
            if (j < 4) {
                const int m = j == 0 ? M_SG : j == 1 ? M_BG : j == 2 ? M_SU : M_BU;
                bulk_g2s(d + 2 * nn * qrow + j * nn * srow + r0 * srow, base[s] + offs[m] + row * srow, nrow * srow,
                         &sbar[s][p]);
            } else {
                const int h = j - 4;
                bulk_g2s(d + h * nn * qrow + r0 * qrow, base[s] + offs[h ? M_QU : M_QG] + row * qrow, nrow * qrow,
                         &sbar[s][p]);
            }
        }
    };

    // ---- before the wait: only what does not depend on the router's output
    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxSeg; ++s)
            for (int p = 0; p < kParts; ++p)
                mbar_init(&sbar[s][p], 1);
        mbar_init(&dbar, 1);
        mbar_init(&xbar, kExThreads);
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
        s_base[k] = A.src.shared;
    }
    for (int e = threadIdx.x; e < A.E; e += kExThreads)
        tab[e] = __ldg(A.src.table + e);
    __syncthreads();
    // the shared expert's units come first in the list: stage them now
    if (warp == NW - 1) {
        const char *base[kMaxSeg] = {A.src.shared, A.src.shared};
        stage_rows([](int i, int kk) { return i == kk; }, base);
    }

    // ---- after the wait: x records and the shared-gate logit are fetched
    // while warp 0 selects the top k; then every copy is issued
    pdl_wait();
    cp_slice(xs, A.xrec + (size_t)rep * A.xrs, (H / 32) * kRec, threadIdx.x, kExThreads);
    cp_arrive(&xbar);
    if (threadIdx.x == 32)
        s_w[kMaxAct] = sigmoid_f(__ldcg(A.R.logits ? A.R.logits + (size_t)rep * A.R.lgs + A.E : A.R.sg_logit));
    if (warp == 0) {
        load_routing(A.R, rep, A.E, k, lane, s_idx, s_w, tks, c == 0);
        if (lane < k)
            s_base[lane] = routed_base(A.src, tab, s_idx[lane]);
    }
    __syncthreads();
    // the copy warp: routed gate/up rows; then, once every gate/up part of
    // this SM has landed (the down rows are needed only after the grid
    // barrier, so they must not compete with the gate/up stream), lane 12 + i
    // copies expert i's down code, scale and bias rows [h0, h1) (lane 12 arms
    // the barrier)
    if (warp == NW - 1) {
        const char *base[kMaxSeg];
        for (int s = 0; s < kMaxSeg; ++s)
            base[s] = s < nseg ? s_base[seg_i[s]] : nullptr;
        stage_rows([](int i, int kk) { return i != kk; }, base);
        for (int s = 0; s < nseg; ++s)
            for (int p = 0; p < kParts; ++p)
                if ((p + 1) * seg_n[s] / kParts > p * seg_n[s] / kParts)
                    mbar_wait0(&sbar[s][p]);
        const int i = lane - 12;
        const char *b = (i >= 0 && i < n_act) ? s_base[i] : nullptr;
        const uint32_t nq = b ? (uint32_t)nr * s_qb[i] : 0u, ns = b ? (uint32_t)(nr * s_ng[i]) * sb : 0u;
        const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, nq + 2 * ns);
        if (lane == 12)
            mbar_expect_tx(&dbar, tot);
        __syncwarp();
        if (b && nq) {
            const size_t *offs = (i == k) ? A.src.off_sh : A.src.off;
            unsigned char *d = down + s_eoff[i];
            bulk_g2s(d, b + offs[M_QD] + (size_t)h0 * s_qb[i], nq, &dbar);
            bulk_g2s(d + nq, b + offs[M_SD] + (size_t)h0 * s_ng[i] * sb, ns, &dbar);
            bulk_g2s(d + nq + ns, b + offs[M_BD] + (size_t)h0 * s_ng[i] * sb, ns, &dbar);
        }
    }
    constexpr int NWC = NW - 1; // gate/up warps

    // ---- gate/up: warp w < NWC computes row pairs w, w + NWC, ... (at most
    // kRowsPerWarp).  Every row's dot products come first, with no wait
    // between rows, so that their loads and dp4a chains overlap; then one
    // transposing reduction sums all 2 kRowsPerWarp partial values across
    // the warp (9 shuffles instead of 10 per row).
    static_assert(kRowsPerWarp == 4 && kParts == 1, "the reduction below assumes 4 rows per warp, 1 part");
    if (!__all_sync(0xFFFFFFFFu, mbar_wait0(&xbar)))
        return;
    // lane l owns chunks NXC l ... of a row; with two chunks, lanes 4-7 of
    // each quarter warp take them in the other order (xv[m] is chunk
    // 2 l + (m ^ sw)), which makes each 16-byte code load conflict-free
    const int sw = NXC == 2 ? (lane >> 2) & 1 : 0;
    Chunk xv[NXC];
    float Xs = 0.f; // sum of this lane's x columns (its quantisation group)
#pragma unroll
    for (int m = 0; m < NXC; ++m) {
        xv[m] = load_chunk(xs + (size_t)(NXC * lane + (m ^ sw)) * kRec);
        Xs += xv[m].X;
    }
    bool landed = warp < NWC;
    if (landed)
        for (int s = 0; s < nseg; ++s)
            landed &= mbar_wait0(&sbar[s][0]);
    landed = __all_sync(0xFFFFFFFFu, landed);
    float v[2 * kRowsPerWarp]; // gate, up partial sums of rows t = 0, 1, ...
#pragma unroll
    for (int t = 0; t < kRowsPerWarp; ++t) {
        const int rp = warp + t * NWC;
        float g = 0.f, u = 0.f;
        if (landed && rp < NR) {
            const int s = (nseg > 1 && rp >= seg_n[0]) ? 1 : 0, r = s ? rp - seg_n[0] : rp;
            if (s_base[seg_i[s]]) {
                const uint32_t nq = (uint32_t)seg_n[s] * qrow;
                const unsigned char *d = smem + seg_off[s];
                // this lane's group of row r: gate scale, gate bias, up scale, up bias
                const TS *sc = reinterpret_cast<const TS *>(d + 2 * nq) + r * HG + ((NXC * lane * 32) >> A.log2G);
                const int na = seg_n[s] * HG;
                const uint4 *qg = reinterpret_cast<const uint4 *>(d + (size_t)r * qrow);
                const uint4 *qu = reinterpret_cast<const uint4 *>(d + nq + (size_t)r * qrow);
                // one quantisation group per lane: sum_m s (sx_m D_m) + b X_m
                float Dg = 0.f, Du = 0.f;
#pragma unroll
                for (int m = 0; m < NXC; ++m) {
                    Dg = fmaf((float)chunk_idot(qg[NXC * lane + (m ^ sw)], xv[m]), xv[m].sx, Dg);
                    Du = fmaf((float)chunk_idot(qu[NXC * lane + (m ^ sw)], xv[m]), xv[m].sx, Du);
                }
                g = fmaf(to_f32(sc[0]), Dg, to_f32(sc[na]) * Xs);
                u = fmaf(to_f32(sc[2 * na]), Du, to_f32(sc[3 * na]) * Xs);
            }
        }
        v[2 * t] = g;
        v[2 * t + 1] = u;
    }
    // round with half-count w: lanes with bit 4 w set keep values [w, 2 w),
    // the others [0, w), each adding its partner's copy of the kept values
#pragma unroll
    for (int w = kRowsPerWarp; w >= 1; w >>= 1) {
        const bool hi = (lane & (4 * w)) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = hi ? v[j] : v[j + w];
            const float keep = hi ? v[j + w] : v[j];
            v[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4 * w);
        }
    }
    v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], 2);
    v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], 1);
    // lane l now holds the total of value 2 t + h, t = (l >> 3) & 3, h = (l >> 2) & 1
    const float up = __shfl_xor_sync(0xFFFFFFFFu, v[0], 4);
    if ((lane & 7) == 0 && warp < NWC) {
        const int rp = warp + (lane >> 3) * NWC;
        if (rp < NR)
            s_a[rp] = v[0] * sigmoid_f(v[0]) * up;
    }
    __syncthreads();
    // each unit writes its quarter of a chunk's record, in kRep copies
    if (threadIdx.x < u1 - u0) {
        const int uu = u0 + threadIdx.x;
        int i, o0;
        unit_of(uu, k, A.I, A.Is, &i, &o0);
        const float *v = s_a + 8 * threadIdx.x;
        float am = 0.f, X = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            am = fmaxf(am, fabsf(v[j]));
            X += v[j];
        }
        const bool nz = am > 0.f && am < INFINITY;
        const float inv = nz ? 32767.0f / am : 0.f;
        uint32_t f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            f[j] = __float_as_uint(fmaf(v[j], inv, 12582912.0f));
        // byte j of he / le: columns 2j (high / low byte); of ho / lo: 2j + 1
        const uint32_t e01 = __byte_perm(f[0], f[2], 0x5140), e23 = __byte_perm(f[4], f[6], 0x5140);
        const uint32_t o01 = __byte_perm(f[1], f[3], 0x5140), o23 = __byte_perm(f[5], f[7], 0x5140);
        const uint32_t he = __byte_perm(e01, e23, 0x7632), le = __byte_perm(e01, e23, 0x5410);
        const uint32_t ho = __byte_perm(o01, o23, 0x7632), lo = __byte_perm(o01, o23, 0x5410);
        const int m = (o0 & 31) >> 3;
        unsigned char *rec = A.arec + (size_t)chunk_index(i, o0 >> 5, k, A.I, A.Is) * kArec + 4 * m;
        const float sx = nz ? am / 32767.0f : 0.f;
        for (int r = 0; r < kRep; ++r) {
            unsigned char *rr = rec + (size_t)r * A.ars;
            *reinterpret_cast<uint32_t *>(rr) = he;
            *reinterpret_cast<uint32_t *>(rr + 16) = le;
            *reinterpret_cast<uint32_t *>(rr + 32) = ho;
            *reinterpret_cast<uint32_t *>(rr + 48) = lo;
            *reinterpret_cast<float *>(rr + 64) = sx;
            *reinterpret_cast<float *>(rr + 80) = X;
        }
    }

    // ---- grid barrier: every record is written
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(A.bar, 1u);
        const uint64_t t0 = global_ns();
        while (ld_acquire_u32(A.bar) < (unsigned int)n) {
            if (global_ns() - t0 > kWaitNs) {
                record_error(MOE_ERR_TIMEOUT);
                break;
            }
        }
    }
    __syncthreads();
    pdl_trigger(); // the next layer call may start its own weight loads now

    // ---- down, item by item: thread t < 2 NC owns chunk j = t % NC (chunk ch
    // of active expert i; its record is loaded into registers) and half the
    // CTA's output rows, [rg RH, rg RH + RH) with rg = t / NC.  It writes w_i
    // times its part of each row to P[row][j]; warp w then sums row w over
    // the chunks in a fixed order, so the result does not depend on where the
    // experts live.
    const int RH = (nr + 1) / 2;
    float *P = reinterpret_cast<float *>(down + ((s_eoff[n_act] + 15) & ~15u)); // [nr][NC]
    const int t = threadIdx.x;
    const bool mine = t < 2 * NC;
    const int j = mine ? t % NC : 0, rg = t / NC;
    int ii, ch;
    if (j < (A.Is >> 5)) {
        ii = k;
        ch = j;
    } else {
        ii = (j - (A.Is >> 5)) / (A.I >> 5);
        ch = (j - (A.Is >> 5)) - ii * (A.I >> 5);
    }
    uint4 rv[6] = {};
    if (mine) {
        const uint4 *src = reinterpret_cast<const uint4 *>(A.arec + (size_t)rep * A.ars + (size_t)j * kArec);
#pragma unroll
        for (int q = 0; q < 6; ++q)
            rv[q] = __ldcg(src + q);
    }
    const bool ready = __all_sync(0xFFFFFFFFu, mbar_wait0(&dbar));
    if (mine) {
        const int r0 = rg * RH, r1 = min(nr, r0 + RH);
        if (ready && s_base[ii]) {
            const int qb = s_qb[ii], ng = s_ng[ii];
            const unsigned char *d = down + s_eoff[ii];
            const TS *sd = reinterpret_cast<const TS *>(d + nr * qb);
            const TS *bd = sd + nr * ng;
            const int g = (ch * 32) >> A.log2G;
            const float wi = ii < k ? s_w[ii] : s_w[kMaxAct];
            const float4 sx = make_float4(__uint_as_float(rv[4].x), __uint_as_float(rv[4].y),
                                          __uint_as_float(rv[4].z), __uint_as_float(rv[4].w));
            const float4 X = make_float4(__uint_as_float(rv[5].x), __uint_as_float(rv[5].y),
                                         __uint_as_float(rv[5].z), __uint_as_float(rv[5].w));
#pragma unroll 4
            for (int r = r0; r < r1; ++r) {
                const uint4 q = reinterpret_cast<const uint4 *>(d + r * qb)[ch];
                P[r * NC + j] = wi * arec_term(q, rv[0], rv[1], rv[2], rv[3], sx, X, ld_sb(sd + r * ng + g),
                                               ld_sb(bd + r * ng + g));
            }
        } else {
            for (int r = r0; r < r1; ++r)
                P[r * NC + j] = 0.f;
        }
    }
    __syncthreads();
    for (int r = warp; r < nr; r += NW) {
        float acc = 0.f;
        for (int q = lane; q < NC; q += 32)
            acc += P[r * NC + q];
        acc = warp_sum(acc);
        if (ready && lane == 0) {
            A.y[h0 + r] = __float2bfloat16_rn(acc);
            if (A.y32)
                A.y32[h0 + r] = acc;
        }
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

// Gate/up units (8 row pairs) and 32-row chunks of a of one token.
static int n_units(const Shape &s) { return s.Is / 8 + s.k * (s.I / 8); }
static int n_chunks(const Shape &s) { return s.Is / 32 + s.k * (s.I / 32); }

// Dynamic shared memory of the experts kernel (the largest CTA share).
static size_t experts_smem(const Shape &s, int n)
{
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    const size_t rowpair = (size_t)s.H + 4 * (size_t)(s.H / s.G) * sb; // gate and up code, scale and bias rows
    const int units = (n_units(s) + n - 1) / n;
    const int nr = (s.H + n - 1) / n;
    size_t w = 0;
    for (int i = 0; i <= s.k; ++i) {
        const int inter = (i == s.k) ? s.Is : s.I;
        w += (size_t)nr * (inter / 2 + 2 * (inter / s.G) * sb);
    }
    w = (w + 15) & ~(size_t)15;
    return 8 * (size_t)units * rowpair + w + sizeof(float) * (size_t)nr * n_chunks(s);
}

constexpr size_t kSmemLimit = 220 * 1024;

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
    if (s.I % 32 || s.Is % 32 || s.G < 64) // one quantisation group per lane of a gate/up row
        return false;
    const int n = sm_count();
    const int units = (n_units(s) + n - 1) / n;
    if (units > kMaxUnits || 8 * units > s.I || 8 * units > s.Is) // at most two segments per CTA
        return false;
    if (2 * n_chunks(s) > kExThreads) // down: one thread per (chunk, half of the rows)
        return false;
    const int nr = (s.H + n - 1) / n;
    if (nr > 2 * (kExThreads / 32)) // down: output rows per CTA
        return false;
    if (8 * units > kRowsPerWarp * (kExThreads / 32 - 1)) // gate/up row pairs per warp
        return false;
    if (12 + s.k + 1 > 32 || 6 * kMaxSeg * kParts > 12) // lanes of the copy warp
        return false;
    return experts_smem(s, n) <= kSmemLimit;
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
    const size_t lg = up256(sizeof(float) * (size_t)(s.E + 1));
    const size_t xr = up256((size_t)kRec * (s.H / 32));
    const size_t ar = up256((size_t)kArec * n_chunks(s));
    return kRep * (lg + xr + ar) + 256;
}

Bufs bufs_carve(const Shape &s, char *base)
{
    const size_t lg = up256(sizeof(float) * (size_t)(s.E + 1));
    const size_t xr = up256((size_t)kRec * (s.H / 32));
    const size_t ar = up256((size_t)kArec * n_chunks(s));
    Bufs b;
    b.lg = reinterpret_cast<float *>(base);
    b.lgs = (int)(lg / sizeof(float));
    b.xrec = reinterpret_cast<unsigned char *>(base + kRep * lg);
    b.xrs = xr;
    b.arec = reinterpret_cast<unsigned char *>(base + kRep * (lg + xr));
    b.ars = ar;
    b.bar = reinterpret_cast<unsigned int *>(base + kRep * (lg + xr + ar));
    return b;
}

cudaError_t launch_router(const Shape &s, const void *x, const void *w_router, const float *bias, const void *w_sg,
                          float *lg, int lgs, int nrep, float *sg, unsigned char *xrec, size_t xrs, unsigned int *bar,
                          cudaStream_t st)
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
                                             nrep, sg, xrec, xrs, bar, row_ctas);
    }
    e = set_carveout(router_tok_kernel<8>, &cv8);
    return e != cudaSuccess ? e
                            : launch_pdl(router_tok_kernel<8>, grid, 128, 0, st, xb, s.E, wr, bias, ws, lg, lgs, nrep,
                                         sg, xrec, xrs, bar, row_ctas);
}

template <int NXC, typename TS>
static cudaError_t experts_go(const ExpertsArgs &A, int n, size_t smem, cudaStream_t st)
{
    static int cur = 0;
    static bool cv = false;
    cudaError_t e = set_carveout(experts_tok_kernel<NXC, TS>, &cv);
    if (e == cudaSuccess)
        e = ensure_smem(experts_tok_kernel<NXC, TS>, smem, &cur);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(experts_tok_kernel<NXC, TS>, n, kExThreads, smem, st, A);
}

cudaError_t launch_experts(const Shape &s, const Bufs &b, const ExpertSrc &src, const Routing &R, void *y,
                           float *y32, cudaStream_t st)
{
    const int n = sm_count();
    ExpertsArgs A{b.xrec, b.xrs, src, R, b.arec, b.ars, b.bar, static_cast<__nv_bfloat16 *>(y), y32,
                  s.E, s.k, s.I, s.Is, log2i(s.G)};
    const size_t smem = experts_smem(s, n);
    const bool f16 = s.qscale == MOE_F16;
    if (s.H == 1024)
        return f16 ? experts_go<1, __half>(A, n, smem, st) : experts_go<1, float>(A, n, smem, st);
    return f16 ? experts_go<2, __half>(A, n, smem, st) : experts_go<2, float>(A, n, smem, st);
}

} // namespace tok
} // namespace moe
