// Single-token (batch-1 decode) path of the routed int4 MoE layer on B300.
//
// Three kernels per layer call, chained with programmatic dependent launch
// (PDL).  Each loads what does not depend on its predecessor's output
// (weights, the slot table) before griddepcontrol.wait, and reads its
// predecessor's outputs and writes its own only after the wait, so a
// successor never races a kernel that still reads a buffer it overwrites.
// A kernel boundary is the device-wide exchange: on B300 it costs about
// half of what a 148-CTA grid barrier inside one kernel does, and it needs no
// co-residency guarantee.
//
//   router_tok  one warp per router row (E experts, then the shared-gate
//               row), the row's bf16 weights held in registers before the
//               wait; after it, x is read and the logits written (in kRep
//               copies).  A few extra CTAs convert x into the fixed-point
//               chunk records the gate/up kernel uses.
//   gateup_tok  one CTA of 512 threads per SM.  Before the wait: the slot
//               table, and this CTA's rows of the shared expert straight into
//               registers.  After it: the top-k of the logits (all warps),
//               then this CTA's share of the routed experts' gate/up row
//               pairs, loaded straight into registers (every load in flight
//               at once, so the dot products run as the bytes arrive), and
//               an L2 prefetch of the W_d rows the down kernel's CTA with the
//               same index will read.  Each warp computes
//                 a = silu(W_g x) * (W_u x)
//               for its row pairs and writes a in fp32 (kRep copies).
//   down_tok    one CTA of 256 threads per SM.  Before the wait: the same
//               top-k.  After it: bulk copies of output rows [h0, h1) of
//               every active expert's W_d (L2-warm), the fixed-point records
//               of a, then
//                 y[h] = sum_r w_r (W_d,r a_r)[h] + sigmoid(s) (W_d,sh a_sh)[h]
//               for h in [h0, h1), summed in a fixed order.
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

constexpr int kMaxAct = 17;    // top_k <= 16 plus the shared expert
constexpr int kMaxE = 512;     // experts the single-token kernels take
constexpr int kRec = 80;       // bytes per fixed-point chunk record
constexpr int kGuWarps = 16;
constexpr int kGuThreads = 32 * kGuWarps;
constexpr int kMaxUnits = 5;   // gate/up units (8 row pairs) a CTA stages: 6 copy lanes each
constexpr int kDnThreads = 384;
constexpr int kMaxRH = 8;      // output rows a down thread computes (half of a CTA's rows)

// Bound on every device wait (ns) and extra arrivals the down kernel's copy
// barrier expects.  Both are test hooks (moe_debug_set_waits): the defaults
// are 0.2 s and 0.
__device__ unsigned long long g_wait_ns = 200ull * 1000 * 1000;
__device__ int g_extra_arrivals = 0;

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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
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

// Fire-and-forget bulk prefetch of global bytes into L2 (16-byte aligned
// address, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
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

// Wait for phase 0 of a single-use barrier for at most g_wait_ns; false (with
// MOE_ERR_TIMEOUT recorded) if it does not complete in time.
__device__ __forceinline__ bool mbar_wait0(uint64_t *bar)
{
    if (mbar_try_wait(bar, 0))
        return true;
    const uint64_t t0 = global_ns(), lim = g_wait_ns;
    for (;;) {
        if (mbar_try_wait(bar, 0))
            return true;
        if (global_ns() - t0 > lim) {
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

// 16 sum_c q_c * (256 xh_c + xl_c) over one chunk of 32 codes (exact
// integer, |value| < 2^28), in four short dp4a chains.  The odd nibbles stay
// in place (16 q, one LOP3 a word instead of a shift and a LOP3): their
// chains carry 16x, so the even chains are scaled by 16 to match.
__device__ __forceinline__ int chunk_idot16(uint4 q, const Chunk &c)
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
        const uint32_t od = w[m] & 0xF0F0F0F0u;
        h0 = dp4a_us(ev, he[m], h0);
        h1 = dp4a_us(od, ho[m], h1);
        l0 = dp4a_uu(ev, le[m], l0);
        l1 = dp4a_uu(od, lo[m], l1);
    }
    return (h0 * 16 + h1) * 256 + (l0 * 16 + l1);
}

// s * sum_c q_c v_c + b * sum_c v_c for one chunk.  (16 D) sx / 16 rounds
// exactly as D sx: scaling by a power of two commutes with rounding.
__device__ __forceinline__ float chunk_term(uint4 q, const Chunk &c, float s, float b)
{
    const float D = (float)chunk_idot16(q, c) * c.sx * 0.0625f;
    return fmaf(s, D, b * c.X);
}

// 8-bit codes of columns 8m..8m+7 (word w0: columns 8m..8m+3, w1: 8m+4..8m+7)
// in the record order: byte j of ev is column 8m+2j, of od column 8m+2j+1.
__device__ __forceinline__ void split8(uint32_t w0, uint32_t w1, uint32_t &ev, uint32_t &od)
{
    ev = __byte_perm(w0, w1, 0x6420);
    od = __byte_perm(w0, w1, 0x7531);
}

// chunk_idot for 8-bit codes: the chunk's 32 codes are the two words qa, qb
// (columns 0..15, 16..31).  Exact: |sum| < 2^29.
__device__ __forceinline__ int chunk_idot8(uint4 qa, uint4 qb, const Chunk &c)
{
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const uint32_t he[4] = {c.he.x, c.he.y, c.he.z, c.he.w};
    const uint32_t le[4] = {c.le.x, c.le.y, c.le.z, c.le.w};
    const uint32_t ho[4] = {c.ho.x, c.ho.y, c.ho.z, c.ho.w};
    const uint32_t lo[4] = {c.lo.x, c.lo.y, c.lo.z, c.lo.w};
    int h0 = 0, h1 = 0, l0 = 0, l1 = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t ev, od;
        split8(w[2 * m], w[2 * m + 1], ev, od);
        h0 = dp4a_us(ev, he[m], h0);
        h1 = dp4a_us(od, ho[m], h1);
        l0 = dp4a_uu(ev, le[m], l0);
        l1 = dp4a_uu(od, lo[m], l1);
    }
    return (h0 + h1) * 256 + (l0 + l1);
}

// The codes of chunk ch of a BITS-bit code row at row (shared memory), as a
// chunk term.
template <int BITS>
__device__ __forceinline__ float row_chunk_term(const unsigned char *row, int ch, const Chunk &c, float s, float b)
{
    const uint4 *q = reinterpret_cast<const uint4 *>(row);
    const float D = BITS == 8 ? (float)chunk_idot8(q[2 * ch], q[2 * ch + 1], c) * c.sx
                              : (float)chunk_idot16(q[ch], c) * c.sx * 0.0625f;
    return fmaf(s, D, b * c.X);
}

// ------------------------------------------------------------ top-k

// 32-bit order key of a logit: unsigned order = float order, NaN as -inf;
// every real key is nonzero.
__device__ __forceinline__ uint32_t ord32(float f)
{
    const uint32_t u = __float_as_uint(isnan(f) ? -INFINITY : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord32_logit(uint32_t u)
{
    u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(u);
}
// Routing key: the order key in the high word, the complement of the expert
// id in the low word, so that the key order is the routing order (logit
// descending, then expert id ascending).
__device__ __forceinline__ unsigned long long route_key(uint32_t u, int e)
{
    return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)e);
}

// Shared scratch of the block top-k.
struct TopkBlk {
    uint32_t gm[32];                   // group maxima
    unsigned long long cand[kMaxE];    // candidates (routing keys)
    unsigned long long sel[16];        // the top k in rank order
    int wcnt[32];                      // candidates per warp
};

// Top k of the E <= EPT NT logits at lg (global memory, written by an earlier
// kernel) by all threads of the CTA; thread t < NT holds experts t + NT j
// (NT a power of two, at least 32; threads past NT hold none).  At most 32
// warps.
//
// The keys are cut into 32 groups of NT / 32 consecutive threads.  T = the
// group maximum of the largest rank <= k - 1 is at most the k-th largest key
// (at least k keys are >= T), so the top k are among the candidates >= T,
// usually about k of them.  Each warp ranks some candidates against all of
// them, 32 at a time by ballot, comparing routing keys; a candidate's rank
// among the candidates is its rank among all keys.
//
// Writes s_idx[r] (r < k), the r-th expert; when s_w is non-NULL also its
// renormalised weight exp(l_r - l_0) / sum_{j<k} exp(l_j - l_0) to s_w[r],
// and, when idx_out is non-NULL, both to idx_out / w_out.  Ends synchronised.
template <int NT, int EPT>
__device__ __forceinline__ void block_topk(const float *lg, int E, int k, TopkBlk &S, int *s_idx, float *s_w,
                                           int32_t *idx_out, float *w_out)
{
    constexpr int GS = NT / 32;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nw = blockDim.x >> 5;
    uint32_t u[EPT], m = 0;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int e = t + NT * j;
        u[j] = (t < NT && e < E) ? ord32(__ldcg(lg + e)) : 0u;
        m = max(m, u[j]);
    }
#pragma unroll
    for (int o = GS / 2; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (t < NT && t % GS == 0)
        S.gm[t / GS] = m;
    __syncthreads();
    const uint32_t g = S.gm[lane];
    int r = 0;
#pragma unroll
    for (int o = 0; o < 32; o += 4) {
        const uint4 q = *reinterpret_cast<const uint4 *>(&S.gm[o]);
        r += (q.x > g ? 1 : 0) + (q.y > g ? 1 : 0) + (q.z > g ? 1 : 0) + (q.w > g ? 1 : 0);
    }
    const unsigned rmax = __reduce_max_sync(0xFFFFFFFFu, r <= k - 1 ? (unsigned)r : 0u);
    const uint32_t T = __shfl_sync(0xFFFFFFFFu, g, __ffs(__ballot_sync(0xFFFFFFFFu, (unsigned)r == rmax)) - 1);
    // candidates: counted per warp, then stored at the warp's offset
    uint32_t bal[EPT];
    int wn = 0;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        bal[j] = __ballot_sync(0xFFFFFFFFu, u[j] != 0u && u[j] >= T);
        wn += __popc(bal[j]);
    }
    if (lane == 0)
        S.wcnt[warp] = wn;
    __syncthreads();
    const int before = (int)__reduce_add_sync(0xFFFFFFFFu, lane < warp && lane < nw ? (unsigned)S.wcnt[lane] : 0u);
    const int C = (int)__reduce_add_sync(0xFFFFFFFFu, lane < nw ? (unsigned)S.wcnt[lane] : 0u);
    int pos = before;
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        if ((bal[j] >> lane) & 1u)
            S.cand[pos + __popc(bal[j] & lt)] = route_key(u[j], t + NT * j);
        pos += __popc(bal[j]);
    }
    __syncthreads();
    for (int i = warp; i < C; i += nw) {
        const unsigned long long ki = S.cand[i];
        int rk = 0;
        for (int b0 = 0; b0 < C; b0 += 32) {
            const unsigned long long v = b0 + lane < C ? S.cand[b0 + lane] : 0ull;
            rk += __popc(__ballot_sync(0xFFFFFFFFu, v > ki));
        }
        if (lane == 0 && rk < k)
            S.sel[rk] = ki;
    }
    __syncthreads();
    if (warp == 0) {
        const unsigned long long q = lane < k ? S.sel[lane] : 0ull;
        const int se = (int)(0xFFFFFFFFu - (uint32_t)q);
        if (lane < k)
            s_idx[lane] = se;
        if (s_w) {
            const float l0 = ord32_logit((uint32_t)(S.sel[0] >> 32));
            const float ex = lane < k ? expf(ord32_logit((uint32_t)(q >> 32)) - l0) : 0.f;
            float sum = ex;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
            const float wv = ex / sum;
            if (lane < k) {
                s_w[lane] = wv;
                if (idx_out) {
                    idx_out[lane] = se;
                    w_out[lane] = wv;
                }
            }
        }
    }
    __syncthreads();
}

// Routing of this token into s_idx (and s_w when non-NULL), shared memory:
// the top-k of logits copy `rep`, or the given idx / w.  All threads; ends
// synchronised.
template <int NT>
__device__ __forceinline__ void load_routing(const Routing &R, int rep, int E, int k, TopkBlk &S, int *s_idx,
                                             float *s_w, bool write_out)
{
    if (R.logits) {
        const float *lg = R.logits + (size_t)rep * R.lgs;
        int32_t *io = write_out ? R.idx_out : nullptr;
        if (E <= NT)
            block_topk<NT, 1>(lg, E, k, S, s_idx, s_w, io, R.w_out);
        else
            block_topk<NT, kMaxE / NT>(lg, E, k, S, s_idx, s_w, io, R.w_out);
    } else {
        if ((int)threadIdx.x < k) {
            s_idx[threadIdx.x] = __ldcg(R.idx + threadIdx.x);
            if (s_w)
                s_w[threadIdx.x] = __ldcg(R.w + threadIdx.x);
        }
        __syncthreads();
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
    float acc = acc0 + acc1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
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

struct TokArgs {
    const unsigned char *xrec; // [kRep][xrs] fixed-point records of x
    size_t xrs;
    ExpertSrc src;
    Routing R;
    unsigned char *arec;       // [kRep][ars] activation records, one per 32-row chunk
    size_t ars;
    __nv_bfloat16 *y;
    float *y32;
    int E, k, I, Is, log2G;
};

// Activation record of one 32-row chunk of a, written 8 rows (a quarter) at
// a time: for quarter m, he[m] le[m] ho[m] lo[m] hold the dp4a bytes of its
// even and odd rows (as in Chunk), sx[m] its step and X[m] its sum.  Quarter
// m occupies bytes 4m of each 16-byte field: he, le, ho, lo, sx[4], X[4].
constexpr int kArec = 96;

// Gate/up unit u of the list [shared expert's units | rank 0's | rank 1's
// ...] (8 row pairs each): active expert *i (k: the shared one), first row *o0.
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

__device__ __forceinline__ void named_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// H = 1024 * NXC; TS = scale/bias type.  One CTA of kGuThreads per SM.
//
// CTA c takes units [c NU / n, (c + 1) NU / n) of the unit list (NU units in
// all).  Each unit is staged in shared memory by six bulk copies (its gate
// and up code rows, its gate/up scale and bias rows) completing on the
// unit's own barrier.  A CTA's shared-expert units are issued before the
// wait; its routed units after the top-k, at most kDepth in flight: the
// group that finds routed unit r landed issues unit r + kDepth, so the units
// land one after another while the groups work on the earlier ones.  Warp
// group g (warps 4g .. 4g + 3) computes units g, g + 4, ...: each warp two
// row pairs of the unit, lane l taking chunks l and l + 32 of the row; then
// lanes 0..7 of the group's first warp write the unit's quarter of its
// chunk's activation record, one copy each.
//
// 72 registers a thread: with the down kernel (384 x 56) and the router (128
// x 56) beside it, each of the SM's four register banks holds its share of
// all three kernels, so each kernel's CTAs are resident before its
// predecessor ends.
template <int NXC, typename TS, int BITS>
__global__ void __maxnreg__(72) gateup_tok_kernel(TokArgs A)
{
    constexpr int H = 1024 * NXC;
    constexpr uint32_t RB = H * BITS / 8; // bytes of one code row
    constexpr int NG = kGuWarps / 4; // warp groups
    constexpr int kDepth = 3;        // routed units in flight
    extern __shared__ __align__(128) unsigned char units[]; // [local unit][unitb]
    __shared__ uint64_t ubar[kMaxUnits], xbar;
    __shared__ int tab[kMaxE];
    __shared__ __align__(16) unsigned char xs[(H / 32) * kRec];
    __shared__ __align__(16) TopkBlk tks;
    __shared__ int s_idx[kMaxAct];
    __shared__ const char *s_base[kMaxAct]; // blob of active expert i (i == k: shared), or nullptr
    __shared__ float s_a[kMaxUnits][8];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = gridDim.x, c = blockIdx.x, rep = c % kRep;
    const int k = A.k;
    const int NU = (A.Is >> 3) + k * (A.I >> 3);
    const int u0 = (int)((long)c * NU / n), nu = (int)((long)(c + 1) * NU / n) - u0;
    const int js = max(0, min(nu, (A.Is >> 3) - u0)); // local units [0, js) are the shared expert's
    const int HG = H >> A.log2G;
    const uint32_t sbr = (uint32_t)HG * (uint32_t)sizeof(TS); // bytes of one scale row
    const uint32_t unitb = 8u * (2u * RB + 4u * sbr);

    // The copies of local unit j, by one warp: lane a < 6 copies array a
    // (gate codes, up codes, gate scales, gate biases, up scales, up biases)
    // of the unit's 8 rows; lane 0 arms the unit's barrier.
    auto stage = [&](int j) {
        int i, o0;
        unit_of(u0 + j, k, A.I, A.Is, &i, &o0);
        const char *b = s_base[i];
        if (lane == 0)
            mbar_expect_tx(&ubar[j], b ? unitb : 0u);
        __syncwarp();
        if (b && lane < 6) {
            const size_t *offs = i == k ? A.src.off_sh : A.src.off;
            unsigned char *d = units + (size_t)j * unitb;
            if (lane < 2)
                bulk_g2s(d + lane * 8 * RB, b + offs[lane ? M_QU : M_QG] + (size_t)o0 * RB, 8u * RB, &ubar[j]);
            else
                bulk_g2s(d + 16 * RB + (lane - 2) * 8 * sbr, b + offs[M_SG + (lane - 2)] + (size_t)o0 * sbr, 8u * sbr,
                         &ubar[j]);
        }
    };

    // ---- before the wait: barriers, the slot table, the shared expert's units
    if (threadIdx.x == 0) {
        for (int j = 0; j < nu; ++j)
            mbar_init(&ubar[j], 1);
        mbar_init(&xbar, 1);
        fence_mbar_init();
        s_base[k] = A.src.shared;
    }
    for (int e = threadIdx.x; e < A.E; e += kGuThreads)
        tab[e] = __ldg(A.src.table + e);
    __syncthreads();
    if (warp == kGuWarps - 1)
        for (int j = 0; j < js; ++j)
            stage(j);

    pdl_wait();
    pdl_trigger(); // the router has completed: the down kernel may start its own top-k

    // ---- x's records, the routing, the first routed units
    if (threadIdx.x == 0) {
        constexpr uint32_t xb = (H / 32) * kRec;
        mbar_expect_tx(&xbar, xb);
        bulk_g2s(xs, A.xrec + (size_t)rep * A.xrs, xb, &xbar);
    }
    load_routing<kGuThreads>(A.R, rep, A.E, k, tks, s_idx, nullptr, false);
    // the staging warp resolves the slots; compute warps read s_base only
    // after a unit barrier it armed (its arrival releases these writes)
    if (warp == kGuWarps - 1) {
        if (lane < k)
            s_base[lane] = routed_base(A.src, tab, s_idx[lane]);
        __syncwarp();
        for (int j = js; j < min(nu, js + kDepth); ++j)
            stage(j);
    }

    // ---- gate/up: this lane's chunks of x, then the group's units
    const bool xok = __all_sync(0xFFFFFFFFu, mbar_wait0(&xbar));
    Chunk xv[NXC];
#pragma unroll
    for (int m = 0; m < NXC; ++m)
        xv[m] = load_chunk(xs + (size_t)(lane + 32 * m) * kRec);
    const int grp = warp >> 2, wq = warp & 3;
    for (int j = grp; j < nu; j += NG) {
        int i, o0;
        unit_of(u0 + j, k, A.I, A.Is, &i, &o0);
        const bool landed = __all_sync(0xFFFFFFFFu, mbar_wait0(&ubar[j]));
        const bool have = xok && landed && s_base[i] != nullptr;
        if (wq == 0 && j >= js && j + kDepth < nu)
            stage(j + kDepth);
        const unsigned char *d = units + (size_t)j * unitb;
        const TS *sc = reinterpret_cast<const TS *>(d + 16 * RB);
        float v[4] = {0.f, 0.f, 0.f, 0.f}; // gate, up of rows 2 wq and 2 wq + 1
        if (have) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = 2 * wq + rr;
#pragma unroll
                for (int m = 0; m < NXC; ++m) {
                    const int ch = lane + 32 * m;
                    const int gi = (ch * 32) >> A.log2G;
                    v[2 * rr] += row_chunk_term<BITS>(d + r * RB, ch, xv[m], to_f32(sc[r * HG + gi]),
                                                      to_f32(sc[8 * HG + r * HG + gi]));
                    v[2 * rr + 1] += row_chunk_term<BITS>(d + (8 + r) * RB, ch, xv[m], to_f32(sc[16 * HG + r * HG + gi]),
                                                          to_f32(sc[24 * HG + r * HG + gi]));
                }
            }
        }
        // transposing reduction of the four sums: lanes with bit 4 set keep
        // values 2, 3, the others 0, 1; then bit 3 splits those
        {
            const bool hi = (lane & 16) != 0;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float send = hi ? v[q] : v[q + 2];
                const float keep = hi ? v[q + 2] : v[q];
                v[q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
            }
            const bool h8 = (lane & 8) != 0;
            const float send = h8 ? v[0] : v[1];
            const float keep = h8 ? v[1] : v[0];
            v[0] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
#pragma unroll
            for (int o = 4; o > 0; o >>= 1)
                v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
        }
        // lane l holds value 2 (l >> 4) + ((l >> 3) & 1): gate or up of row 2 wq + (l >> 4)
        const float up = __shfl_xor_sync(0xFFFFFFFFu, v[0], 8);
        if ((lane & 15) == 0)
            s_a[j][2 * wq + (lane >> 4)] = have ? v[0] * sigmoid_f(v[0]) * up : 0.f;
        named_sync(1 + grp, 128);
        if (wq == 0 && lane < kRep) {
            float a[8], am = 0.f, X = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                a[q] = s_a[j][q];
                am = fmaxf(am, fabsf(a[q]));
                X += a[q];
            }
            const bool nz = am > 0.f && am < INFINITY;
            const float inv = nz ? 32767.0f / am : 0.f;
            uint32_t f[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                f[q] = __float_as_uint(fmaf(a[q], inv, 12582912.0f));
            // byte q of he / le: rows 2q (high / low byte); of ho / lo: 2q + 1
            const uint32_t e01 = __byte_perm(f[0], f[2], 0x5140), e23 = __byte_perm(f[4], f[6], 0x5140);
            const uint32_t o01 = __byte_perm(f[1], f[3], 0x5140), o23 = __byte_perm(f[5], f[7], 0x5140);
            const int mq = (o0 & 31) >> 3;
            unsigned char *rec = A.arec + (size_t)lane * A.ars + (size_t)chunk_index(i, o0 >> 5, k, A.I, A.Is) * kArec + 4 * mq;
            *reinterpret_cast<uint32_t *>(rec) = __byte_perm(e01, e23, 0x7632);
            *reinterpret_cast<uint32_t *>(rec + 16) = __byte_perm(e01, e23, 0x5410);
            *reinterpret_cast<uint32_t *>(rec + 32) = __byte_perm(o01, o23, 0x7632);
            *reinterpret_cast<uint32_t *>(rec + 48) = __byte_perm(o01, o23, 0x5410);
            *reinterpret_cast<float *>(rec + 64) = nz ? am / 32767.0f : 0.f;
            *reinterpret_cast<float *>(rec + 80) = X;
        }
    }
}

// ------------------------------------------------------------ down

// s * sum_c q_c a_c + b * sum_c a_c for one 32-code chunk of a W_d row and an
// activation record's fields he..lo (uint4 each, word m = quarter m), sx, X.
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

// arec_term for 8-bit codes: the chunk's 32 codes are the words qa, qb.
__device__ __forceinline__ float arec_term8(uint4 qa, uint4 qb, uint4 he, uint4 le, uint4 ho, uint4 lo, float4 sx,
                                            float4 X, float s, float b)
{
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const uint32_t H_[4] = {he.x, he.y, he.z, he.w}, L_[4] = {le.x, le.y, le.z, le.w};
    const uint32_t HO[4] = {ho.x, ho.y, ho.z, ho.w}, LO[4] = {lo.x, lo.y, lo.z, lo.w};
    const float S[4] = {sx.x, sx.y, sx.z, sx.w};
    float D = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t ev, od;
        split8(w[2 * m], w[2 * m + 1], ev, od);
        const int h = dp4a_us(od, HO[m], dp4a_us(ev, H_[m], 0));
        const int l = dp4a_uu(od, LO[m], dp4a_uu(ev, L_[m], 0));
        D = fmaf((float)(h * 256 + l), S[m], D);
    }
    return fmaf(s, D, b * ((X.x + X.y) + (X.z + X.w)));
}

// Down projection and combine.  CTA c computes output rows [h0, h1) =
// [c H / n, (c + 1) H / n).  Its W_d rows of every active expert (codes
// [nr][I_i/2], then scales and biases [nr][I_i/G] each, per expert) are bulk-
// copied into shared memory before the wait (weights: not written by the
// kernels this one waits for), the activation records after it.  Thread t
// takes chunk t % NCp of the chunk list [shared | rank 0 | rank 1 | ...]
// (NCp = the chunk count rounded up to 32) for half t / NCp of the output
// rows, and forms w_i times its chunk's term of each of those rows.  Each
// warp sums every row over its 32 chunks by butterfly, then one thread a row
// adds its half's warps in order: a fixed summation order, so the result does
// not depend on where the experts live.  The routing (with weights) is
// computed before the wait.
template <typename TS, int BITS>
__global__ void __maxnreg__(56) down_tok_kernel(TokArgs A, int H)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t dbar, rbar;
    __shared__ int tab[kMaxE];
    __shared__ __align__(16) TopkBlk tks;
    __shared__ int s_idx[kMaxAct];
    __shared__ float s_w[kMaxAct + 1];
    __shared__ const char *s_base[kMaxAct];
    __shared__ uint32_t s_eoff[kMaxAct + 1]; // offset of expert i's rows in the down region
    __shared__ float Pw[2 * kMaxRH][kDnThreads / 32]; // [row][warp] partial sums

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int n = gridDim.x, c = blockIdx.x, rep = c % kRep;
    const int k = A.k, n_act = k + 1;
    const int h0 = (int)((long)c * H / n), nr = (int)((long)(c + 1) * H / n) - h0;
    const int NC = (A.Is >> 5) + k * (A.I >> 5);
    const uint32_t sb = sizeof(TS);

    // ---- before the wait: slot table, routing, region offsets
    if (t == 0) {
        mbar_init(&dbar, 1u + (uint32_t)g_extra_arrivals);
        mbar_init(&rbar, 1);
        fence_mbar_init();
        uint32_t off = 0;
        for (int i = 0; i < n_act; ++i) {
            const int inter = i == k ? A.Is : A.I;
            s_eoff[i] = off;
            off += (uint32_t)nr * ((uint32_t)inter * BITS / 8 + 2 * (uint32_t)(inter >> A.log2G) * sb);
        }
        s_eoff[n_act] = off;
        s_base[k] = A.src.shared;
    }
    for (int e = t; e < A.E; e += kDnThreads)
        tab[e] = __ldg(A.src.table + e);
    load_routing<256>(A.R, rep, A.E, k, tks, s_idx, s_w, false); // keys on the first 256 threads
    if (t < k)
        s_base[t] = routed_base(A.src, tab, s_idx[t]);
    if (t == 32)
        s_w[kMaxAct] = sigmoid_f(__ldcg(A.R.logits ? A.R.logits + (size_t)rep * A.R.lgs + A.E : A.R.sg_logit));
    __syncthreads();

    // ---- the W_d rows [h0, h1) of every active expert (weights: not written
    // by the kernels this one waits for, so copied before the wait)
    unsigned char *down = smem;
    unsigned char *rec = smem + ((s_eoff[n_act] + 127) & ~127u); // [NC][kArec]
    if (warp == 0) {
        const char *b = lane < n_act ? s_base[lane] : nullptr;
        const int inter = lane == k ? A.Is : A.I;
        const uint32_t qb = (uint32_t)inter * BITS / 8, sbb = (uint32_t)(inter >> A.log2G) * sb;
        const uint32_t nq = b ? (uint32_t)nr * qb : 0u, nsb = b ? (uint32_t)nr * sbb : 0u;
        const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, nq + 2 * nsb);
        if (lane == 0)
            mbar_expect_tx(&dbar, tot);
        __syncwarp();
        if (b && nq) {
            const size_t *offs = lane == k ? A.src.off_sh : A.src.off;
            unsigned char *d = down + s_eoff[lane];
            bulk_g2s(d, b + offs[M_QD] + (size_t)h0 * qb, nq, &dbar);
            bulk_g2s(d + nq, b + offs[M_SD] + (size_t)h0 * sbb, nsb, &dbar);
            bulk_g2s(d + nq + nsb, b + offs[M_BD] + (size_t)h0 * sbb, nsb, &dbar);
        }
    }

    pdl_wait(); // the activation records are complete
    pdl_trigger();
    if (c == 0 && A.R.logits && A.R.idx_out && t < k) {
        A.R.idx_out[t] = s_idx[t];
        A.R.w_out[t] = s_w[t];
    }
    if (t == 0) {
        const uint32_t rb = (uint32_t)NC * kArec;
        mbar_expect_tx(&rbar, rb);
        bulk_g2s(rec, A.arec + (size_t)rep * A.ars, rb, &rbar);
    }
    const bool rec_ok = mbar_wait0(&rbar);
    bool ready = mbar_wait0(&dbar);
    if (!ready && t == 0) {
        // supply the arrivals a test asked for, then let the copies land
        for (int j = 0; j < g_extra_arrivals; ++j)
            mbar_arrive(&dbar);
    }
    if (!ready)
        mbar_wait0(&dbar);
    ready = __syncthreads_and(ready && rec_ok);

    // ---- the terms: thread t, chunk j = t % NCp, rows [r0, r0 + nrr) of half hf
    const int NCp = (NC + 31) & ~31;
    const int RH = (nr + 1) >> 1;
    const int hf = t / NCp, j = t - hf * NCp;
    const int r0 = hf * RH, nrr = hf < 2 ? max(0, min(nr, r0 + RH) - r0) : 0; // uniform across a warp
    float v[kMaxRH];
#pragma unroll
    for (int rr = 0; rr < kMaxRH; ++rr)
        v[rr] = 0.f;
    if (ready && hf < 2 && j < NC && nrr > 0) {
        int i, ch;
        if (j < (A.Is >> 5)) {
            i = k;
            ch = j;
        } else {
            i = (j - (A.Is >> 5)) / (A.I >> 5);
            ch = (j - (A.Is >> 5)) - i * (A.I >> 5);
        }
        if (s_base[i]) {
            const uint4 *rv = reinterpret_cast<const uint4 *>(rec + (size_t)j * kArec);
            const uint4 he = rv[0], le = rv[1], ho = rv[2], lo = rv[3], sxu = rv[4], Xu = rv[5];
            const float4 sx = make_float4(__uint_as_float(sxu.x), __uint_as_float(sxu.y), __uint_as_float(sxu.z),
                                          __uint_as_float(sxu.w));
            const float4 X = make_float4(__uint_as_float(Xu.x), __uint_as_float(Xu.y), __uint_as_float(Xu.z),
                                         __uint_as_float(Xu.w));
            const int inter = i == k ? A.Is : A.I;
            const int qb = inter * BITS / 8, ng = inter >> A.log2G;
            const unsigned char *d = down + s_eoff[i];
            const TS *sd = reinterpret_cast<const TS *>(d + nr * qb);
            const TS *bd = sd + nr * ng;
            const int g = (ch * 32) >> A.log2G;
            const float wi = i < k ? s_w[i] : s_w[kMaxAct];
            // straight-line over kMaxRH rows (rows past this half repeat its
            // last row and are dropped), so the rows' chains interleave
#pragma unroll
            for (int rr = 0; rr < kMaxRH; ++rr) {
                const int r = r0 + min(rr, nrr - 1);
                const uint4 *q = reinterpret_cast<const uint4 *>(d + r * qb);
                const float s = to_f32(sd[r * ng + g]), b = to_f32(bd[r * ng + g]);
                const float term = wi * (BITS == 8 ? arec_term8(q[2 * ch], q[2 * ch + 1], he, le, ho, lo, sx, X, s, b)
                                                   : arec_term(q[ch], he, le, ho, lo, sx, X, s, b));
                v[rr] = rr < nrr ? term : 0.f;
            }
        }
    }
    // ---- per warp, each row's sum over the warp's chunks; then per row, its
    // half's warps in order
#pragma unroll
    for (int rr = 0; rr < kMaxRH; ++rr) {
        if (rr < nrr) {
            float x = v[rr];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
            if (lane == 0)
                Pw[r0 + rr][warp] = x;
        }
    }
    __syncthreads();
    if (t < nr) {
        const int wpr = NCp / 32, w0 = (t >= RH ? 1 : 0) * wpr; // warps of each half
        float acc = 0.f;
        for (int w = w0; w < w0 + wpr; ++w)
            acc += Pw[t][w];
        A.y[h0 + t] = __float2bfloat16_rn(acc);
        if (A.y32)
            A.y32[h0 + t] = acc;
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

static int n_chunks(const Shape &s) { return s.Is / 32 + s.k * (s.I / 32); }
static int n_units(const Shape &s) { return s.Is / 8 + s.k * (s.I / 8); }

// Dynamic shared memory of the down kernel (the largest CTA share).
static size_t down_smem(const Shape &s, int n)
{
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    const int nr = (s.H + n - 1) / n;
    size_t w = 0;
    for (int i = 0; i <= s.k; ++i) {
        const int inter = (i == s.k) ? s.Is : s.I;
        w += (size_t)nr * ((size_t)inter * s.bits / 8 + 2 * (inter / s.G) * sb);
    }
    w = (w + 127) & ~(size_t)127;
    return w + (size_t)kArec * n_chunks(s);
}

// Dynamic shared memory of the gate/up kernel: the staged units of the
// largest CTA share.
static size_t gateup_smem(const Shape &s, int n)
{
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    const size_t unitb = 8 * (2 * (size_t)s.H * s.bits / 8 + 4 * (size_t)(s.H / s.G) * sb);
    return (size_t)((n_units(s) + n - 1) / n) * unitb;
}

// With 4-bit codes the gate/up and down kernels share an SM (with their
// static arrays, within its 228 KB).  With 8-bit codes each fits alone: a down
// CTA then starts on an SM as its gate/up CTA ends (nothing waits on their
// being resident together).
constexpr size_t kSmemLimit = 196 * 1024;
constexpr size_t kSmemLimitAlone = 200 * 1024;

bool eligible(const Shape &s)
{
    if (kernel_path() == 1)
        return false;
    if (s.act != MOE_BF16 || s.router != MOE_BF16 || (s.bits != 4 && s.bits != 8))
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
    if ((n_units(s) + n - 1) / n > 5) // six copy lanes a unit, one warp
        return false;
    // down: two threads (row halves) to each chunk, rounded up to whole warps
    if (2 * ((n_chunks(s) + 31) & ~31) > kDnThreads || (s.H + n - 1) / n > 2 * kMaxRH)
        return false;
    if (s.bits == 8)
        return gateup_smem(s, n) <= kSmemLimitAlone && down_smem(s, n) <= kSmemLimitAlone;
    return gateup_smem(s, n) + down_smem(s, n) <= kSmemLimit;
}

// All kernels run with the same (maximal) shared-memory carveout: an SM
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
    return kRep * (lg + xr + ar);
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

template <int NXC, typename TS, int BITS>
static cudaError_t experts_go(const TokArgs &A, int n, size_t gsmem, size_t smem, int H, cudaStream_t st)
{
    static int cur = 0, gcur = 0;
    static bool cvg = false, cvd = false;
    cudaError_t e = set_carveout(gateup_tok_kernel<NXC, TS, BITS>, &cvg);
    if (e == cudaSuccess)
        e = set_carveout(down_tok_kernel<TS, BITS>, &cvd);
    if (e == cudaSuccess)
        e = ensure_smem(down_tok_kernel<TS, BITS>, smem, &cur);
    if (e == cudaSuccess)
        e = ensure_smem(gateup_tok_kernel<NXC, TS, BITS>, gsmem, &gcur);
    if (e == cudaSuccess)
        e = launch_pdl(gateup_tok_kernel<NXC, TS, BITS>, n, kGuThreads, gsmem, st, A);
    if (e == cudaSuccess)
        e = launch_pdl(down_tok_kernel<TS, BITS>, n, kDnThreads, smem, st, A, H);
    return e;
}

template <int BITS>
static cudaError_t experts_bits(const Shape &s, const TokArgs &A, int n, size_t gsmem, size_t smem, cudaStream_t st)
{
    const bool f16 = s.qscale == MOE_F16;
    if (s.H == 1024)
        return f16 ? experts_go<1, __half, BITS>(A, n, gsmem, smem, s.H, st)
                   : experts_go<1, float, BITS>(A, n, gsmem, smem, s.H, st);
    return f16 ? experts_go<2, __half, BITS>(A, n, gsmem, smem, s.H, st)
               : experts_go<2, float, BITS>(A, n, gsmem, smem, s.H, st);
}

cudaError_t launch_experts(const Shape &s, const Bufs &b, const ExpertSrc &src, const Routing &R, void *y,
                           float *y32, cudaStream_t st)
{
    const int n = sm_count();
    TokArgs A{b.xrec, b.xrs, src, R, b.arec, b.ars, static_cast<__nv_bfloat16 *>(y), y32,
              s.E, s.k, s.I, s.Is, log2i(s.G)};
    const size_t smem = down_smem(s, n), gsmem = gateup_smem(s, n);
    return s.bits == 8 ? experts_bits<8>(s, A, n, gsmem, smem, st) : experts_bits<4>(s, A, n, gsmem, smem, st);
}

} // namespace tok
} // namespace moe

extern "C" moe_status moe_debug_set_waits(uint64_t wait_ns, int32_t extra_arrivals)
{
    using namespace moe;
    if (wait_ns == 0 || extra_arrivals < 0 || extra_arrivals > 4)
        return fail(MOE_ERR_INVALID_ARG, "moe_debug_set_waits: wait_ns > 0 and extra_arrivals in [0, 4]");
    const unsigned long long w = wait_ns;
    const int x = extra_arrivals;
    cudaError_t e = cudaMemcpyToSymbol(tok::g_wait_ns, &w, sizeof(w));
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(tok::g_extra_arrivals, &x, sizeof(x));
    return cuda_check(e, "moe_debug_set_waits");
}
