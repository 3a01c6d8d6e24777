// Single-token decode path of the routed int4 MoE layer, built for B300.
//
// Three kernels chained with programmatic dependent launch (PDL), one CTA per
// SM for the expert kernels:
//   router_fast  one warp per router row; the row's weights are loaded before
//                griddepcontrol.wait, so they stream while the previous kernel
//                finishes; writes the logits and the shared-gate logit.
//   gateup_fast  before the wait: bulk-copies (cp.async.bulk + mbarrier) its
//                share of the shared expert's gate/up rows into shared memory
//                and loads x into registers; after the wait: top-k from the
//                logits (every CTA, redundantly: no cross-CTA counter), then
//                bulk-copies its share of the routed rows and computes
//                a = silu(W_g x) * (W_u x) as they land.
//   down_fast    before the wait: top-k again, then bulk-copies its rows of
//                every active expert's W_d (they overlap gate/up's stream);
//                after the wait: loads a and writes
//                y[h] = sum_r w_r (W_d,r a_r)[h] + sigmoid(s) (W_d,sh a_sh)[h]
//                in fixed order.
// Every CTA's share of bytes fits in shared memory at once, so each copy is
// issued exactly once and waited on with a single-phase mbarrier.
//
// Dequantisation: the code q of each weight is placed in the top mantissa
// bits of 1.0f (one PRMT per weight builds 1 + q/16), products are summed
// with packed fp32 FMA (two lanes per instruction), and
//   sum_c (s q_c + b) x_c = 16 s D + (b - 16 s) X,  D = sum_c (1 + q_c/16) x_c,
// with X = sum_c x_c taken once per 32-column chunk.
#include <float.h>
#include <math.h>

#include "internal.h"

namespace moe {
namespace fast {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSeg = 4;          // gate/up segments per CTA (1 shared + up to 3 routed)
constexpr int kMaxAct = 17;         // top_k <= 16 plus the shared expert
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000; // 0.2 s bound on any barrier wait

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

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy; completion is signalled on `bar` as bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
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

// Wait for phase 0 of a single-use barrier, for at most kWaitNs of wall
// time (try_wait may suspend between polls, so the bound is on time, not
// on polls); false, with MOE_ERR_TIMEOUT recorded, if it never completes.
__device__ __forceinline__ bool mbar_wait0(uint64_t *bar)
{
    if (mbar_try_wait(bar, 0))
        return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
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

// ------------------------------------------------------------ arithmetic

// D = sum_{j<32} (1 + q_j/16) * v[j] for the 32 codes of one 16-byte chunk
// (column order: word m holds columns 8m..8m+7, lowest column in the lowest
// nibble).
__device__ __forceinline__ float chunk_dot(uint4 q, const float *v)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        // byte b of lo: 0x80 | code(col 2b) << 3; of hi: 0x80 | code(col 2b+1) << 3
        const uint32_t lo = ((w[m] << 3) & 0x78787878u) | 0x80808080u;
        const uint32_t hi = ((w[m] >> 1) & 0x78787878u) | 0x80808080u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t sel = 0x7044u | (uint32_t)(b << 8);
            const float f0 = __uint_as_float(__byte_perm(lo, 0x3F000000u, sel));
            const float f1 = __uint_as_float(__byte_perm(hi, 0x3F000000u, sel));
            const float2 xv = make_float2(v[8 * m + 2 * b], v[8 * m + 2 * b + 1]);
            if (b & 1)
                acc1 = __ffma2_rn(make_float2(f0, f1), xv, acc1);
            else
                acc0 = __ffma2_rn(make_float2(f0, f1), xv, acc0);
        }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// Group contribution of one chunk: s * sum q x + b * sum x.
__device__ __forceinline__ float chunk_term(float D, float X, float s, float b)
{
    const float s16 = 16.f * s;
    return fmaf(s16, D, (b - s16) * X);
}

template <typename TS> __device__ __forceinline__ float ld_scale(const TS *p) { return to_f32(*p); }

// Does (va, ea) rank before (vb, eb) under (logit descending, id ascending)?
__device__ __forceinline__ bool ranks_before(float va, int ea, float vb, int eb)
{
    return va > vb || (va == vb && ea < eb);
}

// Top-k of E <= 32*PER logits (global, written by an earlier kernel) by one
// warp, under the order (logit descending, id ascending); NaN ranks as -inf.
// Lane r < k returns the r-th expert and its weight exp(l_r - l_0) / sum.
//
// Prefilter: tau = the k-th largest of the 32 lane maxima.  At least k
// logits are >= tau, so every logit of the top k is >= tau; when at most 32
// logits pass, one bitonic sort across the lanes orders them exactly.
// Otherwise (heavy ties) k rounds of warp arg-max select them.  Both give
// the same list.  cand_v / cand_e: 32-entry shared scratch of this warp.
template <int PER>
__device__ __forceinline__ void warp_topk(const float *lg, int E, int k, int lane, float *cand_v, int *cand_e,
                                          int *sel_e, float *sel_w)
{
    float v[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        const float f = e < E ? __ldcg(lg + e) : -INFINITY;
        v[j] = isnan(f) ? -INFINITY : f;
    }
    float m = v[0];
#pragma unroll
    for (int j = 1; j < PER; ++j)
        m = fmaxf(m, v[j]);
    // bitonic sort (descending across lanes) of the lane maxima
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, m, stride);
            const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
            m = keep_max ? fmaxf(m, o) : fminf(m, o);
        }
    const float tau = __shfl_sync(0xFFFFFFFFu, m, k - 1);
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
        cnt += (v[j] >= tau && lane + 32 * j < E) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o)
            incl += u;
    }
    const int C = __shfl_sync(0xFFFFFFFFu, incl, 31);
    float sv;
    int se;
    if (C <= 32 && tau > -INFINITY) {
        int pos = incl - cnt;
#pragma unroll
        for (int j = 0; j < PER; ++j)
            if (v[j] >= tau && lane + 32 * j < E) {
                cand_v[pos] = v[j];
                cand_e[pos] = lane + 32 * j;
                ++pos;
            }
        __syncwarp();
        sv = lane < C ? cand_v[lane] : -INFINITY;
        se = lane < C ? cand_e[lane] : 0x7FFFFFFF;
        __syncwarp();
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, sv, stride);
                const int oe = __shfl_xor_sync(0xFFFFFFFFu, se, stride);
                const bool keep_first = ((lane & stride) == 0) == ((lane & size) == 0);
                const bool other_first = ranks_before(ov, oe, sv, se);
                if (keep_first == other_first) {
                    sv = ov;
                    se = oe;
                }
            }
    } else {
        uint32_t taken = 0;
        sv = 0.f;
        se = 0;
        for (int r = 0; r < k; ++r) {
            float bv = -INFINITY;
            int be = 0x7FFFFFFF;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int e = lane + 32 * j;
                if (e < E && !((taken >> j) & 1u) && ranks_before(v[j], e, bv, be)) {
                    bv = v[j];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
                const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
                if (ranks_before(ov, oe, bv, be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane)
                taken |= 1u << (be >> 5);
            if (lane == r) {
                sv = bv;
                se = be;
            }
        }
    }
    const float lmax = __shfl_sync(0xFFFFFFFFu, sv, 0);
    const float ex = lane < k ? expf(sv - lmax) : 0.f;
    const float den = warp_sum(ex);
    *sel_e = se;
    *sel_w = ex / den;
}

// Fill s_idx / s_w (shared memory) from the routing.  Called by warp 0 only.
__device__ __forceinline__ void load_routing(const Routing &R, int E, int k, int lane, int *s_idx, float *s_w,
                                             float *cand_v, int *cand_e, bool write_out)
{
    if (R.logits) {
        int e;
        float wv;
        if (E <= 256)
            warp_topk<8>(R.logits, E, k, lane, cand_v, cand_e, &e, &wv);
        else if (E <= 512)
            warp_topk<16>(R.logits, E, k, lane, cand_v, cand_e, &e, &wv);
        else
            warp_topk<32>(R.logits, E, k, lane, cand_v, cand_e, &e, &wv);
        if (lane < k) {
            s_idx[lane] = e;
            s_w[lane] = wv;
            if (write_out && R.idx_out) {
                R.idx_out[lane] = e;
                R.w_out[lane] = wv;
            }
        }
    } else if (lane < k) {
        s_idx[lane] = __ldcg(R.idx + lane);
        s_w[lane] = __ldcg(R.w + lane);
    }
    __syncwarp();
}

// Blob address of active expert i (i == k: shared) or nullptr (recorded).
__device__ __forceinline__ const char *active_base(const ExpertSrc &src, const int *s_idx, int k, int i)
{
    if (i == k)
        return src.shared;
    const int e = s_idx[i];
    if (e < 0 || e >= src.n_experts) {
        record_error(MOE_ERR_DEVICE_FAULT);
        return nullptr;
    }
    const int slot = src.table[e];
    if (slot < 0 || slot >= src.n_slots) {
        record_error(MOE_ERR_NOT_RESIDENT);
        return nullptr;
    }
    return src.pool + (size_t)slot * src.stride;
}

// ------------------------------------------------------------ router

// One warp per row: rows 0..E-1 are experts, row E the shared gate.
// grid = ceil((E + has_sg) / 4), 128 threads.  H = 256 * NJ.
template <int NJ>
__global__ void __launch_bounds__(128) router_fast_kernel(const __nv_bfloat16 *__restrict__ x, int E,
                                                         const __nv_bfloat16 *__restrict__ wr,
                                                         const float *__restrict__ bias,
                                                         const __nv_bfloat16 *__restrict__ wsg,
                                                         float *__restrict__ logits, float *__restrict__ sg)
{
    constexpr int H = 256 * NJ;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    const int nrows = E + (wsg ? 1 : 0);
    uint4 wv[NJ];
    const bool active = row < nrows;
    if (active) {
        const __nv_bfloat16 *w = row < E ? wr + (size_t)row * H : wsg;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            wv[j] = __ldg(reinterpret_cast<const uint4 *>(w + (lane + 32 * j) * 8));
    }
    pdl_wait();
    pdl_trigger();
    if (!active)
        return;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + (lane + 32 * j) * 8));
        const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t wa[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            acc = fmaf(__uint_as_float(wa[m] << 16), __uint_as_float(xa[m] << 16), acc);
            acc = fmaf(__uint_as_float(wa[m] & 0xFFFF0000u), __uint_as_float(xa[m] & 0xFFFF0000u), acc);
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) {
        if (row < E)
            logits[row] = acc + (bias ? bias[row] : 0.f);
        else
            *sg = acc;
    }
}

// ------------------------------------------------------------ gate/up

struct GateUpArgs {
    const __nv_bfloat16 *x; // [H]
    ExpertSrc src;
    Routing R;
    float *a;               // [k+1][Imax]
    int E, k, I, Is, Imax, G;
};

// Rows of active expert `i`, [o0, o0 + n), one segment of a CTA's share.
struct Seg {
    int i, o0, n;
    uint32_t off; // shared-memory byte offset of the segment
};

// H = 1024 * NXC; TS = scale/bias type.
//
// Warp 0 waits for the router (griddepcontrol.wait), selects the top k, and
// issues the routed rows' copies (lane s handles segment s); then all warps
// compute, the shared expert's rows first (their copies were issued before
// the wait), the routed rows as they land.  Every segment barrier is armed
// exactly once, with zero bytes when the expert has no slot, so no consumer
// can wait forever.
template <int NXC, typename TS>
__global__ void __launch_bounds__(kThreads, 1) gateup_fast_kernel(GateUpArgs A)
{
    constexpr int H = 1024 * NXC;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bars[kMaxSeg];
    __shared__ int s_idx[kMaxAct];
    __shared__ float s_w[kMaxAct];
    __shared__ const char *s_base[kMaxSeg];
    __shared__ float cand_v[32];
    __shared__ int cand_e[32];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = gridDim.x, c = blockIdx.x;
    const int k = A.k, G = A.G;
    const uint32_t qrow = H / 2;                          // code bytes per row
    const uint32_t srow = (uint32_t)(H / G) * sizeof(TS); // scale (or bias) bytes per row
    const uint32_t rowpair = 2 * qrow + 4 * srow;

    // This CTA's share: shared rows [sh0, sh1) and routed flat rows [r0, r1).
    const int sh0 = (int)((long)c * A.Is / n), sh1 = (int)((long)(c + 1) * A.Is / n);
    const long RT = (long)k * A.I;
    const int r0 = (int)((long)c * RT / n), r1 = (int)((long)(c + 1) * RT / n);
    Seg seg[kMaxSeg];
    int nseg = 0;
    uint32_t off = 0;
    if (sh1 > sh0) {
        seg[nseg++] = {k, sh0, sh1 - sh0, off};
        off += (uint32_t)(sh1 - sh0) * rowpair;
    }
    for (int r = r0; r < r1 && nseg < kMaxSeg;) {
        const int i = r / A.I, o = r - i * A.I;
        const int len = min(r1 - r, A.I - o);
        seg[nseg++] = {i, o, len, off};
        off += (uint32_t)len * rowpair;
        r += len;
    }

    // Six copies of one segment (one thread).
    auto issue = [&](int s, const char *base) {
        const Seg &g = seg[s];
        const size_t *offs = (g.i == k) ? A.src.off_sh : A.src.off;
        const uint32_t n_q = (uint32_t)g.n * qrow, n_s = (uint32_t)g.n * srow;
        unsigned char *d = smem + g.off;
        mbar_arrive_expect_tx(&bars[s], 2 * n_q + 4 * n_s);
        bulk_g2s(d, base + offs[M_QG] + (size_t)g.o0 * qrow, n_q, &bars[s]);
        bulk_g2s(d + n_q, base + offs[M_QU] + (size_t)g.o0 * qrow, n_q, &bars[s]);
        bulk_g2s(d + 2 * n_q, base + offs[M_SG] + (size_t)g.o0 * srow, n_s, &bars[s]);
        bulk_g2s(d + 2 * n_q + n_s, base + offs[M_BG] + (size_t)g.o0 * srow, n_s, &bars[s]);
        bulk_g2s(d + 2 * n_q + 2 * n_s, base + offs[M_SU] + (size_t)g.o0 * srow, n_s, &bars[s]);
        bulk_g2s(d + 2 * n_q + 3 * n_s, base + offs[M_BU] + (size_t)g.o0 * srow, n_s, &bars[s]);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxSeg; ++s)
            mbar_init(&bars[s], 1);
        fence_mbar_init();
        for (int s = 0; s < nseg; ++s)
            if (seg[s].i == k) {
                s_base[s] = A.src.shared;
                issue(s, A.src.shared);
            }
    }
    __syncthreads();

    // x into registers: lane owns 32-column chunks lane + 32 m.
    float xr[NXC][32];
    float xs[NXC];
#pragma unroll
    for (int m = 0; m < NXC; ++m) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(A.x + (lane + 32 * m) * 32);
        xs[m] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldg(xp + q);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                xr[m][8 * q + 2 * t] = __uint_as_float(u[t] << 16);
                xr[m][8 * q + 2 * t + 1] = __uint_as_float(u[t] & 0xFFFF0000u);
            }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
            xs[m] += xr[m][j];
    }

    if (warp == 0) {
        pdl_wait();
        load_routing(A.R, A.E, k, lane, s_idx, s_w, cand_v, cand_e, c == 0);
        if (lane < nseg && seg[lane].i != k) {
            const char *b = active_base(A.src, s_idx, k, seg[lane].i);
            s_base[lane] = b;
            if (b)
                issue(lane, b);
            else
                mbar_arrive_expect_tx(&bars[lane], 0);
        }
    }
    // The routing is settled and every routed copy is in flight: the shared
    // rows (already landed) are computed while the routed rows arrive.
    __syncthreads();
    pdl_trigger();

    int seg_start[kMaxSeg + 1];
    seg_start[0] = 0;
    for (int s = 0; s < kMaxSeg; ++s)
        seg_start[s + 1] = seg_start[s] + (s < nseg ? seg[s].n : 0);
    const int total = seg_start[nseg];
    int waited = -1;
    for (int rho = warp; rho < total; rho += kWarps) {
        int s = 0;
        while (rho >= seg_start[s + 1])
            ++s;
        const Seg &g = seg[s];
        if (waited < s) {
            if (!mbar_wait0(&bars[s]))
                return;
            waited = s;
        }
        const int r = rho - seg_start[s];
        float *dst = A.a + (size_t)g.i * A.Imax + g.o0 + r;
        if (s_base[s] == nullptr) {
            if (lane == 0)
                *dst = 0.f;
            continue;
        }
        const uint32_t n_q = (uint32_t)g.n * qrow, n_s = (uint32_t)g.n * srow;
        const unsigned char *d = smem + g.off;
        const uint4 *qg = reinterpret_cast<const uint4 *>(d + (size_t)r * qrow);
        const uint4 *qu = reinterpret_cast<const uint4 *>(d + n_q + (size_t)r * qrow);
        const TS *sg = reinterpret_cast<const TS *>(d + 2 * n_q) + (size_t)r * (H / G);
        const TS *bg = reinterpret_cast<const TS *>(d + 2 * n_q + n_s) + (size_t)r * (H / G);
        const TS *su = reinterpret_cast<const TS *>(d + 2 * n_q + 2 * n_s) + (size_t)r * (H / G);
        const TS *bu = reinterpret_cast<const TS *>(d + 2 * n_q + 3 * n_s) + (size_t)r * (H / G);
        float gacc = 0.f, uacc = 0.f;
#pragma unroll
        for (int m = 0; m < NXC; ++m) {
            const int ch = lane + 32 * m;
            const int grp = (ch * 32) / G;
            const float dg = chunk_dot(qg[ch], xr[m]);
            const float du = chunk_dot(qu[ch], xr[m]);
            gacc += chunk_term(dg, xs[m], ld_scale(sg + grp), ld_scale(bg + grp));
            uacc += chunk_term(du, xs[m], ld_scale(su + grp), ld_scale(bu + grp));
        }
        const float gv = warp_sum(gacc);
        const float uv = warp_sum(uacc);
        if (lane == 0)
            *dst = gv * sigmoid_f(gv) * uv;
    }
}

// ------------------------------------------------------------ down + combine

struct DownArgs {
    ExpertSrc src;
    Routing R;
    const float *a; // [k+1][Imax]
    __nv_bfloat16 *y;
    float *y32;
    int E, H, k, I, Is, Imax, G, n_act;
};

// grid = n CTAs; CTA c owns output rows [c*H/n, (c+1)*H/n).
//
// Before the wait (the routing is at least two kernels old, so visible): warp
// 0 selects the top k, resolves every active expert's slot in parallel (lane
// i, expert i) and issues its three copies; the shared-gate logit is read
// here too, before this kernel lets the next token's router start.  After the
// wait: a (written by gate/up) is loaded with 16-byte loads.
template <typename TS>
__global__ void __launch_bounds__(kThreads, 1) down_fast_kernel(DownArgs A)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t bar;
    __shared__ int s_idx[kMaxAct];
    __shared__ float s_w[kMaxAct + 1];
    __shared__ const char *s_base[kMaxAct];
    __shared__ uint32_t s_eoff[kMaxAct];
    __shared__ float cand_v[32];
    __shared__ int cand_e[32];

    const int n = gridDim.x, c = blockIdx.x;
    const int h0 = (int)((long)c * A.H / n), h1 = (int)((long)(c + 1) * A.H / n);
    const int nr = h1 - h0;
    const int k = A.k, G = A.G, n_act = A.n_act;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Per-expert shared-memory offsets: codes [nr][inter/2], scales and
    // biases [nr][inter/G] each (identical in every thread).
    auto exp_off = [&](int i) {
        uint32_t o = 0;
        for (int j = 0; j < i; ++j) {
            const int inter = (j == k) ? A.Is : A.I;
            o += (uint32_t)nr * (inter / 2 + 2 * (inter / G) * (uint32_t)sizeof(TS));
        }
        return o;
    };
    const uint32_t wbytes = exp_off(n_act);

    if (warp == 0) {
        float sgl = 0.f;
        if (lane == 0) {
            mbar_init(&bar, 1);
            fence_mbar_init();
            sgl = __ldcg(A.R.sg_logit);
        }
        if (lane < n_act)
            s_eoff[lane] = exp_off(lane);
        load_routing(A.R, A.E, k, lane, s_idx, s_w, cand_v, cand_e, false);
        if (lane == 0)
            s_w[kMaxAct] = sigmoid_f(sgl);
        const char *b = nullptr;
        uint32_t bytes = 0;
        if (lane < n_act) {
            b = active_base(A.src, s_idx, k, lane);
            s_base[lane] = b;
            const int inter = (lane == k) ? A.Is : A.I;
            if (b)
                bytes = (uint32_t)nr * (inter / 2 + 2 * (inter / G) * (uint32_t)sizeof(TS));
        }
        uint32_t total = bytes;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
        if (lane == 0)
            mbar_arrive_expect_tx(&bar, total);
        __syncwarp();
        if (b) {
            const int inter = (lane == k) ? A.Is : A.I;
            const size_t *offs = (lane == k) ? A.src.off_sh : A.src.off;
            const uint32_t nq = (uint32_t)nr * (inter / 2), ns = (uint32_t)nr * (inter / G) * sizeof(TS);
            unsigned char *d = smem + s_eoff[lane];
            bulk_g2s(d, b + offs[M_QD] + (size_t)h0 * (inter / 2), nq, &bar);
            bulk_g2s(d + nq, b + offs[M_SD] + (size_t)h0 * (inter / G) * sizeof(TS), ns, &bar);
            bulk_g2s(d + nq + ns, b + offs[M_BD] + (size_t)h0 * (inter / G) * sizeof(TS), ns, &bar);
        }
    }
    const int pI = A.Imax + (A.Imax >> 5) * 4;
    float *as = reinterpret_cast<float *>(smem + ((wbytes + 15) & ~15u)); // [n_act][pI]
    float *asum = as + n_act * pI;                                          // [n_act][Imax/32]

    pdl_wait();
    pdl_trigger();
    {   // a -> shared memory, 16-byte loads, several in flight per thread
        const int n4 = n_act * A.Imax / 4, q4 = A.Imax / 4;
        const float4 *a4 = reinterpret_cast<const float4 *>(A.a);
        constexpr int U = 8;
        for (int j0 = threadIdx.x; j0 < n4; j0 += U * kThreads) {
            float4 buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u * kThreads;
                if (j < n4)
                    buf[u] = __ldcg(a4 + j);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u * kThreads;
                if (j < n4) {
                    const int i = j / q4, c4 = j - i * q4; // float4 index within the row
                    *reinterpret_cast<float4 *>(as + i * pI + c4 * 4 + (c4 >> 3) * 4) = buf[u];
                }
            }
        }
    }
    __syncthreads();
    const int nchm = A.Imax >> 5;
    for (int j = threadIdx.x; j < n_act * nchm; j += kThreads) {
        const int i = j / nchm, ch = j - i * nchm;
        const float *p = as + i * pI + ch * 36;
        float sacc = 0.f;
#pragma unroll 8
        for (int q = 0; q < 32; ++q)
            sacc += p[q];
        asum[j] = sacc;
    }
    __syncthreads();
    const bool ready = mbar_wait0(&bar);

    // A half-warp per output row: lane l16 takes chunks l16, l16 + 16, ... of
    // every active expert's row and accumulates w_i * (its chunk terms) in
    // expert order (routed by rank, then shared); one reduction per row.
    const int half = lane >> 4, l16 = lane & 15;
    for (int hr0 = 0; hr0 < nr; hr0 += 2 * kWarps) {
        const int hr = hr0 + warp * 2 + half;
        float acc = 0.f;
        if (ready && hr < nr) {
            for (int i = 0; i < n_act; ++i) {
                if (!s_base[i])
                    continue;
                const int inter = (i == k) ? A.Is : A.I;
                const int nch = inter >> 5;
                const uint32_t nq = (uint32_t)nr * (inter / 2), ns = (uint32_t)nr * (inter / G) * sizeof(TS);
                const unsigned char *d = smem + s_eoff[i];
                const uint4 *q = reinterpret_cast<const uint4 *>(d + (size_t)hr * (inter / 2));
                const TS *sd = reinterpret_cast<const TS *>(d + nq) + (size_t)hr * (inter / G);
                const TS *bd = reinterpret_cast<const TS *>(d + nq + ns) + (size_t)hr * (inter / G);
                const float wi = (i < k) ? s_w[i] : s_w[kMaxAct];
                float part = 0.f;
                for (int ch = l16; ch < nch; ch += 16) {
                    const float *v = as + i * pI + ch * 36;
                    float vr[32];
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const float4 f = *reinterpret_cast<const float4 *>(v + 4 * t);
                        vr[4 * t] = f.x;
                        vr[4 * t + 1] = f.y;
                        vr[4 * t + 2] = f.z;
                        vr[4 * t + 3] = f.w;
                    }
                    const int grp = (ch * 32) / G;
                    part += chunk_term(chunk_dot(q[ch], vr), asum[i * nchm + ch], ld_scale(sd + grp),
                                       ld_scale(bd + grp));
                }
                acc = fmaf(wi, part, acc);
            }
        }
        acc = half_warp_sum(acc);
        if (ready && hr < nr && l16 == 0) {
            A.y[h0 + hr] = __float2bfloat16_rn(acc);
            if (A.y32)
                A.y32[h0 + hr] = acc;
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

static size_t gateup_smem(const Shape &s, int n)
{
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    const size_t rowpair = (size_t)s.H + 4 * (size_t)(s.H / s.G) * sb;
    const long RT = (long)s.k * s.I;
    const size_t rows = (size_t)((s.Is + n - 1) / n) + (size_t)((RT + n - 1) / n);
    return rows * rowpair;
}

static size_t down_smem(const Shape &s, int n)
{
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    const int nr = (s.H + n - 1) / n;
    const int n_act = s.k + (s.Is > 0 ? 1 : 0);
    const int imax = s.I > s.Is ? s.I : s.Is;
    size_t w = 0;
    for (int i = 0; i < n_act; ++i) {
        const int inter = (i == s.k) ? s.Is : s.I;
        w += (size_t)nr * (inter / 2 + 2 * (inter / s.G) * sb);
    }
    w = (w + 15) & ~(size_t)15;
    const size_t pI = imax + (imax / 32) * 4;
    return w + sizeof(float) * (n_act * pI + n_act * (imax / 32) + (size_t)nr * n_act);
}

constexpr size_t kSmemBudget = 200 * 1024;

bool eligible(const Shape &s)
{
    if (kernel_path() != 0)
        return false;
    if (s.act != MOE_BF16 || s.router != MOE_BF16)
        return false;
    if (s.H != 1024 && s.H != 2048 && s.H != 4096)
        return false;
    if (s.Is <= 0 || s.k + 1 > kMaxAct)
        return false;
    const int sb = s.qscale == MOE_F16 ? 2 : 4;
    if (((s.H / s.G) * sb) % 16 || ((s.I / s.G) * sb) % 16 || ((s.Is / s.G) * sb) % 16)
        return false;
    if (s.I % 32 || s.Is % 32)
        return false;
    const int n = sm_count();
    if ((long)s.k * s.I / n + 1 > s.I) // a CTA's routed share spans at most two experts
        return false;
    return gateup_smem(s, n) <= kSmemBudget && down_smem(s, n) <= kSmemBudget;
}

cudaError_t launch_router_fast(const Shape &s, const void *x, const void *w_router, const float *bias,
                               const void *w_sg, float *logits, float *sg, cudaStream_t st)
{
    const int rows = s.E + (w_sg ? 1 : 0);
    const int grid = (rows + 3) / 4;
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    const __nv_bfloat16 *wr = static_cast<const __nv_bfloat16 *>(w_router);
    const __nv_bfloat16 *ws = static_cast<const __nv_bfloat16 *>(w_sg);
    switch (s.H) {
    case 1024:
        return launch_pdl(router_fast_kernel<4>, grid, 128, 0, st, xb, s.E, wr, bias, ws, logits, sg);
    case 2048:
        return launch_pdl(router_fast_kernel<8>, grid, 128, 0, st, xb, s.E, wr, bias, ws, logits, sg);
    default:
        return launch_pdl(router_fast_kernel<16>, grid, 128, 0, st, xb, s.E, wr, bias, ws, logits, sg);
    }
}

template <int NXC, typename TS>
static cudaError_t gateup_go(const Shape &s, const GateUpArgs &A, int n, size_t smem, cudaStream_t st)
{
    static int cur = 0;
    cudaError_t e = ensure_smem(gateup_fast_kernel<NXC, TS>, smem, &cur);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(gateup_fast_kernel<NXC, TS>, n, kThreads, smem, st, A);
}

template <typename TS>
static cudaError_t down_go(const DownArgs &A, int n, size_t smem, cudaStream_t st)
{
    static int cur = 0;
    cudaError_t e = ensure_smem(down_fast_kernel<TS>, smem, &cur);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(down_fast_kernel<TS>, n, kThreads, smem, st, A);
}

cudaError_t launch_experts_fast(const Shape &s, const void *x, const ExpertSrc &src, const Routing &R, float *a,
                                void *y, float *y32, cudaStream_t st)
{
    const int n = sm_count();
    const int imax = s.I > s.Is ? s.I : s.Is;
    GateUpArgs g{static_cast<const __nv_bfloat16 *>(x), src, R, a, s.E, s.k, s.I, s.Is, imax, s.G};
    const size_t gs = gateup_smem(s, n);
    cudaError_t e;
    const bool f16 = s.qscale == MOE_F16;
    if (s.H == 1024)
        e = f16 ? gateup_go<1, __half>(s, g, n, gs, st) : gateup_go<1, float>(s, g, n, gs, st);
    else if (s.H == 2048)
        e = f16 ? gateup_go<2, __half>(s, g, n, gs, st) : gateup_go<2, float>(s, g, n, gs, st);
    else
        e = f16 ? gateup_go<4, __half>(s, g, n, gs, st) : gateup_go<4, float>(s, g, n, gs, st);
    if (e != cudaSuccess)
        return e;
    DownArgs d{src, R, a, static_cast<__nv_bfloat16 *>(y), y32, s.E, s.H, s.k, s.I, s.Is, imax, s.G,
               s.k + 1};
    d.R.idx_out = nullptr;
    d.R.w_out = nullptr;
    const size_t ds = down_smem(s, n);
    return f16 ? down_go<__half>(d, n, ds, st) : down_go<float>(d, n, ds, st);
}

} // namespace fast
} // namespace moe
