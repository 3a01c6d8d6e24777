// Router, top-k and the generic expert kernels of the routed MoE layer
// (affine int4 or int8 codes).
//
// Decode is bandwidth-bound: every active expert's packed weights are read
// once per token, so the kernels stream them with 16-byte loads and do the
// affine dequantisation in registers using the group-sum identity
//   sum_c (s*q_c + b) x_c = s * sum_c q_c x_c + b * sum_c x_c
// with sum_c x_c taken once per 32-column chunk.
#include <float.h>
#include <math.h>

#include "internal.h"

namespace moe {

// ---------------------------------------------------------------- router

// One warp per router row (E expert rows, then the shared-gate row), a block
// of TB tokens per CTA.  logits[t,e] = w_router[e] . x[t] + bias[e];
// sg_logit[t] = w_sg . x[t].  fp32 accumulation.
template <typename TA, typename TR, int TB>
__global__ void __launch_bounds__(128) router_kernel(const TA *__restrict__ x, int T, int H, int E,
                                                     const TR *__restrict__ wr,
                                                     const float *__restrict__ bias,
                                                     const TR *__restrict__ wsg,
                                                     float *__restrict__ logits,
                                                     float *__restrict__ sg_logit)
{
    extern __shared__ float xs[]; // [TB][H]
    const int t0 = blockIdx.y * TB;
    const int nt = min(TB, T - t0);
    for (int i = threadIdx.x; i < nt * H; i += blockDim.x)
        xs[i] = to_f32(x[(size_t)t0 * H + i]);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + warp;
    const int nrows = E + (wsg ? 1 : 0);
    if (row >= nrows)
        return;
    const TR *w = row < E ? wr + (size_t)row * H : wsg;
    float acc[TB];
#pragma unroll
    for (int tb = 0; tb < TB; ++tb)
        acc[tb] = 0.f;
    for (int c = lane * 8; c < H; c += 256) {
        float wv[8];
        load8_f32(w + c, wv);
#pragma unroll
        for (int tb = 0; tb < TB; ++tb) {
            if (tb < nt) {
                const float *xp = xs + tb * H + c;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    acc[tb] = fmaf(wv[j], xp[j], acc[tb]);
            }
        }
    }
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
        float v = warp_sum(acc[tb]);
        if (lane == 0 && tb < nt) {
            if (row < E)
                logits[(size_t)(t0 + tb) * E + row] = v + (bias ? bias[row] : 0.f);
            else
                sg_logit[t0 + tb] = v;
        }
    }
}

template <typename TA, typename TR>
static cudaError_t router_dispatch(const Shape &s, const void *x, int T, const void *wr,
                                   const float *bias, const void *wsg, float *logits, float *sg,
                                   cudaStream_t st)
{
    const int rows = s.E + (wsg ? 1 : 0);
    const int warps = 4;
    if (T == 1) {
        dim3 grid((rows + warps - 1) / warps, 1);
        size_t smem = (size_t)s.H * sizeof(float);
        router_kernel<TA, TR, 1><<<grid, warps * 32, smem, st>>>(
            (const TA *)x, T, s.H, s.E, (const TR *)wr, bias, (const TR *)wsg, logits, sg);
    } else {
        constexpr int TB = 8;
        dim3 grid((rows + warps - 1) / warps, (T + TB - 1) / TB);
        size_t smem = (size_t)TB * s.H * sizeof(float);
        auto kern = router_kernel<TA, TR, TB>;
        static int cur_smem = 0;
        cudaError_t e = ensure_smem(kern, smem, &cur_smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, warps * 32, smem, st>>>((const TA *)x, T, s.H, s.E, (const TR *)wr, bias,
                                             (const TR *)wsg, logits, sg);
    }
    return cudaGetLastError();
}

cudaError_t launch_router(const Shape &s, const void *x, int T, const void *w_router,
                          const float *bias, const void *w_sg, float *logits, float *sg_logit,
                          cudaStream_t st)
{
    // the tensor-core GEMM reads x and the router rows through TMA and the
    // shared-gate row with 16-byte loads
    const auto a16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    if (router_gemm_eligible(s, T) && a16(x) && a16(w_router) && a16(w_sg))
        return launch_router_gemm(s, x, T, w_router, bias, w_sg, logits, sg_logit, st);
    if (s.act == MOE_BF16 && s.router == MOE_BF16)
        return router_dispatch<__nv_bfloat16, __nv_bfloat16>(s, x, T, w_router, bias, w_sg, logits, sg_logit, st);
    if (s.act == MOE_F32 && s.router == MOE_F32)
        return router_dispatch<float, float>(s, x, T, w_router, bias, w_sg, logits, sg_logit, st);
    if (s.act == MOE_BF16 && s.router == MOE_F32)
        return router_dispatch<__nv_bfloat16, float>(s, x, T, w_router, bias, w_sg, logits, sg_logit, st);
    return router_dispatch<float, __nv_bfloat16>(s, x, T, w_router, bias, w_sg, logits, sg_logit, st);
}

// ---------------------------------------------------------------- top-k

// One warp per token.  Lane l holds logits l, l+32, ...; k rounds of a warp
// arg-max under the order (logit descending, expert id ascending) select the
// experts; lane r keeps the r-th.  Weights: exp(l_r - l_0) / sum_r.
// NaN logits rank as -inf.
template <int PER>
__global__ void __launch_bounds__(128) topk_kernel(const float *__restrict__ logits, int T, int E,
                                                   int k, int32_t *__restrict__ idx,
                                                   float *__restrict__ w)
{
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T)
        return;
    const float *lg = logits + (size_t)t * E;
    float v[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        int e = lane + 32 * j;
        float f = e < E ? lg[e] : -INFINITY;
        v[j] = isnan(f) ? -INFINITY : f;
    }
    uint32_t taken = 0;
    float sel_v = 0.f;
    int sel_e = 0;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < be))) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane)
            taken |= 1u << (be >> 5);
        if (lane == r) {
            sel_v = bv;
            sel_e = be;
        }
    }
    const float lmax = __shfl_sync(0xFFFFFFFFu, sel_v, 0);
    const float ex = lane < k ? expf(sel_v - lmax) : 0.f;
    const float den = warp_sum(ex);
    if (lane < k) {
        idx[(size_t)t * k + lane] = sel_e;
        w[(size_t)t * k + lane] = ex / den;
    }
}

cudaError_t launch_topk(const Shape &s, const float *logits, int T, int32_t *idx, float *w,
                        cudaStream_t st)
{
    const int threads = 128, per_cta = threads / 32;
    dim3 grid((T + per_cta - 1) / per_cta);
    if (s.E <= 256)
        topk_kernel<8><<<grid, threads, 0, st>>>(logits, T, s.E, s.k, idx, w);
    else if (s.E <= 512)
        topk_kernel<16><<<grid, threads, 0, st>>>(logits, T, s.E, s.k, idx, w);
    else
        topk_kernel<32><<<grid, threads, 0, st>>>(logits, T, s.E, s.k, idx, w);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- experts

// fp32 vectors in shared memory are stored with 4 floats of padding after
// every 32 values, so that lane l reading chunk l with 16-byte loads touches
// distinct banks within each 8-lane phase.
__host__ __device__ __forceinline__ int padded(int c) { return c + (c >> 5) * 4; }

// Dot of one chunk of codes (32 columns, all in one quantisation group) with
// 32 fp32 values at v (padded layout, 16-byte aligned).  BITS = 4: the
// chunk's codes are one 16-byte word q; BITS = 8: two, q then q2.
__device__ __forceinline__ float chunk_code_dot(uint4 q, const float *v)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        float4 v0 = *reinterpret_cast<const float4 *>(v + 8 * m);
        float4 v1 = *reinterpret_cast<const float4 *>(v + 8 * m + 4);
        acc = fmaf(code_f32(w[m], 0), v0.x, acc);
        acc = fmaf(code_f32(w[m], 1), v0.y, acc);
        acc = fmaf(code_f32(w[m], 2), v0.z, acc);
        acc = fmaf(code_f32(w[m], 3), v0.w, acc);
        acc = fmaf(code_f32(w[m], 4), v1.x, acc);
        acc = fmaf(code_f32(w[m], 5), v1.y, acc);
        acc = fmaf(code_f32(w[m], 6), v1.z, acc);
        acc = fmaf(code_f32(w[m], 7), v1.w, acc);
    }
    return acc;
}

// 8-bit code j (byte j) of a word -> exact fp32.
__device__ __forceinline__ float code8_f32(uint32_t word, int j)
{
    return __uint_as_float(((word >> (8 * j)) & 0xFFu) | 0x4B000000u) - 8388608.0f;
}

__device__ __forceinline__ float chunk_code_dot8(uint4 q, uint4 q2, const float *v)
{
    const uint32_t w[8] = {q.x, q.y, q.z, q.w, q2.x, q2.y, q2.z, q2.w};
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float4 v0 = *reinterpret_cast<const float4 *>(v + 4 * m);
        acc = fmaf(code8_f32(w[m], 0), v0.x, acc);
        acc = fmaf(code8_f32(w[m], 1), v0.y, acc);
        acc = fmaf(code8_f32(w[m], 2), v0.z, acc);
        acc = fmaf(code8_f32(w[m], 3), v0.w, acc);
    }
    return acc;
}

// The code dot of chunk ch of a row whose words start at q (BITS-bit codes).
template <int BITS>
__device__ __forceinline__ float row_chunk_dot(const uint4 *q, int ch, const float *v)
{
    if (BITS == 8)
        return chunk_code_dot8(__ldg(q + 2 * ch), __ldg(q + 2 * ch + 1), v);
    return chunk_code_dot(__ldg(q + ch), v);
}

// Gate/up + SwiGLU, one warp per output row o of active expert i of token t:
//   a[t, i, o] = silu(g) * u,  g = W_g[o] . x[t],  u = W_u[o] . x[t].
// grid: (ceil(Imax / 8), n_act, T); 256 threads.
template <typename TA, typename TS, int BITS>
__global__ void __launch_bounds__(256) gateup_kernel(const TA *__restrict__ x, int H, int G, int k,
                                                     int n_act, int I, int Is,
                                                     const int32_t *__restrict__ topk_idx,
                                                     ExpertSrc src, float *__restrict__ a, int Imax)
{
    extern __shared__ __align__(16) float sm[];
    float *xs = sm;                      // padded [H]
    float *xsum = sm + padded(H);        // [H / 32]
    const int t = blockIdx.z, i = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int inter = (i == k) ? Is : I;
    if (blockIdx.x * 8 >= inter)
        return;
    for (int c = threadIdx.x; c < H; c += blockDim.x)
        xs[padded(c)] = to_f32(x[(size_t)t * H + c]);
    __syncthreads();
    const int nch = H >> 5;
    for (int ch = threadIdx.x; ch < nch; ch += blockDim.x) {
        const float *p = xs + ch * 36;
        float s = 0.f;
        for (int j = 0; j < 32; ++j)
            s += p[j];
        xsum[ch] = s;
    }
    __syncthreads();
    const int o = blockIdx.x * 8 + warp;
    if (o >= inter)
        return;
    const char *p[9];
    float *dst = a + ((size_t)t * n_act + i) * Imax + o;
    if (!expert_arrays(src, topk_idx, k, t, i, p)) {
        if (lane == 0)
            *dst = 0.f;
        return;
    }
    const int wpr = H * BITS / 32, gpr = H / G;
    const uint4 *qg = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint32_t *>(p[M_QG]) + (size_t)o * wpr);
    const uint4 *qu = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint32_t *>(p[M_QU]) + (size_t)o * wpr);
    const TS *sg = reinterpret_cast<const TS *>(p[M_SG]) + (size_t)o * gpr;
    const TS *bg = reinterpret_cast<const TS *>(p[M_BG]) + (size_t)o * gpr;
    const TS *su = reinterpret_cast<const TS *>(p[M_SU]) + (size_t)o * gpr;
    const TS *bu = reinterpret_cast<const TS *>(p[M_BU]) + (size_t)o * gpr;
    float gacc = 0.f, uacc = 0.f;
    for (int ch = lane; ch < nch; ch += 32) {
        const int grp = (ch * 32) / G;
        const float *v = xs + ch * 36;
        const float dg = row_chunk_dot<BITS>(qg, ch, v);
        const float du = row_chunk_dot<BITS>(qu, ch, v);
        const float xsm = xsum[ch];
        gacc += to_f32(sg[grp]) * dg + to_f32(bg[grp]) * xsm;
        uacc += to_f32(su[grp]) * du + to_f32(bu[grp]) * xsm;
    }
    const float g = warp_sum(gacc);
    const float u = warp_sum(uacc);
    if (lane == 0)
        *dst = g * sigmoid_f(g) * u;
}

template <typename TS, int BITS>
static cudaError_t gateup_dispatch(const Shape &s, const void *x, int T, int k_eff, int n_act,
                                   const int32_t *idx, const ExpertSrc &src, float *a, int Imax,
                                   cudaStream_t st)
{
    dim3 grid((Imax + 7) / 8, n_act, T);
    size_t smem = (size_t)(s.H + s.H / 8 + s.H / 32) * sizeof(float);
    if (s.act == MOE_BF16) {
        auto kern = gateup_kernel<__nv_bfloat16, TS, BITS>;
        static int cur_smem = 0;
        cudaError_t e = ensure_smem(kern, smem, &cur_smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, 256, smem, st>>>((const __nv_bfloat16 *)x, s.H, s.G, k_eff, n_act, s.I, s.Is, idx, src, a, Imax);
    } else {
        auto kern = gateup_kernel<float, TS, BITS>;
        static int cur_smem = 0;
        cudaError_t e = ensure_smem(kern, smem, &cur_smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, 256, smem, st>>>((const float *)x, s.H, s.G, k_eff, n_act, s.I, s.Is, idx, src, a, Imax);
    }
    return cudaGetLastError();
}

cudaError_t launch_gateup(const Shape &s, const void *x, int T, int k_eff, int n_act,
                          const int32_t *topk_idx, const ExpertSrc &src, float *a, int Imax,
                          cudaStream_t st)
{
    if (s.bits == 8)
        return s.qscale == MOE_F16 ? gateup_dispatch<__half, 8>(s, x, T, k_eff, n_act, topk_idx, src, a, Imax, st)
                                   : gateup_dispatch<float, 8>(s, x, T, k_eff, n_act, topk_idx, src, a, Imax, st);
    if (s.qscale == MOE_F16)
        return gateup_dispatch<__half, 4>(s, x, T, k_eff, n_act, topk_idx, src, a, Imax, st);
    return gateup_dispatch<float, 4>(s, x, T, k_eff, n_act, topk_idx, src, a, Imax, st);
}

// Down projection + weighted combine.  A warp owns two output rows; each
// half-warp computes W_d,i[h] . a[t, i] for one row, active experts taken in
// order i = 0..n_act-1 (routed by rank, then shared), and the half's lane 0
// accumulates weight_i * dot_i in that fixed order:
//   y[t, h] = sum_{r<k} w[t,r] dot_r + sigmoid(gate_logit[t]) dot_shared.
// topk_w == NULL means weight 1; gate_logit == NULL means shared weight 1.
// grid: (H / 16, T); 256 threads.
template <typename TA, typename TS, int BITS>
__global__ void __launch_bounds__(256) down_kernel(const float *__restrict__ a, int H, int G, int k,
                                                   int n_act, int I, int Is, int Imax,
                                                   const int32_t *__restrict__ topk_idx,
                                                   const float *__restrict__ topk_w,
                                                   const float *__restrict__ gate_logit,
                                                   ExpertSrc src, TA *__restrict__ y,
                                                   float *__restrict__ y32)
{
    extern __shared__ __align__(16) float sm[];
    const int t = blockIdx.y;
    const int pI = padded(Imax);
    const char **bases = reinterpret_cast<const char **>(sm);   // [n_act][9] addresses
    float *as = sm + ((n_act * 9 * 2 + 3) & ~3);                 // [n_act][padded Imax]
    float *asum = as + (size_t)n_act * pI;                       // [n_act][Imax / 32]
    for (int j = threadIdx.x; j < n_act * Imax; j += blockDim.x) {
        const int i = j / Imax, c = j - i * Imax;
        as[i * pI + padded(c)] = a[((size_t)t * n_act + i) * Imax + c];
    }
    if (threadIdx.x < n_act) {
        const char *p[9];
        const bool ok = expert_arrays(src, topk_idx, k, t, threadIdx.x, p);
#pragma unroll
        for (int m = 0; m < 9; ++m)
            bases[threadIdx.x * 9 + m] = ok ? p[m] : nullptr;
    }
    __syncthreads();
    const int nchm = Imax >> 5;
    for (int j = threadIdx.x; j < n_act * nchm; j += blockDim.x) {
        const int i = j / nchm, ch = j - i * nchm;
        const float *p = as + i * pI + ch * 36;
        float s = 0.f;
        for (int q = 0; q < 32; ++q)
            s += p[q];
        asum[i * nchm + ch] = s;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, l16 = lane & 15;
    const int h = blockIdx.x * 16 + warp * 2 + half;
    float acc = 0.f;
    for (int i = 0; i < n_act; ++i) {
        const int inter = (i == k) ? Is : I;
        const char *const *p = bases + i * 9;
        float dot = 0.f;
        if (p[M_QD] != nullptr && h < H) {
            const int wpr = inter * BITS / 32, gpr = inter / G, nch = inter >> 5;
            const uint4 *qd = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint32_t *>(p[M_QD]) + (size_t)h * wpr);
            const TS *sd = reinterpret_cast<const TS *>(p[M_SD]) + (size_t)h * gpr;
            const TS *bd = reinterpret_cast<const TS *>(p[M_BD]) + (size_t)h * gpr;
            for (int ch = l16; ch < nch; ch += 16) {
                const int grp = (ch * 32) / G;
                const float d = row_chunk_dot<BITS>(qd, ch, as + i * pI + ch * 36);
                dot += to_f32(sd[grp]) * d + to_f32(bd[grp]) * asum[i * nchm + ch];
            }
        }
        dot = half_warp_sum(dot);
        float wi;
        if (i < k)
            wi = topk_w ? topk_w[(size_t)t * k + i] : 1.f;
        else
            wi = gate_logit ? sigmoid_f(gate_logit[t]) : 1.f;
        acc = fmaf(wi, dot, acc);
    }
    if (l16 == 0 && h < H) {
        y[(size_t)t * H + h] = from_f32<TA>(acc);
        if (y32)
            y32[(size_t)t * H + h] = acc;
    }
}

template <typename TS, int BITS>
static cudaError_t down_dispatch(const Shape &s, const float *a, int T, int k_eff, int n_act,
                                 int Imax, const int32_t *idx, const float *w, const float *gl,
                                 const ExpertSrc &src, void *y, float *y32, cudaStream_t st)
{
    dim3 grid((s.H + 15) / 16, T);
    size_t smem = (size_t)(((n_act * 9 * 2 + 3) & ~3) + n_act * (padded(Imax) + Imax / 32)) * sizeof(float);
    if (s.act == MOE_BF16) {
        auto kern = down_kernel<__nv_bfloat16, TS, BITS>;
        static int cur_smem = 0;
        cudaError_t e = ensure_smem(kern, smem, &cur_smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, 256, smem, st>>>(a, s.H, s.G, k_eff, n_act, s.I, s.Is, Imax, idx, w, gl, src,
                                      (__nv_bfloat16 *)y, y32);
    } else {
        auto kern = down_kernel<float, TS, BITS>;
        static int cur_smem = 0;
        cudaError_t e = ensure_smem(kern, smem, &cur_smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, 256, smem, st>>>(a, s.H, s.G, k_eff, n_act, s.I, s.Is, Imax, idx, w, gl, src,
                                      (float *)y, y32);
    }
    return cudaGetLastError();
}

cudaError_t launch_down(const Shape &s, const float *a, int T, int k_eff, int n_act, int Imax,
                        const int32_t *topk_idx, const float *topk_w, const float *gate_logit,
                        const ExpertSrc &src, void *y, float *y32, cudaStream_t st)
{
    if (s.bits == 8)
        return s.qscale == MOE_F16
                   ? down_dispatch<__half, 8>(s, a, T, k_eff, n_act, Imax, topk_idx, topk_w, gate_logit, src, y, y32, st)
                   : down_dispatch<float, 8>(s, a, T, k_eff, n_act, Imax, topk_idx, topk_w, gate_logit, src, y, y32, st);
    if (s.qscale == MOE_F16)
        return down_dispatch<__half, 4>(s, a, T, k_eff, n_act, Imax, topk_idx, topk_w, gate_logit, src, y, y32, st);
    return down_dispatch<float, 4>(s, a, T, k_eff, n_act, Imax, topk_idx, topk_w, gate_logit, src, y, y32, st);
}

} // namespace moe
