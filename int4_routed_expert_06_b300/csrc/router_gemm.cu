// Router logits of many tokens as one dense GEMM on the tensor cores.
//
// For T tokens the router is logits[T, E] = x[T, H] . w_router[E, H]^T + b,
// together with the shared-gate logit sg[T] = x[T, H] . w_sg[H]: one bf16 GEMM
// against E + 1 weight rows (8.6 GFLOP for a 4096-token 80B prefill), fp32
// accumulation.  CTA tile 128 tokens x 128 weight rows, K steps of 32, staged
// in shared memory by cp.async (two stages, rows padded to 40 elements so
// that every ldmatrix phase is free of bank conflicts), 8 warps of 64 x 32 each
// on mma.sync m16n8k16.  The epilogue adds the bias and writes weight row E to
// sg.
#include "internal.h"

namespace moe {
namespace rgemm {

constexpr int BM = 128, BN = 128, BK = 32, LDS = BK + 8; // smem row: 40 bf16 = 80 B
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 16-byte copy global -> shared, zero-filled when `valid` is false.
__device__ __forceinline__ void cp16z(void *dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr(dst)), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(saddr(p)));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Weight row n of the router-plus-shared-gate matrix (E rows, then w_sg).
__device__ __forceinline__ const __nv_bfloat16 *wrow(const __nv_bfloat16 *wr, const __nv_bfloat16 *wsg, int n,
                                                     int E, int H)
{
    return n < E ? wr + (size_t)n * H : wsg;
}

__global__ void __launch_bounds__(kThreads) router_gemm_kernel(const __nv_bfloat16 *__restrict__ x, int T, int H,
                                                               int E, const __nv_bfloat16 *__restrict__ wr,
                                                               const __nv_bfloat16 *__restrict__ wsg,
                                                               const float *__restrict__ bias,
                                                               float *__restrict__ logits, float *__restrict__ sg)
{
    __shared__ __align__(128) __nv_bfloat16 As[2][BM][LDS];
    __shared__ __align__(128) __nv_bfloat16 Bs[2][BN][LDS];
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int N = E + (wsg ? 1 : 0);
    const int wm = (warp >> 2) * 64, wn = (warp & 3) * 32; // warp tile origin in the CTA tile

    // stage K step kk into buffer b: 128 rows x 4 pieces of 16 B, for A and B
    auto stage = [&](int b, int kk) {
        for (int p = t; p < BM * 4; p += kThreads) {
            const int r = p >> 2, c = (p & 3) * 8;
            const int m = m0 + r, n = n0 + r;
            cp16z(&As[b][r][c], x + (size_t)min(m, T - 1) * H + kk + c, m < T);
            cp16z(&Bs[b][r][c], wrow(wr, wsg, min(n, N - 1), E, H) + kk + c, n < N);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    float acc[4][4][4] = {}; // [m16 tile][n8 tile][fragment]
    const int nk = H / BK;
    stage(0, 0);
    for (int ks = 0; ks < nk; ++ks) {
        const int b = ks & 1;
        if (ks + 1 < nk)
            stage(b ^ 1, (ks + 1) * BK);
        else
            asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();
#pragma unroll
        for (int k16 = 0; k16 < BK; k16 += 16) {
            uint32_t a[4][4], bf[2][4];
            const int q = lane >> 3, rr = lane & 7;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                ldsm_x4(&As[b][wm + 16 * i + rr + 8 * (q & 1)][k16 + 8 * (q >> 1)], a[i][0], a[i][1], a[i][2],
                        a[i][3]);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) // n8 tiles 2 jj and 2 jj + 1
                ldsm_x4(&Bs[b][wn + 16 * jj + rr + 8 * (q >> 1)][k16 + 8 * (q & 1)], bf[jj][0], bf[jj][1],
                        bf[jj][2], bf[jj][3]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16(acc[i][j], a[i], bf[j >> 1][2 * (j & 1)], bf[j >> 1][2 * (j & 1) + 1]);
        }
        __syncthreads(); // buffer b is restaged by the next iteration's copies
    }

    // epilogue: fragment c0, c1 = (row g, cols 2u, 2u + 1), c2, c3 = row g + 8
    const int g = lane >> 2, u = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = m0 + wm + 16 * i + g + 8 * h;
                if (m >= T)
                    continue;
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int n = n0 + wn + 8 * j + 2 * u + v;
                    const float val = acc[i][j][2 * h + v];
                    if (n < E)
                        logits[(size_t)m * E + n] = val + (bias ? bias[n] : 0.f);
                    else if (n == E && wsg)
                        sg[m] = val;
                }
            }
}

} // namespace rgemm

bool router_gemm_eligible(const Shape &s, int T)
{
    return T >= kRouterGemmMinTokens && s.act == MOE_BF16 && s.router == MOE_BF16 && s.H % rgemm::BK == 0 &&
           kernel_path() != 1;
}

cudaError_t launch_router_gemm(const Shape &s, const void *x, int T, const void *w_router, const float *bias,
                               const void *w_sg, float *logits, float *sg_logit, cudaStream_t st)
{
    const int N = s.E + (w_sg ? 1 : 0);
    const dim3 grid((T + rgemm::BM - 1) / rgemm::BM, (N + rgemm::BN - 1) / rgemm::BN);
    rgemm::router_gemm_kernel<<<grid, rgemm::kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(x), T, s.H, s.E, static_cast<const __nv_bfloat16 *>(w_router),
        static_cast<const __nv_bfloat16 *>(w_sg), bias, logits, sg_logit);
    return cudaGetLastError();
}

} // namespace moe
