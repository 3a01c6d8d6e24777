// Router logits of many tokens as one dense GEMM on the tensor cores.
//
// For T tokens the router is logits[T, E] = x[T, H] . w_router[E, H]^T, a
// plain bf16 GEMM (8.6 GFLOP for a 4096-token 80B prefill), so it goes to
// cuBLAS with fp32 accumulation; one small kernel then adds the router bias
// and computes the shared-gate logit w_sg . x[t] (a GEMV per token).  Calls
// made inside moe_layer_forward_noalloc keep the hand-written router kernel,
// since a cuBLAS handle allocates device memory when it is created.
#include <cublas_v2.h>
#include <mutex>

#include "internal.h"

namespace moe {

static thread_local int t_no_alloc_depth = 0;
NoAllocScope::NoAllocScope() { ++t_no_alloc_depth; }
NoAllocScope::~NoAllocScope() { --t_no_alloc_depth; }
bool in_no_alloc_scope() { return t_no_alloc_depth > 0; }

namespace rgemm {

constexpr int kBlasDevices = 64;
std::mutex g_blas_mu;
cublasHandle_t g_blas[kBlasDevices] = {nullptr};

// One warp per token: logits[t, :] += bias; sg[t] = w_sg . x[t].
__global__ void __launch_bounds__(128) router_tail_kernel(const __nv_bfloat16 *__restrict__ x, int T, int H, int E,
                                                          const float *__restrict__ bias,
                                                          const __nv_bfloat16 *__restrict__ wsg,
                                                          float *__restrict__ logits, float *__restrict__ sg)
{
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (t >= T)
        return;
    if (bias) {
        float *row = logits + (size_t)t * E;
        for (int e = lane; e < E; e += 32)
            row[e] += bias[e];
    }
    if (wsg) {
        const __nv_bfloat16 *xr = x + (size_t)t * H;
        float acc = 0.f;
        for (int c = lane * 8; c < H; c += 256) {
            float a[8], b[8];
            load8_f32(xr + c, a);
            load8_f32(wsg + c, b);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                acc = fmaf(a[j], b[j], acc);
        }
        acc = warp_sum(acc);
        if (lane == 0)
            sg[t] = acc;
    }
}

} // namespace rgemm

bool router_gemm_eligible(const Shape &s, int T)
{
    return T >= kRouterGemmMinTokens && s.act == MOE_BF16 && s.router == MOE_BF16 && s.H % 8 == 0 &&
           kernel_path() == 0 && !in_no_alloc_scope();
}

cudaError_t launch_router_gemm(const Shape &s, const void *x, int T, const void *w_router, const float *bias,
                               const void *w_sg, float *logits, float *sg_logit, cudaStream_t st)
{
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return ce;
    if (dev < 0 || dev >= rgemm::kBlasDevices)
        return cudaErrorInvalidDevice;
    {
        using namespace rgemm;
        std::lock_guard<std::mutex> g(g_blas_mu);
        if (!g_blas[dev] && cublasCreate(&g_blas[dev]) != CUBLAS_STATUS_SUCCESS) {
            g_blas[dev] = nullptr;
            return cudaErrorUnknown;
        }
        cublasHandle_t h = g_blas[dev];
        // column-major view: logits^T [E, T] (ld E) = w_router [E, H] x^T [H, T]
        const float one = 1.f, zero = 0.f;
        if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS ||
            cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, s.E, T, s.H, &one, w_router, CUDA_R_16BF, s.H, x,
                         CUDA_R_16BF, s.H, &zero, logits, CUDA_R_32F, s.E, CUBLAS_COMPUTE_32F,
                         CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
            return cudaErrorUnknown;
    }
    if (bias || w_sg) {
        const int threads = 128, per = threads / 32;
        rgemm::router_tail_kernel<<<(T + per - 1) / per, threads, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(x), T, s.H, s.E, bias, static_cast<const __nv_bfloat16 *>(w_sg),
            logits, sg_logit);
    }
    return cudaGetLastError();
}

} // namespace moe
