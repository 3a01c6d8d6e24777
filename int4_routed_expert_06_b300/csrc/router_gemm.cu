// Router logits of many tokens as one dense GEMM on the 5th-generation tensor
// cores.
//
// For T tokens the router is logits[T, E] = x[T, H] . w_router[E, H]^T + b
// (8.6 GFLOP for a 4096-token 80B prefill), bf16 operands, fp32 accumulation
// in TMEM.  CTA tile: 128 tokens x 128 router rows; K in 64-column steps (one
// 128-byte swizzle atom of bf16), both operands brought in by TMA into a
// 4-stage ring; one elected lane of the MMA warp issues tcgen05.mma (M = 128,
// N = 128, K = 16) and commits each stage back to the producer; after the
// last stage the four warps read the accumulator out of TMEM, add the bias
// and write the logits.  The shared-gate logit sg[T] = x[T, H] . w_sg[H] is a warp-per-token
// GEMV beside it.  (This file is included after prefill.cu in the library's
// single translation unit and uses its TMA, mbarrier and TMEM helpers.)
#include "internal.h"

namespace moe {
namespace rgemm {

constexpr int TBM = 128, TBN = 128, TBK = 64, TST = 4;
constexpr int kThreads = 128;
constexpr uint32_t kTileA = TBM * TBK * 2; // 16 KB
constexpr uint32_t kTileB = TBN * TBK * 2; // 16 KB
constexpr uint32_t kSmem = TST * (kTileA + kTileB) + 1024;

// D (TMEM) += A . B, both K-major in shared memory (128-byte swizzle), issued
// by the elected lane of a converged warp.
__device__ __forceinline__ void mma_ss_elect(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw, int T, int E,
                     int K, const float *__restrict__ bias, float *__restrict__ logits)
{
    using namespace prefill;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint64_t full[TST], empty[TST], done;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int s_fail;
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    unsigned char *a_tiles = smem, *b_tiles = smem + TST * kTileA;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * TBM, n0 = blockIdx.y * TBN, nk = K / TBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TST; ++s) {
            bar_init(&full[s], 1);
            bar_init(&empty[s], 1);
        }
        bar_init(&done, 1);
        s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_u32(&tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: x rows [m0, m0 + 128) and router rows [n0, n0 + 128)
        // (rows past T or E read as zero)
        for (int k = 0; k < nk; ++k) {
            const int s = k % TST;
            if (!bar_wait(&empty[s], ((k / TST) & 1) ^ 1)) {
                s_fail = 1;
                break;
            }
            bar_expect(&full[s], kTileA + kTileB);
            tma_load_2d(a_tiles + s * kTileA, &mx, k * TBK, m0, &full[s]);
            tma_load_2d(b_tiles + s * kTileB, &mw, k * TBK, n0, &full[s]);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: the whole warp runs the loop (operands warp-uniform),
        // one elected lane issues; descriptors formed once, then offset
        const uint32_t idesc = idesc_bf16(TBM, TBN);
        const uint64_t ad0 = sw128_desc(smem_u32(a_tiles)), bd0 = sw128_desc(smem_u32(b_tiles));
        for (int k = 0; k < nk; ++k) {
            const int s = k % TST;
            if (!__all_sync(0xFFFFFFFFu, bar_wait(&full[s], (k / TST) & 1))) {
                s_fail = 1;
                break;
            }
            tc_fence_after();
            const uint64_t ad = ad0 + (uint64_t)(s * (kTileA >> 4)), bd = bd0 + (uint64_t)(s * (kTileB >> 4));
#pragma unroll
            for (int kk = 0; kk < TBK / 16; ++kk)
                mma_ss_elect(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (k > 0 || kk > 0) ? 1u : 0u);
            mma_commit_elect(&empty[s]);
        }
        mma_commit_elect(&done);
    }
    __syncwarp();
    // ---- epilogue: warp w reads TMEM lanes 32 w .. + 31 (tokens), 128 columns
    const bool ok = __all_sync(0xFFFFFFFFu, bar_wait(&done, 0) && !s_fail); // tcgen05.ld is warp-collective
    tc_fence_after();
    const int m = m0 + warp * 32 + lane;
    const bool vec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0; // rows 16-byte aligned
    if (ok) {
        for (int c0 = 0; c0 < TBN; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
            if (m < T) {
                const int nb = n0 + c0;
                float *row = logits + (size_t)m * E;
                if (vec && nb + 16 <= E) { // four 16-byte stores
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        float4 o;
                        o.x = __uint_as_float(v[j]) + (bias ? bias[nb + j] : 0.f);
                        o.y = __uint_as_float(v[j + 1]) + (bias ? bias[nb + j + 1] : 0.f);
                        o.z = __uint_as_float(v[j + 2]) + (bias ? bias[nb + j + 2] : 0.f);
                        o.w = __uint_as_float(v[j + 3]) + (bias ? bias[nb + j + 3] : 0.f);
                        *reinterpret_cast<float4 *>(row + nb + j) = o;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (nb + j < E)
                            row[nb + j] = __uint_as_float(v[j]) + (bias ? bias[nb + j] : 0.f);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem) : "memory");
    }
}

// sg[t] = x[t] . w_sg, one warp a token, fp32 accumulation (H a multiple of 8).
__global__ void __launch_bounds__(256) shared_gate_kernel(const __nv_bfloat16 *__restrict__ x,
                                                          const __nv_bfloat16 *__restrict__ w, int T, int H,
                                                          float *__restrict__ sg)
{
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T)
        return;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * H), *wr = reinterpret_cast<const uint4 *>(w);
    float acc = 0.f;
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 a = __ldg(xr + c), b = __ldg(wr + c);
        const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc = fmaf(__uint_as_float(aa[j] << 16), __uint_as_float(bb[j] << 16), acc);
            acc = fmaf(__uint_as_float(aa[j] & 0xFFFF0000u), __uint_as_float(bb[j] & 0xFFFF0000u), acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0)
        sg[t] = acc;
}

// 2-D map over a row-major bf16 matrix [rows, cols]: boxes of `box_rows` rows
// x 64 columns, 128-byte swizzle.
static bool make_map_rows(CUtensorMap *m, const void *base, long rows, int cols, int box_rows)
{
    prefill::EncodeTiledFn fn = prefill::encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)TBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

} // namespace rgemm

bool router_gemm_eligible(const Shape &s, int T)
{
    return T >= kRouterGemmMinTokens && s.act == MOE_BF16 && s.router == MOE_BF16 && s.H % rgemm::TBK == 0 &&
           kernel_path() != 1 && prefill::encode_fn() != nullptr;
}

cudaError_t launch_router_gemm(const Shape &s, const void *x, int T, const void *w_router, const float *bias,
                               const void *w_sg, float *logits, float *sg_logit, cudaStream_t st)
{
    CUtensorMap mx, mw;
    if (!rgemm::make_map_rows(&mx, x, T, s.H, rgemm::TBM) || !rgemm::make_map_rows(&mw, w_router, s.E, s.H, rgemm::TBN))
        return cudaErrorInvalidValue;
    static int cur = 0;
    cudaError_t e = ensure_smem(rgemm::router_tc_kernel, rgemm::kSmem, &cur);
    if (e != cudaSuccess)
        return e;
    const dim3 grid((T + rgemm::TBM - 1) / rgemm::TBM, (s.E + rgemm::TBN - 1) / rgemm::TBN);
    rgemm::router_tc_kernel<<<grid, rgemm::kThreads, rgemm::kSmem, st>>>(mx, mw, T, s.E, s.H, bias, logits);
    if (w_sg && sg_logit)
        rgemm::shared_gate_kernel<<<(T + 7) / 8, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(x),
                                                               static_cast<const __nv_bfloat16 *>(w_sg), T, s.H,
                                                               sg_logit);
    return cudaGetLastError();
}

} // namespace moe
