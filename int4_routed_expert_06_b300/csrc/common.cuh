// Device helpers shared by the kernels of the routed int4 MoE layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_int4.h"

namespace moe {

// Per-device error word: the first fault a kernel records wins; the host
// reads and clears it with moe_get_device_error().  The library is a single
// translation unit, so this is its only definition.
__device__ int g_device_error = 0;

__device__ __forceinline__ void record_error(int code)
{
    atomicCAS(&g_device_error, 0, code);
}

// ------------------------------------------------------------ conversions

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// 8 consecutive elements -> fp32 (16-byte vector loads for bf16, two for f32).
__device__ __forceinline__ void load8_f32(const __nv_bfloat16 *p, float *out)
{
    uint4 v = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        out[2 * j] = __uint_as_float(w[j] << 16);
        out[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void load8_f32(const float *p, float *out)
{
    float4 a = *reinterpret_cast<const float4 *>(p);
    float4 b = *reinterpret_cast<const float4 *>(p + 4);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}

// 4-bit code -> exact fp32 via the exponent-bias method (OR the code into the
// mantissa of 2^23, then subtract 2^23).
__device__ __forceinline__ float code_f32(uint32_t word, int j)
{
    return __uint_as_float(((word >> (4 * j)) & 0xFu) | 0x4B000000u) - 8388608.0f;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Sum over aligned groups of 16 lanes.
__device__ __forceinline__ float half_warp_sum(float v)
{
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + __expf(-v)); }

// Raise a kernel's dynamic shared-memory limit to at least `bytes`, calling
// the runtime only when the limit grows (so that repeated launches, including
// those made during stream capture, do not touch function attributes).  The
// limit is raised even below 48 KB: the default covers static plus dynamic
// shared memory, so a kernel with static arrays needs it sooner.
template <typename F>
static cudaError_t ensure_smem(F *kern, size_t bytes, int *cur)
{
    if ((int)bytes <= *cur)
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess)
        *cur = (int)bytes;
    return e;
}

// ------------------------------------------------------------ expert lookup

// Where the nine arrays of each active expert live.  Active index i < k is
// the routed expert topk_idx[t, i]; i == k is the shared expert.  In
// explicit mode the single active expert is given by `ptr`.
struct ExpertSrc {
    const char *pool;
    size_t stride;
    const int32_t *table;
    int32_t n_slots;
    int32_t n_experts;
    const char *shared;
    size_t off[9];      // routed blob offsets
    size_t off_sh[9];   // shared blob offsets
    const void *ptr[9]; // explicit single expert
    int explicit_mode;
};

enum { M_QG = 0, M_QU, M_QD, M_SG, M_BG, M_SU, M_BU, M_SD, M_BD };

// The nine array addresses of active expert i of token t.  Returns false
// (and records MOE_ERR_NOT_RESIDENT or MOE_ERR_DEVICE_FAULT) if a routed
// expert has no valid slot.
__device__ __forceinline__ bool expert_arrays(const ExpertSrc &src, const int32_t *topk_idx,
                                              int k, int t, int i, const char *p[9])
{
    if (src.explicit_mode) {
#pragma unroll
        for (int m = 0; m < 9; ++m)
            p[m] = static_cast<const char *>(src.ptr[m]);
        return true;
    }
    const char *base;
    const size_t *off;
    if (i == k) {
        base = src.shared;
        off = src.off_sh;
    } else {
        int e = topk_idx[t * k + i];
        if (e < 0 || e >= src.n_experts) {
            record_error(MOE_ERR_DEVICE_FAULT);
            return false;
        }
        int slot = src.table[e];
        if (slot < 0 || slot >= src.n_slots) {
            record_error(MOE_ERR_NOT_RESIDENT);
            return false;
        }
        base = src.pool + (size_t)slot * src.stride;
        off = src.off;
    }
#pragma unroll
    for (int m = 0; m < 9; ++m)
        p[m] = base + off[m];
    return true;
}

} // namespace moe
