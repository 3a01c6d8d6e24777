// Allocation-free variant of moe_layer_forward.
//
// Some callers cannot allocate device memory at the point where they run the
// layer: an engine plugin whose host owns every byte of device memory and
// hands out none, code on a latency-critical path that must not take
// cudaMalloc's implicit device-wide synchronisation, or a caller with no
// allocator of its own.  moe_layer_forward_noalloc serves them: its scratch
// is a fixed array in this library's device image instead of a
// caller-provided workspace.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  Its device address is looked up
// once per device (cudaGetSymbolAddress, with that device current) on the
// first call made on that device; the host-side name of the array is only a
// stand-in and is never handed to a kernel.  Every call on a device shares the
// one array: calls whose GPU work overlaps (different streams, no ordering
// between them) race on it.  The layer's kernels need no part of their
// scratch to start at zero, so nothing is cleared between calls.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20; // 4 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};

} // namespace

extern "C" moe_status moe_layer_forward_noalloc(const moe_config *cfg, const moe_layer *layer, const void *x,
                                                int32_t T, void *y, float *y_f32, int32_t *topk_idx_out,
                                                float *topk_w_out, cudaStream_t stream)
{
    using namespace moe;
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (T < 0)
        return fail(MOE_ERR_INVALID_ARG, "moe_layer_forward_noalloc: T %d out of range", T);
    const size_t need = moe_layer_workspace_bytes(cfg, T);
    if (need > kNoAllocScratchBytes)
        return fail(MOE_ERR_OOM,
                    "moe_layer_forward_noalloc: T=%d needs %zu bytes of scratch; the built-in scratch holds %zu "
                    "bytes (use moe_layer_forward with a caller workspace for larger T)",
                    T, need, kNoAllocScratchBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_check(e, "moe_layer_forward_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(MOE_ERR_UNSUPPORTED, "moe_layer_forward_noalloc: device %d beyond %d", dev, kMaxDevices);
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> g(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess)
                return cuda_check(e, "moe_layer_forward_noalloc: cudaGetSymbolAddress");
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    return moe_layer_forward(cfg, layer, x, T, y, y_f32, topk_idx_out, topk_w_out, scratch, kNoAllocScratchBytes,
                             stream);
}
