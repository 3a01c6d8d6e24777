// Single translation unit of libmoe_int4.so: the per-device error word is one
// __device__ variable shared by every kernel, so all sources compile together.
#include "api.cu"
#include "kernels_decode.cu"
#include "kernels_token.cu"
#include "prefill.cu"
#include "router_gemm.cu" // uses prefill.cu's TMA / TMEM helpers
#include "bucket.cu"
#include "slot_pool.cu"
#include "noalloc.cu"
