// Many-token (prefill) path of the routed int4 MoE layer: the expert MLPs
// as grouped GEMMs on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA-fed operands).
//
//   route      router logits (tcgen05 router GEMM) and top-k per token
//   bucket     stable counting sort of the T*k (token, rank) pairs by expert
//   gather     X_sorted[p] = x[token of pair p]           (bf16 rows)
//   pairs      per sorted row: its routing weight, and the inverse permutation
//   plan       work units (expert, feature tile, token chunk), largest first
//   gemm gu    act[p, f] = silu(W_g x_p)_f * (W_u x_p)_f   (bf16)
//   gemm down  P[p, h]   = (W_d act_p)_h                   (fp32)
//   combine    y[t] = sum_r w_p P[p] over p = pair(t, r), + g_t P[shared row t],
//              each product rounded to fp32, summed in that fixed order
//
// The GEMMs run "swap-AB": the M = 128 side of each MMA is a tile of weight
// rows, dequantised from int4 by 16 warps straight into TMEM (tcgen05.st), the
// A operand of the MMA; the N side is the expert's tokens (rounded up to 16,
// at most 192 per unit), brought into shared memory by TMA with a 128-byte
// swizzle.  Skewed routing then costs at most 15 padded token columns per unit
// instead of a 128-row tile.  The shared expert is one more group, over all T
// tokens.
#include <cuda.h>
#include <mutex>

#include "internal.h"

namespace moe {
namespace prefill {

constexpr int kNch = 192;        // tokens per unit (MMA N <= 256)
constexpr int kAtomK = 64;       // K of one 128-byte swizzle atom of bf16
constexpr int kBK = 128;         // K per pipeline stage: two atoms, so that the per-stage
                                 // synchronisation is paid once per 128 K
constexpr int kSub = kBK / kAtomK;
constexpr int kStages = 2;       // A (dequantised, in TMEM) and B (token, in shared memory) stages
constexpr int kCStages = 3;      // staged code tiles (run ahead of the dequant)
constexpr int kCK = 256;         // K of one code stage: 128-byte row pieces (whole lines)
constexpr int kBoxRows = 32;     // TMA box: 32 rows x 64 bf16
// warps 0-15 dequant, 16 weight TMA, 17 token TMA, 18 MMA, 19-22 epilogue
constexpr int kDqWarps = 16, kCodeWarp = 16, kRowWarp = 17, kMmaWarp = 18;
constexpr int kThreads = 32 * 23;
constexpr uint32_t kACols = kBK / 2;           // TMEM columns of one A stage: 128 rows x kBK bf16
constexpr uint32_t kAccCols = kNch;            // TMEM columns of one fp32 accumulator
constexpr uint32_t kACol0 = 2 * kAccCols;      // the A stages follow the two accumulators
static_assert(kACol0 + kStages * kACols <= 512, "TMEM columns of one CTA");
constexpr uint32_t kBTile = kNch * kBK * 2;    // 32 KB: kSub atoms of [kNch rows][128 B]
constexpr uint32_t kCTile = 128 * (kCK / 2);   // 16 KB: 128 rows x 256 codes
constexpr uint32_t kSTile = 16 * 1024;         // a unit's scale and bias rows (at most 4 x 64 rows x 64 B)
constexpr uint32_t kPTile = 16 * 1024;         // the same as (scale, bias) pairs [group][128 rows] (<= 32 groups)
constexpr uint32_t kSmem = kStages * kBTile + kCStages * kCTile + kSTile + kPTile + 1024;
static_assert(kCK % kBK == 0, "a code stage holds whole pipeline stages");
static_assert(kSmem <= 232448, "dynamic shared memory of one CTA");
constexpr uint64_t kWaitNs = 500ull * 1000 * 1000; // 0.5 s bound on any single wait

struct Unit {
    int e;    // expert id, -1 = shared expert
    int ft;   // feature tile: gate/up 64 features (128 interleaved rows), down 128 output rows
    int j0;   // first row of the unit in the B source (sorted pair index, or token for the shared expert)
    int n;    // tokens (1..256)
    int slot; // pool slot of the expert (0 for the shared expert), -1 when not resident
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtime()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void bar_init(uint64_t *b, uint32_t n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void bar_expect(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool bar_try(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(b)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// The same test, but a thread whose phase has not completed is suspended
// until it completes or about `hint_ns` nanoseconds have passed, instead of
// returning at once: a waiting warp then takes no issue slots from the warps
// that share its scheduler.
__device__ __forceinline__ bool bar_try_suspend(uint64_t *b, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(b)), "r"(parity), "r"(hint_ns)
                 : "memory");
    return ok != 0;
}

constexpr uint32_t kSuspendNs = 20u * 1000; // one suspended test: well inside kWaitNs

// Wait until the phase of parity `parity` has completed, for at most kWaitNs.
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t parity)
{
    if (bar_try(b, parity))
        return true;
    const uint64_t t0 = gtime();
    for (;;) {
        if (bar_try_suspend(b, parity, kSuspendNs))
            return true;
        if (gtime() - t0 > kWaitNs) {
            record_error(MOE_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
                     smem_u32(dst)),
                 "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
                 : "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle,
// 8-row groups 1024 bytes apart (SBO), version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);          // start address
    d |= (uint64_t)1 << 16;                           // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 x bf16 -> fp32, both K-major.
__host__ __device__ __forceinline__ uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Store 16 columns of this warp's 32 TMEM lanes (one row a thread).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (TMEM) += A (TMEM: 128 lanes = rows, two bf16 of K a column) . B (shared
// memory descriptor), issued by one lane of a converged warp (and below, the
// commit of the MMAs issued so far): elect.sync picks the lowest active lane,
// so a warp that runs with all lanes always issues from lane 0, and a commit
// tracks the MMAs that lane issued.
__device__ __forceinline__ void mma_bf16_ta_elect(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
                 "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint64_t *bar)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------ small kernels

// X_sorted[p] = x[perm_tok[p]], rows of H bf16: a warp a row, its lanes over
// the row's 16-byte chunks (no index division).
__global__ void gather_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ perm_tok, int P,
                                   int row16, uint4 *__restrict__ xs)
{
    const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    for (int p = blockIdx.x * wpb + (threadIdx.x >> 5); p < P; p += gridDim.x * wpb) {
        const uint4 *src = x + (long)perm_tok[p] * row16;
        uint4 *dst = xs + (long)p * row16;
        for (int c = lane; c < row16; c += 32)
            dst[c] = __ldg(src + c);
    }
}

// Per sorted row: the routing weight (shared rows: sigmoid of the gate logit)
// and the inverse permutation inv[t*k + r] = sorted index of pair (t, r).
__global__ void pair_prep_kernel(const int32_t *__restrict__ perm_tok, const int32_t *__restrict__ perm_rank,
                                 const float *__restrict__ topk_w, const float *__restrict__ sg, int T, int k,
                                 float *__restrict__ wpair, int32_t *__restrict__ inv)
{
    const int P = T * k;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P + T; p += gridDim.x * blockDim.x) {
        if (p < P) {
            const int t = perm_tok[p], r = perm_rank[p];
            wpair[p] = topk_w[t * k + r];
            inv[t * k + r] = p;
        } else {
            wpair[p] = sg ? 1.f / (1.f + __expf(-sg[p - P])) : 1.f;
        }
    }
}

// Units of both GEMM kinds from one ranking.  Every CTA ranks the experts by
// token count (descending, ties by id: a bitonic sort of 64-bit keys in
// shared memory) and scans their token chunks of up to kNch tokens; CTA b then
// writes units b, b + grid, ... of each list: the shared expert's first, then
// the experts' in rank order, token chunk major and feature tile minor within
// an expert.  The unit count of a kind is n_ft x chunks, so one chunk scan
// serves both kinds.  E <= 1024.
constexpr int kPlanCtas = 16;

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *__restrict__ counts,
                                                    const int32_t *__restrict__ offsets,
                                                    const int32_t *__restrict__ table, int n_slots, int E, int T,
                                                    int n_ft0, int n_ft_sh0, int n_ft1, int n_ft_sh1, int has_shared,
                                                    Unit *__restrict__ units0, Unit *__restrict__ units1,
                                                    int32_t *__restrict__ n_units)
{
    __shared__ unsigned long long s_key[1024];
    __shared__ int s_ord[1024];  // expert at each rank position
    __shared__ int s_scan[1024]; // inclusive scan of token chunks by rank position
    __shared__ int s_slot[1024]; // slot of the expert at each rank position
    const int e = threadIdx.x;
    // ascending keys = (count descending, id ascending); past E: the largest key
    s_key[e] = e < E ? ((unsigned long long)(0x7FFFFFFF - counts[e]) << 32) | (unsigned)e : ~0ull;
    __syncthreads();
    for (int k = 2; k <= 1024; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int ixj = e ^ j;
            if (ixj > e) {
                const unsigned long long a = s_key[e], b = s_key[ixj];
                if ((a > b) == ((e & k) == 0)) {
                    s_key[e] = b;
                    s_key[ixj] = a;
                }
            }
            __syncthreads();
        }
    int ch = 0, ex = -1;
    if (e < E) {
        ex = (int)(s_key[e] & 0xFFFFFFFFu);
        ch = (counts[ex] + kNch - 1) / kNch;
        const int sl = table[ex];
        s_slot[e] = sl >= 0 && sl < n_slots ? sl : -1;
    }
    s_ord[e] = ex;
    s_scan[e] = ch;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) { // inclusive scan (Hillis-Steele)
        const int v = e >= o ? s_scan[e - o] : 0;
        __syncthreads();
        s_scan[e] += v;
        __syncthreads();
    }
    const int n_ch_sh = has_shared ? (T + kNch - 1) / kNch : 0, chunks = s_scan[1023];
    const int gt = blockIdx.x * blockDim.x + e, gs = gridDim.x * blockDim.x;
    for (int kind = 0; kind < 2; ++kind) {
        const int n_ft = kind ? n_ft1 : n_ft0, n_ft_sh = kind ? n_ft_sh1 : n_ft_sh0;
        Unit *units = kind ? units1 : units0;
        const int sh_units = n_ft_sh * n_ch_sh, total = sh_units + n_ft * chunks;
        for (int u = gt; u < total; u += gs) {
            if (u < sh_units) {
                const int c = u / n_ft_sh, ft = u - c * n_ft_sh;
                units[u] = {-1, ft, c * kNch, min(kNch, T - c * kNch), 0};
            } else {
                const int v = u - sh_units, q = v / n_ft, ft = v - q * n_ft; // global chunk q
                int lo = 0, hi = E - 1; // first rank position p with s_scan[p] > q
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (s_scan[mid] > q)
                        hi = mid;
                    else
                        lo = mid + 1;
                }
                const int p = lo, ex2 = s_ord[p], cnt = counts[ex2];
                const int c = q - (s_scan[p] - (cnt + kNch - 1) / kNch);
                units[u] = {ex2, ft, offsets[ex2] + c * kNch, min(kNch, cnt - c * kNch), s_slot[p]};
            }
        }
        if (blockIdx.x == 0 && e == 0)
            n_units[kind] = total;
    }
}

// y[t, h] = sum_r w[p] P[p, h] with p = inv[t, r], + w[T*k + t] P[T*k + t, h]:
// the routing weight of each pair (and the shared expert's gate) times its
// down-projection row, each product rounded to fp32 and summed in rank order;
// bf16 y and optional fp32, one output a thread (any alignment of y and y32).
__global__ void combine_scalar_kernel(const float *__restrict__ P, const float *__restrict__ wpair,
                                      const int32_t *__restrict__ inv, int T, int k, int H, int has_shared,
                                      __nv_bfloat16 *__restrict__ y, float *__restrict__ y32)
{
    const long n = (long)T * H;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int t = (int)(i / H), h = (int)(i - (long)t * H);
        float acc = 0.f;
        for (int r = 0; r < k; ++r) {
            const int p = inv[t * k + r];
            acc += __fmul_rn(__ldg(wpair + p), __ldg(P + (long)p * H + h));
        }
        if (has_shared) {
            const long p = (long)T * k + t;
            acc += __fmul_rn(__ldg(wpair + p), __ldg(P + p * H + h));
        }
        y[i] = __float2bfloat16_rn(acc);
        if (y32)
            y32[i] = acc;
    }
}

// The same sum in the same order, four consecutive h a thread (16-byte loads;
// H a multiple of 4, y 8-byte and y32 16-byte aligned).
__global__ void combine_kernel(const float *__restrict__ P, const float *__restrict__ wpair,
                               const int32_t *__restrict__ inv, int T, int k, int H, int has_shared,
                               __nv_bfloat16 *__restrict__ y, float *__restrict__ y32)
{
    const int H4 = H >> 2;
    const int n = T * H4; // T <= 65536 and H <= 32768: fits 32 bits
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int t = i / H4, h4 = i - t * H4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < k; ++r) {
            const int p = inv[t * k + r];
            const float w = __ldg(wpair + p);
            const float4 v = __ldg(reinterpret_cast<const float4 *>(P + (long)p * H) + h4);
            acc.x += __fmul_rn(w, v.x);
            acc.y += __fmul_rn(w, v.y);
            acc.z += __fmul_rn(w, v.z);
            acc.w += __fmul_rn(w, v.w);
        }
        if (has_shared) {
            const long p = (long)T * k + t;
            const float w = __ldg(wpair + p);
            const float4 v = __ldg(reinterpret_cast<const float4 *>(P + p * H) + h4);
            acc.x += __fmul_rn(w, v.x);
            acc.y += __fmul_rn(w, v.y);
            acc.z += __fmul_rn(w, v.z);
            acc.w += __fmul_rn(w, v.w);
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(y + (long)t * H)[h4] = packed;
        if (y32)
            reinterpret_cast<float4 *>(y32 + (long)t * H)[h4] = acc;
    }
}

// ------------------------------------------------------------ grouped GEMM

struct GemmArgs {
    const Unit *units;
    const int32_t *n_units;
    ExpertSrc src;
    int mode;            // 0 gate/up, 1 down
    int H, I, Is, G, T, k;
    int act_ld;          // row length of the activation buffer (max(I, Is))
    __nv_bfloat16 *act;  // gate/up output [T*k + T, act_ld]
    float *pout;         // down output [T*k + T, H], unweighted
};

// Tensor maps of the weight side of one GEMM kind, over the fixed-stride
// pool (3-D: bytes or scale groups of a row, rows, slot) and over the shared
// blob (slot extent 1).  Gate/up: codes of W_g, W_u (boxes of 64 rows x 128
// bytes = 256 K: whole 128-byte lines), and the scale and bias rows of W_g,
// W_u (64 rows x all groups).  Down: codes of W_d (128 rows x 128 bytes), its
// scale and bias rows (128 rows x all groups).
struct WMaps {
    CUtensorMap routed[6]; // gate/up: qg qu sg bg su bu; down: qd sd bd
    CUtensorMap shared[6];
};

// 32 codes of one weight row (four code words, one quantisation group) ->
// 32 bf16 w = s q + b (fp32 arithmetic, one rounding), packed two a word in K
// order: out[j] holds columns 2j, 2j + 1.
__device__ __forceinline__ void dequant_32(uint4 qw, float s, float b, uint32_t (&out)[16])
{
    const uint32_t w[4] = {qw.x, qw.y, qw.z, qw.w};
    const float s16 = 16.f * s, b16 = b - s16;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) { // one code word = 8 columns
        const uint32_t word = w[cc];
        const uint32_t lo = ((word << 3) & 0x78787878u) | 0x80808080u;
        const uint32_t hi = ((word >> 1) & 0x78787878u) | 0x80808080u;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
            const uint32_t sel = 0x7044u | (uint32_t)(bb << 8);
            const float f0 = __uint_as_float(__byte_perm(lo, 0x3F000000u, sel)); // 1 + q/16, column 2bb
            const float f1 = __uint_as_float(__byte_perm(hi, 0x3F000000u, sel)); // column 2bb + 1
            const float2 wv = __ffma2_rn(make_float2(f0, f1), make_float2(s16, s16), make_float2(b16, b16));
            __nv_bfloat162 h2 = __floats2bfloat162_rn(wv.x, wv.y);
            out[4 * cc + bb] = *reinterpret_cast<uint32_t *>(&h2);
        }
    }
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
                     smem_u32(dst)),
                 "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void dq_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kDqWarps * 32) : "memory"); }

// A unit's scale and bias of one weight row and group.
template <typename TS> struct SBPair {
    TS s, b;
};

template <typename TS>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_rows, const __grid_constant__ CUtensorMap tm_shared,
                        const __grid_constant__ WMaps wm, GemmArgs A)
{
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint64_t a_full[kStages], b_full[kStages], ab_empty[kStages];
    __shared__ uint64_t c_full[kCStages], c_empty[kCStages], s_full, s_empty;
    __shared__ uint64_t acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ volatile int s_abort;
    __shared__ volatile int s_dq_fail; // set only: a dequant wait gave up (read only after dq_sync)

    // 1024-byte aligned tiles, as an offset from the shared array, so that the
    // compiler keeps every access in the shared window (no generic accesses)
    const uint32_t raw_base = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw_base + 1023u) & ~1023u) - raw_base);
    unsigned char *b_tiles = smem;
    unsigned char *c_ring = b_tiles + kStages * kBTile;
    unsigned char *s_raw = c_ring + kCStages * kCTile;
    SBPair<TS> *s_pair = reinterpret_cast<SBPair<TS> *>(s_raw + kSTile); // [group][128 rows]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nu = *A.n_units;
    const int G = A.G, grid = gridDim.x;
    const uint32_t sb = sizeof(TS);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            bar_init(&a_full[s], kDqWarps);
            bar_init(&b_full[s], 1);
            bar_init(&ab_empty[s], 1);
        }
        for (int s = 0; s < kCStages; ++s) {
            bar_init(&c_full[s], 1);
            bar_init(&c_empty[s], kDqWarps);
        }
        bar_init(&s_full, 1);
        bar_init(&s_empty, 1);
        for (int b = 0; b < 2; ++b) {
            bar_init(&acc_full[b], 1);
            bar_init(&acc_empty[b], 128);
        }
        s_abort = 0;
        s_dq_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) { // TMEM: 2 accumulators x 256 fp32 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    auto kdim = [&](const Unit &u) { return A.mode == 0 ? A.H : (u.e < 0 ? A.Is : A.I); };
    // the unit descriptor after ui (this CTA's next), loaded a unit ahead
    auto next_unit = [&](int ui, const Unit &cur) { return ui + grid < nu ? A.units[ui + grid] : cur; };

    if (warp < kDqWarps) {
        // ---------------- dequant: warp w writes TMEM lanes 32 (w % 4) .. + 31
        // (one weight row a thread), K part w / 4 (32 K) of each stage, with
        // tcgen05.st into the stage's A columns.  The named barrier dq_sync
        // joins exactly these warps, so they leave the unit loop together: a
        // failed wait sets s_dq_fail, and the decision to stop is read after
        // the next dq_sync.
        const int t = threadIdx.x, qd = warp & 3, part = warp >> 2, r = qd * 32 + lane;
        const int gshift = (G & (G - 1)) == 0 ? __ffs(G) - 1 : -1; // group size a power of two: shift, not divide
        const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16) + kACol0 + (uint32_t)part * (kACols / 4);
        int cs = 0, as = 0;
        uint32_t cph = 0, aph = 0, sph = 0;
        Unit u = blockIdx.x < nu ? A.units[blockIdx.x] : Unit{};
        for (int ui = blockIdx.x; ui < nu; ui += grid) {
            const Unit nx = next_unit(ui, u);
            const int K = kdim(u), ng = K / G;
            const bool ok = u.slot >= 0;
            if (!ok && t == 0)
                record_error(MOE_ERR_NOT_RESIDENT);
            // the unit's scale rows -> (scale, bias) pairs [group][row]
            if (!bar_wait(&s_full, sph))
                s_dq_fail = 1;
            sph ^= 1;
            dq_sync(); // every dequant thread is done with the previous unit's pairs
            if (s_dq_fail) {
                s_abort = 1;
                break;
            }
            {
                const TS *raw = reinterpret_cast<const TS *>(s_raw);
                // a warp takes 32 rows of one pass j, row rr its group
                // (j + rot(rr)) mod ng: each row still visits every group once,
                // but the lanes' 2-byte reads of the row-major scale rows now
                // spread over the banks (at most 2-way conflicts for 8, 16 or
                // 32 groups; with one group a warp they were 4- to 16-way), and
                // the pair writes, one row a lane, stay conflict-free
                // (a thread's row rr = t mod 128 is the same on every pass)
                static_assert((kDqWarps * 32) % 128 == 0, "one row a thread across the passes");
                const int rot = ((t & 127) >> 1) + (((t & 127) >> 4) << 1), rot_ng = rot % ng;
                for (int e = t; e < 128 * ng; e += kDqWarps * 32) {
                    const int j = e >> 7, rr = e & 127;
                    const int g = j + rot_ng < ng ? j + rot_ng : j + rot_ng - ng;
                    int si, bi;
                    if (A.mode == 0) { // raw: sg, bg, su, bu, each [64 rows][ng]; rows interleave gate / up
                        const int m = rr & 1, f = rr >> 1;
                        si = (2 * m) * 64 * ng + f * ng + g;
                        bi = si + 64 * ng;
                    } else {           // raw: sd, bd, each [128 rows][ng]
                        si = rr * ng + g;
                        bi = si + 128 * ng;
                    }
                    s_pair[g * 128 + rr] = SBPair<TS>{raw[si], raw[bi]};
                }
            }
            dq_sync(); // the pairs are complete and the raw rows free
            if (t == 0)
                bar_arrive(&s_empty);
            // this row's code piece (kCK / 2 bytes, 16-byte chunks 128-byte
            // swizzled by the copy) in a code stage
            const int brow = A.mode == 0 ? (r >> 1) : r; // row within its box
            const int coff = (A.mode == 0 ? (r & 1) * (kCTile / 2) : 0) + brow * (kCK / 2);
            bool wfail = false; // warp-uniform
            for (int kc = 0; kc < K && !wfail; kc += kCK) {
                if (!__all_sync(0xFFFFFFFFu, bar_wait(&c_full[cs], cph))) {
                    s_dq_fail = 1;
                    s_abort = 1;
                    break;
                }
                const unsigned char *cp = c_ring + cs * kCTile + coff;
                for (int k0 = kc; k0 < min(K, kc + kCK); k0 += kBK) {
                    // warp-uniform, so that a give-up never splits the warp at __syncwarp
                    if (!__all_sync(0xFFFFFFFFu, bar_wait(&ab_empty[as], aph ^ 1))) {
                        s_dq_fail = 1;
                        s_abort = 1;
                        wfail = true;
                        break;
                    }
                    uint32_t packed[16];
                    if (ok) {
                        const int c16 = ((k0 - kc) >> 5) + part; // 16-byte chunk of the row piece
                        const uint4 qw = *reinterpret_cast<const uint4 *>(cp + ((c16 ^ (brow & 7)) << 4));
                        const int kp = k0 + 32 * part, gi = gshift >= 0 ? kp >> gshift : kp / G;
                        const SBPair<TS> p = s_pair[gi * 128 + r];
                        dequant_32(qw, to_f32(p.s), to_f32(p.b), packed);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            packed[j] = 0u;
                    }
                    tmem_st16(trow + (uint32_t)as * kACols, packed);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        bar_arrive(&a_full[as]);
                    if (++as == kStages) {
                        as = 0;
                        aph ^= 1;
                    }
                }
                __syncwarp();
                if (lane == 0)
                    bar_arrive(&c_empty[cs]);
                if (++cs == kCStages) {
                    cs = 0;
                    cph ^= 1;
                }
            }
            u = nx;
        }
    } else if (warp == kCodeWarp) {
        // ---------------- TMA producer of the weight side: a unit's scale rows
        // (issued as soon as the buffer is free, while the unit before is
        // still in flight), then its code stages
        if (lane == 0) {
            int cs = 0;
            uint32_t cph = 0, sph = 0;
            int sui = blockIdx.x; // next unit whose scale rows are to be loaded
            auto issue_scales = [&](const Unit &v) {
                const CUtensorMap *mp = v.e < 0 ? wm.shared : wm.routed;
                const int z = v.slot < 0 ? 0 : v.slot, ng = kdim(v) / G;
                if (A.mode == 0) {
                    const uint32_t part = 64u * (uint32_t)ng * sb;
                    bar_expect(&s_full, 4 * part);
                    for (int j = 0; j < 4; ++j) // sg bg su bu
                        tma_load_3d(s_raw + j * part, &mp[2 + j], 0, v.ft * 64, z, &s_full);
                } else {
                    const uint32_t part = 128u * (uint32_t)ng * sb;
                    bar_expect(&s_full, 2 * part);
                    for (int j = 0; j < 2; ++j) // sd bd
                        tma_load_3d(s_raw + j * part, &mp[1 + j], 0, v.ft * 128, z, &s_full);
                }
                sph ^= 1;
                sui += grid;
            };
            Unit u = blockIdx.x < nu ? A.units[blockIdx.x] : Unit{};
            for (int ui = blockIdx.x; ui < nu && !s_abort; ui += grid) {
                const Unit nx = next_unit(ui, u);
                if (sui == ui) { // this unit's scale rows: wait for the buffer
                    if (!bar_wait(&s_empty, sph ^ 1)) {
                        s_abort = 1;
                        break;
                    }
                    issue_scales(u);
                }
                const int K = kdim(u);
                const int z = u.slot < 0 ? 0 : u.slot;
                const CUtensorMap *mp = u.e < 0 ? wm.shared : wm.routed;
                for (int kc = 0; kc < K; kc += kCK) {
                    if (sui == ui + grid && sui < nu && bar_try(&s_empty, sph ^ 1))
                        issue_scales(nx);
                    if (!bar_wait(&c_empty[cs], cph ^ 1)) {
                        s_abort = 1;
                        break;
                    }
                    // a piece past the row end (K not a multiple of kCK) is
                    // zero-filled by the copy and never read
                    unsigned char *cd = c_ring + cs * kCTile;
                    bar_expect(&c_full[cs], kCTile);
                    if (A.mode == 0) {
                        tma_load_3d(cd, &mp[0], kc / 2, u.ft * 64, z, &c_full[cs]);
                        tma_load_3d(cd + kCTile / 2, &mp[1], kc / 2, u.ft * 64, z, &c_full[cs]);
                    } else {
                        tma_load_3d(cd, &mp[0], kc / 2, u.ft * 128, z, &c_full[cs]);
                    }
                    if (++cs == kCStages) {
                        cs = 0;
                        cph ^= 1;
                    }
                }
                u = nx;
            }
        }
    } else if (warp == kRowWarp) {
        // ---------------- TMA producer for the token operand
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            Unit u = blockIdx.x < nu ? A.units[blockIdx.x] : Unit{};
            for (int ui = blockIdx.x; ui < nu && !s_abort; ui += grid) {
                const Unit nx = next_unit(ui, u);
                const int K = kdim(u);
                const int nbox = (u.n + kBoxRows - 1) / kBoxRows;
                // rows: gate/up routed -> sorted x; gate/up shared -> x; down -> activations
                const CUtensorMap *map = (A.mode == 0 && u.e < 0) ? &tm_shared : &tm_rows;
                const int row0 = (A.mode == 1 && u.e < 0) ? A.T * A.k + u.j0 : u.j0;
                for (int k0 = 0; k0 < K; k0 += kBK) {
                    if (!bar_wait(&ab_empty[stage], ph ^ 1)) {
                        s_abort = 1;
                        break;
                    }
                    bar_expect(&b_full[stage], (uint32_t)(nbox * kSub) * kBoxRows * 128);
                    unsigned char *tile = b_tiles + stage * kBTile;
                    for (int j = 0; j < kSub; ++j)
                        for (int bx = 0; bx < nbox; ++bx)
                            tma_load_2d(tile + j * (kNch * 128) + bx * kBoxRows * 128, map, k0 + j * kAtomK,
                                        row0 + bx * kBoxRows, &b_full[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1;
                    }
                }
                u = nx;
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer
        // The whole warp runs the loop, so that every MMA operand is
        // warp-uniform, and one elected lane (the same one throughout)
        // issues each tcgen05.mma and commit.  The B descriptors are formed
        // once: a stage and a 16-column step only add a constant to the start
        // address field.
        int stage = 0, acc = 0;
        uint32_t ph = 0, acc_ph = 0;
        const uint64_t bdesc0 = sw128_desc(smem_u32(b_tiles));
        Unit u = blockIdx.x < nu ? A.units[blockIdx.x] : Unit{};
        for (int ui = blockIdx.x; ui < nu; ui += grid) {
            if (__any_sync(0xFFFFFFFFu, s_abort))
                break;
            const Unit nx = next_unit(ui, u);
            const int K = kdim(u);
            const int N = (u.n + 15) & ~15;
            const uint32_t idesc = idesc_bf16(128, N);
            const uint32_t d_tmem = tmem + (uint32_t)acc * kAccCols;
            if (!__all_sync(0xFFFFFFFFu, bar_wait(&acc_empty[acc], acc_ph ^ 1))) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            bool fail = false;
            for (int k0 = 0; k0 < K; k0 += kBK) {
                if (!__all_sync(0xFFFFFFFFu, bar_wait(&a_full[stage], ph) && bar_wait(&b_full[stage], ph))) {
                    s_abort = 1;
                    fail = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a_t = tmem + kACol0 + (uint32_t)stage * kACols;
                const uint64_t bd = bdesc0 + (uint64_t)(stage * (kBTile >> 4));
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) { // B atom kk / 4, 16-column step kk % 4 within it
                    const uint32_t bo = (uint32_t)(kk / 4) * (kNch * 128) + (uint32_t)(kk % 4) * 32;
                    mma_bf16_ta_elect(d_tmem, a_t + (uint32_t)kk * 8, bd + (bo >> 4), idesc,
                                      (k0 > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit_elect(&ab_empty[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    ph ^= 1;
                }
            }
            if (fail)
                break;
            mma_commit_elect(&acc_full[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_ph ^= 1;
            }
            u = nx;
        }
    } else {
        // ---------------- epilogue: 4 warps, TMEM lanes 32*(warp%4) ..
        const int quad = warp & 3;
        const int r = quad * 32 + lane; // tile row of this thread
        int acc = 0;
        uint32_t acc_ph = 0;
        Unit u = blockIdx.x < nu ? A.units[blockIdx.x] : Unit{};
        for (int ui = blockIdx.x; ui < nu && !s_abort; ui += grid) {
            const Unit nx = next_unit(ui, u);
            if (!bar_wait(&acc_full[acc], acc_ph)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)acc * kAccCols;
            const int rowb = (u.e < 0) ? A.T * A.k + u.j0 : u.j0; // first output row of the unit
            for (int c0 = 0; c0 < u.n; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(t_row + (uint32_t)c0, v);
                if (A.mode == 0) {
                    // rows 2f (gate) and 2f + 1 (up) of feature f sit in a lane
                    // pair: the even lane finishes column j, the odd lane
                    // column j + 1, each with one exchange
                    const int f = u.ft * 64 + (r >> 1);
                    const bool odd = r & 1;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float c_j = __uint_as_float(v[j]), c_j1 = __uint_as_float(v[j + 1]);
                        const float got = __shfl_xor_sync(0xFFFFFFFFu, odd ? c_j : c_j1, 1);
                        const float g = odd ? got : c_j, up = odd ? c_j1 : got;
                        const int col = c0 + j + (odd ? 1 : 0);
                        if (col < u.n) {
                            const float a = g / (1.f + __expf(-g)) * up;
                            A.act[(size_t)(rowb + col) * A.act_ld + f] = __float2bfloat16_rn(a);
                        }
                    }
                } else {
                    // the routing weight is applied by the combine
                    const int h = u.ft * 128 + r;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < u.n)
                            A.pout[(size_t)(rowb + c0 + j) * A.H + h] = __uint_as_float(v[j]);
                }
            }
            tc_fence_before();
            bar_arrive(&acc_empty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_ph ^= 1;
            }
            u = nx;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

// ------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2D map over a row-major bf16 matrix [rows, cols]: boxes of 32 rows x 64
// columns with the 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *base, long rows, int cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kAtomK, (cuuint32_t)kBoxRows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over one weight array of every slot of a pool: elements of a
// row (inner), rows, slots; no swizzle.
static bool make_wmap(CUtensorMap *m, CUtensorMapDataType dt, size_t esz, const char *base, uint64_t inner,
                      uint64_t rows, uint64_t slots, uint64_t slot_stride, uint32_t box_inner, uint32_t box_rows,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {inner, rows, slots};
    cuuint64_t strides[2] = {inner * esz, slot_stride};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<char *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The weight-side maps of one GEMM kind (mode 0 gate/up, 1 down), for the
// routed pool and the shared blob.
static bool make_wmaps(const Shape &s, const ExpertSrc &src, int mode, WMaps *w)
{
    const CUtensorMapDataType sdt = s.qscale == MOE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const size_t sb = s.qscale == MOE_F16 ? 2 : 4;
    for (int side = 0; side < 2; ++side) {
        const char *base = side ? src.shared : src.pool;
        const size_t *off = side ? src.off_sh : src.off;
        const uint64_t inter = side ? s.Is : s.I, slots = side ? 1 : src.n_slots;
        const uint64_t stride = side ? (uint64_t)s.H * inter : src.stride; // one slot: any valid stride
        CUtensorMap *m = side ? w->shared : w->routed;
        bool ok;
        if (mode == 0) {
            ok = make_wmap(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base + off[M_QG], s.H / 2, inter, slots, stride,
                           kCK / 2, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_wmap(&m[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base + off[M_QU], s.H / 2, inter, slots, stride,
                           kCK / 2, 64, CU_TENSOR_MAP_SWIZZLE_128B);
            const size_t so[4] = {off[M_SG], off[M_BG], off[M_SU], off[M_BU]};
            for (int j = 0; ok && j < 4; ++j)
                ok = make_wmap(&m[2 + j], sdt, sb, base + so[j], s.H / s.G, inter, slots, stride, s.H / s.G, 64);
        } else {
            ok = make_wmap(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base + off[M_QD], inter / 2, s.H, slots, stride,
                           kCK / 2, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
                 make_wmap(&m[1], sdt, sb, base + off[M_SD], inter / s.G, s.H, slots, stride, inter / s.G, 128) &&
                 make_wmap(&m[2], sdt, sb, base + off[M_BD], inter / s.G, s.H, slots, stride, inter / s.G, 128);
        }
        if (!ok)
            return false;
    }
    return true;
}

static int sm_count()
{
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 148;
}

static size_t a256(size_t v) { return (v + 255) & ~(size_t)255; }

Layout layout(const Shape &s, int T)
{
    Layout L{};
    const long P = (long)T * s.k;
    const int imax = s.I > s.Is ? s.I : s.Is;
    const int nft = s.I / 64, nft_sh = s.Is / 64, hft = s.H / 128;
    const long max_u_gu = (long)nft * (s.E + P / kNch + 1) + (long)nft_sh * (T / kNch + 1);
    const long max_u_dn = (long)hft * (s.E + P / kNch + 1) + (long)hft * (T / kNch + 1);
    size_t o = 0;
    L.counts = o;   o += a256(4 * (size_t)s.E);
    L.offsets = o;  o += a256(4 * (size_t)(s.E + 1));
    L.perm_tok = o; o += a256(4 * (size_t)P);
    L.perm_rank = o; o += a256(4 * (size_t)P);
    L.hist = o;     o += a256(4 * (size_t)bucket_chunks((int)P) * s.E);
    L.inv = o;      o += a256(4 * (size_t)P);
    L.wpair = o;    o += a256(4 * (size_t)(P + T));
    L.units_gu = o; o += a256(sizeof(Unit) * (size_t)max_u_gu);
    L.units_dn = o; o += a256(sizeof(Unit) * (size_t)max_u_dn);
    L.n_units = o;  o += 256;
    L.xs = o;       o += a256(2 * (size_t)P * s.H + 2 * (size_t)kNch * s.H);   // + slack rows for full boxes
    L.act = o;      o += a256(2 * (size_t)(P + T + kNch) * imax);
    L.pout = o;     o += a256(4 * (size_t)(P + T) * s.H);
    L.total = o;
    return L;
}

int min_tokens() { return kernel_path() == 2 ? 2 : kMinTokens; }

bool wanted(const Shape &s, int T)
{
    if (kernel_path() == 1 || T < min_tokens() || T > 65536)
        return false;
    return s.act == MOE_BF16 && s.bits == 4 && s.H % 128 == 0 && s.I % kBK == 0 && s.Is % kBK == 0 && s.Is > 0;
}

bool eligible(const Shape &s, int T)
{
    if (!wanted(s, T))
        return false;
    // the weight-side staging: a half stage (32 K) in one group; a unit's
    // scale and bias rows (16-byte rows, at most 256 elements) in one buffer
    const int sb = s.qscale == MOE_F16 ? 2 : 4;
    if (s.G % 32 || s.H / s.G > 256 || s.I / s.G > 256 || s.Is / s.G > 256)
        return false;
    if ((s.H / s.G * sb) % 16 || (s.I / s.G * sb) % 16 || (s.Is / s.G * sb) % 16)
        return false;
    if (256u * (s.H / s.G) * sb > kSTile || 256u * (s.I / s.G) * sb > kSTile || 256u * (s.Is / s.G) * sb > kSTile)
        return false;
    if (128u * 2 * sb * (s.H / s.G) > kPTile || 128u * 2 * sb * (s.I / s.G) > kPTile ||
        128u * 2 * sb * (s.Is / s.G) > kPTile)
        return false;
    if (encode_fn() == nullptr)
        return false;
    int dev = 0, major = 0, minor = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10;
}

template <typename TS>
static cudaError_t gemm_go(const CUtensorMap &rows, const CUtensorMap &shared, const WMaps &wm, const GemmArgs &g,
                           cudaStream_t st)
{
    static int cur = 0;
    cudaError_t e = ensure_smem(grouped_gemm_kernel<TS>, kSmem, &cur);
    if (e != cudaSuccess)
        return e;
    grouped_gemm_kernel<TS><<<sm_count(), kThreads, kSmem, st>>>(rows, shared, wm, g);
    return cudaGetLastError();
}

// Expert part of the layer for T tokens given the routing (idx, w, sg).
cudaError_t experts_forward(const Shape &s, const ExpertSrc &src, const void *x, int T, const int32_t *idx,
                            const float *topk_w, const float *sg, void *y, float *y32, char *ws, cudaStream_t st)
{
    const Layout L = layout(s, T);
    const long P = (long)T * s.k;
    const int imax = s.I > s.Is ? s.I : s.Is;
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *perm_tok = reinterpret_cast<int32_t *>(ws + L.perm_tok);
    int32_t *perm_rank = reinterpret_cast<int32_t *>(ws + L.perm_rank);
    int32_t *inv = reinterpret_cast<int32_t *>(ws + L.inv);
    float *wpair = reinterpret_cast<float *>(ws + L.wpair);
    Unit *u_gu = reinterpret_cast<Unit *>(ws + L.units_gu);
    Unit *u_dn = reinterpret_cast<Unit *>(ws + L.units_dn);
    int32_t *n_units = reinterpret_cast<int32_t *>(ws + L.n_units);
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(ws + L.xs);
    __nv_bfloat16 *act = reinterpret_cast<__nv_bfloat16 *>(ws + L.act);
    float *pout = reinterpret_cast<float *>(ws + L.pout);

    cudaError_t e = launch_bucket(s, idx, T, counts, offsets, perm_tok, perm_rank,
                                  reinterpret_cast<int32_t *>(ws + L.hist), st);
    if (e != cudaSuccess)
        return e;
    const int row16 = s.H / 8;
    gather_rows_kernel<<<4 * sm_count(), 256, 0, st>>>(static_cast<const uint4 *>(x), perm_tok, (int)P, row16,
                                                      reinterpret_cast<uint4 *>(xs));
    pair_prep_kernel<<<(int)((P + T + 255) / 256), 256, 0, st>>>(perm_tok, perm_rank, topk_w, sg, T, s.k, wpair,
                                                                 inv);
    plan_kernel<<<kPlanCtas, 1024, 0, st>>>(counts, offsets, src.table, src.n_slots, s.E, T, s.I / 64, s.Is / 64,
                                            s.H / 128, s.H / 128, 1, u_gu, u_dn, n_units);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;

    CUtensorMap m_xs, m_x, m_act;
    WMaps w_gu, w_dn;
    if (!make_map(&m_xs, xs, P + kNch, s.H) || !make_map(&m_x, x, T, s.H) ||
        !make_map(&m_act, act, P + T + kNch, imax) || !make_wmaps(s, src, 0, &w_gu) || !make_wmaps(s, src, 1, &w_dn))
        return cudaErrorInvalidValue;
    GemmArgs g{};
    g.src = src;
    g.H = s.H;
    g.I = s.I;
    g.Is = s.Is;
    g.G = s.G;
    g.T = T;
    g.k = s.k;
    g.act_ld = imax;
    g.act = act;
    g.pout = pout;
    g.units = u_gu;
    g.n_units = n_units;
    g.mode = 0;
    e = (s.qscale == MOE_F16) ? gemm_go<__half>(m_xs, m_x, w_gu, g, st) : gemm_go<float>(m_xs, m_x, w_gu, g, st);
    if (e != cudaSuccess)
        return e;
    g.units = u_dn;
    g.n_units = n_units + 1;
    g.mode = 1;
    e = (s.qscale == MOE_F16) ? gemm_go<__half>(m_act, m_act, w_dn, g, st)
                              : gemm_go<float>(m_act, m_act, w_dn, g, st);
    if (e != cudaSuccess)
        return e;
    if ((reinterpret_cast<uintptr_t>(y) & 7) == 0 && (reinterpret_cast<uintptr_t>(y32) & 15) == 0)
        combine_kernel<<<4 * sm_count(), 256, 0, st>>>(pout, wpair, inv, T, s.k, s.H, 1,
                                                        static_cast<__nv_bfloat16 *>(y), y32);
    else
        combine_scalar_kernel<<<4 * sm_count(), 256, 0, st>>>(pout, wpair, inv, T, s.k, s.H, 1,
                                                               static_cast<__nv_bfloat16 *>(y), y32);
    return cudaGetLastError();
}

} // namespace prefill
} // namespace moe
