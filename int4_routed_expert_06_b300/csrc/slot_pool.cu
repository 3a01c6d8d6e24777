// Bounded HBM expert slot pool with LFU + recency eviction.
//
// The Swiftlet pages keep hot routed experts in a bounded pool of slots,
// fetch a missing expert with one read of its fixed-stride blob, and evict by
// "LFU plus recency" (Swiftlet README "How it works" and "Relation to
// TurboFieldfare").  Here the pool lives in HBM, the backing store is pinned
// host memory, a fill is one cudaMemcpyAsync per expert on a side stream, and
// the policy runs on the host:
//   hit  -> use count + 1, stamp = lookup clock (one tick per lookup);
//   miss -> lowest empty slot, else evict the expert not needed by this
//           lookup with the smallest (use count, stamp, slot id); the filled
//           slot starts at use count 1.
// Two comparison rules are selectable for studies (slot_pool_set_policy):
// LRU, the smallest (stamp, slot id), and LFU, the smallest (use count, slot id).
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <chrono>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "internal.h"

namespace {

constexpr int kMaxUpdates = 32;

struct TableUpdate {
    int32_t n;
    int32_t expert[kMaxUpdates];  // installed expert
    int32_t slot[kMaxUpdates];    // its slot
    int32_t evicted[kMaxUpdates]; // expert removed from that slot, -1 = none
};

// Device-table update for one layer: evictions first, then installs.
__global__ void table_update_kernel(int32_t *__restrict__ row, int E, TableUpdate u)
{
    const int j = threadIdx.x;
    if (j < u.n && u.evicted[j] >= 0 && u.evicted[j] < E)
        row[u.evicted[j]] = -1;
    __syncthreads();
    if (j < u.n && u.expert[j] >= 0 && u.expert[j] < E)
        row[u.expert[j]] = u.slot[j];
}

struct Fill {
    int32_t expert, slot, evicted;
};

enum { C_CLOCK = 0, C_LOOKUPS, C_HITS, C_MISSES, C_EVICTIONS, C_BYTES, C_N };

constexpr int kLookupThreads = 256;
constexpr int kMaxUniq = 1024; // distinct experts one device lookup takes

// Victim key of the device lookup, compared lexicographically.
struct VKey {
    int cls;
    long long a, b;
    int slot;
    __device__ bool less(const VKey &o) const
    {
        if (cls != o.cls)
            return cls < o.cls;
        if (a != o.a)
            return a < o.a;
        if (b != o.b)
            return b < o.b;
        return slot < o.slot;
    }
};

// The pool rule on one layer's device state, for the n expert ids at ids
// (device): the same steps, in the same order, as slot_pool_lookup on the
// host.  Distinct ids in order of first appearance; hits are counted and
// stamped; each miss takes the lowest empty slot, else the slot whose expert
// the lookup does not need with the smallest key (policy), ties to the lowest
// slot id.  The (expert, slot) pairs to fill go to fills (count first).  One
// CTA.
__global__ void __launch_bounds__(kLookupThreads) pool_lookup_kernel(const int32_t *__restrict__ ids, int n, int E,
                                                                     int S, int policy, int32_t *__restrict__ table,
                                                                     int32_t *__restrict__ owner,
                                                                     long long *__restrict__ freq,
                                                                     long long *__restrict__ stamp,
                                                                     long long *__restrict__ ctr,
                                                                     int32_t *__restrict__ fills, long long blob_bytes)
{
    __shared__ int32_t uniq[kMaxUniq], miss[kMaxUniq];
    __shared__ int n_uniq, n_miss, bad;
    __shared__ long long clock;
    __shared__ VKey wbest[kLookupThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (t == 0) {
        int nu = 0, b = 0;
        for (int j = 0; j < n && !b; ++j) {
            const int e = ids[j];
            if (e < 0 || e >= E) {
                b = MOE_ERR_DEVICE_FAULT;
                break;
            }
            bool seen = false;
            for (int u = 0; u < nu; ++u)
                seen |= uniq[u] == e;
            if (!seen) {
                if (nu == S || nu == kMaxUniq) {
                    b = MOE_ERR_POOL_EXHAUSTED;
                    break;
                }
                uniq[nu++] = e;
            }
        }
        bad = b;
        n_uniq = nu;
        fills[0] = 0;
        if (!b) {
            clock = ++ctr[C_CLOCK];
            ctr[C_LOOKUPS] += 1;
            int nm = 0;
            for (int u = 0; u < nu; ++u) {
                const int e = uniq[u], sl = table[e];
                if (sl >= 0) {
                    freq[sl] += 1;
                    stamp[sl] = clock;
                    ctr[C_HITS] += 1;
                } else {
                    miss[nm++] = e;
                }
            }
            n_miss = nm;
        } else {
            n_miss = 0;
        }
    }
    __syncthreads();
    if (bad) {
        if (t == 0)
            moe::record_error(bad);
        return;
    }
    const int nu = n_uniq, nm = n_miss;
    for (int m = 0; m < nm; ++m) {
        // victim search: key (class, a, b, slot), smallest first; class 0 =
        // empty slot, 1 = a slot whose expert this lookup does not need,
        // 2 = not a candidate; (a, b) = (use count, stamp) under LFU +
        // recency, (stamp, 0) under LRU, (use count, 0) under LFU
        VKey best{2, 0, 0, 0x7FFFFFFF};
        for (int j = t; j < S; j += kLookupThreads) {
            const int o = owner[j];
            VKey kj{0, 0, 0, j};
            if (o >= 0) {
                bool needed = false;
                for (int u = 0; u < nu; ++u)
                    needed |= uniq[u] == o;
                kj.cls = needed ? 2 : 1;
                kj.a = policy == MOE_POOL_LRU ? stamp[j] : freq[j];
                kj.b = policy == MOE_POOL_LFU_RECENCY ? stamp[j] : 0;
            }
            if (kj.less(best))
                best = kj;
        }
        for (int o = 16; o > 0; o >>= 1) {
            VKey v{__shfl_xor_sync(0xFFFFFFFFu, best.cls, o), __shfl_xor_sync(0xFFFFFFFFu, best.a, o),
                   __shfl_xor_sync(0xFFFFFFFFu, best.b, o), __shfl_xor_sync(0xFFFFFFFFu, best.slot, o)};
            if (v.less(best))
                best = v;
        }
        if (lane == 0)
            wbest[warp] = best;
        __syncthreads();
        if (t == 0) {
            for (int w = 1; w < kLookupThreads / 32; ++w)
                if (wbest[w].less(best))
                    best = wbest[w];
            if (best.cls == 2) { // cannot happen with n_uniq <= S
                moe::record_error(MOE_ERR_DEVICE_FAULT);
                n_miss = m;
                break;
            }
            const int sl = best.slot;
            const int e = miss[m], ev = owner[sl];
            if (ev >= 0) {
                table[ev] = -1;
                ctr[C_EVICTIONS] += 1;
            }
            owner[sl] = e;
            table[e] = sl;
            freq[sl] = 1;
            stamp[sl] = clock;
            ctr[C_MISSES] += 1;
            ctr[C_BYTES] += blob_bytes;
            fills[1 + 2 * m] = e;
            fills[2 + 2 * m] = sl;
        }
        __syncthreads();
    }
    if (t == 0)
        fills[0] = nm;
}

// Copy the blobs of the last lookup's fills from the backing store (host
// memory the device reads through the mapping) into their slots: 16-byte
// pieces, grid-stride over (fill, piece).
__global__ void __launch_bounds__(256) pool_fill_kernel(const int32_t *__restrict__ fills, const char *backing,
                                                        char *__restrict__ pool, size_t stride, size_t blob_bytes,
                                                        int E)
{
    const int nf = fills[0];
    const size_t per = blob_bytes / 16;
    const size_t total = (size_t)nf * per;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int f = (int)(i / per);
        const size_t c = i - (size_t)f * per;
        const int e = fills[1 + 2 * f], sl = fills[2 + 2 * f];
        reinterpret_cast<uint4 *>(pool + (size_t)sl * stride)[c] =
            __ldcs(reinterpret_cast<const uint4 *>(backing + (size_t)e * stride) + c);
    }
}

} // namespace

struct slot_pool {
    moe::Shape s;
    int32_t L = 0, S = 0;
    char *pool = nullptr;
    const char *backing = nullptr;
    size_t stride = 0, blob_bytes = 0;
    cudaStream_t side = nullptr;
    std::vector<int32_t> table;          // [L*E] expert -> slot
    std::vector<int32_t> owner;          // [L*S] slot -> expert
    std::vector<int64_t> freq, stamp;    // [L*S]
    std::vector<std::vector<Fill>> pending; // per layer: fills of its last lookup
    int64_t clock = 0;
    int32_t *table_dev = nullptr;
    moe_pool_stats st{};
    int32_t policy = MOE_POOL_LFU_RECENCY;
    std::mutex mu;
    // moe_pooled_layer_forward: pinned readback of the routed ids, scratch
    // lists, and events that time the compute stream's wait for fills.
    int32_t *pinned_ids = nullptr;
    size_t pinned_cap = 0;
    std::vector<int32_t> tmp_slots, tmp_miss;
    cudaEvent_t fill_done = nullptr, wait_begin = nullptr, wait_end = nullptr;
    bool pending_exposure = false;
    // device-side policy (slot_pool_enable_device): the same rule on device
    // copies of the policy state, fills read from the mapped backing store
    bool device_mode = false;
    const char *backing_dev = nullptr;
    int32_t *d_owner = nullptr;            // [L*S]
    long long *d_freq = nullptr, *d_stamp = nullptr; // [L*S]
    long long *d_ctr = nullptr;            // clock, lookups, hits, misses, evictions, bytes_filled
    int32_t *d_fills = nullptr;            // [L][1 + 2*S]: count, then (expert, slot) pairs of the last lookup
    // storage tier (slot_pool_create_file): blobs read from a file of
    // fixed-stride records into pinned staging buffers, then copied to slots
    int fd = -1;
    bool direct = false;                   // opened with O_DIRECT
    size_t file_stride = 0, file_off0 = 0;
    int n_readers = 0;
    std::vector<char *> staging;           // pinned, file_stride bytes each
    std::vector<cudaEvent_t> staging_ev;   // the copy out of each buffer
    int64_t read_ns = 0, bytes_read = 0;
};

extern "C" moe_status slot_pool_create(const moe_config *cfg, int32_t n_layers, int32_t slots_per_layer,
                                       void *pool_dev, size_t pool_bytes, const void *backing_host,
                                       size_t expert_stride, cudaStream_t side_stream, slot_pool **out)
{
    using namespace moe;
    if (!out)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create: out is NULL");
    *out = nullptr;
    Shape s;
    moe_status cs = check_config(cfg, &s);
    if (cs != MOE_OK)
        return cs;
    if (n_layers <= 0 || slots_per_layer <= 0)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create: n_layers and slots_per_layer must be > 0");
    if (!pool_dev || (reinterpret_cast<uintptr_t>(pool_dev) & 255))
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create: pool_dev must be non-NULL and 256-byte aligned");
    if (!backing_host)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create: backing_host is NULL");
    moe_blob_layout lay;
    moe_blob_layout_get(cfg, cfg->inter, &lay);
    if (expert_stride < lay.bytes || (expert_stride & 255))
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create: expert_stride %zu must be a multiple of 256 and >= %zu",
                    expert_stride, lay.bytes);
    if (pool_bytes / expert_stride < (size_t)n_layers * slots_per_layer)
        return fail(MOE_ERR_OOM, "slot_pool_create: pool_bytes %zu < %d layers x %d slots x %zu", pool_bytes,
                    n_layers, slots_per_layer, expert_stride);
    slot_pool *p = new (std::nothrow) slot_pool();
    if (!p)
        return fail(MOE_ERR_OOM, "slot_pool_create: host allocation failed");
    p->s = s;
    p->L = n_layers;
    p->S = slots_per_layer;
    p->pool = static_cast<char *>(pool_dev);
    p->backing = static_cast<const char *>(backing_host);
    p->stride = expert_stride;
    p->blob_bytes = lay.bytes;
    p->side = side_stream;
    p->table.assign((size_t)n_layers * s.E, -1);
    p->owner.assign((size_t)n_layers * slots_per_layer, -1);
    p->freq.assign((size_t)n_layers * slots_per_layer, 0);
    p->stamp.assign((size_t)n_layers * slots_per_layer, 0);
    p->pending.resize(n_layers);
    *out = p;
    return MOE_OK;
}

// The device table is allocated (all -1) on first use, so that the host
// policy needs no device work until something is filled or read.
static moe_status ensure_table_dev(slot_pool *p)
{
    using namespace moe;
    if (p->table_dev)
        return MOE_OK;
    const size_t tb = sizeof(int32_t) * (size_t)p->L * p->s.E;
    int32_t *t = nullptr;
    cudaError_t e = cudaMalloc(&t, tb);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(t, 0xFF, tb, p->side);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(p->side);
    if (e != cudaSuccess) {
        if (t)
            cudaFree(t);
        return cuda_check(e, "slot pool device table");
    }
    p->table_dev = t;
    return MOE_OK;
}

// ------------------------------------------------------------ storage tier

constexpr int kStaging = 16;   // pinned staging buffers (one blob each)
constexpr size_t kIoAlign = 4096;

static size_t up_io(size_t v) { return (v + kIoAlign - 1) / kIoAlign * kIoAlign; }

// Read `bytes` at `off` of the pool's file into dst, whole: pread until done.
static bool read_full(int fd, char *dst, size_t bytes, off_t off)
{
    size_t got = 0;
    while (got < bytes) {
        const ssize_t r = pread(fd, dst + got, bytes - got, off + (off_t)got);
        if (r <= 0)
            return false;
        got += (size_t)r;
    }
    return true;
}

// The fills of one lookup from the file: in batches of kStaging, each blob
// read (by n_readers threads) into a staging buffer whose previous copy has
// finished, then copied to its slot on the side stream.  Called with p->mu held.
static moe_status file_fill(slot_pool *p, int32_t layer, const std::vector<Fill> &fills)
{
    using namespace moe;
    if (p->staging.empty()) {
        for (int i = 0; i < kStaging; ++i) {
            char *b = nullptr;
            cudaEvent_t ev = nullptr;
            cudaError_t e = cudaHostAlloc(reinterpret_cast<void **>(&b), p->file_stride, cudaHostAllocDefault);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e != cudaSuccess) {
                if (b)
                    cudaFreeHost(b);
                return cuda_check(e, "slot_pool_fill: staging buffers");
            }
            p->staging.push_back(b);
            p->staging_ev.push_back(ev);
        }
    }
    const size_t rb = p->direct ? up_io(p->blob_bytes) : p->blob_bytes; // bytes one read takes
    const int E = p->s.E;
    for (size_t b0 = 0; b0 < fills.size(); b0 += kStaging) {
        const int nb = (int)std::min(fills.size() - b0, (size_t)kStaging);
        for (int i = 0; i < nb; ++i) { // the buffer's last copy must have finished
            cudaError_t e = cudaEventSynchronize(p->staging_ev[i]);
            if (e != cudaSuccess)
                return cuda_check(e, "slot_pool_fill: staging reuse");
        }
        const auto t0 = std::chrono::steady_clock::now();
        std::vector<char> ok(nb, 0);
        auto work = [&](int w) {
            for (int i = w; i < nb; i += p->n_readers) {
                const Fill &f = fills[b0 + i];
                const off_t off = (off_t)(p->file_off0 + ((size_t)layer * E + f.expert) * p->file_stride);
                ok[i] = read_full(p->fd, p->staging[i], rb, off) ? 1 : 0;
            }
        };
        std::vector<std::thread> th;
        for (int w = 1; w < std::min(p->n_readers, nb); ++w)
            th.emplace_back(work, w);
        work(0);
        for (auto &t : th)
            t.join();
        p->read_ns += (int64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(
                          std::chrono::steady_clock::now() - t0)
                          .count();
        for (int i = 0; i < nb; ++i) {
            if (!ok[i])
                return fail(MOE_ERR_CUDA, "slot_pool_fill: read of expert %d of layer %d from the file failed",
                            fills[b0 + i].expert, layer);
            char *dst = p->pool + ((size_t)layer * p->S + fills[b0 + i].slot) * p->stride;
            cudaError_t e = cudaMemcpyAsync(dst, p->staging[i], p->blob_bytes, cudaMemcpyHostToDevice, p->side);
            if (e == cudaSuccess)
                e = cudaEventRecord(p->staging_ev[i], p->side);
            if (e != cudaSuccess)
                return cuda_check(e, "slot_pool_fill: copy");
            p->st.bytes_filled += (int64_t)p->blob_bytes;
            p->bytes_read += (int64_t)rb;
        }
    }
    return MOE_OK;
}

extern "C" moe_status slot_pool_create_file(const moe_config *cfg, int32_t n_layers, int32_t slots_per_layer,
                                            void *pool_dev, size_t pool_bytes, const char *path, size_t file_offset,
                                            size_t file_stride, int32_t readers, cudaStream_t side_stream,
                                            slot_pool **out)
{
    using namespace moe;
    if (!out || !path)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create_file: NULL argument");
    *out = nullptr;
    if (readers < 1 || readers > 64)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create_file: readers %d outside [1, 64]", readers);
    if (file_stride % kIoAlign || file_offset % kIoAlign)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create_file: file_stride and file_offset must be multiples of %zu",
                    kIoAlign);
    moe_blob_layout lay;
    moe_status ls = moe_blob_layout_get(cfg, cfg ? cfg->inter : 0, &lay);
    if (ls != MOE_OK)
        return ls;
    if (file_stride < up_io(lay.bytes))
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create_file: file_stride %zu < %zu (blob rounded to 4 KiB)",
                    file_stride, up_io(lay.bytes));
    bool direct = true;
    int fd = open(path, O_RDONLY | O_DIRECT);
    if (fd < 0) { // a file system without direct I/O: buffered reads
        direct = false;
        fd = open(path, O_RDONLY);
    }
    if (fd < 0)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create_file: cannot open %s", path);
    struct stat sbuf;
    const size_t need = file_offset + (size_t)n_layers * (size_t)(cfg->n_experts > 0 ? cfg->n_experts : 0) * file_stride;
    if (fstat(fd, &sbuf) != 0 || (size_t)sbuf.st_size < need) {
        close(fd);
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_create_file: %s holds fewer than the %zu bytes of %d layers",
                    path, need, n_layers);
    }
    // the pool itself, with a placeholder backing address (never read in this mode)
    moe_status st = slot_pool_create(cfg, n_layers, slots_per_layer, pool_dev, pool_bytes, pool_dev,
                                     lay.bytes <= 256 ? 256 : (lay.bytes + 255) / 256 * 256, side_stream, out);
    if (st != MOE_OK) {
        close(fd);
        return st;
    }
    slot_pool *p = *out;
    p->backing = nullptr;
    p->fd = fd;
    p->direct = direct;
    p->file_stride = file_stride;
    p->file_off0 = file_offset;
    p->n_readers = readers;
    return MOE_OK;
}

extern "C" moe_status slot_pool_file_stats(slot_pool *p, int64_t *bytes_read, int64_t *read_ns, int32_t *direct)
{
    using namespace moe;
    if (!p || !bytes_read || !read_ns || !direct)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_file_stats: NULL argument");
    std::lock_guard<std::mutex> g(p->mu);
    if (p->fd < 0)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_file_stats: the pool has no file tier");
    *bytes_read = p->bytes_read;
    *read_ns = p->read_ns;
    *direct = p->direct ? 1 : 0;
    return MOE_OK;
}

extern "C" moe_status slot_pool_lookup(slot_pool *p, int32_t layer, const int32_t *expert_ids, int32_t n,
                                       int32_t *slots_out, int32_t *miss_ids, int32_t *n_miss)
{
    using namespace moe;
    if (!p || !n_miss || (n > 0 && (!expert_ids || !slots_out || !miss_ids)))
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_lookup: NULL argument");
    if (layer < 0 || layer >= p->L || n < 0)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_lookup: layer %d or n %d out of range", layer, n);
    std::lock_guard<std::mutex> g(p->mu);
    if (p->device_mode)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_lookup: the pool runs its policy on the device");
    const int E = p->s.E, S = p->S;
    std::vector<int32_t> uniq;
    for (int j = 0; j < n; ++j) {
        const int e = expert_ids[j];
        if (e < 0 || e >= E)
            return fail(MOE_ERR_INVALID_ARG, "slot_pool_lookup: expert id %d outside [0, %d)", e, E);
        bool seen = false;
        for (int u : uniq)
            seen |= (u == e);
        if (!seen)
            uniq.push_back(e);
    }
    if ((int)uniq.size() > S)
        return fail(MOE_ERR_POOL_EXHAUSTED, "slot_pool_lookup: %zu distinct experts, %d slots", uniq.size(), S);
    p->clock += 1;
    p->st.lookups += 1;
    int32_t *tab = &p->table[(size_t)layer * E];
    int32_t *own = &p->owner[(size_t)layer * S];
    int64_t *fr = &p->freq[(size_t)layer * S];
    int64_t *sp = &p->stamp[(size_t)layer * S];
    std::vector<int32_t> missing;
    for (int e : uniq) {
        const int s = tab[e];
        if (s >= 0) {
            fr[s] += 1;
            sp[s] = p->clock;
            p->st.hits += 1;
        } else {
            missing.push_back(e);
        }
    }
    std::vector<Fill> &fills = p->pending[layer];
    fills.clear();
    for (int e : missing) {
        int s = -1;
        for (int j = 0; j < S && s < 0; ++j)
            if (own[j] < 0)
                s = j;
        int evicted = -1;
        if (s < 0) {
            for (int j = 0; j < S; ++j) {
                bool needed = false;
                for (int u : uniq)
                    needed |= (own[j] == u);
                if (needed)
                    continue;
                // a candidate replaces the current victim only when its key
                // is strictly smaller, so on equal keys the lower slot id stays
                bool smaller = s < 0;
                if (!smaller) {
                    if (p->policy == MOE_POOL_LRU)
                        smaller = sp[j] < sp[s];
                    else if (p->policy == MOE_POOL_LFU)
                        smaller = fr[j] < fr[s];
                    else
                        smaller = fr[j] < fr[s] || (fr[j] == fr[s] && sp[j] < sp[s]);
                }
                if (smaller)
                    s = j;
            }
            evicted = own[s];
            tab[evicted] = -1;
            p->st.evictions += 1;
        }
        own[s] = e;
        tab[e] = s;
        fr[s] = 1;
        sp[s] = p->clock;
        p->st.misses += 1;
        fills.push_back({e, s, evicted});
    }
    for (int j = 0; j < n; ++j)
        slots_out[j] = tab[expert_ids[j]];
    *n_miss = (int32_t)fills.size();
    for (size_t j = 0; j < fills.size(); ++j)
        miss_ids[j] = fills[j].expert;
    return MOE_OK;
}

extern "C" moe_status slot_pool_set_policy(slot_pool *p, int32_t policy)
{
    using namespace moe;
    if (!p)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_set_policy: NULL pool");
    if (policy != MOE_POOL_LFU_RECENCY && policy != MOE_POOL_LRU && policy != MOE_POOL_LFU)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_set_policy: unknown policy %d", policy);
    std::lock_guard<std::mutex> g(p->mu);
    p->policy = policy;
    return MOE_OK;
}

extern "C" moe_status slot_pool_fill(slot_pool *p, int32_t layer, const int32_t *miss_ids, int32_t n_miss,
                                     cudaEvent_t done)
{
    using namespace moe;
    if (!p || (n_miss > 0 && !miss_ids))
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_fill: NULL argument");
    if (layer < 0 || layer >= p->L)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_fill: layer %d out of range", layer);
    std::lock_guard<std::mutex> g(p->mu);
    std::vector<Fill> &fills = p->pending[layer];
    if ((size_t)n_miss != fills.size())
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_fill: %d misses given, last lookup of layer %d had %zu",
                    n_miss, layer, fills.size());
    for (int j = 0; j < n_miss; ++j)
        if (miss_ids[j] != fills[j].expert)
            return fail(MOE_ERR_INVALID_ARG, "slot_pool_fill: miss %d is expert %d, lookup assigned expert %d", j,
                        miss_ids[j], fills[j].expert);
    moe_status ts = ensure_table_dev(p);
    if (ts != MOE_OK)
        return ts;
    const int E = p->s.E;
    if (p->fd >= 0) {
        moe_status fs = file_fill(p, layer, fills);
        if (fs != MOE_OK)
            return fs;
    } else {
        for (const Fill &f : fills) {
            char *dst = p->pool + ((size_t)layer * p->S + f.slot) * p->stride;
            const char *src = p->backing + ((size_t)layer * E + f.expert) * p->stride;
            cudaError_t e = cudaMemcpyAsync(dst, src, p->blob_bytes, cudaMemcpyHostToDevice, p->side);
            if (e != cudaSuccess)
                return cuda_check(e, "slot_pool_fill: copy");
            p->st.bytes_filled += (int64_t)p->blob_bytes;
        }
    }
    for (size_t j0 = 0; j0 < fills.size(); j0 += kMaxUpdates) {
        TableUpdate u{};
        u.n = (int32_t)std::min(fills.size() - j0, (size_t)kMaxUpdates);
        for (int j = 0; j < u.n; ++j) {
            u.expert[j] = fills[j0 + j].expert;
            u.slot[j] = fills[j0 + j].slot;
            u.evicted[j] = fills[j0 + j].evicted;
        }
        table_update_kernel<<<1, kMaxUpdates, 0, p->side>>>(p->table_dev + (size_t)layer * E, E, u);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return cuda_check(e, "slot_pool_fill: table update");
    }
    fills.clear();
    if (done) {
        cudaError_t e = cudaEventRecord(done, p->side);
        if (e != cudaSuccess)
            return cuda_check(e, "slot_pool_fill: event record");
    }
    return MOE_OK;
}

extern "C" moe_status slot_pool_layer(slot_pool *p, int32_t layer, const int32_t **table_dev,
                                      const void **pool_base_dev)
{
    using namespace moe;
    if (!p || !table_dev || !pool_base_dev)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_layer: NULL argument");
    if (layer < 0 || layer >= p->L)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_layer: layer %d out of range", layer);
    std::lock_guard<std::mutex> g(p->mu);
    moe_status ts = ensure_table_dev(p);
    if (ts != MOE_OK)
        return ts;
    *table_dev = p->table_dev + (size_t)layer * p->s.E;
    *pool_base_dev = p->pool + (size_t)layer * p->S * p->stride;
    return MOE_OK;
}

extern "C" moe_status slot_pool_table_host(slot_pool *p, int32_t layer, int32_t *table_host)
{
    using namespace moe;
    if (!p || !table_host)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_table_host: NULL argument");
    if (layer < 0 || layer >= p->L)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_table_host: layer %d out of range", layer);
    std::lock_guard<std::mutex> g(p->mu);
    if (p->device_mode)
        return cuda_check(cudaMemcpy(table_host, p->table_dev + (size_t)layer * p->s.E, sizeof(int32_t) * p->s.E,
                                     cudaMemcpyDeviceToHost),
                          "slot_pool_table_host: device table");
    for (int e = 0; e < p->s.E; ++e)
        table_host[e] = p->table[(size_t)layer * p->s.E + e];
    return MOE_OK;
}

// Add the last pooled forward's fill wait to the stats once it has finished.
static void harvest_exposure(slot_pool *p)
{
    if (!p->pending_exposure)
        return;
    float ms = 0.f;
    if (cudaEventSynchronize(p->wait_end) == cudaSuccess &&
        cudaEventElapsedTime(&ms, p->wait_begin, p->wait_end) == cudaSuccess)
        p->st.exposed_copy_ns += (int64_t)(ms * 1.0e6);
    p->pending_exposure = false;
}

static moe_status device_step(slot_pool *p, int32_t layer, const int32_t *ids_dev, int32_t n, cudaStream_t stream);

extern "C" moe_status slot_pool_stats(slot_pool *p, moe_pool_stats *out)
{
    using namespace moe;
    if (!p || !out)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_stats: NULL argument");
    std::lock_guard<std::mutex> g(p->mu);
    if (p->device_mode) {
        long long c[C_N];
        cudaError_t e = cudaMemcpy(c, p->d_ctr, sizeof(c), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess)
            return cuda_check(e, "slot_pool_stats: device counters");
        *out = moe_pool_stats{c[C_LOOKUPS], c[C_HITS], c[C_MISSES], c[C_EVICTIONS], c[C_BYTES], 0};
        return MOE_OK;
    }
    harvest_exposure(p);
    *out = p->st;
    return MOE_OK;
}

extern "C" moe_status moe_pooled_layer_forward(const moe_config *cfg, slot_pool *p, int32_t layer,
                                               const moe_resident_weights *w, const void *x, int32_t T, void *y,
                                               float *y_f32, int32_t *topk_idx_out, void *workspace,
                                               size_t ws_bytes, cudaStream_t stream)
{
    using namespace moe;
    Shape s;
    moe_status st = check_config(cfg, &s);
    if (st != MOE_OK)
        return st;
    if (!p || !w || !w->w_router)
        return fail(MOE_ERR_INVALID_ARG, "moe_pooled_layer_forward: NULL pool, weights or router");
    if (s.H != p->s.H || s.E != p->s.E || s.k != p->s.k || s.I != p->s.I || s.G != p->s.G ||
        s.qscale != p->s.qscale)
        return fail(MOE_ERR_INVALID_ARG, "moe_pooled_layer_forward: config differs from the pool's");
    if (layer < 0 || layer >= p->L)
        return fail(MOE_ERR_INVALID_ARG, "moe_pooled_layer_forward: layer %d out of range", layer);
    if (T < 0 || T > 65535)
        return fail(MOE_ERR_INVALID_ARG, "moe_pooled_layer_forward: T %d out of range", T);
    if (T == 0)
        return MOE_OK;
    const Ws ws = layer_ws(s, T);
    if (!workspace || ws_bytes < ws.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return fail(MOE_ERR_OOM, "moe_pooled_layer_forward: workspace needs %zu bytes (256-byte aligned), got %zu",
                    ws.total, ws_bytes);
    char *wsp = static_cast<char *>(workspace);
    int32_t *idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t *>(wsp + ws.idx);
    float *tw = reinterpret_cast<float *>(wsp + ws.w);
    float *sg = s.Is > 0 ? reinterpret_cast<float *>(wsp + ws.sg) : nullptr;
    float *logits = reinterpret_cast<float *>(wsp + ws.logits);
    st = moe_route(cfg, x, T, w->w_router, w->router_bias, s.Is > 0 ? w->w_shared_gate : nullptr, idx, tw, sg,
                   logits, nullptr, 0, stream);
    if (st != MOE_OK)
        return st;

    const size_t n_ids = (size_t)T * s.k;
    if (p->device_mode) {
        // no host round trip: lookup and fills are kernels on `stream`
        st = device_step(p, layer, idx, (int32_t)n_ids, stream);
        if (st != MOE_OK)
            return st;
        moe_layer L{w->w_router, w->router_bias, w->w_shared_gate, w->shared_blob,
                    p->pool + (size_t)layer * p->S * p->stride, p->stride, p->table_dev + (size_t)layer * s.E, p->S};
        return moe_experts_forward(cfg, &L, x, T, idx, tw, sg, y, y_f32, workspace, ws_bytes, stream);
    }
    {
        std::lock_guard<std::mutex> g(p->mu);
        moe_status ts = ensure_table_dev(p);
        if (ts != MOE_OK)
            return ts;
        cudaError_t e = cudaSuccess;
        if (!p->fill_done) {
            e = cudaEventCreateWithFlags(&p->fill_done, cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreate(&p->wait_begin);
            if (e == cudaSuccess)
                e = cudaEventCreate(&p->wait_end);
        }
        if (e == cudaSuccess && n_ids > p->pinned_cap) {
            if (p->pinned_ids)
                cudaFreeHost(p->pinned_ids);
            p->pinned_ids = nullptr;
            p->pinned_cap = 0;
            e = cudaHostAlloc(reinterpret_cast<void **>(&p->pinned_ids), n_ids * sizeof(int32_t),
                              cudaHostAllocDefault);
            if (e == cudaSuccess)
                p->pinned_cap = n_ids;
        }
        if (e != cudaSuccess)
            return cuda_check(e, "moe_pooled_layer_forward: host buffers");
        harvest_exposure(p);
    }
    cudaError_t e = cudaMemcpyAsync(p->pinned_ids, idx, n_ids * sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return cuda_check(e, "moe_pooled_layer_forward: routing readback");

    p->tmp_slots.resize(n_ids);
    p->tmp_miss.resize(n_ids);
    int32_t n_miss = 0;
    st = slot_pool_lookup(p, layer, p->pinned_ids, (int32_t)n_ids, p->tmp_slots.data(), p->tmp_miss.data(),
                          &n_miss);
    if (st != MOE_OK)
        return st;
    if (n_miss > 0) {
        st = slot_pool_fill(p, layer, p->tmp_miss.data(), n_miss, p->fill_done);
        if (st != MOE_OK)
            return st;
        e = cudaEventRecord(p->wait_begin, stream);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(stream, p->fill_done, 0);
        if (e == cudaSuccess)
            e = cudaEventRecord(p->wait_end, stream);
        if (e != cudaSuccess)
            return cuda_check(e, "moe_pooled_layer_forward: fill ordering");
        std::lock_guard<std::mutex> g(p->mu);
        p->pending_exposure = true;
    }
    moe_layer L{w->w_router, w->router_bias, w->w_shared_gate, w->shared_blob,
                p->pool + (size_t)layer * p->S * p->stride, p->stride, p->table_dev + (size_t)layer * s.E, p->S};
    return moe_experts_forward(cfg, &L, x, T, idx, tw, sg, y, y_f32, workspace, ws_bytes, stream);
}

// ------------------------------------------------------------ device-side policy

extern "C" moe_status slot_pool_enable_device(slot_pool *p)
{
    using namespace moe;
    if (!p)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_enable_device: NULL pool");
    std::lock_guard<std::mutex> g(p->mu);
    if (p->device_mode)
        return MOE_OK;
    if (p->st.lookups != 0)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_enable_device: the pool has already served host lookups");
    if (p->S > kMaxUniq * 2)
        return fail(MOE_ERR_UNSUPPORTED, "slot_pool_enable_device: %d slots per layer (at most %d)", p->S,
                    kMaxUniq * 2);
    if (p->fd >= 0)
        return fail(MOE_ERR_UNSUPPORTED, "slot_pool_enable_device: a file-backed pool fills from the host");
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p->backing) != cudaSuccess || at.type != cudaMemoryTypeHost ||
        !at.devicePointer) {
        cudaGetLastError();
        return fail(MOE_ERR_UNSUPPORTED, "slot_pool_enable_device: the backing store is not pinned host memory "
                                         "the device can read");
    }
    moe_status ts = ensure_table_dev(p);
    if (ts != MOE_OK)
        return ts;
    const size_t LS = (size_t)p->L * p->S;
    cudaError_t e = cudaMalloc(&p->d_owner, LS * sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMalloc(&p->d_freq, LS * sizeof(long long));
    if (e == cudaSuccess)
        e = cudaMalloc(&p->d_stamp, LS * sizeof(long long));
    if (e == cudaSuccess)
        e = cudaMalloc(&p->d_ctr, C_N * sizeof(long long));
    if (e == cudaSuccess)
        e = cudaMalloc(&p->d_fills, (size_t)p->L * (1 + 2 * (size_t)p->S) * sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMemset(p->d_owner, 0xFF, LS * sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaMemset(p->d_freq, 0, LS * sizeof(long long));
    if (e == cudaSuccess)
        e = cudaMemset(p->d_stamp, 0, LS * sizeof(long long));
    if (e == cudaSuccess)
        e = cudaMemset(p->d_ctr, 0, C_N * sizeof(long long));
    if (e == cudaSuccess)
        e = cudaMemset(p->d_fills, 0, (size_t)p->L * (1 + 2 * (size_t)p->S) * sizeof(int32_t));
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_check(e, "slot_pool_enable_device: device state");
    p->backing_dev = static_cast<const char *>(at.devicePointer);
    p->device_mode = true;
    return MOE_OK;
}

// Lookup + fills of one layer on `stream` (device mode; the caller holds no lock).
static moe_status device_step(slot_pool *p, int32_t layer, const int32_t *ids_dev, int32_t n, cudaStream_t stream)
{
    using namespace moe;
    const int E = p->s.E, S = p->S;
    int32_t *fills = p->d_fills + (size_t)layer * (1 + 2 * (size_t)S);
    pool_lookup_kernel<<<1, kLookupThreads, 0, stream>>>(
        ids_dev, n, E, S, p->policy, p->table_dev + (size_t)layer * E, p->d_owner + (size_t)layer * S,
        p->d_freq + (size_t)layer * S, p->d_stamp + (size_t)layer * S, p->d_ctr, fills, (long long)p->blob_bytes);
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    pool_fill_kernel<<<4 * (sms > 0 ? sms : 148), 256, 0, stream>>>(
        fills, p->backing_dev + (size_t)layer * E * p->stride, p->pool + (size_t)layer * S * p->stride, p->stride,
        p->blob_bytes, E);
    return cuda_check(cudaGetLastError(), "slot pool device step");
}

extern "C" moe_status slot_pool_step_device(slot_pool *p, int32_t layer, const int32_t *ids_dev, int32_t n,
                                            cudaStream_t stream)
{
    using namespace moe;
    if (!p || (n > 0 && !ids_dev))
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_step_device: NULL argument");
    if (!p->device_mode)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_step_device: the pool is not in device mode");
    if (layer < 0 || layer >= p->L || n < 0 || n > 65535 * 16)
        return fail(MOE_ERR_INVALID_ARG, "slot_pool_step_device: layer %d or n %d out of range", layer, n);
    if (n == 0)
        return MOE_OK;
    return device_step(p, layer, ids_dev, n, stream);
}

extern "C" void slot_pool_destroy(slot_pool *p)
{
    if (!p)
        return;
    if (p->pending_exposure && p->wait_end)
        cudaEventSynchronize(p->wait_end);
    if (p->table_dev)
        cudaFree(p->table_dev);
    for (void *d : {(void *)p->d_owner, (void *)p->d_freq, (void *)p->d_stamp, (void *)p->d_ctr, (void *)p->d_fills})
        if (d)
            cudaFree(d);
    if (p->pinned_ids)
        cudaFreeHost(p->pinned_ids);
    for (size_t i = 0; i < p->staging.size(); ++i) {
        cudaEventSynchronize(p->staging_ev[i]);
        cudaEventDestroy(p->staging_ev[i]);
        cudaFreeHost(p->staging[i]);
    }
    if (p->fd >= 0)
        close(p->fd);
    if (p->fill_done)
        cudaEventDestroy(p->fill_done);
    if (p->wait_begin)
        cudaEventDestroy(p->wait_begin);
    if (p->wait_end)
        cudaEventDestroy(p->wait_end);
    delete p;
}
