// kvb_api.cpp -- host side of the KV backup / restore engine: the C ABI of
// include/kvb.h.  Validation, handle and IPC-mapping registries, fences, and
// the launch plan of each operation.  All data movement happens in the
// kernels of kvb_kernels.cu (and, in STAGED mode, in copy-engine memcpys).
//
// Pages this follows (by title and section):
//   [RFC] "[Feature] [RFC] [HiCache] Out-of-process HiCache data plane with
//         device-memory IPC": §Device IPC data path, §Ownership, §Failure and
//         lifecycle handling.
//   [PR]  "[PP + HiCache] Add PP Prefetch Tickets for eager cross-stage
//         storage prefetch": §PP Prefetch Ticket Path (layer-wise H2D).
//   [LMC] "LMCacheRawCudaIPCWrapper深度解析": §共享与重建的完整链路,
//         §发送端校验, §重建生命周期与引用计数, §为什么不做_share_cuda_回退.
#include "kvb.h"
#include "kvb_internal.h"
#include "kvb_ring_internal.h"

#include <cuda.h>   // CUresult / CUdeviceptr types only; the function comes from the runtime
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <ctime>
#include <mutex>
#include <sched.h>
#include <string>
#include <unistd.h>
#include <unordered_map>
#include <vector>

using namespace kvb;

namespace {

// ------------------------------------------------------------------ errors

thread_local std::string t_err;

kv_status fail(kv_status st, const char *fmt, ...) {
    char buf[768];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return st;
}

kv_status cuda_fail(cudaError_t e, const char *what) {
    kv_status st = fail(KV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                        cudaGetErrorString(e));
    (void)cudaGetLastError();   // a non-sticky error must not resurface at a later launch
    return st;
}

// ----------------------------------------------------------- fault injection
// Host-side failure drills ("[PP + HiCache] Add PP Prefetch Tickets",
// §Targeted fault-injection validation: injected allocation failures must fall
// back and leave the service running).  The next `count` passes through a
// point fail as if the CUDA call there had failed ("launch_nth": only the
// count-th pass from now fails); nothing touches the GPU.  "chain_stall" is
// the one drill that reaches a kernel: the next overlapped restore chains its
// fence on a sequence number its predecessor never stores, so its bounded
// wait runs out (2 s) and the kernel reports it through the error word.
enum FaultPoint { FP_STAGING_ALLOC, FP_FENCE_RESERVE, FP_LAUNCH, FP_IPC_OPEN, FP_HOST_REGISTER,
                  FP_LAUNCH_NTH, FP_CHAIN_STALL, FP_COUNT };
const char *const kFaultNames[FP_COUNT] = {"staging_alloc", "fence_reserve", "launch", "ipc_open",
                                           "host_register", "launch_nth", "chain_stall"};
std::atomic<uint32_t> g_fault[FP_COUNT];
std::once_flag g_fault_env_once;

void load_fault_env() {
    // KVB_FAULT="point:count[,point:count...]"
    const char *v = getenv("KVB_FAULT");
    if (v == nullptr) return;
    std::string spec(v);
    size_t pos = 0;
    while (pos < spec.size()) {
        size_t end = spec.find(',', pos);
        if (end == std::string::npos) end = spec.size();
        const std::string item = spec.substr(pos, end - pos);
        const size_t colon = item.find(':');
        const std::string name = item.substr(0, colon);
        const uint32_t count = colon == std::string::npos ? 1u
                                                          : (uint32_t)strtoul(item.c_str() + colon + 1,
                                                                              nullptr, 10);
        for (int i = 0; i < FP_COUNT; ++i)
            if (name == kFaultNames[i]) g_fault[i].store(count);
        pos = end + 1;
    }
}

bool fault_hit(FaultPoint p) {
    std::call_once(g_fault_env_once, load_fault_env);
    uint32_t c = g_fault[p].load();
    while (c > 0)
        if (g_fault[p].compare_exchange_weak(c, c - 1)) return p == FP_LAUNCH_NTH ? c == 1 : true;
    return false;
}

// ---------------------------------------------------------------- geometry

struct Geo {
    uint64_t L, C, P, T, H, B;
    uint32_t order, heads;
    uint64_t cb;   // chunk bytes: T*H*B (one page or slot, one layer, one component)
    uint64_t pb;   // page bytes: L*C*cb
};

bool mul_ok(uint64_t a, uint64_t b, uint64_t lim, uint64_t *out) {
    if (a != 0 && b > lim / a) return false;
    *out = a * b;
    return true;
}

// Layout checks shared by every entry point ([LMC] §发送端校验: reject, never guess).
kv_status check_layout(const kv_layout *lay, Geo *g) {
    if (lay == nullptr) return fail(KV_ERR_INVALID_ARG, "layout is NULL");
    if (lay->num_layers == 0 || lay->num_comps == 0 || lay->num_pages == 0 ||
        lay->page_tokens == 0 || lay->num_heads == 0 || lay->head_bytes == 0)
        return fail(KV_ERR_LAYOUT,
                    "layout has a zero dimension (L=%u C=%u P=%u T=%u H=%u B=%u)",
                    lay->num_layers, lay->num_comps, lay->num_pages, lay->page_tokens,
                    lay->num_heads, lay->head_bytes);
    if (lay->order > KV_PAGE_FIRST || lay->heads > KV_HND || lay->reserved != 0)
        return fail(KV_ERR_LAYOUT, "layout has unknown order %u / heads %u or reserved %u != 0",
                    lay->order, lay->heads, lay->reserved);
    if (lay->head_bytes % 16 != 0)
        return fail(KV_ERR_ALIGNMENT, "head_bytes %u is not a multiple of 16", lay->head_bytes);
    Geo r{lay->num_layers, lay->num_comps, lay->num_pages, lay->page_tokens, lay->num_heads,
          lay->head_bytes, lay->order, lay->heads, 0, 0};
    uint64_t th, lc, pool;
    const uint64_t lim = 1ull << 62;
    if (!mul_ok(r.T, r.H, lim, &th) || !mul_ok(th, r.B, lim, &r.cb) ||
        !mul_ok(r.L, r.C, lim, &lc) || !mul_ok(lc, r.cb, lim, &r.pb) ||
        !mul_ok(r.pb, r.P, lim, &pool))
        return fail(KV_ERR_LAYOUT, "layout sizes overflow 64-bit byte offsets");
    if (r.cb / 16 >= (1ull << 31))
        return fail(KV_ERR_LAYOUT, "one (page, layer, component) chunk of %llu bytes is too large",
                    (unsigned long long)r.cb);
    *g = r;
    return KV_OK;
}

bool same_slot_geometry(const Geo &a, const Geo &b) {
    return a.L == b.L && a.C == b.C && a.T == b.T && a.H == b.H && a.B == b.B;
}

// --------------------------------------------------------------- handles

struct PoolObj {
    Geo g{};
    kv_layout layout;
    char *dev;           // device address of the pool's first byte
    uint64_t nbytes;
    int device;
    uint64_t instance_id, generation;
    bool imported;
    std::string ipc_key; // handle bytes of the mapping (imported pools)
    std::vector<std::string> ipc_keys;   // imported split pools: each distinct mapping, once
    // split pools: one device buffer per (layer, component); the table of their
    // addresses (entry l * C + c) lives in device memory for the kernels
    unsigned long long *table_dev = nullptr;
    std::vector<unsigned long long> table_host;   // the same table, for copy-engine moves
};

struct HostObj {
    Geo g{};               // slot geometry (P unused)
    uint32_t heads;      // head order of the tier
    uint32_t num_slots;
    char *host;
    char *dev_view;      // device-visible address of `host`
    uint64_t bytes;
};

struct Mapping {
    void *base;
    int refs;
    int device;
};

constexpr int kRing = 4096;       // fence words / events per device
constexpr int kMaxDevices = 64;
constexpr uint64_t kSeqMask = (1ull << 56) - 1;

struct DevState {
    bool init = false;
    unsigned long long *words = nullptr;     // host view of the fence words
    unsigned long long *words_dev = nullptr; // device view
    unsigned long long *status = nullptr;    // host view: status[k] == seq -> op gave up
    unsigned long long *status_dev = nullptr;
    uint32_t *err = nullptr;                 // sticky "kernel met a bad id" word
    uint32_t *err_dev = nullptr;
    uint32_t *counters = nullptr;            // device: finished-CTA counters, one per slot
    uint32_t *aux = nullptr;                 // device: per-slot layer counters, kRing each of
                                             // done / published / work / lock (progressive)
    bool wait_value = false;                 // GPU-side waits on fence words supported
    cudaEvent_t ev[kRing] = {};
    uint64_t slot_seq[kRing] = {};
    int sms = 0;
    char *staging = nullptr;                 // STAGED mode buffer, two halves
    uint64_t staging_bytes = 0;
    cudaEvent_t staging_free[2] = {nullptr, nullptr};
    bool staging_used[2] = {false, false};
    // STAGED ops of several chunks: each half is two ping-pong buffers; the HBM
    // kernels run on side[half] (a backup's and a restore's apart, so the two
    // can run at once) while the copy engine works on the caller's stream
    cudaStream_t side[2] = {nullptr, nullptr};
    cudaEvent_t op_start = nullptr;          // caller's stream at the op's start
    cudaEvent_t moved[2][2] = {};            // [half][buffer]: kernel done with it
    cudaEvent_t copied[2][2] = {};           // [half][buffer]: copy engine done with it
    // Progressive restores of more than kMaxItems pages: their ids go through a
    // pinned buffer and a device buffer (a then b, n each) instead of the launch
    int32_t *gids = nullptr;                 // device
    int32_t *gids_host = nullptr;            // pinned
    uint64_t gids_cap = 0;                   // int32 entries in each
    cudaEvent_t gids_copied = nullptr;       // the pinned -> device copy is done
    cudaEvent_t gids_free = nullptr;         // the kernel reading the device ids is done
    bool gids_used = false;
    // KV_CFG_OVERLAP_RESTORES / _BACKUPS: per stream, the run of zero-copy
    // restores and backups of one pool issued there since the last op that
    // waited for its predecessor; any other op of this library on the stream
    // erases it.  Each overlapped kernel may start while its predecessors still
    // run (each lets the next launch early), so a new op may overlap only if no
    // byte it touches is written by an op of the run whose fence is not yet
    // complete, and it writes no byte such an op reads (ops_conflict).
    struct ChainOp {
        int k;                      // fence slot and sequence number
        uint64_t seq;
        int kind;                   // 0 backup (reads pages, writes slots), 1 restore
        int32_t layer;              // -1 = every layer
        std::vector<int32_t> pages; // pool pages it reads (backup) or writes (restore), sorted
        std::vector<int32_t> slots; // host slots it writes (backup) or reads (restore), sorted
    };
    struct Chain {
        uint64_t pool;              // pool handle id
        std::vector<ChainOp> ops;   // in call order; the last is the stream's last op
    };
    std::unordered_map<void *, Chain> chains;
};

std::mutex g_mu;
std::unordered_map<uint64_t, PoolObj *> g_pools;   // handle id -> object
std::unordered_map<uint64_t, HostObj *> g_hosts;
std::unordered_map<std::string, Mapping> g_maps;   // IPC handle bytes -> mapping
std::unordered_map<uint64_t, uint64_t> g_floor;    // instance -> lowest live generation
uint64_t g_next_handle = 1;                         // handle ids are never reused
uint64_t g_next_seq = 1;
DevState g_dev[kMaxDevices];
kv_config g_cfg = {KV_MODE_ZERO_COPY, 0, 0, 0, 0};
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_overlapped{0};   // ops issued overlapped

constexpr uint64_t kDefaultStaging = 256ull << 20;
constexpr uint64_t kMaxReadyTimeoutNs = 60ull * 1000 * 1000 * 1000;   // gate waits at most 60 s

uint64_t handle_id(const void *h) { return (uint64_t)(uintptr_t)h; }

PoolObj *find_pool(kv_pool p) {
    auto it = g_pools.find(handle_id(p));
    return it == g_pools.end() ? nullptr : it->second;
}

HostObj *find_host(kv_host h) {
    auto it = g_hosts.find(handle_id(h));
    return it == g_hosts.end() ? nullptr : it->second;
}

struct DeviceGuard {
    int prev = -1;
    int want;
    explicit DeviceGuard(int d) : want(d) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != want) cudaSetDevice(want);
    }
    ~DeviceGuard() {
        if (prev >= 0 && prev != want) cudaSetDevice(prev);
    }
};

typedef CUresult (*GetAddressRangeFn)(CUdeviceptr *, size_t *, CUdeviceptr);

kv_status address_range(const void *p, uintptr_t *base, size_t *size) {
    static GetAddressRangeFn fn = nullptr;
    if (fn == nullptr) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || f == nullptr)
            return fail(KV_ERR_CUDA, "cuMemGetAddressRange entry point unavailable");
        fn = (GetAddressRangeFn)f;
    }
    CUdeviceptr b = 0;
    size_t s = 0;
    CUresult r = fn(&b, &s, (CUdeviceptr)(uintptr_t)p);
    if (r != CUDA_SUCCESS)
        return fail(KV_ERR_INVALID_ARG, "pointer %p is not inside a device allocation (CUresult %d)",
                    p, (int)r);
    *base = (uintptr_t)b;
    *size = s;
    return KV_OK;
}

// Driver entry points fetched through the runtime (no link-time libcuda).
typedef CUresult (*StreamWaitValue64Fn)(CUstream, CUdeviceptr, cuuint64_t, unsigned int);
typedef CUresult (*DeviceGetFn)(CUdevice *, int);
typedef CUresult (*DeviceGetAttributeFn)(int *, CUdevice_attribute, CUdevice);

void *driver_fn(const char *name) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return f;
}

StreamWaitValue64Fn g_wait_value64 = nullptr;

// GPU-side waits on a 64-bit word (a stream waits until fence word >= seq)
// need the driver's 64-bit stream memory operations.
bool stream_wait_value_supported(int ordinal) {
    auto get = (DeviceGetFn)driver_fn("cuDeviceGet");
    auto attr = (DeviceGetAttributeFn)driver_fn("cuDeviceGetAttribute");
    g_wait_value64 = (StreamWaitValue64Fn)driver_fn("cuStreamWaitValue64");
    if (get == nullptr || attr == nullptr || g_wait_value64 == nullptr) return false;
    CUdevice dev;
    int v = 0;
    if (get(&dev, ordinal) != CUDA_SUCCESS) return false;
    if (attr(&v, CU_DEVICE_ATTRIBUTE_CAN_USE_64_BIT_STREAM_MEM_OPS, dev) != CUDA_SUCCESS) return false;
    return v != 0;
}

kv_status init_device(int d) {
    if (d < 0 || d >= kMaxDevices) return fail(KV_ERR_INVALID_ARG, "device %d out of range", d);
    DevState &s = g_dev[d];
    if (s.init) return KV_OK;
    DeviceGuard guard(d);
    // every kernel loaded before the first launch: a lazy load behind a waiting
    // kernel (gate, resident server) would wait for that kernel to end
    cudaError_t e0 = preload_kernels();
    if (e0 == cudaSuccess) e0 = preload_ring_kernels();
    if (e0 != cudaSuccess) return cuda_fail(e0, "loading the library's kernels");
    // mapped pinned table: kRing fence words, kRing status words, the error word
    const size_t table = 2 * kRing * sizeof(unsigned long long) + 64;
    void *mem = nullptr;
    cudaError_t e = cudaHostAlloc(&mem, table, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc(fence words)");
    std::memset(mem, 0, table);
    void *dmem = nullptr;
    e = cudaHostGetDevicePointer(&dmem, mem, 0);
    if (e != cudaSuccess) {
        cudaFreeHost(mem);
        return cuda_fail(e, "cudaHostGetDevicePointer(fence words)");
    }
    void *cnt = nullptr;
    e = cudaMalloc(&cnt, 5 * kRing * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(cnt, 0, 5 * kRing * sizeof(uint32_t));
    if (e != cudaSuccess) {
        if (cnt) cudaFree(cnt);
        cudaFreeHost(mem);
        return cuda_fail(e, "cudaMalloc(completion counters)");
    }
    s.aux = (uint32_t *)cnt + kRing;
    s.wait_value = stream_wait_value_supported(d);
    s.words = (unsigned long long *)mem;
    s.words_dev = (unsigned long long *)dmem;
    s.status = s.words + kRing;
    s.status_dev = s.words_dev + kRing;
    s.err = (uint32_t *)(s.words + 2 * kRing);
    s.err_dev = (uint32_t *)(s.words_dev + 2 * kRing);
    s.counters = (uint32_t *)cnt;
    cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, d);
    if (s.sms <= 0) s.sms = 1;
    s.init = true;
    return KV_OK;
}

// ------------------------------------------------------------------ fences

unsigned long long load_acquire(const unsigned long long *p) {
    return __atomic_load_n(p, __ATOMIC_ACQUIRE);
}

double now_ns() {
    timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return ts.tv_sec * 1e9 + ts.tv_nsec;
}

// Fences.  An operation first reserves the next sequence number and its ring
// slot (waiting, bounded, if the slot's previous op is still in flight); its
// last kernel then stores the number into the slot's mapped word -- fused into
// the move kernel, or by kv_mark_kernel after copy-engine work -- and
// commit_fence records the slot's event and publishes the fence.  Both run
// with g_mu held and the device current, so a failed operation simply never
// commits and its number is reused.
struct FenceSlot {
    uint64_t seq;
    int k;
};

kv_status reserve_fence(int d, FenceSlot *out) {
    if (fault_hit(FP_FENCE_RESERVE))
        return fail(KV_ERR_NO_MEMORY, "fence ring exhausted: injected failure");
    DevState &s = g_dev[d];
    const uint64_t seq = g_next_seq;
    if (seq > kSeqMask) return fail(KV_ERR_NO_MEMORY, "fence sequence space exhausted");
    const int k = (int)(seq % kRing);
    if (s.slot_seq[k] != 0 && load_acquire(&s.words[k]) < s.slot_seq[k]) {
        // The op that last used this slot (kRing fences ago) is still running.
        const double deadline = now_ns() + 30e9;
        while (load_acquire(&s.words[k]) < s.slot_seq[k]) {
            if (now_ns() > deadline)
                return fail(KV_ERR_NO_MEMORY, "%d fences in flight: fence ring exhausted", kRing);
            sched_yield();
        }
    }
    if (s.ev[k] == nullptr) {
        cudaError_t e = cudaEventCreateWithFlags(&s.ev[k], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            s.ev[k] = nullptr;
            return cuda_fail(e, "cudaEventCreate(fence)");
        }
    }
    out->seq = seq;
    out->k = k;
    return KV_OK;
}

// Reserves `count` consecutive sequence numbers (count <= kRing / 2), each
// slot free; returns the first.  Nothing is committed.
kv_status reserve_fence_range(int d, uint32_t count, uint64_t *seq0) {
    if (fault_hit(FP_FENCE_RESERVE))
        return fail(KV_ERR_NO_MEMORY, "fence ring exhausted: injected failure");
    DevState &s = g_dev[d];
    const uint64_t first = g_next_seq;
    if (first + count > kSeqMask) return fail(KV_ERR_NO_MEMORY, "fence sequence space exhausted");
    for (uint32_t j = 0; j < count; ++j) {
        const int k = (int)((first + j) % kRing);
        if (s.slot_seq[k] != 0 && load_acquire(&s.words[k]) < s.slot_seq[k]) {
            const double deadline = now_ns() + 30e9;
            while (load_acquire(&s.words[k]) < s.slot_seq[k]) {
                if (now_ns() > deadline)
                    return fail(KV_ERR_NO_MEMORY, "%d fences in flight: fence ring exhausted",
                                kRing);
                sched_yield();
            }
        }
        if (s.ev[k] == nullptr) {
            cudaError_t e = cudaEventCreateWithFlags(&s.ev[k], cudaEventDisableTiming);
            if (e != cudaSuccess) {
                s.ev[k] = nullptr;
                return cuda_fail(e, "cudaEventCreate(fence)");
            }
        }
    }
    *seq0 = first;
    return KV_OK;
}

kv_status commit_fence(int d, const FenceSlot &f, bool need_mark, cudaStream_t stream,
                       kv_fence *out) {
    DevState &s = g_dev[d];
    if (need_mark) {
        cudaError_t e = launch_mark(s.words_dev + f.k, f.seq, stream);
        if (e != cudaSuccess) return cuda_fail(e, "launch of the completion marker");
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    cudaError_t e = cudaEventRecord(s.ev[f.k], stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fence)");
    s.slot_seq[f.k] = f.seq;
    g_next_seq = f.seq + 1;
    *out = ((uint64_t)d << 56) | f.seq;
    return KV_OK;
}

kv_status issue_fence(int d, cudaStream_t stream, kv_fence *out) {
    FenceSlot f;
    kv_status st = reserve_fence(d, &f);
    if (st != KV_OK) return st;
    return commit_fence(d, f, true, stream, out);
}

// Decodes a fence; returns KV_OK with done set, or an error.
kv_status fence_state(kv_fence f, bool *done, int *dev, int *slot, bool *aborted) {
    const int d = (int)(f >> 56);
    const uint64_t seq = f & kSeqMask;
    if (seq == 0 || d >= kMaxDevices) return fail(KV_ERR_INVALID_ARG, "invalid fence %llu",
                                                  (unsigned long long)f);
    unsigned long long *words;
    uint64_t next;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_dev[d].init || seq >= g_next_seq)
            return fail(KV_ERR_INVALID_ARG, "fence %llu was never issued", (unsigned long long)f);
        words = g_dev[d].words;
        next = g_next_seq;
    }
    const int k = (int)(seq % kRing);
    const bool recycled = next - seq > (uint64_t)kRing;
    *done = recycled || load_acquire(&words[k]) >= seq;
    *aborted = !recycled && *done && load_acquire(&g_dev[d].status[k]) == seq;
    *dev = d;
    *slot = k;
    return KV_OK;
}

// -------------------------------------------------------------- validation

struct DupStamp {
    std::vector<uint32_t> stamp;
    uint32_t epoch = 0;
};
thread_local DupStamp t_dup;

kv_status check_ids(const char *what, const int32_t *ids, uint32_t n, uint64_t limit,
                    bool no_dups) {
    if (no_dups) {
        if (t_dup.stamp.size() < limit) t_dup.stamp.assign(limit, 0u);
        if (++t_dup.epoch == 0) {
            std::fill(t_dup.stamp.begin(), t_dup.stamp.end(), 0u);
            t_dup.epoch = 1;
        }
    }
    for (uint32_t i = 0; i < n; ++i) {
        const int32_t v = ids[i];
        if (v < 0 || (uint64_t)v >= limit)
            return fail(KV_ERR_OUT_OF_RANGE, "%s[%u] = %d is outside [0, %llu)", what, i, v,
                        (unsigned long long)limit);
        if (no_dups) {
            if (t_dup.stamp[v] == t_dup.epoch)
                return fail(KV_ERR_DUPLICATE, "%s[%u] = %d appears twice: one call may write a "
                            "page or slot only once", what, i, v);
            t_dup.stamp[v] = t_dup.epoch;
        }
    }
    return KV_OK;
}

// kind 0 = backup (a = src pages, b = slots), 1 = restore (a = slots, b = dst pages)
kv_status check_op(const Geo &g, uint64_t num_slots, int kind, const int32_t *a, const int32_t *b,
                   uint32_t n, int32_t layer) {
    if (kind != 0 && kind != 1) return fail(KV_ERR_INVALID_ARG, "unknown operation kind %d", kind);
    if (n > 0 && (a == nullptr || b == nullptr))
        return fail(KV_ERR_INVALID_ARG, "id arrays must be non-NULL when n = %u", n);
    if (n > (1u << 30)) return fail(KV_ERR_INVALID_ARG, "n = %u is too large", n);
    if (layer < -1 || (layer >= 0 && (uint64_t)layer >= g.L))
        return fail(KV_ERR_OUT_OF_RANGE, "layer %d is outside [-1, %llu)", layer,
                    (unsigned long long)g.L);
    if (kind == 0) {
        if (layer != -1) return fail(KV_ERR_INVALID_ARG, "backup always moves every layer");
        kv_status st = check_ids("src_pages", a, n, g.P, false);
        if (st != KV_OK) return st;
        return check_ids("host_slots", b, n, num_slots, true);
    }
    kv_status st = check_ids("host_slots", a, n, num_slots, false);
    if (st != KV_OK) return st;
    return check_ids("dst_pages", b, n, g.P, true);
}

// ------------------------------------------------------ overlapped ops

// Any library work on `stream` other than a zero-copy restore ends the run of
// restores there that a later one may overlap.  That work waits for the
// stream's previous kernel, whose completion implies every earlier restore of
// the run is in place (each published its fence only after its predecessor's).
void forget_stream(DevState &ds, void *stream) {
    if (!ds.chains.empty()) ds.chains.erase(stream);
}

// True when two sorted, duplicate-free page lists have no page in common.
bool sorted_disjoint(const std::vector<int32_t> &x, const std::vector<int32_t> &y) {
    size_t i = 0, j = 0;
    while (i < x.size() && j < y.size()) {
        if (x[i] == y[j]) return false;
        if (x[i] < y[j]) ++i; else ++j;
    }
    return true;
}

constexpr size_t kMaxChain = 256;   // ops of one run checked against a new one

// Whether ops x and y touch a common byte that one of them writes.  A backup
// reads the pool pages and writes the host slots it names (every layer); a
// restore reads the slots and writes the pages (one layer, or every layer).
// Two one-layer ops on different layers touch no common byte.
bool ops_conflict(const DevState::ChainOp &x, const DevState::ChainOp &y) {
    if (x.layer >= 0 && y.layer >= 0 && x.layer != y.layer) return false;
    const bool pool_written = x.kind == 1 || y.kind == 1;    // restores write the pool
    const bool host_written = x.kind == 0 || y.kind == 0;    // backups write the host tier
    if (pool_written && !sorted_disjoint(x.pages, y.pages)) return true;
    if (host_written && !sorted_disjoint(x.slots, y.slots)) return true;
    return false;
}

// Whether op `y` of `pool` on `stream` may overlap the run there; sets *pred to
// the run's last op (the fence it chains on).  Drops ops of the run whose fence
// the host already sees complete: their bytes are in place.
bool may_overlap(DevState &ds, void *stream, uint64_t pool, const DevState::ChainOp &y,
                 const DevState::ChainOp **pred) {
    auto it = ds.chains.find(stream);
    if (it == ds.chains.end() || it->second.pool != pool || it->second.ops.empty()) return false;
    std::vector<DevState::ChainOp> &ops = it->second.ops;
    size_t keep = 0;
    bool last_done = false;   // the last op stays as the chain's anchor even when done
    for (size_t i = 0; i < ops.size(); ++i) {
        const bool last = i + 1 == ops.size();
        const bool done = load_acquire(&ds.words[ops[i].k]) >= ops[i].seq;
        if (done && !last) continue;
        if (last) last_done = done;
        if (keep != i) ops[keep] = std::move(ops[i]);
        ++keep;
    }
    ops.resize(keep);
    if (ops.size() >= kMaxChain) return false;
    for (size_t i = 0; i < ops.size(); ++i) {
        if (i + 1 == ops.size() && last_done) break;   // its bytes are in place
        if (ops_conflict(ops[i], y)) return false;
    }
    *pred = &ops.back();
    return true;
}

// ---------------------------------------------------------- launch planning

Side pool_side(const PoolObj &p) {
    const Geo &g = p.g;
    Side s{};
    s.base = (uint64_t)(uintptr_t)p.dev;
    if (g.order == KV_PAGE_FIRST) {   // [P][L][C] chunks
        s.s_id = g.L * g.C * g.cb;
        s.s_l = g.C * g.cb;
        s.s_c = g.cb;
    } else {                          // [L][C][P] chunks
        s.s_id = g.cb;
        s.s_l = g.C * g.P * g.cb;
        s.s_c = g.P * g.cb;
    }
    s.hnd = g.heads;
    s.id_limit = (uint32_t)std::min<uint64_t>(g.P, 0xffffffffull);
    if (p.table_dev != nullptr) {     // split pool: [P][chunk] inside each buffer
        s.lc_base = p.table_dev;
        s.base = 0;
        s.s_id = g.cb;
        s.s_l = 0;
        s.s_c = 0;
    }
    return s;
}

Side host_side(const HostObj &h) {
    const Geo &g = h.g;
    Side s{};
    s.base = (uint64_t)(uintptr_t)h.dev_view;
    s.s_id = g.pb;                    // [S][L][C] chunks
    s.s_l = g.C * g.cb;
    s.s_c = g.cb;
    s.hnd = h.heads;
    s.id_limit = h.num_slots;
    return s;
}

// Staging buffer in host layout for items 0..m-1, layers [l0, l0+nl).
Side staging_side(char *base, const Geo &g, uint32_t heads, uint32_t nl, uint32_t l0,
                  uint32_t m) {
    Side s{};
    s.s_id = (uint64_t)nl * g.C * g.cb;
    s.s_l = g.C * g.cb;
    s.s_c = g.cb;
    s.base = (uint64_t)(uintptr_t)base - (uint64_t)l0 * s.s_l;   // index layers from l0
    s.hnd = heads;
    s.id_limit = m;
    return s;
}

struct Plan {
    MoveDesc d;
    uint32_t max_items;   // items per launch
    bool bulk = false;    // launch the bulk-copy kernel
    bool tsp = false;     // launch the transposing bulk kernel
    int threads = kMoveThreads;   // CTA size of the register kernel
};

// Which kernel a plan is for: the register kernel (kSegPieces x 16-byte warp
// segments), the bulk-copy kernel (identity chunks, kBulkBytes segments) or
// the transposing bulk kernel (one work item per chunk).
enum PlanKernel { PK_REG = 0, PK_BULK = 1, PK_TSP = 2 };

kv_status plan(const Geo &g, const Side &src, const Side &dst, uint32_t nl, uint32_t l0,
               uint32_t *err_dev, bool iter_dst, Plan *out, int kernel = PK_REG) {
    const bool bulk = kernel == PK_BULK;
    MoveDesc d{};
    d.src = src;
    d.dst = dst;
    d.nl = nl;
    d.l0 = l0;
    d.C = (uint32_t)g.C;
    d.cb16 = (uint32_t)(g.cb / 16);
    d.segs = kernel == PK_TSP ? 1u
             : bulk           ? (uint32_t)((g.cb + kBulkBytes - 1) / kBulkBytes)
                              : (d.cb16 + kSegPieces - 1) / kSegPieces;
    d.H = (uint32_t)g.H;
    d.T = (uint32_t)g.T;
    d.B16 = (uint32_t)(g.B / 16);
    d.transpose = (src.hnd != dst.hnd && g.H > 1 && g.T > 1) ? 1u : 0u;
    d.iter_dst = iter_dst ? 1u : 0u;
    const uint64_t per_item = (uint64_t)nl * g.C * d.segs;
    if (per_item == 0 || per_item > 0xffffffffull || (uint64_t)nl * g.C > 0xffffffffull)
        return fail(KV_ERR_LAYOUT, "one page needs %llu warp segments: too large",
                    (unsigned long long)per_item);
    // keep every launch's segment count below 2^31 so no grid-stride index wraps
    uint64_t m = 0x7fffffffull / per_item;
    if (m == 0)
        return fail(KV_ERR_LAYOUT, "one page needs %llu segments: too large",
                    (unsigned long long)per_item);
    out->max_items = (uint32_t)std::min<uint64_t>(m, (uint64_t)kMaxItems);
    out->bulk = bulk;
    out->tsp = kernel == PK_TSP;
    d.div_segs = make_fastdiv(d.segs);
    d.div_lc = make_fastdiv(nl * d.C);
    d.div_c = make_fastdiv(d.C);
    d.div_b16 = make_fastdiv(d.B16);
    d.div_T = make_fastdiv(d.T);
    d.div_H = make_fastdiv(d.H);
    d.err = err_dev;
    out->d = d;
    return KV_OK;
}

// CTAs of a move kernel.  Host-link moves saturate the link with few threads
// (measured on GB300: 16 CTAs of 256 threads reach the D2H peak, 32 the H2D
// peak; every shape from 8 x 1024 to 64 x 256 reaches both solo peaks).  The
// shape matters when a backup and a restore run at once, and there the best
// shape depends on the kernel variant: moves that change head order (the
// TRT-LLM HND pool) reach 338-341 GB/s, 99-100% of the bidirectional memcpy
// peak, with 64 CTAs of 256 per direction on every box measured (16 x 1024:
// 246-338 from box to box), while identity moves reach 322-326 GB/s with 16
// CTAs of 1024 (64 x 256: 305-310; more warps in flight per direction, e.g.
// 32 x 1024 or 128 x 256, lose on every layout: 292-301).  Compute beside the
// moves runs as fast with either shape (one-layer restores pipelined with a
// GEMM per layer: 3.75 ms; write-through backups: within 1%).  HBM-only moves
// use 4 CTAs of 256 per SM.
constexpr int kLinkCtas = 64;       // CTAs of kMoveThreads
constexpr int kLinkWideCtas = 16;   // CTAs of kWideThreads (cta_threads = 1024)
// Progressive layer restores exist to run beside each layer's forward: 8 wide
// CTAs (8 SMs) still reach 98% of the H2D peak and cut the time of a 61-layer
// restore pipelined with a per-layer GEMM from 4.26 ms (16 CTAs) to 3.54 ms.
constexpr int kOverlapWideCtas = 8;
// Overlapped restores (KV_CFG_OVERLAP_RESTORES) keep the link busy across
// calls, so fewer SMs carry it: 61 one-layer restores on GB300 (MLA pool;
// TRT-LLM HND pool) reach 98.8% / 98.7% of the H2D peak with 6 wide CTAs
// alone, and pipelined with a GEMM per layer take 3.69 / 2.47 ms, as fast as
// non-overlapped calls (3.70 / 2.44); 8 CTAs: 99.3% alone but 3.76 / 2.57 ms
// pipelined; 16: 4.03 / 2.56 ms; 4: 88.8% alone.  Head-order changes use
// 1,024-thread CTAs here too (32 x 256: 2.66 ms pipelined).
constexpr int kOverlapRestoreCtas = 6;

int link_threads(bool transpose) {
    if (g_cfg.cta_threads) return (int)g_cfg.cta_threads;
    return transpose ? kMoveThreads : kWideThreads;
}
int progressive_threads() {
    return g_cfg.cta_threads ? (int)g_cfg.cta_threads : kWideThreads;
}

// Turns a plan into a progressive multi-layer plan for n items (one launch).
kv_status plan_layer_major(Plan &p, uint32_t n, const DevState &ds, uint64_t seq0,
                           bool device_ids = false) {
    MoveDesc &d = p.d;
    const uint64_t pls = (uint64_t)n * d.C * d.segs;
    if ((n > p.max_items && !device_ids) || pls * d.nl > 0x7fffffffull || pls == 0)
        return fail(KV_ERR_OUT_OF_RANGE, "%u pages x %u layers is too large for one progressive "
                    "restore", n, d.nl);
    d.layer_major = 1;
    d.per_layer_segs = (uint32_t)pls;
    d.div_pls = make_fastdiv((uint32_t)pls);
    d.div_cs = make_fastdiv(d.C * d.segs);
    d.lay_words = ds.words_dev;
    d.lay_seq0 = seq0;
    d.lay_ring = kRing;
    const uint32_t k_last = (uint32_t)((seq0 + d.nl - 1) % kRing);
    d.lay_done = ds.aux;                        // done[k] for each layer's slot k
    d.lay_published = ds.aux + kRing + k_last;
    d.lay_work = ds.aux + 2 * kRing + k_last;
    d.lay_lock = ds.aux + 3 * kRing + k_last;
    return KV_OK;
}

int default_ctas(const DevState &s, bool touches_host, int kernel = PK_REG,
                 int link_cta_threads = kMoveThreads) {
    if (g_cfg.max_ctas != 0) return (int)g_cfg.max_ctas;
    if (kernel == PK_BULK) return 3 * s.sms;   // 3 x 64 KiB rings fit one SM's shared memory
    if (kernel == PK_TSP) return s.sms;        // one 192 KiB ring per SM
    if (!touches_host) return 4 * s.sms;
    return link_cta_threads == kWideThreads ? std::min(kLinkWideCtas, s.sms)
                                          : std::min(kLinkCtas, 4 * s.sms);
}

// HBM-only moves go through the bulk-copy kernels unless the caller turned
// them off (KV_CFG_NO_BULK): identity chunks through kv_bulk_kernel, chunks
// whose head order changes (and fit the shared-memory ring) through
// kv_tsp_kernel, the rest through the register kernel.
int hbm_kernel(const Geo &g, const Side &a, const Side &b) {
    if ((g_cfg.flags & KV_CFG_NO_BULK) != 0) return PK_REG;
    const bool transpose = a.hnd != b.hnd && g.H > 1 && g.T > 1;
    if (!transpose) return PK_BULK;
    return g.cb <= kTspMaxChunk ? PK_TSP : PK_REG;
}

// Launches the move for items [0, n) of (a, b) in slices of at most max_items.
// b_is_index: the destination id of item i is i itself (a staging position).
// fence: when non-null, the last slice's kernel completes that fence itself.
kv_status run_moves(Plan &p, const int32_t *a, const int32_t *b, uint32_t n, int ctas_cap,
                    cudaStream_t stream, bool b_is_index, const DevState *ds = nullptr,
                    const FenceSlot *fence = nullptr) {
    static thread_local MoveIds ids;
    if (p.d.gid_a != nullptr) {   // ids already in device memory: one launch for all n
        p.d.fence_word = nullptr;
        p.d.fence_count = nullptr;
        p.d.n = n;
        p.d.total_segs = n * p.d.nl * p.d.C * p.d.segs;
        const uint32_t per_cta = (uint32_t)(p.threads / 32);
        const uint64_t need = ((uint64_t)p.d.total_segs + per_cta - 1) / per_cta;
        const int ctas = (int)std::max<uint64_t>(1, std::min<uint64_t>(need, (uint64_t)ctas_cap));
        if (fault_hit(FP_LAUNCH) || fault_hit(FP_LAUNCH_NTH))
            return fail(KV_ERR_CUDA, "launch of the move kernel: injected failure");
        cudaError_t e = launch_move(p.d, ids, ctas, p.threads, stream);
        if (e != cudaSuccess) return cuda_fail(e, "launch of the move kernel");
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return KV_OK;
    }
    // Only an op's first launch overlaps its start with the previous kernel's
    // end (programmatic dependent launch); the further slices of an op above
    // kMaxItems pages launch plainly: with a move in the other direction running
    // at once, early-launched slices cost the pair 5% of its throughput
    // (310 vs 325 GB/s for 4,096 x 1 MiB both ways), and one op gains nothing
    // from overlapping its own slices' launches.
    const uint32_t pdl0 = p.d.pdl;
    unsigned long long *const ext_word = p.d.ext_word;   // the last slice's, with the fence
    for (uint32_t i0 = 0; i0 < n; i0 += p.max_items) {
        const uint32_t m = std::min(p.max_items, n - i0);
        const bool last = i0 + m >= n;
        p.d.pdl = i0 == 0 ? pdl0 : 0u;
        if (last && fence != nullptr) {
            p.d.fence_word = ds->words_dev + fence->k;
            p.d.fence_seq = fence->seq;
            p.d.fence_count = ds->counters + fence->k;
            p.d.ext_word = ext_word;
        } else {
            p.d.fence_word = nullptr;
            p.d.fence_count = nullptr;
            p.d.ext_word = nullptr;
        }
        std::memcpy(ids.a, a + i0, m * sizeof(int32_t));
        if (b_is_index)
            for (uint32_t k = 0; k < m; ++k) ids.b[k] = (int32_t)(i0 + k);
        else
            std::memcpy(ids.b, b + i0, m * sizeof(int32_t));
        p.d.n = m;
        p.d.total_segs = m * p.d.nl * p.d.C * p.d.segs;
        const uint32_t per_cta = (p.bulk || p.tsp) ? 1u : (uint32_t)(p.threads / 32);
        const uint64_t need = ((uint64_t)p.d.total_segs + per_cta - 1) / per_cta;
        const int ctas = (int)std::max<uint64_t>(1, std::min<uint64_t>(need, (uint64_t)ctas_cap));
        if ((i0 == 0 && fault_hit(FP_LAUNCH)) || fault_hit(FP_LAUNCH_NTH)) {
            p.d.pdl = pdl0;
            return fail(KV_ERR_CUDA, "launch of the move kernel: injected failure");
        }
        cudaError_t e = p.tsp    ? launch_tsp(p.d, ids, ctas, stream)
                        : p.bulk ? launch_bulk(p.d, ids, ctas, stream)
                                 : launch_move(p.d, ids, ctas, p.threads, stream);
        if (e != cudaSuccess) {
            p.d.pdl = pdl0;
            return cuda_fail(e, "launch of the move kernel");
        }
        g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    p.d.pdl = pdl0;
    p.d.ext_word = ext_word;
    return KV_OK;
}

kv_status ensure_staging(DevState &s) {
    const uint64_t want = g_cfg.staging_bytes ? g_cfg.staging_bytes : kDefaultStaging;
    if (s.staging != nullptr && s.staging_bytes == want) return KV_OK;
    if (s.staging != nullptr) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize (staging resize)");
        cudaFree(s.staging);
        s.staging = nullptr;
        s.staging_used[0] = s.staging_used[1] = false;
    }
    void *p = nullptr;
    if (fault_hit(FP_STAGING_ALLOC))
        return fail(KV_ERR_NO_MEMORY, "staging buffer of %llu bytes: injected failure",
                    (unsigned long long)want);
    cudaError_t e = cudaMalloc(&p, want);
    if (e != cudaSuccess) return fail(KV_ERR_NO_MEMORY, "staging buffer of %llu bytes: %s",
                                      (unsigned long long)want, cudaGetErrorString(e));
    s.staging = (char *)p;
    s.staging_bytes = want;
    auto make_event = [](cudaEvent_t *ev) {
        return *ev != nullptr ? cudaSuccess : cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    };
    for (int h = 0; h < 2; ++h) {
        e = make_event(&s.staging_free[h]);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            e = make_event(&s.moved[h][b]);
            if (e == cudaSuccess) e = make_event(&s.copied[h][b]);
        }
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate(staging)");
    }
    if (e == cudaSuccess) e = make_event(&s.op_start);
    for (int h = 0; h < 2 && e == cudaSuccess; ++h)
        if (s.side[h] == nullptr) e = cudaStreamCreateWithFlags(&s.side[h], cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "staging stream / events");
    return KV_OK;
}

// Puts the ids of a progressive restore of more than kMaxItems pages into the
// device buffer (a at [0, n), b at [n, 2n)): host copy into the pinned buffer,
// then one copy to the device on `stream`.  The previous large restore's kernel
// must be done with the device buffer (stream wait on gids_free) and its copy
// done with the pinned buffer (host wait on gids_copied, normally long done).
kv_status stage_ids(DevState &s, const int32_t *a, const int32_t *b, uint32_t n,
                    cudaStream_t stream) {
    const uint64_t need = 2ull * n;
    cudaError_t e = cudaSuccess;
    auto make_event = [](cudaEvent_t *ev) {
        return *ev != nullptr ? cudaSuccess : cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    };
    e = make_event(&s.gids_copied);
    if (e == cudaSuccess) e = make_event(&s.gids_free);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate(ids)");
    if (s.gids_used) {
        e = cudaEventSynchronize(s.gids_copied);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, s.gids_free, 0);
        if (e != cudaSuccess) return cuda_fail(e, "waiting for the id buffers");
    }
    if (need > s.gids_cap) {
        if (s.gids_used) {   // nothing may still read the old buffers
            e = cudaEventSynchronize(s.gids_free);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize(ids)");
        }
        if (s.gids) cudaFree(s.gids);
        if (s.gids_host) cudaFreeHost(s.gids_host);
        s.gids = nullptr;
        s.gids_host = nullptr;
        s.gids_cap = 0;
        const uint64_t cap = std::max<uint64_t>(need, 1ull << 16);
        void *dptr = nullptr, *hptr = nullptr;
        e = cudaMalloc(&dptr, cap * sizeof(int32_t));
        if (e == cudaSuccess) e = cudaHostAlloc(&hptr, cap * sizeof(int32_t), cudaHostAllocDefault);
        if (e != cudaSuccess) {
            if (dptr) cudaFree(dptr);
            return fail(KV_ERR_NO_MEMORY, "id buffers of %llu entries: %s",
                        (unsigned long long)cap, cudaGetErrorString(e));
        }
        s.gids = (int32_t *)dptr;
        s.gids_host = (int32_t *)hptr;
        s.gids_cap = cap;
    }
    std::memcpy(s.gids_host, a, (size_t)n * sizeof(int32_t));
    std::memcpy(s.gids_host + n, b, (size_t)n * sizeof(int32_t));
    e = cudaMemcpyAsync(s.gids, s.gids_host, need * sizeof(int32_t), cudaMemcpyHostToDevice,
                        stream);
    if (e == cudaSuccess) e = cudaEventRecord(s.gids_copied, stream);
    if (e != cudaSuccess) return cuda_fail(e, "copying the ids to the device");
    // From here the next large restore waits for this copy (host buffer) and for
    // gids_free, which the caller records after its launch, failed or not.
    s.gids_used = true;
    return KV_OK;
}

// Copies between a host tier and the staging buffer, one memcpy per run of
// consecutive slots.  `lb` = bytes per item moved (whole page or one layer),
// `host_off` = byte offset of the moved part inside a slot.
kv_status staged_copies(const HostObj &h, char *staging, const int32_t *slots, uint32_t m,
                        uint64_t lb, uint64_t host_off, bool to_host, cudaStream_t stream) {
    const uint64_t pb = h.g.pb;
    uint32_t i = 0;
    while (i < m) {
        uint32_t j = i + 1;
        while (j < m && slots[j] == slots[j - 1] + 1) ++j;
        const uint32_t run = j - i;
        char *hp = h.host + (uint64_t)slots[i] * pb + host_off;
        char *sp = staging + (uint64_t)i * lb;
        cudaError_t e;
        if (lb == pb) {
            e = to_host ? cudaMemcpyAsync(hp, sp, run * lb, cudaMemcpyDeviceToHost, stream)
                        : cudaMemcpyAsync(sp, hp, run * lb, cudaMemcpyHostToDevice, stream);
        } else {
            e = to_host ? cudaMemcpy2DAsync(hp, pb, sp, lb, lb, run, cudaMemcpyDeviceToHost, stream)
                        : cudaMemcpy2DAsync(sp, lb, hp, pb, lb, run, cudaMemcpyHostToDevice, stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "staged cudaMemcpyAsync");
        i = j;
    }
    return KV_OK;
}

// One (page, layer, component) chunk between the pool and a host slot through
// the copy engine.  Same head order (or H = 1 or T = 1): one copy of cb bytes.
// Otherwise the chunk is transposed with min(H, T) pitched copies of B-byte
// rows: per head, T rows; or per token, H rows.
kv_status ce_chunk(const Geo &g, char *dst, uint32_t dst_hnd, const char *src, uint32_t src_hnd,
                   cudaMemcpyKind kind, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    const uint64_t B = g.B, H = g.H, T = g.T;
    if (src_hnd == dst_hnd || H == 1 || T == 1) {
        e = cudaMemcpyAsync(dst, src, g.cb, kind, stream);
    } else if (H <= T) {
        // per head h: the T vectors are contiguous in HND ([H][T][B]) and H*B apart in NHD
        for (uint64_t h = 0; h < H && e == cudaSuccess; ++h) {
            const bool to_nhd = dst_hnd == KV_NHD;
            char *dp = dst + (to_nhd ? h * B : h * T * B);
            const char *sp = src + (to_nhd ? h * T * B : h * B);
            e = cudaMemcpy2DAsync(dp, to_nhd ? H * B : B, sp, to_nhd ? B : H * B, B, T, kind,
                                  stream);
        }
    } else {
        // per token t: the H vectors are contiguous in NHD ([T][H][B]) and T*B apart in HND
        for (uint64_t t = 0; t < T && e == cudaSuccess; ++t) {
            const bool to_nhd = dst_hnd == KV_NHD;
            char *dp = dst + (to_nhd ? t * H * B : t * B);
            const char *sp = src + (to_nhd ? t * B : t * H * B);
            e = cudaMemcpy2DAsync(dp, to_nhd ? B : T * B, sp, to_nhd ? T * B : B, B, H, kind,
                                  stream);
        }
    }
    return e == cudaSuccess ? KV_OK : cuda_fail(e, "copy-engine cudaMemcpy*Async");
}

// KV_MODE_COPY_ENGINE: the backup (pool -> host) or restore (host -> pool) of
// items [0, n), layers [l0, l0 + nl), issued as copy-engine copies of the
// pinned host tier.  `pages` / `slots` are the validated ids.  One contiguous
// pool with the host's head order: one pitched copy per item (its nl x C
// chunks are evenly spaced on both sides), or one copy for a run of items whose
// pages and slots both step by one and whose spans are contiguous.  Split pools
// and head-order changes: per chunk (ce_chunk).
kv_status ce_copies(const PoolObj &pool, const HostObj &host, bool backup, const int32_t *pages,
                    const int32_t *slots, uint32_t n, uint32_t nl, uint32_t l0,
                    cudaStream_t stream) {
    const Geo &g = pool.g;
    const cudaMemcpyKind kind = backup ? cudaMemcpyDeviceToHost : cudaMemcpyHostToDevice;
    const Side ps = pool_side(pool);
    const uint64_t nchunks = (uint64_t)nl * g.C;
    const bool same_heads = pool.g.heads == host.heads || g.H == 1 || g.T == 1;
    auto dev_chunk = [&](uint64_t p, uint64_t l, uint64_t c) -> char * {
        if (!pool.table_host.empty())
            return (char *)(uintptr_t)pool.table_host[l * g.C + c] + p * g.cb;
        return pool.dev + p * ps.s_id + l * ps.s_l + c * ps.s_c;
    };
    auto host_chunk = [&](uint64_t s, uint64_t l, uint64_t c) -> char * {
        return host.host + s * g.pb + (l * g.C + c) * g.cb;
    };
    if (!same_heads || !pool.table_host.empty()) {
        for (uint32_t i = 0; i < n; ++i)
            for (uint64_t l = l0; l < l0 + nl; ++l)
                for (uint64_t c = 0; c < g.C; ++c) {
                    char *dp = dev_chunk((uint64_t)pages[i], l, c);
                    char *hp = host_chunk((uint64_t)slots[i], l, c);
                    kv_status st = backup ? ce_chunk(g, hp, host.heads, dp, pool.g.heads, kind, stream)
                                          : ce_chunk(g, dp, pool.g.heads, hp, host.heads, kind, stream);
                    if (st != KV_OK) return st;
                }
        return KV_OK;
    }
    // chunk j = (l - l0) * C + c sits at j * s_c in the pool (s_l = C * s_c in both
    // orders) and at j * cb in the slot
    const uint64_t dev_pitch = ps.s_c;
    const bool contiguous = nchunks == 1 || dev_pitch == g.cb;   // one run on both sides
    const uint64_t span = nchunks * g.cb;
    const bool mergeable = contiguous && ps.s_id == span && g.pb == span;
    for (uint32_t i = 0; i < n;) {
        uint32_t j = i + 1;
        if (mergeable)
            while (j < n && pages[j] == pages[j - 1] + 1 && slots[j] == slots[j - 1] + 1) ++j;
        char *dp = dev_chunk((uint64_t)pages[i], l0, 0);
        char *hp = host_chunk((uint64_t)slots[i], l0, 0);
        cudaError_t e;
        if (contiguous) {
            const uint64_t bytes = (uint64_t)(j - i) * span;
            e = backup ? cudaMemcpyAsync(hp, dp, bytes, kind, stream)
                       : cudaMemcpyAsync(dp, hp, bytes, kind, stream);
        } else {
            e = backup ? cudaMemcpy2DAsync(hp, g.cb, dp, dev_pitch, g.cb, nchunks, kind, stream)
                       : cudaMemcpy2DAsync(dp, dev_pitch, hp, g.cb, g.cb, nchunks, kind, stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "copy-engine cudaMemcpy*Async");
        i = j;
    }
    return KV_OK;
}

// Issues one backup (kind 0) or restore (kind 1).  g_mu held.
// `ready` (device-visible, or NULL): BACKUP's ready_fence -- the move starts
// only once *ready >= ready_value, waited for on the GPU for at most
// ready_timeout_ns; on time-out nothing moves and the fence reports ABORTED.
// `ext_word` (device-visible, or NULL): a second completion word the move
// kernel stores `ext_value` to right after the fence; *ext_fused says whether
// it could (a zero-copy op with pages to move).
kv_status issue(kv_pool pool_h, kv_host host_h, int kind, const int32_t *a, const int32_t *b,
                uint32_t n, int32_t layer, void *stream_v, kv_fence *fence,
                const unsigned long long *ready = nullptr, uint64_t ready_value = 0,
                uint64_t ready_timeout_ns = 0, unsigned long long *ext_word = nullptr,
                uint64_t ext_value = 0, int *ext_fused = nullptr) {
    if (ext_fused != nullptr) *ext_fused = 0;
    if (fence == nullptr) return fail(KV_ERR_INVALID_ARG, "fence output pointer is NULL");
    if (pool_h == nullptr || host_h == nullptr)
        return fail(KV_ERR_INVALID_ARG, "pool or host handle is NULL");
    PoolObj *pool = find_pool(pool_h);
    if (pool == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    HostObj *host = find_host(host_h);
    if (host == nullptr) return fail(KV_ERR_CLOSED, "host handle is closed or unknown");
    auto fl = g_floor.find(pool->instance_id);
    if (fl != g_floor.end() && pool->generation < fl->second)
        return fail(KV_ERR_STALE, "pool generation %llu of instance %llu is retired (floor %llu)",
                    (unsigned long long)pool->generation, (unsigned long long)pool->instance_id,
                    (unsigned long long)fl->second);
    if (!same_slot_geometry(pool->g, host->g))
        return fail(KV_ERR_LAYOUT, "pool and host tier have different page geometry");
    kv_status st = check_op(pool->g, host->num_slots, kind, a, b, n, layer);
    if (st != KV_OK) return st;

    const int d = pool->device;
    DeviceGuard guard(d);
    st = init_device(d);
    if (st != KV_OK) return st;
    DevState &ds = g_dev[d];
    cudaStream_t stream = (cudaStream_t)stream_v;
    const bool backup = kind == 0;
    const uint32_t nl = layer < 0 ? (uint32_t)pool->g.L : 1u;
    const uint32_t l0 = layer < 0 ? 0u : (uint32_t)layer;
    FenceSlot fs;
    st = reserve_fence(d, &fs);
    if (st != KV_OK) return st;
    // A gate on the stream records a give-up under the op's sequence number.  Once
    // it is launched, a failure further on must not hand that number to the next
    // op (whose moves the stale record would skip): the number is consumed.
    bool gated = false;
    auto gate = [&]() -> kv_status {
        cudaError_t e = launch_gate(ready, ready_value, ready_timeout_ns, ds.status_dev + fs.k,
                                    fs.seq, stream);
        if (e != cudaSuccess) return cuda_fail(e, "launch of the ready-fence gate");
        g_launches.fetch_add(1, std::memory_order_relaxed);
        gated = true;
        return KV_OK;
    };
    auto bail = [&](kv_status err) {
        if (gated) g_next_seq = fs.seq + 1;
        return err;
    };
    bool fused = false;

    // Overlapped ops (KV_CFG_OVERLAP_RESTORES, KV_CFG_OVERLAP_BACKUPS): a
    // zero-copy op may start moving while the previous kernel on its stream
    // still runs when that kernel is the last op this library issued there, of
    // the same pool, and the new op conflicts with no unfinished op of the run
    // (ops_conflict: no common byte that one of them writes).
    const uint32_t kind_flag = backup ? KV_CFG_OVERLAP_BACKUPS : KV_CFG_OVERLAP_RESTORES;
    const bool overlap_cfg = (g_cfg.flags & kind_flag) != 0 &&
                             (g_cfg.flags & KV_CFG_NO_PDL) == 0;
    // Not on the legacy default stream nor the special handles (0, 1, 2): the
    // legacy stream also waits on every blocking stream, so work the library
    // cannot see may sit between two of its ops there.
    const bool plain_stream = (uintptr_t)stream_v > 2u;
    const bool run_kind = ready == nullptr && n > 0 && g_cfg.mode == KV_MODE_ZERO_COPY &&
                          plain_stream;   // an op that may take part in a run
    bool chain = false, overlapped = false;
    int chain_k = 0;
    uint64_t chain_seq = 0;
    static thread_local DevState::ChainOp me;
    if (overlap_cfg && run_kind) {
        const int32_t *pages = backup ? a : b, *slots = backup ? b : a;
        me.kind = backup ? 0 : 1;
        me.layer = layer;
        me.pages.assign(pages, pages + n);
        me.slots.assign(slots, slots + n);
        std::sort(me.pages.begin(), me.pages.end());
        std::sort(me.slots.begin(), me.slots.end());
        // a backup's source pages may repeat (duplicate sources are allowed)
        me.pages.erase(std::unique(me.pages.begin(), me.pages.end()), me.pages.end());
        const DevState::ChainOp *pred = nullptr;
        if (may_overlap(ds, stream_v, handle_id(pool_h), me, &pred)) {
            chain = true;
            chain_k = pred->k;
            chain_seq = pred->seq;
        }
    }
    // the stream's run, kept aside: re-recorded below once this op is committed
    DevState::Chain run;
    if (chain) run = std::move(ds.chains[stream_v]);
    forget_stream(ds, stream_v);

    if (n > 0 && (g_cfg.mode == KV_MODE_ZERO_COPY || ready != nullptr)) {
        const Side ps = pool_side(*pool), hs = host_side(*host);
        Plan p;
        st = plan(pool->g, backup ? ps : hs, backup ? hs : ps, nl, l0, ds.err_dev,
                  /*iter_dst=*/backup, &p);
        if (st != KV_OK) return st;
        if (ready != nullptr) {
            st = gate();
            if (st != KV_OK) return st;
            p.d.skip_word = ds.status_dev + fs.k;
            p.d.skip_tag = fs.seq;
        }
        p.threads = link_threads(p.d.transpose != 0);
        if (overlap_cfg && run_kind && g_cfg.cta_threads == 0) p.threads = kWideThreads;
        p.d.pdl = (g_cfg.flags & KV_CFG_NO_PDL) ? 0u : 1u;
        if (overlap_cfg && run_kind) {
            p.d.early_trigger = 1u;
            // one launch only: the op's fence and its overlap sit in the same kernel
            if (chain && n <= p.max_items) {
                p.d.overlap = 1u;
                p.d.chain_word = ds.words_dev + chain_k;
                p.d.chain_seq = fault_hit(FP_CHAIN_STALL) ? ~0ull : chain_seq;
                overlapped = true;
            }
        }
        p.d.ext_word = ext_word;
        p.d.ext_value = ext_value;
        int ctas = default_ctas(ds, true, PK_REG, p.threads);
        if (overlap_cfg && run_kind && g_cfg.max_ctas == 0)
            ctas = p.threads == kWideThreads ? std::min(kOverlapRestoreCtas, ds.sms)
                                             : std::min(4 * kOverlapRestoreCtas, 4 * ds.sms);
        st = run_moves(p, a, b, n, ctas, stream, false, &ds, &fs);
        if (st != KV_OK) return bail(st);
        fused = true;
    } else if (ready != nullptr) {   // an empty gated op: its fence follows the gate
        st = gate();
        if (st != KV_OK) return st;
    } else if (n > 0 && g_cfg.mode == KV_MODE_COPY_ENGINE) {
        st = backup ? ce_copies(*pool, *host, true, a, b, n, nl, l0, stream)
                    : ce_copies(*pool, *host, false, b, a, n, nl, l0, stream);
        if (st != KV_OK) return st;
    } else if (n > 0) {
        st = ensure_staging(ds);
        if (st != KV_OK) return st;
        // STAGED: the op is cut into chunks (layer groups x item slices) that fit
        // one of the half's two ping-pong buffers.  Backup: the gather of chunk k
        // (HBM kernel, side stream) runs while chunk k-1 crosses the host link
        // (copy engine, caller's stream); restore: the copy of chunk k runs while
        // chunk k-1 is scattered.  Events order each buffer's reuse; the op ends
        // on the caller's stream (its fence and the half's staging_free event).
        const int half = backup ? 0 : 1;
        const uint64_t half_bytes = ds.staging_bytes / 2;
        const uint64_t buf_bytes = (half_bytes / 2) & ~(uint64_t)255;
        char *const bufs[2] = {ds.staging + (uint64_t)half * half_bytes,
                               ds.staging + (uint64_t)half * half_bytes + buf_bytes};
        const uint64_t layer_bytes = pool->g.C * pool->g.cb;        // one layer of one page
        // layers per group: the whole range if one page fits, else as many as fit
        const uint32_t gl = (uint32_t)std::min<uint64_t>(nl, buf_bytes / layer_bytes);
        if (gl == 0)
            return fail(KV_ERR_NO_MEMORY, "staging buffer of %llu bytes holds no layer of %llu "
                        "bytes", (unsigned long long)buf_bytes, (unsigned long long)layer_bytes);
        const uint64_t lb = (uint64_t)gl * layer_bytes;              // staged bytes per item
        const uint32_t fit = (uint32_t)std::min<uint64_t>(buf_bytes / lb, n);   // items per fill
        const uint64_t chunks = (uint64_t)((nl + gl - 1) / gl) * ((n + fit - 1) / fit);
        const bool pipelined = chunks > 1;
        cudaStream_t ks = pipelined ? ds.side[half] : stream;        // kernels' stream
        auto ck = [](cudaError_t e, const char *what) {
            return e == cudaSuccess ? KV_OK : cuda_fail(e, what);
        };
        if (ds.staging_used[half])
            st = ck(cudaStreamWaitEvent(stream, ds.staging_free[half], 0),
                    "cudaStreamWaitEvent(staging)");
        if (st == KV_OK && pipelined) {
            st = ck(cudaEventRecord(ds.op_start, stream), "cudaEventRecord(staging start)");
            if (st == KV_OK)
                st = ck(cudaStreamWaitEvent(ks, ds.op_start, 0), "cudaStreamWaitEvent(staging)");
        }
        if (st != KV_OK) return st;
        const Side ps = pool_side(*pool);
        static thread_local std::vector<int32_t> idx;
        // A failure after chunks were enqueued: the caller's stream still waits for
        // every kernel already on the side stream and marks the half busy until
        // then, so the next op of this direction cannot reuse a buffer in use.
        auto fail_after_enqueue = [&](kv_status err) {
            if (pipelined && cudaEventRecord(ds.op_start, ks) == cudaSuccess)
                (void)cudaStreamWaitEvent(stream, ds.op_start, 0);
            if (cudaEventRecord(ds.staging_free[half], stream) == cudaSuccess)
                ds.staging_used[half] = true;
            return err;
        };
        uint64_t k = 0;
        for (uint32_t la = l0; la < l0 + nl; la += gl) {
            const uint32_t g_n = std::min(gl, l0 + nl - la);          // layers in this group
            const uint64_t host_off = (uint64_t)la * layer_bytes;
            const uint64_t gb = (uint64_t)g_n * layer_bytes;
            for (uint32_t i0 = 0; i0 < n; i0 += fit, ++k) {
                const uint32_t m = std::min(fit, n - i0);
                const int bi = (int)(k & 1);
                char *stg = bufs[bi];
                const Side ss = staging_side(stg, pool->g, host->heads, g_n, la, m);
                const int kernel = hbm_kernel(pool->g, ps, ss);
                Plan p;
                st = plan(pool->g, backup ? ps : ss, backup ? ss : ps, g_n, la, ds.err_dev, backup,
                          &p, kernel);
                if (st != KV_OK) return k ? fail_after_enqueue(st) : st;
                const int ctas = default_ctas(ds, false, kernel);
                if (backup) {
                    if (pipelined && k >= 2)   // chunk k-2's copy has left this buffer
                        st = ck(cudaStreamWaitEvent(ks, ds.copied[half][bi], 0), "staging wait");
                    if (st == KV_OK) st = run_moves(p, a + i0, nullptr, m, ctas, ks, true);
                    if (st == KV_OK && pipelined) {
                        st = ck(cudaEventRecord(ds.moved[half][bi], ks), "staging record");
                        if (st == KV_OK)
                            st = ck(cudaStreamWaitEvent(stream, ds.moved[half][bi], 0),
                                    "staging wait");
                    }
                    if (st == KV_OK)
                        st = staged_copies(*host, stg, b + i0, m, gb, host_off, true, stream);
                    if (st == KV_OK && pipelined)
                        st = ck(cudaEventRecord(ds.copied[half][bi], stream), "staging record");
                } else {
                    if (pipelined && k >= 2)   // chunk k-2's scatter has read this buffer
                        st = ck(cudaStreamWaitEvent(stream, ds.moved[half][bi], 0), "staging wait");
                    if (st == KV_OK)
                        st = staged_copies(*host, stg, a + i0, m, gb, host_off, false, stream);
                    if (st == KV_OK && pipelined) {
                        st = ck(cudaEventRecord(ds.copied[half][bi], stream), "staging record");
                        if (st == KV_OK)
                            st = ck(cudaStreamWaitEvent(ks, ds.copied[half][bi], 0),
                                    "staging wait");
                    }
                    if (st == KV_OK) {
                        // staging item j -> dst page b[i0 + j]: a = staging index, b = page
                        idx.resize(m);
                        for (uint32_t j = 0; j < m; ++j) idx[j] = (int32_t)j;
                        st = run_moves(p, idx.data(), b + i0, m, ctas, ks, false);
                    }
                    if (st == KV_OK && pipelined)
                        st = ck(cudaEventRecord(ds.moved[half][bi], ks), "staging record");
                }
                if (st != KV_OK) return fail_after_enqueue(st);
            }
        }
        if (pipelined && !backup) {   // the last scatters end on the caller's stream too
            for (int bi = 0; bi < 2 && st == KV_OK; ++bi)
                st = ck(cudaStreamWaitEvent(stream, ds.moved[half][bi], 0), "staging wait");
            if (st != KV_OK) return fail_after_enqueue(st);
        }
        cudaError_t e = cudaEventRecord(ds.staging_free[half], stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(staging)");
        ds.staging_used[half] = true;
    }
    st = commit_fence(d, fs, !fused, stream, fence);
    if (st != KV_OK) return bail(st);
    if (ext_fused != nullptr) *ext_fused = fused && ext_word != nullptr ? 1 : 0;
    if (overlapped) g_overlapped.fetch_add(1, std::memory_order_relaxed);
    if (overlap_cfg && run_kind && fused) {
        // an op that did not overlap waited for all before it: it starts a new run
        if (!overlapped) run.ops.clear();
        run.pool = handle_id(pool_h);
        me.k = fs.k;
        me.seq = fs.seq;
        run.ops.push_back(me);
        if (ds.chains.size() >= 4096) ds.chains.clear();   // streams come and go
        ds.chains[stream_v] = std::move(run);
    }
    return KV_OK;
}

// Device gather (kind 0) / scatter (kind 1) between the pool and a caller's
// device buffer in host-tier layout.  g_mu held.  fence == NULL: stream order
// only -- no fence is reserved and the kernel skips the fused completion.
kv_status issue_device(kv_pool pool_h, void *buf, uint64_t buf_bytes, uint32_t buf_heads, int kind,
                       const int32_t *pages, uint32_t n, int32_t layer, void *stream_v,
                       kv_fence *fence) {
    if (pool_h == nullptr) return fail(KV_ERR_INVALID_ARG, "pool handle is NULL");
    PoolObj *pool = find_pool(pool_h);
    if (pool == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    auto fl = g_floor.find(pool->instance_id);
    if (fl != g_floor.end() && pool->generation < fl->second)
        return fail(KV_ERR_STALE, "pool generation %llu of instance %llu is retired",
                    (unsigned long long)pool->generation, (unsigned long long)pool->instance_id);
    if (buf_heads > KV_HND) return fail(KV_ERR_LAYOUT, "unknown buffer head order %u", buf_heads);
    if (n > 0 && (pages == nullptr || buf == nullptr))
        return fail(KV_ERR_INVALID_ARG, "page list and buffer must be non-NULL when n = %u", n);
    if (((uintptr_t)buf) % 16 != 0)
        return fail(KV_ERR_ALIGNMENT, "buffer %p is not 16-byte aligned", buf);
    const Geo &g = pool->g;
    if (kind == 0 && layer != -1) return fail(KV_ERR_INVALID_ARG, "a gather moves every layer");
    if (layer < -1 || (layer >= 0 && (uint64_t)layer >= g.L))
        return fail(KV_ERR_OUT_OF_RANGE, "layer %d is outside [-1, %llu)", layer,
                    (unsigned long long)g.L);
    const uint32_t nl = layer < 0 ? (uint32_t)g.L : 1u;
    const uint32_t l0 = layer < 0 ? 0u : (uint32_t)layer;
    const uint64_t item = (uint64_t)nl * g.C * g.cb;
    if (buf_bytes / item < n)
        return fail(KV_ERR_OUT_OF_RANGE, "buffer of %llu bytes cannot hold %u items of %llu bytes",
                    (unsigned long long)buf_bytes, n, (unsigned long long)item);
    kv_status st = check_ids(kind == 0 ? "src_pages" : "dst_pages", pages, n, g.P, kind == 1);
    if (st != KV_OK) return st;
    const int d = pool->device;
    DeviceGuard guard(d);
    st = init_device(d);
    if (st != KV_OK) return st;
    DevState &ds = g_dev[d];
    cudaStream_t stream = (cudaStream_t)stream_v;
    forget_stream(ds, stream_v);
    if (n > 0) {
        cudaPointerAttributes attr;
        cudaError_t e = cudaPointerGetAttributes(&attr, buf);
        if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(buffer)");
        if (attr.type != cudaMemoryTypeDevice || attr.device != d)
            return fail(KV_ERR_INVALID_ARG, "buffer %p is not device memory of device %d", buf, d);
        const Side ps = pool_side(*pool);
        const Side bs = staging_side((char *)buf, g, buf_heads, nl, l0, n);
        const int kernel = hbm_kernel(g, ps, bs);
        Plan p;
        st = plan(g, kind == 0 ? ps : bs, kind == 0 ? bs : ps, nl, l0, ds.err_dev, kind == 0, &p,
                  kernel);
        if (st != KV_OK) return st;
        FenceSlot fs;
        if (fence != nullptr) {
            st = reserve_fence(d, &fs);
            if (st != KV_OK) return st;
        }
        p.d.pdl = (g_cfg.flags & KV_CFG_NO_PDL) ? 0u : 1u;
        const int ctas = default_ctas(ds, false, kernel);
        const DevState *fds = fence != nullptr ? &ds : nullptr;
        const FenceSlot *ffs = fence != nullptr ? &fs : nullptr;
        if (kind == 0) {
            st = run_moves(p, pages, nullptr, n, ctas, stream, true, fds, ffs);
        } else {
            static thread_local std::vector<int32_t> idx;
            idx.resize(n);
            for (uint32_t k = 0; k < n; ++k) idx[k] = (int32_t)k;
            st = run_moves(p, idx.data(), pages, n, ctas, stream, false, fds, ffs);
        }
        if (st != KV_OK || fence == nullptr) return st;
        return commit_fence(d, fs, false, stream, fence);
    }
    return fence != nullptr ? issue_fence(d, stream, fence) : KV_OK;
}

}  // namespace

// ------------------------------------------- staged backup with no allocation

namespace kvb {

int set_last_error(int status, const char *msg) { return fail((kv_status)status, "%s", msg); }

int ring_issue(const void *pool_handle, const void *host_handle, int kind, const int32_t *a,
               const int32_t *b, uint32_t n, int32_t layer, void *stream,
               unsigned long long *done_word, unsigned long long ticket, uint64_t *fence,
               int *fused) {
    std::lock_guard<std::mutex> lk(g_mu);
    return issue((kv_pool)pool_handle, (kv_host)host_handle, kind, a, b, n, layer, stream,
                 (kv_fence *)fence, nullptr, 0, 0, done_word, ticket, fused);
}

int pool_device_of(const void *pool_handle, int *device) {
    std::lock_guard<std::mutex> lk(g_mu);
    PoolObj *p = find_pool((kv_pool)pool_handle);
    if (p == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    *device = p->device;
    return KV_OK;
}

int ring_server_view(const kv_pool *pools, uint32_t npools, kv_host host_h, RingPoolK *table,
                     Side *host_side_out, uint32_t *num_slots, int *device) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (npools == 0 || pools == nullptr)
        return fail(KV_ERR_INVALID_ARG, "a resident server needs at least one pool");
    if (host_h == nullptr) return fail(KV_ERR_INVALID_ARG, "host handle is NULL");
    HostObj *host = find_host(host_h);
    if (host == nullptr) return fail(KV_ERR_CLOSED, "host handle is closed or unknown");
    int dev = -1;
    for (uint32_t i = 0; i < npools; ++i) {
        PoolObj *p = pools[i] != nullptr ? find_pool(pools[i]) : nullptr;
        if (p == nullptr) return fail(KV_ERR_CLOSED, "pool %u of the table is closed or unknown", i);
        auto fl = g_floor.find(p->instance_id);
        if (fl != g_floor.end() && p->generation < fl->second)
            return fail(KV_ERR_STALE, "pool %u: generation %llu of instance %llu is retired", i,
                        (unsigned long long)p->generation, (unsigned long long)p->instance_id);
        if (!same_slot_geometry(p->g, host->g))
            return fail(KV_ERR_LAYOUT, "pool %u and the host tier have different page geometry", i);
        if (dev >= 0 && p->device != dev)
            return fail(KV_ERR_INVALID_ARG, "the pools of one server live on different devices");
        dev = p->device;
        const Geo &g = p->g;
        RingPoolK &k = table[i];
        k = RingPoolK{};
        k.pool = pool_side(*p);
        k.L = (uint32_t)g.L;
        k.C = (uint32_t)g.C;
        k.P = (uint32_t)std::min<uint64_t>(g.P, 0xffffffffull);
        k.H = (uint32_t)g.H;
        k.T = (uint32_t)g.T;
        k.B16 = (uint32_t)(g.B / 16);
        k.cb16 = (uint32_t)(g.cb / 16);
        k.segs = (k.cb16 + kSegPieces - 1) / kSegPieces;
        // the segments of the largest descriptor (every id, every layer) must count in 32 bits
        if ((uint64_t)KV_RING_MAX_IDS * g.L * g.C * k.segs > 0xffffffffull)
            return fail(KV_ERR_LAYOUT, "pool %u: a descriptor of %d pages would need more than "
                        "2^32 warp segments", i, KV_RING_MAX_IDS);
        k.transpose = (g.heads != host->heads && g.H > 1 && g.T > 1) ? 1u : 0u;
        k.div_segs = make_fastdiv(k.segs);
        k.div_lc_all = make_fastdiv(k.L * k.C);
        k.div_lc_one = make_fastdiv(k.C);
        k.div_c = make_fastdiv(k.C);
        k.div_b16 = make_fastdiv(k.B16);
        k.div_T = make_fastdiv(k.T);
        k.div_H = make_fastdiv(k.H);
    }
    // The fence state must exist before the resident kernel is launched: creating
    // it (pinned allocation, memset) would wait for that kernel to end.
    {
        DeviceGuard guard(dev);
        kv_status st = init_device(dev);
        if (st != KV_OK) return st;
    }
    *host_side_out = host_side(*host);
    *num_slots = host->num_slots;
    *device = dev;
    return KV_OK;
}

int ring_launch_server(int device, const RingKDesc &k, int ctas, cudaStream_t stream,
                       kv_fence *fence) {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceGuard guard(device);
    kv_status st = init_device(device);
    if (st != KV_OK) return st;
    forget_stream(g_dev[device], (void *)stream);
    // the fence's slot (and its event) before the launch, its marker after
    FenceSlot fs;
    st = reserve_fence(device, &fs);
    if (st != KV_OK) return st;
    cudaError_t e = launch_ring_server(k, ctas, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launch of the resident ring server");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return commit_fence(device, fs, true, stream, fence);
}

int enqueue_staged_backup_noalloc(const void *pool_handle, const void *host_handle,
                                  const int32_t *src, const int32_t *slots, uint32_t n,
                                  void *staging, uint64_t staging_bytes, cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (pool_handle == nullptr || host_handle == nullptr)
        return fail(KV_ERR_INVALID_ARG, "pool or host handle is NULL");
    PoolObj *pool = find_pool((kv_pool)pool_handle);
    if (pool == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    HostObj *host = find_host((kv_host)host_handle);
    if (host == nullptr) return fail(KV_ERR_CLOSED, "host handle is closed or unknown");
    auto fl = g_floor.find(pool->instance_id);
    if (fl != g_floor.end() && pool->generation < fl->second)
        return fail(KV_ERR_STALE, "pool generation %llu of instance %llu is retired",
                    (unsigned long long)pool->generation, (unsigned long long)pool->instance_id);
    if (!same_slot_geometry(pool->g, host->g))
        return fail(KV_ERR_LAYOUT, "pool and host tier have different page geometry");
    if (n > 0 && (src == nullptr || slots == nullptr))
        return fail(KV_ERR_INVALID_ARG, "id arrays must be non-NULL when n = %u", n);
    const Geo &g = pool->g;
    if (n > (uint32_t)kMaxItems)
        return fail(KV_ERR_OUT_OF_RANGE, "n = %u exceeds the %d pages one allocation-free backup "
                    "may move", n, kMaxItems);
    if ((uint64_t)n * g.pb > staging_bytes)
        return fail(KV_ERR_OUT_OF_RANGE, "%u pages of %llu bytes exceed the %llu-byte static "
                    "staging area of the allocation-free backup", n, (unsigned long long)g.pb,
                    (unsigned long long)staging_bytes);
    // range checks, then duplicate slots by sorting a stack copy (no heap)
    int32_t sorted[kMaxItems];
    for (uint32_t i = 0; i < n; ++i) {
        if (src[i] < 0 || (uint64_t)src[i] >= g.P)
            return fail(KV_ERR_OUT_OF_RANGE, "src_pages[%u] = %d is outside [0, %llu)", i, src[i],
                        (unsigned long long)g.P);
        if (slots[i] < 0 || (uint32_t)slots[i] >= host->num_slots)
            return fail(KV_ERR_OUT_OF_RANGE, "host_slots[%u] = %d is outside [0, %u)", i, slots[i],
                        host->num_slots);
        sorted[i] = slots[i];
    }
    std::sort(sorted, sorted + n);
    for (uint32_t i = 1; i < n; ++i)
        if (sorted[i] == sorted[i - 1])
            return fail(KV_ERR_DUPLICATE, "host slot %d appears twice: one call may write a slot "
                        "only once", sorted[i]);
    if (n == 0) return KV_OK;
    if (g_dev[pool->device].init) forget_stream(g_dev[pool->device], (void *)stream);
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, pool->device);
    const Side ps = pool_side(*pool);
    const Side ss = staging_side((char *)staging, g, host->heads, (uint32_t)g.L, 0, n);
    Plan p;
    kv_status st = plan(g, ps, ss, (uint32_t)g.L, 0, nullptr, true, &p);
    if (st != KV_OK) return st;
    MoveIds ids;   // on the stack: the ids travel inside the launch
    std::memcpy(ids.a, src, n * sizeof(int32_t));
    for (uint32_t k = 0; k < n; ++k) ids.b[k] = (int32_t)k;
    p.d.n = n;
    p.d.total_segs = n * p.d.nl * p.d.C * p.d.segs;
    const uint32_t per_cta = kMoveThreads / 32;
    const uint64_t need = (p.d.total_segs + per_cta - 1) / per_cta;
    const int cap = g_cfg.max_ctas ? (int)g_cfg.max_ctas : 4 * std::max(sms, 1);
    const int ctas = (int)std::max<uint64_t>(1, std::min<uint64_t>(need, (uint64_t)cap));
    cudaError_t e = launch_move(p.d, ids, ctas, kMoveThreads, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launch of the move kernel");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return staged_copies(*host, (char *)staging, slots, n, g.pb, 0, true, stream);
}

int fence_gate_word(kv_fence f, const unsigned long long **word, unsigned long long *tag) {
    const int d = (int)(f >> 56);
    const uint64_t seq = f & kSeqMask;
    std::lock_guard<std::mutex> lk(g_mu);
    if (seq == 0 || d >= kMaxDevices || !g_dev[d].init || seq >= g_next_seq)
        return fail(KV_ERR_INVALID_ARG, "invalid fence %llu", (unsigned long long)f);
    *word = g_dev[d].status_dev + (seq % kRing);
    *tag = seq;
    return KV_OK;
}

}  // namespace kvb

// =================================================================== C ABI

extern "C" {

uint32_t kv_abi_version(void) { return KVB_ABI_VERSION; }

kv_status kv_fault_inject(const char *point, uint32_t count) {
    std::call_once(g_fault_env_once, load_fault_env);
    if (point == nullptr) return fail(KV_ERR_INVALID_ARG, "fault point is NULL");
    for (int i = 0; i < FP_COUNT; ++i)
        if (std::strcmp(point, kFaultNames[i]) == 0) {
            g_fault[i].store(count);
            return KV_OK;
        }
    return fail(KV_ERR_INVALID_ARG, "unknown fault point \"%s\"", point);
}

const char *kv_last_error(void) { return t_err.c_str(); }

uint64_t kv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t kv_overlap_count(void) { return g_overlapped.load(std::memory_order_relaxed); }

kv_status kv_layout_page_bytes(const kv_layout *layout, uint64_t *out) {
    if (out == nullptr) return fail(KV_ERR_INVALID_ARG, "output pointer is NULL");
    Geo g{};
    kv_status st = check_layout(layout, &g);
    if (st != KV_OK) return st;
    *out = g.pb;
    return KV_OK;
}

kv_status kv_config_get(kv_config *out) {
    if (out == nullptr) return fail(KV_ERR_INVALID_ARG, "output pointer is NULL");
    std::lock_guard<std::mutex> lk(g_mu);
    *out = g_cfg;
    return KV_OK;
}

kv_status kv_config_set(const kv_config *cfg) {
    if (cfg == nullptr) return fail(KV_ERR_INVALID_ARG, "config is NULL");
    if (cfg->mode > KV_MODE_COPY_ENGINE) return fail(KV_ERR_INVALID_ARG, "unknown mode %u", cfg->mode);
    if (cfg->max_ctas > 65535) return fail(KV_ERR_INVALID_ARG, "max_ctas %u > 65535", cfg->max_ctas);
    if (cfg->staging_bytes != 0 && (cfg->staging_bytes < (2ull << 20) || cfg->staging_bytes % 512))
        return fail(KV_ERR_INVALID_ARG, "staging_bytes must be 0 or a multiple of 512 >= 2 MiB");
    if ((cfg->flags & ~(uint32_t)(KV_CFG_NO_BULK | KV_CFG_NO_PDL | KV_CFG_OVERLAP_RESTORES |
                                  KV_CFG_OVERLAP_BACKUPS)) != 0)
        return fail(KV_ERR_INVALID_ARG, "unknown config flags %#x", cfg->flags);
    if (cfg->cta_threads != 0 && cfg->cta_threads != (uint32_t)kMoveThreads &&
        cfg->cta_threads != (uint32_t)kWideThreads)
        return fail(KV_ERR_INVALID_ARG, "cta_threads must be 0, %d or %d", kMoveThreads,
                    kWideThreads);
    std::lock_guard<std::mutex> lk(g_mu);
    g_cfg = *cfg;
    return KV_OK;
}

kv_status kv_op_validate(const kv_layout *layout, uint32_t num_slots, int kind, const int32_t *a,
                         const int32_t *b, uint32_t n, int32_t layer) {
    Geo g{};
    kv_status st = check_layout(layout, &g);
    if (st != KV_OK) return st;
    return check_op(g, num_slots, kind, a, b, n, layer);
}

kv_status kv_pool_register(const kv_layout *layout, void *base, uint64_t offset,
                           uint64_t instance_id, uint64_t generation, kv_pool *out) {
    if (out == nullptr) return fail(KV_ERR_INVALID_ARG, "output handle pointer is NULL");
    Geo g{};
    kv_status st = check_layout(layout, &g);
    if (st != KV_OK) return st;
    if (base == nullptr) return fail(KV_ERR_INVALID_ARG, "pool base is NULL");
    char *start = (char *)base + offset;
    if (((uintptr_t)start) % 16 != 0)
        return fail(KV_ERR_ALIGNMENT, "pool start %p (base + %llu) is not 16-byte aligned",
                    (void *)start, (unsigned long long)offset);
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, start);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(pool)");
    if (attr.type != cudaMemoryTypeDevice)
        return fail(KV_ERR_INVALID_ARG, "pool start %p is not device memory", (void *)start);
    uintptr_t ab;
    size_t as;
    {
        DeviceGuard guard(attr.device);
        st = address_range(start, &ab, &as);
    }
    if (st != KV_OK) return st;
    const uint64_t nbytes = g.pb * g.P;
    if ((uintptr_t)start + nbytes > ab + as || (uintptr_t)start + nbytes < (uintptr_t)start)
        return fail(KV_ERR_OUT_OF_RANGE, "pool of %llu bytes at offset %llu overruns its "
                    "allocation (%llu bytes from %p)", (unsigned long long)nbytes,
                    (unsigned long long)((uintptr_t)start - ab), (unsigned long long)as,
                    (void *)ab);
    PoolObj *p = new (std::nothrow) PoolObj{g, *layout, start, nbytes, attr.device, instance_id,
                                            generation, false, std::string()};
    if (p == nullptr) return fail(KV_ERR_NO_MEMORY, "out of host memory");
    std::lock_guard<std::mutex> lk(g_mu);
    const uint64_t id = g_next_handle++;
    g_pools[id] = p;
    *out = (kv_pool)(uintptr_t)id;
    return KV_OK;
}

kv_status kv_pool_register_split(const kv_layout *layout, void *const *bases,
                                 uint64_t instance_id, uint64_t generation, kv_pool *out) {
    if (out == nullptr) return fail(KV_ERR_INVALID_ARG, "output handle pointer is NULL");
    Geo g{};
    kv_status st = check_layout(layout, &g);
    if (st != KV_OK) return st;
    if (g.order != KV_LAYER_FIRST)
        return fail(KV_ERR_LAYOUT, "a split pool is layer-first: one buffer per layer and "
                    "component");
    if (bases == nullptr) return fail(KV_ERR_INVALID_ARG, "buffer table is NULL");
    const uint64_t nb = g.L * g.C;
    if (nb > (1u << 20)) return fail(KV_ERR_LAYOUT, "too many layer buffers");
    const uint64_t buf_bytes = g.P * g.cb;   // [P][T][H][B] or [P][H][T][B]
    for (uint64_t i = 0; i < nb; ++i) {
        if (bases[i] == nullptr)
            return fail(KV_ERR_INVALID_ARG, "buffer of layer %llu component %llu is NULL",
                        (unsigned long long)(i / g.C), (unsigned long long)(i % g.C));
        if (((uintptr_t)bases[i]) % 16 != 0)
            return fail(KV_ERR_ALIGNMENT, "buffer %p is not 16-byte aligned", bases[i]);
    }
    int device = -1;
    for (uint64_t i = 0; i < nb; ++i) {
        cudaPointerAttributes attr;
        cudaError_t e = cudaPointerGetAttributes(&attr, bases[i]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(layer buffer)");
        if (attr.type != cudaMemoryTypeDevice)
            return fail(KV_ERR_INVALID_ARG, "layer buffer %p is not device memory", bases[i]);
        if (device >= 0 && attr.device != device)
            return fail(KV_ERR_INVALID_ARG, "layer buffers live on different devices");
        device = attr.device;
        uintptr_t ab;
        size_t as;
        {
            DeviceGuard guard(device);
            st = address_range(bases[i], &ab, &as);
        }
        if (st != KV_OK) return st;
        if ((uintptr_t)bases[i] + buf_bytes > ab + as)
            return fail(KV_ERR_OUT_OF_RANGE, "layer buffer %p of %llu bytes overruns its "
                        "allocation", bases[i], (unsigned long long)buf_bytes);
    }
    std::vector<unsigned long long> table(nb);
    for (uint64_t i = 0; i < nb; ++i) table[i] = (unsigned long long)(uintptr_t)bases[i];
    void *tdev = nullptr;
    {
        DeviceGuard guard(device);
        cudaError_t e = cudaMalloc(&tdev, nb * sizeof(unsigned long long));
        if (e == cudaSuccess)
            e = cudaMemcpy(tdev, table.data(), nb * sizeof(unsigned long long),
                           cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            if (tdev) cudaFree(tdev);
            return cuda_fail(e, "copying the split pool's buffer table to the device");
        }
    }
    PoolObj *p = new (std::nothrow) PoolObj{g, *layout, (char *)bases[0], buf_bytes * nb, device,
                                            instance_id, generation, false, std::string()};
    if (p == nullptr) {
        cudaFree(tdev);
        return fail(KV_ERR_NO_MEMORY, "out of host memory");
    }
    p->table_dev = (unsigned long long *)tdev;
    p->table_host.swap(table);
    std::lock_guard<std::mutex> lk(g_mu);
    const uint64_t id = g_next_handle++;
    g_pools[id] = p;
    *out = (kv_pool)(uintptr_t)id;
    return KV_OK;
}

kv_status kv_pool_export(kv_pool pool_h, kv_ipc_desc *out) {
    if (out == nullptr) return fail(KV_ERR_INVALID_ARG, "output descriptor pointer is NULL");
    std::lock_guard<std::mutex> lk(g_mu);
    PoolObj *p = find_pool(pool_h);
    if (p == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    if (p->table_dev != nullptr)
        return fail(KV_ERR_LAYOUT, "a split pool spans several allocations: export it with "
                    "kv_pool_export_split");
    DeviceGuard guard(p->device);
    uintptr_t ab;
    size_t as;
    kv_status st = address_range(p->dev, &ab, &as);
    if (st != KV_OK) return st;
    cudaIpcMemHandle_t h;
    cudaError_t e = cudaIpcGetMemHandle(&h, (void *)ab);
    if (e != cudaSuccess) return cuda_fail(e, "cudaIpcGetMemHandle(allocation base)");
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, p->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    kv_ipc_desc dsc;
    std::memset(&dsc, 0, sizeof dsc);
    dsc.magic = KVB_IPC_MAGIC;
    dsc.version = KVB_ABI_VERSION;
    static_assert(sizeof(h.reserved) == sizeof(dsc.handle), "IPC handle size");
    std::memcpy(dsc.handle, h.reserved, sizeof dsc.handle);
    dsc.alloc_offset = (uint64_t)((uintptr_t)p->dev - ab);
    dsc.nbytes = p->nbytes;
    dsc.instance_id = p->instance_id;
    dsc.generation = p->generation;
    dsc.exporter_pid = (int64_t)getpid();
    std::memcpy(dsc.device_uuid, prop.uuid.bytes, sizeof dsc.device_uuid);
    dsc.layout = p->layout;
    *out = dsc;
    return KV_OK;
}

kv_status kv_pool_import(const kv_ipc_desc *desc, kv_pool *out) {
    if (desc == nullptr || out == nullptr) return fail(KV_ERR_INVALID_ARG, "NULL argument");
    if (desc->magic == KVB_IPC_MAGIC_SPLIT)
        return fail(KV_ERR_INVALID_ARG, "descriptor of a split pool: import it with "
                    "kv_pool_import_split");
    if (desc->magic != KVB_IPC_MAGIC || desc->version != KVB_ABI_VERSION)
        return fail(KV_ERR_INVALID_ARG, "descriptor magic/version %08x/%u not recognised",
                    desc->magic, desc->version);
    Geo g{};
    kv_status st = check_layout(&desc->layout, &g);
    if (st != KV_OK) return st;
    if (desc->nbytes != g.pb * g.P)
        return fail(KV_ERR_LAYOUT, "descriptor nbytes %llu != pool size %llu",
                    (unsigned long long)desc->nbytes, (unsigned long long)(g.pb * g.P));
    if (desc->alloc_offset % 16 != 0)
        return fail(KV_ERR_ALIGNMENT, "alloc_offset %llu is not 16-byte aligned",
                    (unsigned long long)desc->alloc_offset);
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    int device = -1;
    for (int i = 0; i < ndev && device < 0; ++i) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, i) == cudaSuccess &&
            std::memcmp(prop.uuid.bytes, desc->device_uuid, 16) == 0)
            device = i;
    }
    if (device < 0) return fail(KV_ERR_INVALID_ARG, "no visible device has the descriptor's UUID");
    std::lock_guard<std::mutex> lk(g_mu);
    auto fl = g_floor.find(desc->instance_id);
    if (fl != g_floor.end() && desc->generation < fl->second)
        return fail(KV_ERR_STALE, "descriptor generation %llu of instance %llu is retired",
                    (unsigned long long)desc->generation, (unsigned long long)desc->instance_id);
    const std::string key((const char *)desc->handle, sizeof desc->handle);
    auto it = g_maps.find(key);
    void *base = nullptr;
    if (it != g_maps.end()) {
        if (it->second.device != device)   // addresses of another device's context
            return fail(KV_ERR_INVALID_ARG, "the allocation is already mapped on device %d, not "
                        "on the descriptor's device %d", it->second.device, device);
        base = it->second.base;
    } else {
        DeviceGuard guard(device);
        cudaIpcMemHandle_t h;
        std::memcpy(h.reserved, desc->handle, sizeof desc->handle);
        if (fault_hit(FP_IPC_OPEN)) return fail(KV_ERR_CUDA, "cudaIpcOpenMemHandle: injected failure");
        e = cudaIpcOpenMemHandle(&base, h, cudaIpcMemLazyEnablePeerAccess);
        if (e != cudaSuccess) return cuda_fail(e, "cudaIpcOpenMemHandle");
    }
    char *start = (char *)base + desc->alloc_offset;
    if (((uintptr_t)start) % 16 != 0) {
        if (it == g_maps.end()) cudaIpcCloseMemHandle(base);
        return fail(KV_ERR_ALIGNMENT, "imported pool start %p is not 16-byte aligned", (void *)start);
    }
    {   // the descriptor's extent must lie inside the allocation the handle maps
        uintptr_t ab = 0;
        size_t as = 0;
        DeviceGuard guard(device);
        st = address_range(base, &ab, &as);
        if (st == KV_OK && (desc->alloc_offset > as || desc->nbytes > as - desc->alloc_offset))
            st = fail(KV_ERR_OUT_OF_RANGE, "descriptor extent (offset %llu + %llu bytes) overruns "
                      "the imported allocation of %llu bytes",
                      (unsigned long long)desc->alloc_offset, (unsigned long long)desc->nbytes,
                      (unsigned long long)as);
        if (st != KV_OK) {
            if (it == g_maps.end()) cudaIpcCloseMemHandle(base);
            return st;
        }
    }
    PoolObj *p = new (std::nothrow) PoolObj{g, desc->layout, start, desc->nbytes, device,
                                            desc->instance_id, desc->generation, true, key};
    if (p == nullptr) {
        if (it == g_maps.end()) cudaIpcCloseMemHandle(base);
        return fail(KV_ERR_NO_MEMORY, "out of host memory");
    }
    if (it != g_maps.end())
        it->second.refs += 1;
    else
        g_maps[key] = Mapping{base, 1, device};
    const uint64_t id = g_next_handle++;
    g_pools[id] = p;
    *out = (kv_pool)(uintptr_t)id;
    return KV_OK;
}

kv_status kv_pool_export_split(kv_pool pool_h, kv_ipc_desc *out, kv_ipc_buffer *bufs,
                               uint32_t nbufs) {
    if (out == nullptr || bufs == nullptr) return fail(KV_ERR_INVALID_ARG, "NULL argument");
    std::lock_guard<std::mutex> lk(g_mu);
    PoolObj *p = find_pool(pool_h);
    if (p == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    if (p->table_dev == nullptr)
        return fail(KV_ERR_LAYOUT, "not a split pool: export it with kv_pool_export");
    const uint64_t nb = p->g.L * p->g.C;
    if (nbufs != nb)
        return fail(KV_ERR_INVALID_ARG, "%u buffer entries for a pool of %llu buffers", nbufs,
                    (unsigned long long)nb);
    DeviceGuard guard(p->device);
    std::vector<kv_ipc_buffer> tmp(nb);
    std::unordered_map<uintptr_t, cudaIpcMemHandle_t> handles;   // one handle per allocation
    for (uint64_t i = 0; i < nb; ++i) {
        const uintptr_t ptr = (uintptr_t)p->table_host[i];
        uintptr_t ab;
        size_t as;
        kv_status st = address_range((const void *)ptr, &ab, &as);
        if (st != KV_OK) return st;
        auto h = handles.find(ab);
        if (h == handles.end()) {
            cudaIpcMemHandle_t hd;
            cudaError_t e = cudaIpcGetMemHandle(&hd, (void *)ab);
            if (e != cudaSuccess) return cuda_fail(e, "cudaIpcGetMemHandle(layer buffer allocation)");
            h = handles.emplace(ab, hd).first;
        }
        static_assert(sizeof(h->second.reserved) == sizeof(tmp[i].handle), "IPC handle size");
        std::memcpy(tmp[i].handle, h->second.reserved, sizeof tmp[i].handle);
        tmp[i].alloc_offset = (uint64_t)(ptr - ab);
    }
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, p->device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    kv_ipc_desc dsc;
    std::memset(&dsc, 0, sizeof dsc);
    dsc.magic = KVB_IPC_MAGIC_SPLIT;
    dsc.version = KVB_ABI_VERSION;
    std::memcpy(dsc.handle, tmp[0].handle, sizeof dsc.handle);
    dsc.alloc_offset = tmp[0].alloc_offset;
    dsc.nbytes = p->nbytes;
    dsc.instance_id = p->instance_id;
    dsc.generation = p->generation;
    dsc.exporter_pid = (int64_t)getpid();
    std::memcpy(dsc.device_uuid, prop.uuid.bytes, sizeof dsc.device_uuid);
    dsc.layout = p->layout;
    *out = dsc;
    std::memcpy(bufs, tmp.data(), nb * sizeof(kv_ipc_buffer));
    return KV_OK;
}

kv_status kv_pool_import_split(const kv_ipc_desc *desc, const kv_ipc_buffer *bufs, uint32_t nbufs,
                               kv_pool *out) {
    if (desc == nullptr || bufs == nullptr || out == nullptr)
        return fail(KV_ERR_INVALID_ARG, "NULL argument");
    if (desc->magic != KVB_IPC_MAGIC_SPLIT || desc->version != KVB_ABI_VERSION)
        return fail(KV_ERR_INVALID_ARG, "not a split-pool descriptor (magic/version %08x/%u)",
                    desc->magic, desc->version);
    Geo g{};
    kv_status st = check_layout(&desc->layout, &g);
    if (st != KV_OK) return st;
    if (g.order != KV_LAYER_FIRST)
        return fail(KV_ERR_LAYOUT, "a split pool is layer-first: one buffer per layer and "
                    "component");
    const uint64_t nb = g.L * g.C;
    if (nb > (1u << 20)) return fail(KV_ERR_LAYOUT, "too many layer buffers");
    if (nbufs != nb)
        return fail(KV_ERR_INVALID_ARG, "%u buffer entries for a pool of %llu buffers", nbufs,
                    (unsigned long long)nb);
    const uint64_t buf_bytes = g.P * g.cb;
    if (desc->nbytes != buf_bytes * nb)
        return fail(KV_ERR_LAYOUT, "descriptor nbytes %llu != %llu buffers of %llu bytes",
                    (unsigned long long)desc->nbytes, (unsigned long long)nb,
                    (unsigned long long)buf_bytes);
    for (uint64_t i = 0; i < nb; ++i)
        if (bufs[i].alloc_offset % 16 != 0)
            return fail(KV_ERR_ALIGNMENT, "buffer %llu: alloc_offset %llu is not 16-byte aligned",
                        (unsigned long long)i, (unsigned long long)bufs[i].alloc_offset);
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    int device = -1;
    for (int i = 0; i < ndev && device < 0; ++i) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, i) == cudaSuccess &&
            std::memcmp(prop.uuid.bytes, desc->device_uuid, 16) == 0)
            device = i;
    }
    if (device < 0) return fail(KV_ERR_INVALID_ARG, "no visible device has the descriptor's UUID");
    std::lock_guard<std::mutex> lk(g_mu);
    auto fl = g_floor.find(desc->instance_id);
    if (fl != g_floor.end() && desc->generation < fl->second)
        return fail(KV_ERR_STALE, "descriptor generation %llu of instance %llu is retired",
                    (unsigned long long)desc->generation, (unsigned long long)desc->instance_id);
    DeviceGuard guard(device);
    // each distinct allocation: its mapping (existing, or opened here) and size
    struct Mapped {
        void *base;
        size_t size;
        bool opened;
    };
    std::unordered_map<std::string, Mapped> mapped;
    std::vector<std::string> keys;
    auto undo = [&]() {
        for (auto &m : mapped)
            if (m.second.opened) cudaIpcCloseMemHandle(m.second.base);
    };
    std::vector<unsigned long long> table(nb);
    for (uint64_t i = 0; i < nb; ++i) {
        const std::string key((const char *)bufs[i].handle, sizeof bufs[i].handle);
        auto m = mapped.find(key);
        if (m == mapped.end()) {
            Mapped mp{nullptr, 0, false};
            auto it = g_maps.find(key);
            if (it != g_maps.end()) {
                if (it->second.device != device) {   // addresses of another device's context
                    undo();
                    return fail(KV_ERR_INVALID_ARG, "buffer %llu's allocation is already mapped "
                                "on device %d, not on the descriptor's device %d",
                                (unsigned long long)i, it->second.device, device);
                }
                mp.base = it->second.base;
            } else {
                cudaIpcMemHandle_t h;
                std::memcpy(h.reserved, bufs[i].handle, sizeof bufs[i].handle);
                if (fault_hit(FP_IPC_OPEN)) {
                    undo();
                    return fail(KV_ERR_CUDA, "cudaIpcOpenMemHandle: injected failure");
                }
                e = cudaIpcOpenMemHandle(&mp.base, h, cudaIpcMemLazyEnablePeerAccess);
                if (e != cudaSuccess) {
                    undo();
                    return cuda_fail(e, "cudaIpcOpenMemHandle(layer buffer allocation)");
                }
                mp.opened = true;
            }
            uintptr_t ab = 0;
            st = address_range(mp.base, &ab, &mp.size);
            m = mapped.emplace(key, mp).first;   // recorded first, so undo() closes it
            if (st != KV_OK) {
                undo();
                return st;
            }
            keys.push_back(key);
        }
        const uint64_t off = bufs[i].alloc_offset;
        if (off > m->second.size || buf_bytes > m->second.size - off) {
            undo();
            return fail(KV_ERR_OUT_OF_RANGE, "buffer %llu (offset %llu + %llu bytes) overruns its "
                        "imported allocation of %llu bytes", (unsigned long long)i,
                        (unsigned long long)off, (unsigned long long)buf_bytes,
                        (unsigned long long)m->second.size);
        }
        table[i] = (unsigned long long)((uintptr_t)m->second.base + off);
    }
    void *tdev = nullptr;
    e = cudaMalloc(&tdev, nb * sizeof(unsigned long long));
    if (e == cudaSuccess)
        e = cudaMemcpy(tdev, table.data(), nb * sizeof(unsigned long long), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        if (tdev) cudaFree(tdev);
        undo();
        return cuda_fail(e, "copying the imported split pool's buffer table to the device");
    }
    PoolObj *p = new (std::nothrow) PoolObj{g, desc->layout, (char *)(uintptr_t)table[0],
                                            desc->nbytes, device, desc->instance_id,
                                            desc->generation, true, std::string()};
    if (p == nullptr) {
        cudaFree(tdev);
        undo();
        return fail(KV_ERR_NO_MEMORY, "out of host memory");
    }
    p->table_dev = (unsigned long long *)tdev;
    p->table_host.swap(table);
    p->ipc_keys = keys;
    for (const std::string &key : keys) {
        auto it = g_maps.find(key);
        if (it != g_maps.end())
            it->second.refs += 1;
        else
            g_maps[key] = Mapping{mapped[key].base, 1, device};
    }
    const uint64_t id = g_next_handle++;
    g_pools[id] = p;
    *out = (kv_pool)(uintptr_t)id;
    return KV_OK;
}

kv_status kv_pool_close(kv_pool pool_h) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_pools.find(handle_id(pool_h));
    if (it == g_pools.end()) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    PoolObj *p = it->second;
    g_pools.erase(it);
    kv_status st = KV_OK;
    if (p->table_dev != nullptr) {
        DeviceGuard guard(p->device);
        if (cudaFree(p->table_dev) != cudaSuccess)
            st = cuda_fail(cudaErrorUnknown, "cudaFree(split pool table)");
    }
    if (p->imported) {
        std::vector<std::string> keys = p->ipc_keys;
        if (keys.empty()) keys.push_back(p->ipc_key);
        for (const std::string &key : keys) {
            auto m = g_maps.find(key);
            if (m != g_maps.end() && --m->second.refs == 0) {
                DeviceGuard guard(m->second.device);
                cudaError_t e = cudaIpcCloseMemHandle(m->second.base);
                g_maps.erase(m);
                if (e != cudaSuccess) st = cuda_fail(e, "cudaIpcCloseMemHandle (mapping dropped)");
            }
        }
    }
    delete p;
    return st;
}

kv_status kv_pool_retire(uint64_t instance_id, uint64_t min_generation) {
    std::lock_guard<std::mutex> lk(g_mu);
    uint64_t &f = g_floor[instance_id];
    f = std::max(f, min_generation);
    return KV_OK;
}

kv_status kv_pool_info(kv_pool pool_h, kv_layout *layout, void **dev_ptr, uint64_t *nbytes) {
    std::lock_guard<std::mutex> lk(g_mu);
    PoolObj *p = find_pool(pool_h);
    if (p == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    if (layout) *layout = p->layout;
    if (dev_ptr) *dev_ptr = p->dev;
    if (nbytes) *nbytes = p->nbytes;
    return KV_OK;
}

kv_status kv_host_register(void *host, uint64_t bytes, uint32_t num_slots, uint32_t host_heads,
                           const kv_layout *pool_layout, kv_host *out) {
    if (out == nullptr) return fail(KV_ERR_INVALID_ARG, "output handle pointer is NULL");
    Geo g{};
    kv_status st = check_layout(pool_layout, &g);
    if (st != KV_OK) return st;
    if (host_heads > KV_HND) return fail(KV_ERR_LAYOUT, "unknown host head order %u", host_heads);
    if (host == nullptr || num_slots == 0)
        return fail(KV_ERR_INVALID_ARG, "host tier pointer is NULL or has no slots");
    if (((uintptr_t)host) % 16 != 0)
        return fail(KV_ERR_ALIGNMENT, "host tier %p is not 16-byte aligned", host);
    uint64_t need;
    if (!mul_ok(g.pb, num_slots, 1ull << 62, &need) || bytes < need)
        return fail(KV_ERR_OUT_OF_RANGE, "host tier of %llu bytes cannot hold %u slots of %llu bytes",
                    (unsigned long long)bytes, num_slots, (unsigned long long)g.pb);
    cudaPointerAttributes attr;
    if (fault_hit(FP_HOST_REGISTER))
        return fail(KV_ERR_CUDA, "host tier registration: injected failure");
    cudaError_t e = cudaPointerGetAttributes(&attr, host);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(host tier)");
    if (attr.type != cudaMemoryTypeHost)
        return fail(KV_ERR_INVALID_ARG, "host tier %p is not page-locked host memory known to CUDA",
                    host);
    void *dv = attr.devicePointer;
    if (dv == nullptr) {
        e = cudaHostGetDevicePointer(&dv, host, 0);
        if (e != cudaSuccess || dv == nullptr)
            return fail(KV_ERR_INVALID_ARG, "host tier %p is not mapped into the device", host);
    }
    HostObj *h = new (std::nothrow) HostObj{g, host_heads, num_slots, (char *)host, (char *)dv, bytes};
    if (h == nullptr) return fail(KV_ERR_NO_MEMORY, "out of host memory");
    std::lock_guard<std::mutex> lk(g_mu);
    const uint64_t id = g_next_handle++;
    g_hosts[id] = h;
    *out = (kv_host)(uintptr_t)id;
    return KV_OK;
}

kv_status kv_host_close(kv_host host_h) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_hosts.find(handle_id(host_h));
    if (it == g_hosts.end()) return fail(KV_ERR_CLOSED, "host handle is closed or unknown");
    delete it->second;
    g_hosts.erase(it);
    return KV_OK;
}

kv_status kv_backup(kv_pool pool, kv_host host, const int32_t *src_pages,
                    const int32_t *host_slots, uint32_t n, void *stream, kv_fence *fence) {
    std::lock_guard<std::mutex> lk(g_mu);
    return issue(pool, host, 0, src_pages, host_slots, n, -1, stream, fence);
}

namespace {
// Checks a ready word and returns its device-visible address (or an error).
kv_status ready_word_dev(const uint64_t *ready_word, uint64_t ready_timeout_ns,
                         const void **dev_word) {
    if (ready_word == nullptr) return fail(KV_ERR_INVALID_ARG, "ready_word is NULL");
    if (((uintptr_t)ready_word) % 8 != 0)
        return fail(KV_ERR_ALIGNMENT, "ready_word %p is not 8-byte aligned", (const void *)ready_word);
    if (ready_timeout_ns > kMaxReadyTimeoutNs)
        return fail(KV_ERR_INVALID_ARG, "ready_timeout_ns %llu exceeds the %llu ns limit",
                    (unsigned long long)ready_timeout_ns, (unsigned long long)kMaxReadyTimeoutNs);
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, ready_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(ready_word)");
    *dev_word = nullptr;
    if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged)
        *dev_word = ready_word;
    else if (attr.type == cudaMemoryTypeHost)
        *dev_word = attr.devicePointer;
    if (*dev_word == nullptr)
        return fail(KV_ERR_INVALID_ARG, "ready_word %p is not visible to the GPU (use device or "
                    "pinned mapped host memory)", (const void *)ready_word);
    return KV_OK;
}
}  // namespace

kv_status kv_restore_when_ready(kv_pool pool, kv_host host, const int32_t *host_slots,
                                const int32_t *dst_pages, uint32_t n, int32_t layer,
                                const uint64_t *ready_word, uint64_t ready_value,
                                uint64_t ready_timeout_ns, void *stream, kv_fence *fence) {
    const void *dev_word = nullptr;
    kv_status st = ready_word_dev(ready_word, ready_timeout_ns, &dev_word);
    if (st != KV_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    return issue(pool, host, 1, host_slots, dst_pages, n, layer, stream, fence,
                 (const unsigned long long *)dev_word, ready_value, ready_timeout_ns);
}

kv_status kv_backup_when_ready(kv_pool pool, kv_host host, const int32_t *src_pages,
                               const int32_t *host_slots, uint32_t n, const uint64_t *ready_word,
                               uint64_t ready_value, uint64_t ready_timeout_ns, void *stream,
                               kv_fence *fence) {
    const void *dev_word = nullptr;
    kv_status st = ready_word_dev(ready_word, ready_timeout_ns, &dev_word);
    if (st != KV_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    return issue(pool, host, 0, src_pages, host_slots, n, -1, stream, fence,
                 (const unsigned long long *)dev_word, ready_value, ready_timeout_ns);
}

kv_status kv_restore_layers(kv_pool pool_h, kv_host host_h, const int32_t *host_slots,
                            const int32_t *dst_pages, uint32_t n, uint32_t first_layer,
                            uint32_t num_layers, void *stream_v, kv_fence *fences) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (fences == nullptr) return fail(KV_ERR_INVALID_ARG, "fence output array is NULL");
    if (pool_h == nullptr || host_h == nullptr)
        return fail(KV_ERR_INVALID_ARG, "pool or host handle is NULL");
    PoolObj *pool = find_pool(pool_h);
    if (pool == nullptr) return fail(KV_ERR_CLOSED, "pool handle is closed or unknown");
    HostObj *host = find_host(host_h);
    if (host == nullptr) return fail(KV_ERR_CLOSED, "host handle is closed or unknown");
    auto fl = g_floor.find(pool->instance_id);
    if (fl != g_floor.end() && pool->generation < fl->second)
        return fail(KV_ERR_STALE, "pool generation %llu of instance %llu is retired",
                    (unsigned long long)pool->generation, (unsigned long long)pool->instance_id);
    if (!same_slot_geometry(pool->g, host->g))
        return fail(KV_ERR_LAYOUT, "pool and host tier have different page geometry");
    if (num_layers == 0 || num_layers > kRing / 2 || (uint64_t)first_layer + num_layers > pool->g.L)
        return fail(KV_ERR_OUT_OF_RANGE, "layers [%u, %u + %u) are not inside [0, %llu) or exceed "
                    "%d", first_layer, first_layer, num_layers, (unsigned long long)pool->g.L,
                    kRing / 2);
    kv_status st = check_op(pool->g, host->num_slots, 1, host_slots, dst_pages, n, -1);
    if (st != KV_OK) return st;
    const int d = pool->device;
    DeviceGuard guard(d);
    st = init_device(d);
    if (st != KV_OK) return st;
    DevState &ds = g_dev[d];
    cudaStream_t stream = (cudaStream_t)stream_v;
    forget_stream(ds, stream_v);
    uint64_t seq0 = 0;
    st = reserve_fence_range(d, num_layers, &seq0);
    if (st != KV_OK) return st;
    if (n > 0) {
        // Counters of this call, zeroed in stream order.  The last slot's previous
        // user must have fully finished (its kernel may still be fetching tickets
        // after publishing its last fence): wait for that op's event first.
        const uint32_t k0 = (uint32_t)(seq0 % kRing);
        const uint32_t k_last = (uint32_t)((seq0 + num_layers - 1) % kRing);
        cudaError_t e = cudaSuccess;
        if (ds.slot_seq[k_last] != 0) e = cudaStreamWaitEvent(stream, ds.ev[k_last], 0);
        const uint32_t first_run = std::min<uint32_t>(num_layers, kRing - k0);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(ds.aux + k0, 0, first_run * sizeof(uint32_t), stream);
        if (e == cudaSuccess && first_run < num_layers)
            e = cudaMemsetAsync(ds.aux, 0, (num_layers - first_run) * sizeof(uint32_t), stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(ds.aux + kRing + k_last, 0, sizeof(uint32_t), stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(ds.aux + 2 * kRing + k_last, 0, sizeof(uint32_t), stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(ds.aux + 3 * kRing + k_last, 0, sizeof(uint32_t), stream);
        if (e != cudaSuccess) return cuda_fail(e, "zeroing the layer counters");
        const Side ps = pool_side(*pool), hs = host_side(*host);
        Plan p;
        st = plan(pool->g, hs, ps, num_layers, first_layer, ds.err_dev, false, &p);
        // above one launch's id capacity the ids go through device memory, so
        // that one kernel still publishes every layer of the whole op in order
        const bool device_ids = st == KV_OK && n > p.max_items;
        if (st == KV_OK) st = plan_layer_major(p, n, ds, seq0, device_ids);
        bool staged = false;
        if (st == KV_OK && device_ids) {
            st = stage_ids(ds, host_slots, dst_pages, n, stream);
            staged = st == KV_OK;
            p.d.gid_a = ds.gids;
            p.d.gid_b = ds.gids + n;
        }
        p.threads = progressive_threads();
        const int ctas = g_cfg.max_ctas ? (int)g_cfg.max_ctas
                         : p.threads == kWideThreads ? std::min(kOverlapWideCtas, ds.sms)
                                                     : default_ctas(ds, true, PK_REG, p.threads);
        if (st == KV_OK) st = run_moves(p, host_slots, dst_pages, n, ctas, stream, false);
        if (staged) {   // the id buffers are busy up to here in stream order, launched or not
            cudaError_t e2 = cudaEventRecord(ds.gids_free, stream);
            if (e2 != cudaSuccess) return cuda_fail(e2, "cudaEventRecord(ids)");
        }
        if (st != KV_OK) return st;
    } else {
        for (uint32_t j = 0; j < num_layers; ++j) {   // nothing to move: mark every layer
            cudaError_t e = launch_mark(ds.words_dev + (seq0 + j) % kRing, seq0 + j, stream);
            if (e != cudaSuccess) return cuda_fail(e, "launch of the completion marker");
            g_launches.fetch_add(1, std::memory_order_relaxed);
        }
    }
    for (uint32_t j = 0; j < num_layers; ++j) {
        const int k = (int)((seq0 + j) % kRing);
        cudaError_t e = cudaEventRecord(ds.ev[k], stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fence)");
        ds.slot_seq[k] = seq0 + j;
        fences[j] = ((uint64_t)d << 56) | (seq0 + j);
    }
    g_next_seq = seq0 + num_layers;
    return KV_OK;
}

kv_status kv_restore(kv_pool pool, kv_host host, const int32_t *host_slots,
                     const int32_t *dst_pages, uint32_t n, int32_t layer, void *stream,
                     kv_fence *fence) {
    std::lock_guard<std::mutex> lk(g_mu);
    return issue(pool, host, 1, host_slots, dst_pages, n, layer, stream, fence);
}

kv_status kv_device_gather(kv_pool pool, void *buf, uint64_t buf_bytes, uint32_t buf_heads,
                           const int32_t *src_pages, uint32_t n, void *stream, kv_fence *fence) {
    std::lock_guard<std::mutex> lk(g_mu);
    return issue_device(pool, buf, buf_bytes, buf_heads, 0, src_pages, n, -1, stream, fence);
}

kv_status kv_device_scatter(kv_pool pool, const void *buf, uint64_t buf_bytes, uint32_t buf_heads,
                            const int32_t *dst_pages, uint32_t n, int32_t layer, void *stream,
                            kv_fence *fence) {
    std::lock_guard<std::mutex> lk(g_mu);
    return issue_device(pool, (void *)buf, buf_bytes, buf_heads, 1, dst_pages, n, layer, stream,
                        fence);
}

kv_status kv_fence_query(kv_fence f) {
    bool done = false, aborted = false;
    int d = 0, k = 0;
    kv_status st = fence_state(f, &done, &d, &k, &aborted);
    if (st != KV_OK) return st;
    if (aborted)
        return fail(KV_ERR_ABORTED, "fence %llu: the ready fence was not reached in time; the "
                    "operation moved nothing", (unsigned long long)f);
    const uint32_t kerr = g_dev[d].err != nullptr ? __atomic_load_n(g_dev[d].err, __ATOMIC_ACQUIRE)
                                                  : 0u;
    if (kerr == 3u)
        return fail(KV_ERR_TIMEOUT, "an overlapped restore gave up waiting (2 s of GPU time) for "
                    "the previous restore's fence and published its own anyway: fences may have "
                    "completed out of call order");
    if (kerr != 0u)
        return fail(KV_ERR_OUT_OF_RANGE, "a transfer kernel met an out-of-range id and skipped it");
    return done ? KV_OK : KV_ERR_TIMEOUT;
}

kv_status kv_fence_wait(kv_fence f, uint64_t timeout_ns) {
    bool done = false, aborted = false;
    int d = 0, k = 0;
    kv_status st = fence_state(f, &done, &d, &k, &aborted);   // validates the fence once
    if (st != KV_OK) return st;
    // Poll the fence's mapped word directly (no lock): busy for the first 50 us
    // (small operations finish in a few microseconds), then yield the core
    // between polls up to 20 ms, then sleep.  A sleeping poller wakes tens of
    // microseconds after the word changes, which a caller that waits on every
    // step pays once per step: yielding up to 20 ms took the end-to-end
    // Llama-8B step from 199.4-200.5 to 201.2-201.3 GB/s and 61 one-layer MLA
    // restores from 203.7-204.0 to 207.9-208.0 GB/s.
    const unsigned long long *word = &g_dev[d].words[k];
    const uint64_t seq = f & kSeqMask;
    const double t0 = now_ns(), deadline = t0 + (double)timeout_ns;
    while (!done) {
        if (load_acquire(word) >= seq) break;
        const double t = now_ns();
        if (t >= deadline)
            return fail(KV_ERR_TIMEOUT, "fence %llu not complete after %llu ns",
                        (unsigned long long)f, (unsigned long long)timeout_ns);
        if (t - t0 < 50e3) continue;
        if (t - t0 < 20e6) {
            sched_yield();
        } else {
            timespec ts{0, 20000};
            nanosleep(&ts, nullptr);
        }
    }
    return kv_fence_query(f);   // complete: report aborted ops and kernel id errors
}

kv_status kv_fence_stream_wait(kv_fence f, void *stream) {
    bool done = false, aborted = false;
    int d = 0, k = 0;
    kv_status st = fence_state(f, &done, &d, &k, &aborted);
    if (st != KV_OK) return st;
    if (done) return KV_OK;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceGuard guard(d);
    DevState &ds = g_dev[d];
    if (ds.wait_value) {
        // Wait on the GPU for the fence word itself: right for fences that a
        // kernel publishes before it ends (progressive layers), and slot reuse
        // only ever raises the word, so it is never early.
        CUresult r = g_wait_value64((CUstream)stream, (CUdeviceptr)(uintptr_t)(ds.words_dev + k),
                                    (cuuint64_t)(f & kSeqMask), CU_STREAM_WAIT_VALUE_GEQ);
        if (r != CUDA_SUCCESS)
            return fail(KV_ERR_CUDA, "cuStreamWaitValue64(fence word) failed (CUresult %d)", (int)r);
        return KV_OK;
    }
    // The slot's event is this fence's, or a later one recorded only after this
    // fence completed (slots are reused only then): never too early.
    cudaError_t e = cudaStreamWaitEvent((cudaStream_t)stream, ds.ev[k], 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(fence)");
    return KV_OK;
}

}  // extern "C"
