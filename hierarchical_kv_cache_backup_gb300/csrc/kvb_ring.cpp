// kvb_ring.cpp -- shared-memory descriptor ring between a submitting process
// (the scheduler) and a serving process (the data plane).
//
// "[Feature] [RFC] [HiCache] Out-of-process HiCache data plane with
// device-memory IPC", §Device IPC data path: after the pool is registered once,
// operations only carry descriptors (page IDs, keys, fences), over a control
// path such as shared-memory submission / completion rings, NVMe-style; and
// device-memory sharing and cross-process synchronization are separate
// capabilities.  Here the bulk bytes never leave the GPU / host tier, the
// ring carries descriptors, and completion is written by the GPU straight into
// the shared page the submitter polls.
//
// Layout of the shared segment (page-aligned regions):
//   [0, 4096)            RingHeader (with the ready words of gated descriptors)
//   [comp_off, +C)       CompRec[slots]   (registered with CUDA by the server)
//   [entry_off, +E)      kv_ring_op[slots]
// Ticket t (1, 2, ...) uses slot (t - 1) % slots.  tail = last ticket published
// by the submitter, head = last ticket taken by the server.  A slot is reused
// for ticket t only when t - slots has been taken and completed.
#include "kvb.h"
#include "kvb_internal.h"
#include "kvb_ring_internal.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cerrno>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <ctime>
#include <fcntl.h>
#include <mutex>
#include <sched.h>
#include <string>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>
#include <unordered_map>
#include <vector>

namespace {

constexpr uint32_t kRingMagic = 0x4B565252u;   // "KVRR"
constexpr uint32_t kRingVersion = 2u;   // 2: ready words, gated descriptors
constexpr uint32_t kMaxSlots = 4096;
constexpr size_t kPage = 4096;

struct RingHeader {
    uint32_t magic, version, slots, entry_bytes;
    uint64_t comp_off, entry_off, total_bytes;
    int64_t creator_pid;
    alignas(64) uint64_t tail;        // last published ticket
    alignas(64) uint64_t head;        // last taken ticket
    alignas(64) int64_t server_pid;   // last server that took a descriptor
    alignas(64) uint64_t ready[KV_RING_READY_WORDS];   // ready fences of gated descriptors
};
static_assert(sizeof(RingHeader) <= kPage, "ring header fits one page");

// Completion records (kvb::CompRec): `done` is written by the GPU (or the CPU)
// when ticket `done` is complete; err_ticket / err before it when it failed.
using kvb::CompRec;
constexpr uint32_t kMaxServerPools = 64;

struct RingObj {
    std::string name;
    bool creator;
    int fd;
    void *base;
    size_t bytes;
    RingHeader *h;
    CompRec *comp;
    kv_ring_op *ops;
    std::mutex mu;                  // one submitter / one server thread at a time
    char *seg_dev = nullptr;        // device view of the whole segment once a server registered it
    CompRec *comp_dev = nullptr;    // device view of the completion records
    bool registered = false;
    // GPU-resident server (kv_ring_serve_device): scratch on its device
    int srv_device = -1;
    kvb::RingCtl *srv_ctl = nullptr;
    int32_t *srv_ids = nullptr;
    kvb::RingPoolK *srv_pools = nullptr;
    uint32_t *srv_result = nullptr;       // mapped pinned: served, status
    uint32_t *srv_result_dev = nullptr;
    kv_fence srv_fence = 0;               // completes when the last resident server ended
    // Stores into the segment queued on streams (ready words set from a stream,
    // completion marks of the host server): per (stream, device), an event
    // recorded after the last one; close waits for them before unmapping.
    struct PendingStore {
        void *stream;
        int device;
        cudaEvent_t ev;
    };
    std::vector<PendingStore> stores;
};

std::mutex g_rings_mu;
std::unordered_map<uint64_t, RingObj *> g_rings;
uint64_t g_next_ring = 1;

kv_status err(kv_status st, const char *msg) {
    return (kv_status)kvb::set_last_error(st, msg);
}

double now_ns() {
    timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return ts.tv_sec * 1e9 + ts.tv_nsec;
}

// Busy for the first 50 us of a wait, then yield until 20 ms, then sleep.
void backoff(int &spins) {
    static thread_local double t0;
    if (spins++ == 0) t0 = now_ns();
    const double t = now_ns() - t0;
    if (t < 50e3) return;
    if (t < 20e6) {
        sched_yield();
    } else {
        timespec ts{0, 10000};
        nanosleep(&ts, nullptr);
    }
}

uint64_t ld(const uint64_t *p) { return __atomic_load_n(p, __ATOMIC_ACQUIRE); }
void st(uint64_t *p, uint64_t v) { __atomic_store_n(p, v, __ATOMIC_RELEASE); }

size_t round_page(size_t x) { return (x + kPage - 1) / kPage * kPage; }

bool valid_name(const char *name) {
    if (name == nullptr || name[0] != '/' || name[1] == '\0') return false;
    const size_t n = strnlen(name, 256);
    if (n >= 255) return false;
    return std::strchr(name + 1, '/') == nullptr;
}

RingObj *find(kv_ring r) {
    std::lock_guard<std::mutex> lk(g_rings_mu);
    auto it = g_rings.find((uint64_t)(uintptr_t)r);
    return it == g_rings.end() ? nullptr : it->second;
}

kv_ring publish(RingObj *o) {
    std::lock_guard<std::mutex> lk(g_rings_mu);
    const uint64_t id = g_next_ring++;
    g_rings[id] = o;
    return (kv_ring)(uintptr_t)id;
}

void bind(RingObj *o) {
    char *b = (char *)o->base;
    o->h = (RingHeader *)b;
    o->comp = (CompRec *)(b + o->h->comp_off);
    o->ops = (kv_ring_op *)(b + o->h->entry_off);
}

// The completion and entry regions of a header lie, in order and page-aligned,
// between the header page and the end of the segment.
bool regions_fit(const RingHeader *h) {
    const uint64_t comp_end = h->comp_off + (uint64_t)h->slots * sizeof(CompRec);
    const uint64_t entry_end = h->entry_off + (uint64_t)h->slots * sizeof(kv_ring_op);
    return h->comp_off >= kPage && h->comp_off % kPage == 0 && h->entry_off % kPage == 0 &&
           h->comp_off <= h->total_bytes && h->entry_off <= h->total_bytes &&
           comp_end <= h->entry_off && entry_end <= h->total_bytes;
}

// The whole segment becomes device-visible (once): the GPU stores each
// ticket into its completion record, and a resident server reads the header
// and the entries too.
kv_status register_segment(RingObj *o) {
    if (o->registered) return KV_OK;
    cudaError_t e = cudaHostRegister(o->base, o->bytes,
                                     cudaHostRegisterMapped | cudaHostRegisterPortable);
    void *dv = nullptr;
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dv, o->base, 0);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return err(KV_ERR_CUDA, "registering the ring segment with CUDA failed");
    }
    o->seg_dev = (char *)dv;
    o->comp_dev = (CompRec *)(o->seg_dev + o->h->comp_off);
    o->registered = true;
    return KV_OK;
}

// After a store into the segment was launched on `stream` (current device):
// records that stream's event, so close can tell when the store has run.
// Caller holds o->mu.
kv_status note_store(RingObj *o, void *stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return err(KV_ERR_CUDA, "cudaGetDevice failed");
    }
    RingObj::PendingStore *ps = nullptr;
    for (auto &x : o->stores)
        if (x.stream == stream && x.device == dev) ps = &x;
    if (ps == nullptr) {
        cudaEvent_t ev = nullptr;
        if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            return err(KV_ERR_CUDA, "cudaEventCreate for a ring store failed");
        }
        o->stores.push_back(RingObj::PendingStore{stream, dev, ev});
        ps = &o->stores.back();
    }
    if (cudaEventRecord(ps->ev, (cudaStream_t)stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return err(KV_ERR_CUDA, "cudaEventRecord after a ring store failed");
    }
    return KV_OK;
}

// Runs f() with `device` current, then restores the caller's device.
template <class F>
void on_device(int device, F f) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != device) cudaSetDevice(device);
    f();
    if (prev >= 0 && prev != device) cudaSetDevice(prev);
}

// Whether every store queued into the segment has run, polling for at most
// timeout_ns (each event queried with its own device current).
bool stores_done(RingObj *o, double timeout_ns) {
    const double deadline = now_ns() + timeout_ns;
    for (auto &x : o->stores) {
        bool done = false, expired = false;
        on_device(x.device, [&] {
            for (;;) {
                const cudaError_t e = cudaEventQuery(x.ev);
                if (e == cudaSuccess) {
                    done = true;
                    return;
                }
                if (e != cudaErrorNotReady) {   // a broken context: nothing will run any more
                    (void)cudaGetLastError();
                    done = true;
                    return;
                }
                if (now_ns() >= deadline) {
                    expired = true;
                    return;
                }
                timespec ts{0, 50000};
                nanosleep(&ts, nullptr);
            }
        });
        if (expired && !done) return false;
    }
    return true;
}

uint32_t slot_of(const RingObj *o, uint64_t t) { return (uint32_t)((t - 1) % o->h->slots); }

// A gated descriptor names a ready word that does not exist or a wait above 60 s.
bool bad_gate(const kv_ring_op &op) {
    return op.ready_value != 0 &&
           (op.ready_index >= KV_RING_READY_WORDS || op.ready_timeout_ms > 60000u);
}

// CPU completion of ticket t with status s (error record first, then done).
void complete_cpu(RingObj *o, uint64_t t, kv_status s) {
    CompRec &c = o->comp[slot_of(o, t)];
    if (s != KV_OK) {
        c.err = (int32_t)s;
        st(&c.err_ticket, t);
    }
    st(&c.done, t);
}

}  // namespace

extern "C" {

kv_status kv_ring_create(const char *name, uint32_t slots, kv_ring *out) {
    if (out == nullptr) return err(KV_ERR_INVALID_ARG, "output handle pointer is NULL");
    if (!valid_name(name)) return err(KV_ERR_INVALID_ARG, "ring name must be \"/name\"");
    if (slots < 2 || slots > kMaxSlots) return err(KV_ERR_INVALID_ARG, "slots must be 2..4096");
    const size_t comp_off = kPage;
    const size_t comp_bytes = round_page(slots * sizeof(CompRec));
    const size_t entry_off = comp_off + comp_bytes;
    const size_t total = entry_off + round_page((size_t)slots * sizeof(kv_ring_op));
    const int fd = shm_open(name, O_CREAT | O_EXCL | O_RDWR, 0600);
    if (fd < 0)
        return err(KV_ERR_INVALID_ARG, errno == EEXIST ? "a ring of that name already exists"
                                                       : "shm_open failed");
    if (ftruncate(fd, (off_t)total) != 0) {
        close(fd);
        shm_unlink(name);
        return err(KV_ERR_NO_MEMORY, "ftruncate of the ring failed");
    }
    void *base = mmap(nullptr, total, PROT_READ | PROT_WRITE, MAP_SHARED, fd, 0);
    if (base == MAP_FAILED) {
        close(fd);
        shm_unlink(name);
        return err(KV_ERR_NO_MEMORY, "mmap of the ring failed");
    }
    std::memset(base, 0, total);
    RingHeader *h = (RingHeader *)base;
    h->slots = slots;
    h->entry_bytes = (uint32_t)sizeof(kv_ring_op);
    h->comp_off = comp_off;
    h->entry_off = entry_off;
    h->total_bytes = total;
    h->creator_pid = (int64_t)getpid();
    h->version = kRingVersion;
    __atomic_store_n(&h->magic, kRingMagic, __ATOMIC_RELEASE);   // last: marks it initialised
    RingObj *o = new RingObj{name, true, fd, base, total, nullptr, nullptr, nullptr, {}};
    bind(o);
    *out = publish(o);
    return KV_OK;
}

kv_status kv_ring_attach(const char *name, kv_ring *out) {
    if (out == nullptr) return err(KV_ERR_INVALID_ARG, "output handle pointer is NULL");
    if (!valid_name(name)) return err(KV_ERR_INVALID_ARG, "ring name must be \"/name\"");
    const int fd = shm_open(name, O_RDWR, 0600);
    if (fd < 0) return err(KV_ERR_INVALID_ARG, "no ring of that name");
    struct stat sb;
    if (fstat(fd, &sb) != 0 || (size_t)sb.st_size < kPage) {
        close(fd);
        return err(KV_ERR_INVALID_ARG, "ring segment too small");
    }
    void *base = mmap(nullptr, (size_t)sb.st_size, PROT_READ | PROT_WRITE, MAP_SHARED, fd, 0);
    if (base == MAP_FAILED) {
        close(fd);
        return err(KV_ERR_NO_MEMORY, "mmap of the ring failed");
    }
    RingHeader *h = (RingHeader *)base;
    if (__atomic_load_n(&h->magic, __ATOMIC_ACQUIRE) != kRingMagic || h->version != kRingVersion ||
        h->entry_bytes != sizeof(kv_ring_op) || h->total_bytes != (uint64_t)sb.st_size ||
        h->slots < 2 || h->slots > kMaxSlots || !regions_fit(h)) {
        munmap(base, (size_t)sb.st_size);
        close(fd);
        return err(KV_ERR_INVALID_ARG, "segment is not a ring of this version");
    }
    RingObj *o = new RingObj{name, false, fd, base, (size_t)sb.st_size, nullptr, nullptr, nullptr,
                             {}};
    bind(o);
    *out = publish(o);
    return KV_OK;
}

kv_status kv_ring_close(kv_ring r) {
    RingObj *o;
    const uint64_t id = (uint64_t)(uintptr_t)r;
    {
        std::lock_guard<std::mutex> lk(g_rings_mu);
        auto it = g_rings.find(id);
        if (it == g_rings.end()) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
        o = it->second;
        g_rings.erase(it);
    }
    // A store into the segment still queued on a stream would land in unmapped
    // memory after munmap: wait (bounded) for each, else keep the ring open.
    if (!stores_done(o, 2e9)) {
        std::lock_guard<std::mutex> lk(g_rings_mu);
        g_rings[id] = o;
        return err(KV_ERR_TIMEOUT, "a store into the ring's segment queued on a stream "
                   "(kv_ring_ready_stream_set, or a completion of kv_ring_serve) has not run "
                   "within 2 s: the ring stays open; close it again once that stream's work "
                   "has finished");
    }
    for (auto &x : o->stores) on_device(x.device, [&] { cudaEventDestroy(x.ev); });
    o->stores.clear();
    kv_status s = KV_OK;
    if (o->srv_fence != 0 && kv_fence_query(o->srv_fence) == KV_ERR_TIMEOUT) {
        // a resident server still reads the segment: ask it to stop, and never
        // unmap under it (if it has not ended in time, everything is left mapped)
        __atomic_store_n(&o->srv_result[2], 1u, __ATOMIC_RELEASE);
        if (kv_fence_wait(o->srv_fence, 120ull * 1000 * 1000 * 1000) == KV_ERR_TIMEOUT)
            return err(KV_ERR_TIMEOUT, "the ring's resident server did not stop: the ring is "
                       "closed but its memory stays mapped");
    }
    if (o->srv_ctl != nullptr) {   // one allocation: control block, ids, pool table
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != o->srv_device) cudaSetDevice(o->srv_device);
        cudaFree(o->srv_ctl);
        if (prev >= 0 && prev != o->srv_device) cudaSetDevice(prev);
    }
    if (o->srv_result != nullptr) cudaFreeHost(o->srv_result);
    if (o->registered && cudaHostUnregister(o->base) != cudaSuccess) {
        (void)cudaGetLastError();
        s = err(KV_ERR_CUDA, "cudaHostUnregister of the ring segment failed");
    }
    munmap(o->base, o->bytes);
    close(o->fd);
    if (o->creator) shm_unlink(o->name.c_str());
    delete o;
    return s;
}

kv_status kv_ring_submit(kv_ring r, const kv_ring_op *op, uint64_t timeout_ns, uint64_t *ticket) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (op == nullptr || ticket == nullptr) return err(KV_ERR_INVALID_ARG, "NULL argument");
    if (op->kind > KV_RING_OP_RESTORE) return err(KV_ERR_INVALID_ARG, "unknown operation kind");
    if (op->n > KV_RING_MAX_IDS) return err(KV_ERR_INVALID_ARG, "n exceeds KV_RING_MAX_IDS");
    if (bad_gate(*op))
        return err(KV_ERR_INVALID_ARG, "gated descriptor: ready_index must be below "
                   "KV_RING_READY_WORDS and ready_timeout_ms at most 60000");
    std::lock_guard<std::mutex> lk(o->mu);
    RingHeader *h = o->h;
    const uint64_t t = ld(&h->tail) + 1;
    const uint64_t slots = h->slots;
    const double deadline = now_ns() + (double)timeout_ns;
    int spins = 0;
    // the slot's previous ticket (t - slots) must be taken and completed
    while (t > slots && (ld(&h->head) < t - slots ||
                         ld(&o->comp[slot_of(o, t)].done) < t - slots)) {
        if (now_ns() >= deadline) return err(KV_ERR_TIMEOUT, "ring full: the server is behind");
        backoff(spins);
    }
    kv_ring_op &e = o->ops[slot_of(o, t)];
    std::memcpy(&e, op, offsetof(kv_ring_op, a));
    std::memcpy(e.a, op->a, op->n * sizeof(int32_t));
    std::memcpy(e.b, op->b, op->n * sizeof(int32_t));
    st(&h->tail, t);
    *ticket = t;
    return KV_OK;
}

kv_status kv_ring_wait(kv_ring r, uint64_t ticket, uint64_t timeout_ns, kv_status *op_status) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (ticket == 0 || ticket > ld(&o->h->tail))
        return err(KV_ERR_INVALID_ARG, "ticket was never submitted");
    CompRec &c = o->comp[slot_of(o, ticket)];
    const double deadline = now_ns() + (double)timeout_ns;
    int spins = 0;
    while (ld(&c.done) < ticket) {
        if (now_ns() >= deadline) return err(KV_ERR_TIMEOUT, "ticket not complete in time");
        backoff(spins);
    }
    if (op_status != nullptr)
        *op_status = ld(&c.err_ticket) == ticket ? (kv_status)__atomic_load_n(&c.err,
                                                                             __ATOMIC_ACQUIRE)
                                                 : KV_OK;
    return KV_OK;
}

kv_status kv_ring_pop(kv_ring r, uint64_t timeout_ns, kv_ring_op *op, uint64_t *ticket) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (op == nullptr || ticket == nullptr) return err(KV_ERR_INVALID_ARG, "NULL argument");
    std::lock_guard<std::mutex> lk(o->mu);
    RingHeader *h = o->h;
    const uint64_t t = ld(&h->head) + 1;
    const double deadline = now_ns() + (double)timeout_ns;
    int spins = 0;
    while (ld(&h->tail) < t) {
        if (now_ns() >= deadline) return err(KV_ERR_TIMEOUT, "no descriptor in time");
        backoff(spins);
    }
    const kv_ring_op &e = o->ops[slot_of(o, t)];
    std::memcpy(op, &e, offsetof(kv_ring_op, a));
    // The entry comes from another process's memory: a descriptor that
    // kv_ring_submit would have refused is taken and failed here, not served.
    const bool malformed = op->n > KV_RING_MAX_IDS || op->kind > KV_RING_OP_RESTORE ||
                           bad_gate(*op);
    const uint32_t n = malformed ? 0 : op->n;
    std::memcpy(op->a, e.a, n * sizeof(int32_t));
    std::memcpy(op->b, e.b, n * sizeof(int32_t));
    __atomic_store_n(&h->server_pid, (int64_t)getpid(), __ATOMIC_RELAXED);
    st(&h->head, t);   // the slot may now be refilled (after t completes)
    *ticket = t;
    if (malformed) {
        op->n = 0;
        complete_cpu(o, t, KV_ERR_INVALID_ARG);
        return err(KV_ERR_INVALID_ARG, "descriptor with an unknown kind, n above "
                   "KV_RING_MAX_IDS or a bad gate: taken and completed with INVALID_ARG");
    }
    return KV_OK;
}

kv_status kv_ring_complete(kv_ring r, uint64_t ticket, kv_status op_status) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (ticket == 0 || ticket > ld(&o->h->head))
        return err(KV_ERR_INVALID_ARG, "ticket was never taken");
    complete_cpu(o, ticket, op_status);
    return KV_OK;
}

kv_status kv_ring_ready_set(kv_ring r, uint32_t index, uint64_t value) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (index >= KV_RING_READY_WORDS)
        return err(KV_ERR_INVALID_ARG, "ready index must be below KV_RING_READY_WORDS");
    st(&o->h->ready[index], value);
    return KV_OK;
}

kv_status kv_ring_ready_stream_set(kv_ring r, uint32_t index, uint64_t value, void *stream) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (index >= KV_RING_READY_WORDS)
        return err(KV_ERR_INVALID_ARG, "ready index must be below KV_RING_READY_WORDS");
    std::lock_guard<std::mutex> lk(o->mu);
    kv_status rs = register_segment(o);
    if (rs != KV_OK) return rs;
    unsigned long long *word =
        (unsigned long long *)(o->seg_dev + offsetof(RingHeader, ready)) + index;
    cudaError_t e = kvb::launch_mark(word, value, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return err(KV_ERR_CUDA, "launch of the ready-word store failed");
    }
    return note_store(o, stream);
}

kv_status kv_ring_serve(kv_ring r, const kv_pool *pools, uint32_t npools, kv_host host,
                        void *stream, uint32_t max_ops, uint64_t idle_timeout_ns,
                        uint32_t *served) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (served == nullptr || (npools > 0 && pools == nullptr))
        return err(KV_ERR_INVALID_ARG, "NULL argument");
    *served = 0;
    kv_status rs;
    {
        std::lock_guard<std::mutex> lk(o->mu);
        rs = register_segment(o);
    }
    if (rs != KV_OK) return rs;
    static thread_local kv_ring_op op;
    for (uint32_t k = 0; k < max_ops; ++k) {
        uint64_t t = 0;
        kv_status s = kv_ring_pop(r, k == 0 ? idle_timeout_ns : 0, &op, &t);
        if (s == KV_ERR_TIMEOUT) break;
        if (s == KV_ERR_INVALID_ARG && t != 0) {   // malformed: already completed by pop
            ++*served;
            continue;
        }
        if (s != KV_OK) return s;
        ++*served;
        if (op.pool_index >= npools) {
            complete_cpu(o, t, KV_ERR_INVALID_ARG);
            continue;
        }
        kv_fence f = 0;
        const bool gated = op.ready_value != 0;
        const uint64_t *ready = (const uint64_t *)(o->seg_dev + offsetof(RingHeader, ready)) +
                                op.ready_index;
        const uint64_t ready_ns =
            (uint64_t)(op.ready_timeout_ms ? op.ready_timeout_ms : 10000u) * 1000000ull;
        CompRec *cd = &o->comp_dev[slot_of(o, t)];
        // An ungated op's move kernel completes the ticket itself, right after its
        // fence (no marker kernel between consecutive ops on the stream, so
        // restores overlapped under KV_CFG_OVERLAP_RESTORES stay overlapped).
        int fused = 0;
        if (op.kind == KV_RING_OP_BACKUP)
            s = op.layer != -1 ? KV_ERR_INVALID_ARG
                : gated ? kv_backup_when_ready(pools[op.pool_index], host, op.a, op.b, op.n, ready,
                                               op.ready_value, ready_ns, stream, &f)
                        : (kv_status)kvb::ring_issue(pools[op.pool_index], host, 0, op.a, op.b,
                                                     op.n, -1, stream,
                                                     (unsigned long long *)&cd->done, t, &f,
                                                     &fused);
        else
            s = gated ? kv_restore_when_ready(pools[op.pool_index], host, op.a, op.b, op.n,
                                              op.layer, ready, op.ready_value, ready_ns, stream,
                                              &f)
                      : (kv_status)kvb::ring_issue(pools[op.pool_index], host, 1, op.a, op.b,
                                                   op.n, op.layer, stream,
                                                   (unsigned long long *)&cd->done, t, &f, &fused);
        if (s != KV_OK) {
            complete_cpu(o, t, s);
            continue;
        }
        int device = 0;
        kvb::pool_device_of(pools[op.pool_index], &device);
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != device) cudaSetDevice(device);
        cudaError_t e = cudaSuccess;
        kv_status fail_st = KV_OK;   // completed from the CPU with this status instead
        if (gated) {   // the ticket reports a gate that gave up (ABORTED)
            const unsigned long long *status = nullptr;
            unsigned long long tag = 0;
            const int gs = kvb::fence_gate_word(f, &status, &tag);
            if (gs != KV_OK)
                fail_st = (kv_status)gs;   // never report a gated op OK without its gate's word
            else
                e = kvb::launch_ring_mark((unsigned long long *)&cd->done,
                                          (unsigned long long *)&cd->err_ticket, &cd->err, t,
                                          status, tag, (cudaStream_t)stream);
        } else if (!fused) {
            e = kvb::launch_mark((unsigned long long *)&cd->done, t, (cudaStream_t)stream);
        }
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            fail_st = KV_ERR_CUDA;
        } else if (fail_st == KV_OK) {
            std::lock_guard<std::mutex> lk(o->mu);
            fail_st = note_store(o, stream);
            if (fail_st != KV_OK) {
                // the store is queued but close could not see it: let it run first
                cudaStreamSynchronize((cudaStream_t)stream);
                fail_st = KV_OK;
            }
        }
        if (prev >= 0 && prev != device) cudaSetDevice(prev);
        if (fail_st != KV_OK) {
            kv_fence_wait(f, 60ull * 1000 * 1000 * 1000);   // the bytes land; report the failure
            complete_cpu(o, t, fail_st);
        }
    }
    return KV_OK;
}

kv_status kv_ring_serve_device(kv_ring r, const kv_pool *pools, uint32_t npools, kv_host host,
                               void *stream, uint32_t max_ops, uint64_t idle_timeout_ns,
                               kv_fence *fence) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (fence == nullptr) return err(KV_ERR_INVALID_ARG, "fence output pointer is NULL");
    if (npools > kMaxServerPools) return err(KV_ERR_INVALID_ARG, "more than 64 pools");
    if (idle_timeout_ns > 60ull * 1000 * 1000 * 1000)
        return err(KV_ERR_INVALID_ARG, "idle_timeout_ns exceeds the 60 s limit");
    kvb::RingPoolK table[kMaxServerPools];
    kvb::Side host_side;
    uint32_t num_slots = 0;
    int device = -1;
    kv_status st = (kv_status)kvb::ring_server_view(pools, npools, host, table, &host_side,
                                                    &num_slots, &device);
    if (st != KV_OK) return st;
    std::lock_guard<std::mutex> lk(o->mu);
    if (o->srv_fence != 0 && kv_fence_query(o->srv_fence) == KV_ERR_TIMEOUT)
        return err(KV_ERR_INVALID_ARG, "a resident server is still running on this ring");
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != device) cudaSetDevice(device);
    struct Restore {
        int prev, device;
        ~Restore() {
            if (prev >= 0 && prev != device) cudaSetDevice(prev);
        }
    } restore{prev, device};
    // Everything that may synchronize with the device (registration, allocations)
    // happens before the launch: afterwards it would wait for the server to end.
    st = register_segment(o);
    if (st != KV_OK) return st;
    auto ck = [](cudaError_t e, const char *what) {
        if (e == cudaSuccess) return KV_OK;
        (void)cudaGetLastError();
        return err(KV_ERR_CUDA, what);
    };
    if (o->srv_ctl != nullptr && o->srv_device != device) {   // scratch of another device
        cudaSetDevice(o->srv_device);
        cudaFree(o->srv_ctl);
        cudaSetDevice(device);
        o->srv_ctl = nullptr;
    }
    const size_t ids_off = 256, pools_off = ids_off + 2 * KV_RING_MAX_IDS * sizeof(int32_t);
    static_assert(sizeof(kvb::RingCtl) <= 256, "control block fits its slot");
    if (o->srv_ctl == nullptr) {
        void *p = nullptr;
        st = ck(cudaMalloc(&p, pools_off + kMaxServerPools * sizeof(kvb::RingPoolK)),
                "cudaMalloc of the resident server's scratch failed");
        if (st != KV_OK) return st;
        o->srv_ctl = (kvb::RingCtl *)p;
        o->srv_ids = (int32_t *)((char *)p + ids_off);
        o->srv_pools = (kvb::RingPoolK *)((char *)p + pools_off);
        o->srv_device = device;
    }
    if (o->srv_result == nullptr) {
        void *h = nullptr, *d = nullptr;
        st = ck(cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable),
                "cudaHostAlloc of the resident server's result words failed");
        if (st != KV_OK) return st;
        st = ck(cudaHostGetDevicePointer(&d, h, 0), "mapping the result words failed");
        if (st != KV_OK) {
            cudaFreeHost(h);
            return st;
        }
        o->srv_result = (uint32_t *)h;
        o->srv_result_dev = (uint32_t *)d;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    // leader + movers: kRingMovers, or the configured CTA cap of move kernels
    kv_config cfg{};
    const int want = kv_config_get(&cfg) == KV_OK && cfg.max_ctas != 0 ? (int)cfg.max_ctas
                                                                      : kvb::kRingMovers;
    const int ctas = 1 + std::max(1, std::min(want, sms - 1));
    cudaStream_t s = (cudaStream_t)stream;
    o->srv_result[0] = 0;
    o->srv_result[1] = (uint32_t)KV_OK;
    __atomic_store_n(&o->srv_result[2], 0u, __ATOMIC_RELEASE);   // no stop request
    st = ck(cudaMemcpyAsync(o->srv_pools, table, npools * sizeof(kvb::RingPoolK),
                            cudaMemcpyHostToDevice, s), "copying the pool table failed");
    if (st == KV_OK)
        st = ck(cudaMemsetAsync(o->srv_ctl, 0, sizeof(kvb::RingCtl), s),
                "zeroing the control block failed");
    if (st != KV_OK) return st;
    kvb::RingKDesc k{};
    k.tail = (const unsigned long long *)(o->seg_dev + offsetof(RingHeader, tail));
    k.ready = (const unsigned long long *)(o->seg_dev + offsetof(RingHeader, ready));
    k.head = (unsigned long long *)(o->seg_dev + offsetof(RingHeader, head));
    k.server_pid = (long long *)(o->seg_dev + offsetof(RingHeader, server_pid));
    k.ops = (const kv_ring_op *)(o->seg_dev + o->h->entry_off);
    k.comp = o->comp_dev;
    k.slots = o->h->slots;
    k.max_ops = max_ops;
    k.first_ticket = ld(&o->h->head) + 1;
    k.idle_ns = idle_timeout_ns;
    k.pid = (long long)getpid();
    k.host = host_side;
    k.num_slots = num_slots;
    k.npools = npools;
    k.pools = o->srv_pools;
    k.ctl = o->srv_ctl;
    k.ids = o->srv_ids;
    k.result = o->srv_result_dev;
    st = (kv_status)kvb::ring_launch_server(device, k, ctas, s, fence);
    if (st != KV_OK) return st;
    o->srv_fence = *fence;
    return KV_OK;
}

kv_status kv_ring_device_stop(kv_ring r) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    std::lock_guard<std::mutex> lk(o->mu);
    if (o->srv_fence == 0) return err(KV_ERR_INVALID_ARG, "no resident server was started");
    __atomic_store_n(&o->srv_result[2], 1u, __ATOMIC_RELEASE);
    return KV_OK;
}

kv_status kv_ring_device_result(kv_ring r, uint32_t *served, kv_status *status) {
    RingObj *o = find(r);
    if (o == nullptr) return err(KV_ERR_CLOSED, "ring handle is closed or unknown");
    if (served == nullptr || status == nullptr) return err(KV_ERR_INVALID_ARG, "NULL argument");
    std::lock_guard<std::mutex> lk(o->mu);
    if (o->srv_fence == 0) return err(KV_ERR_INVALID_ARG, "no resident server was started");
    if (kv_fence_query(o->srv_fence) == KV_ERR_TIMEOUT)
        return err(KV_ERR_TIMEOUT, "the resident server is still running");
    *served = __atomic_load_n(&o->srv_result[0], __ATOMIC_ACQUIRE);
    *status = (kv_status)__atomic_load_n(&o->srv_result[1], __ATOMIC_ACQUIRE);
    return KV_OK;
}

}  // extern "C"
