// kvb_l3.cpp -- the hop below the host tier: whole pages between host-tier
// slots and fixed-size records of a file descriptor (a regular file, a block
// device or a memfd).
//
// "[Feature] [RFC] [HiCache] Out-of-process HiCache data plane with
// device-memory IPC": §Summary draws the daemon with a host tier and "external
// L3 storage clients" below it, and §Relationship to existing SGLang work
// (#24542, the standalone L3 StorageServer) keeps the bulk bytes of that tier
// in shared memfd host memory.  A record store here is the plainest such
// tier: record r is the page-sized byte range [base + r * RB, base + (r+1) * RB)
// of the descriptor, RB = the host tier's page bytes, and a put / get copies
// whole pages between slots and records without looking at them.
//
// Engine: a persistent pool of worker threads per store.  A call is split into
// runs of consecutive records (at most 1,024 pages and 64 MiB per run) and the
// workers take runs from an atomic counter.  A regular file or memfd opened
// read-write (without O_DIRECT) is mapped shared once, and a run is plain
// memcpy between slots and the mapping: buffered write() to one file takes the
// inode lock, so parallel pwritev calls would run one at a time.  Block
// devices, O_DIRECT and read- or write-only descriptors take the syscall path:
// one pwritev / preadv per run, gathering / scattering the run's slots.  Before
// a mapped call the file size is checked (a put grows the file to its last
// record, a get past the end fails), so no copy touches a page past the end.
// Calls on one store are serialised; calls block until every byte has moved or
// an error stops them.
#include "kvb.h"
#include "kvb_internal.h"

#include <algorithm>
#include <atomic>
#include <cerrno>
#include <cstdarg>
#include <condition_variable>
#include <cstdio>
#include <cstring>
#include <limits.h>
#include <memory>
#include <mutex>
#include <string>
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <sys/uio.h>
#include <thread>
#include <unistd.h>
#include <unordered_map>
#include <vector>

namespace {

constexpr uint32_t kRunPages = 1024;             // iovecs per pwritev / preadv
constexpr uint64_t kRunBytes = 64ull << 20;      // bytes per run (load balance)
constexpr uint32_t kMaxThreads = 64;
constexpr uint32_t kDefaultThreads = 8;

kv_status err(kv_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
kv_status err(kv_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return (kv_status)kvb::set_last_error(st, buf);
}

struct Run {
    uint64_t file_off;   // first byte in the file
    uint32_t first;      // index of the run's first item in the call
    uint32_t count;      // items in the run (consecutive records)
};

struct Job {
    bool put;
    char *host;
    uint64_t rb;
    const int32_t *slots;
    std::vector<Run> runs;
    std::atomic<uint32_t> next{0};
    std::atomic<int> failed{0};
    int err_no = 0;            // first failure (under Store::mu)
    uint64_t err_off = 0;
    bool short_read = false;
};

struct Store {
    int fd;
    uint64_t base, rb, nrec;
    char *map = nullptr;       // mapped store region (record 0 at map + skew), or null
    uint64_t map_len = 0, skew = 0;
    std::mutex call_mu;        // one call at a time
    bool closed = false;       // set under call_mu by kv_l3_close
    std::mutex mu;             // job hand-off
    std::condition_variable cv_work, cv_done;
    Job *job = nullptr;
    uint64_t job_gen = 0;
    uint32_t busy = 0;         // workers inside the current job
    bool stop = false;
    std::vector<std::thread> workers;

    ~Store() {   // kv_l3_close has joined the workers; this covers a failed open
        {
            std::lock_guard<std::mutex> lk(mu);
            stop = true;
        }
        cv_work.notify_all();
        for (auto &w : workers)
            if (w.joinable()) w.join();
        if (map != nullptr) munmap(map - skew, map_len);
    }
};

std::mutex g_mu;
// Never destroyed: a store left open at exit keeps its (idle) workers until
// the process ends instead of being torn down during static destruction.
auto &g_stores = *new std::unordered_map<uint64_t, std::shared_ptr<Store>>();
uint64_t g_next = 1;

std::shared_ptr<Store> find(kv_l3 h) {
    auto it = g_stores.find((uint64_t)(uintptr_t)h);
    return it == g_stores.end() ? nullptr : it->second;
}

// Moves one run fully: memcpy through the mapping, or repeated pwritev /
// preadv until every byte is done.
void do_run(Store &s, Job &j, const Run &r) {
    if (s.map != nullptr) {
        char *rec = s.map + (r.file_off - s.base);
        for (uint32_t k = 0; k < r.count; ++k, rec += j.rb) {
            char *slot = j.host + (uint64_t)j.slots[r.first + k] * j.rb;
            if (j.put)
                std::memcpy(rec, slot, j.rb);
            else
                std::memcpy(slot, rec, j.rb);
        }
        return;
    }
    iovec iov[kRunPages];
    for (uint32_t k = 0; k < r.count; ++k) {
        iov[k].iov_base = j.host + (uint64_t)j.slots[r.first + k] * j.rb;
        iov[k].iov_len = j.rb;
    }
    uint32_t k0 = 0;
    uint64_t off = r.file_off;
    while (k0 < r.count) {
        const int cnt = (int)std::min<uint32_t>(r.count - k0, (uint32_t)IOV_MAX);
        const ssize_t got = j.put ? pwritev(s.fd, iov + k0, cnt, (off_t)off)
                                  : preadv(s.fd, iov + k0, cnt, (off_t)off);
        if (got < 0 && errno == EINTR) continue;
        if (got <= 0) {
            std::lock_guard<std::mutex> lk(s.mu);
            if (j.failed.fetch_add(1) == 0) {
                j.err_no = got < 0 ? errno : 0;
                j.err_off = off;
                j.short_read = got == 0;
            }
            return;
        }
        off += (uint64_t)got;
        uint64_t left = (uint64_t)got;   // advance past fully and partly moved iovecs
        while (left > 0 && k0 < r.count) {
            if (left >= iov[k0].iov_len) {
                left -= iov[k0].iov_len;
                ++k0;
            } else {
                iov[k0].iov_base = (char *)iov[k0].iov_base + left;
                iov[k0].iov_len -= left;
                left = 0;
            }
        }
        if (j.failed.load(std::memory_order_relaxed) != 0) return;
    }
}

void worker(Store *s) {
    uint64_t seen = 0;
    std::unique_lock<std::mutex> lk(s->mu);
    for (;;) {
        s->cv_work.wait(lk, [&] { return s->stop || s->job_gen != seen; });
        if (s->stop) return;
        seen = s->job_gen;
        Job *j = s->job;
        if (j == nullptr) continue;   // woke after that job was already finished
        ++s->busy;
        lk.unlock();
        for (;;) {
            const uint32_t r = j->next.fetch_add(1);
            if (r >= j->runs.size() || j->failed.load(std::memory_order_relaxed) != 0) break;
            do_run(*s, *j, j->runs[r]);
        }
        lk.lock();
        if (--s->busy == 0) s->cv_done.notify_all();
    }
}

// Checks ids against their limits; rejects a repeated write target.
kv_status check(const char *what, const int32_t *ids, uint32_t n, uint64_t limit, bool no_dups) {
    for (uint32_t i = 0; i < n; ++i) {
        const int32_t v = ids[i];
        if (v < 0 || (uint64_t)v >= limit)
            return err(KV_ERR_OUT_OF_RANGE, "%s[%u] = %d is outside [0, %llu)", what, i, v,
                       (unsigned long long)limit);
    }
    if (no_dups && n > 1) {
        std::vector<int32_t> v(ids, ids + n);
        std::sort(v.begin(), v.end());
        for (uint32_t i = 1; i < n; ++i)
            if (v[i] == v[i - 1])
                return err(KV_ERR_DUPLICATE, "%s holds %d twice: one call may write a record "
                           "or slot only once", what, v[i]);
    }
    return KV_OK;
}

kv_status transfer(kv_l3 h, bool put, void *host, uint64_t host_slots, const int32_t *slots,
                   const int32_t *records, uint32_t n) {
    std::shared_ptr<Store> s;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        s = find(h);
    }
    if (s == nullptr) return err(KV_ERR_CLOSED, "L3 store handle is closed or unknown");
    if (n == 0) return KV_OK;
    if (host == nullptr || slots == nullptr || records == nullptr)
        return err(KV_ERR_INVALID_ARG, "host tier and id arrays must be non-NULL when n = %u", n);
    if (host_slots == 0 || host_slots > UINT64_MAX / s->rb)
        return err(KV_ERR_INVALID_ARG, "host tier of %llu slots of %llu bytes",
                   (unsigned long long)host_slots, (unsigned long long)s->rb);
    kv_status st = check("host_slots", slots, n, host_slots, !put);
    if (st == KV_OK) st = check("records", records, n, s->nrec, put);
    if (st != KV_OK) return st;

    std::lock_guard<std::mutex> call(s->call_mu);
    if (s->closed) return err(KV_ERR_CLOSED, "L3 store handle is closed or unknown");
    if (s->map != nullptr) {
        // the mapping may only be touched inside the file: grow it for a put,
        // refuse a get of a record past its end
        const int32_t last = *std::max_element(records, records + n);
        const uint64_t end = s->base + ((uint64_t)last + 1) * s->rb;
        struct stat sb;
        if (fstat(s->fd, &sb) != 0)
            return err(KV_ERR_IO, "fstat of the store: %s", strerror(errno));
        if ((uint64_t)sb.st_size < end) {
            if (!put)
                return err(KV_ERR_IO, "kv_l3_get: the file ends at byte %llu, before record %d "
                           "(a record never written)", (unsigned long long)sb.st_size, last);
            if (ftruncate(s->fd, (off_t)end) != 0)
                return err(KV_ERR_IO, "growing the store to %llu bytes: %s",
                           (unsigned long long)end, strerror(errno));
        }
    }
    Job j;
    j.put = put;
    j.host = (char *)host;
    j.rb = s->rb;
    j.slots = slots;
    const uint32_t per_run = (uint32_t)std::max<uint64_t>(
        1, std::min<uint64_t>(kRunPages, kRunBytes / s->rb));
    for (uint32_t i = 0; i < n;) {
        uint32_t k = i + 1;
        while (k < n && k - i < per_run && records[k] == records[k - 1] + 1) ++k;
        j.runs.push_back({s->base + (uint64_t)records[i] * s->rb, i, k - i});
        i = k;
    }
    {
        std::unique_lock<std::mutex> lk(s->mu);
        s->job = &j;
        ++s->job_gen;
        s->cv_work.notify_all();
        // wait until every run is taken and every worker has left the job
        s->cv_done.wait(lk, [&] {
            return s->busy == 0 && (j.next.load() >= j.runs.size() || j.failed.load() != 0);
        });
        s->job = nullptr;
    }
    if (j.failed.load() != 0) {
        if (j.short_read)
            return err(KV_ERR_IO, "%s: the file ends before byte %llu (a record never written)",
                       put ? "kv_l3_put" : "kv_l3_get", (unsigned long long)j.err_off);
        return err(KV_ERR_IO, "%s at file byte %llu: %s", put ? "pwritev" : "preadv",
                   (unsigned long long)j.err_off, strerror(j.err_no));
    }
    return KV_OK;
}

}  // namespace

extern "C" {

kv_status kv_l3_open(int fd, uint64_t base_offset, uint64_t record_bytes, uint64_t num_records,
                     uint32_t threads, kv_l3 *out) {
    if (out == nullptr) return err(KV_ERR_INVALID_ARG, "output pointer is NULL");
    if (record_bytes == 0 || num_records == 0)
        return err(KV_ERR_INVALID_ARG, "record_bytes and num_records must be positive");
    if (threads > kMaxThreads) return err(KV_ERR_INVALID_ARG, "threads %u > %u", threads,
                                          kMaxThreads);
    if (num_records > (uint64_t)INT32_MAX + 1 || record_bytes > (uint64_t)INT64_MAX / num_records ||
        base_offset > (uint64_t)INT64_MAX - record_bytes * num_records)
        return err(KV_ERR_OUT_OF_RANGE, "store of %llu records of %llu bytes at %llu overflows "
                   "a file offset", (unsigned long long)num_records,
                   (unsigned long long)record_bytes, (unsigned long long)base_offset);
    struct stat sb;
    if (fd < 0 || fstat(fd, &sb) != 0)
        return err(KV_ERR_INVALID_ARG, "fd %d is not an open descriptor", fd);
    if (!S_ISREG(sb.st_mode) && !S_ISBLK(sb.st_mode))
        return err(KV_ERR_INVALID_ARG, "fd %d is neither a regular file (or memfd) nor a block "
                   "device", fd);
    std::shared_ptr<Store> s(new (std::nothrow) Store());
    if (s == nullptr) return err(KV_ERR_NO_MEMORY, "out of host memory");
    s->fd = fd;
    s->base = base_offset;
    s->rb = record_bytes;
    s->nrec = num_records;
    const int fl = fcntl(fd, F_GETFL);
    if (S_ISREG(sb.st_mode) && fl >= 0 && (fl & O_ACCMODE) == O_RDWR && (fl & O_DIRECT) == 0) {
        const uint64_t pg = (uint64_t)sysconf(_SC_PAGESIZE);
        s->skew = base_offset % pg;
        s->map_len = s->skew + record_bytes * num_records;
        void *m = mmap(nullptr, s->map_len, PROT_READ | PROT_WRITE, MAP_SHARED, fd,
                       (off_t)(base_offset - s->skew));
        if (m != MAP_FAILED)
            s->map = (char *)m + s->skew;   // else: the syscall path
    }
    const uint32_t nt = threads ? threads : kDefaultThreads;
    try {
        for (uint32_t t = 0; t < nt; ++t) s->workers.emplace_back(worker, s.get());
    } catch (...) {
        return err(KV_ERR_NO_MEMORY, "could not start %u worker threads", nt);   // ~Store joins
    }
    std::lock_guard<std::mutex> lk(g_mu);
    const uint64_t id = g_next++;
    g_stores[id] = s;
    *out = (kv_l3)(uintptr_t)id;
    return KV_OK;
}

kv_status kv_l3_close(kv_l3 h) {
    std::shared_ptr<Store> s;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        s = find(h);
        if (s == nullptr) return err(KV_ERR_CLOSED, "L3 store handle is closed or unknown");
        g_stores.erase((uint64_t)(uintptr_t)h);
    }
    {
        std::lock_guard<std::mutex> call(s->call_mu);   // a call in flight finishes first
        s->closed = true;
        std::lock_guard<std::mutex> lk(s->mu);
        s->stop = true;
    }
    s->cv_work.notify_all();
    for (auto &w : s->workers) w.join();
    return KV_OK;   // the store is freed with its last reference
}

kv_status kv_l3_put(kv_l3 store, const void *host, uint64_t host_slots, const int32_t *slots,
                    const int32_t *records, uint32_t n) {
    return transfer(store, true, const_cast<void *>(host), host_slots, slots, records, n);
}

kv_status kv_l3_get(kv_l3 store, void *host, uint64_t host_slots, const int32_t *records,
                    const int32_t *slots, uint32_t n) {
    return transfer(store, false, host, host_slots, slots, records, n);
}

}  // extern "C"
