// kvb_ring_kernels.cu -- the GPU-resident server of the descriptor ring.
//
// "[Feature] [RFC] [HiCache] Out-of-process HiCache data plane with
// device-memory IPC", §Device IPC data path: once the pool is registered,
// BACKUP / RESTORE travel as descriptors, and a high-frequency path may want
// an NVMe-style submission / completion queue.  Here the queue's consumer is
// the GPU itself: one cooperative grid stays resident.  Its leader CTA polls
// the ring's tail in the shared segment (pinned host memory mapped into the
// GPU; on GB300 the reads are coherent over NVLink-C2C), takes each descriptor,
// validates it exactly as the host engine does, and releases it to the mover
// CTAs; they move the pages and the mover that finishes last writes the ticket
// into the slot's completion record.  The leader moves nothing: while the
// movers move descriptor t it already takes and checks t + 1.  No host thread
// and no launch per operation: the submitter's descriptor store and its
// completion poll are the only CPU work.
//
// Accepted descriptors run one after another in ticket order (as the host
// server's single stream runs them); a rejected one is completed as soon as
// it is checked.  Every wait is bounded: the leader waits at most idle_ns for
// a descriptor, then ends the server; any other wait gives up after idle_ns +
// 5 s, records it and returns.  Nothing traps.
//
// Memory model.  Pages and host slots may be written by one descriptor and
// read by the next inside this one launch, so payload and ids are loaded
// through L2 (ld.global.cg) or with strong loads, never through the
// non-coherent read-only path.  A descriptor is released with a gpu-scope
// release after every writer's fence; a CTA arrives at a descriptor's end
// after a device-scope fence of its stores, with an acq_rel count, so the
// completion record the last arriver stores (system scope, release: cumulative
// over what it acquired) covers every byte of the operation.
#include "kvb_ring_internal.h"

namespace kvb {

namespace {

constexpr uint32_t kMaxIds = KV_RING_MAX_IDS;
constexpr int kThreads = kRingThreads;
constexpr int kIdsPerThread = (int)kMaxIds / kThreads;   // ids a leader thread holds
static_assert(kMaxIds == (uint32_t)(kIdsPerThread * kThreads), "ids split evenly over threads");
constexpr unsigned long long kSlackNs = 5000000000ull;   // bound on the non-idle waits
constexpr int kUnroll = kSegPieces / 32;                  // 16-byte pieces per lane per segment

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    const uint32_t t = __umulhi(n, f.m);
    return (uint32_t)(((uint64_t)t + n) >> f.s);
}

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned long long ld_acquire_sys(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int32_t ld_relaxed_sys(const int32_t *p) {
    int32_t v;
    asm volatile("ld.relaxed.sys.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_sys_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_sys_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int32_t ld_relaxed_gpu(const int32_t *p) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_sys(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_sys64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_sys32(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16-byte payload access: loads through L2 (the bytes may have been written
// earlier in this launch), streaming stores.
__device__ __forceinline__ uint4 load16(const char *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void store16(char *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Piece index on the other side of a head-order permutation: q is a 16-byte
// piece of a chunk in head order `from_hnd` (NHD [T][H][B] or HND [H][T][B]).
__device__ __forceinline__ uint32_t permute_piece(uint32_t q, uint32_t from_hnd,
                                                  const RingPoolK &p) {
    const uint32_t j = fdiv(q, p.div_b16);
    const uint32_t r = q - j * p.B16;
    uint32_t h, t;
    if (from_hnd) {
        h = fdiv(j, p.div_T);
        t = j - h * p.T;
        return (t * p.H + h) * p.B16 + r;
    }
    t = fdiv(j, p.div_H);
    h = j - t * p.H;
    return (h * p.T + t) * p.B16 + r;
}

__device__ __forceinline__ uint64_t chunk_addr(const Side &s, uint32_t id, uint64_t l, uint32_t c,
                                               uint32_t C) {
    if (s.lc_base != nullptr) return __ldg(s.lc_base + l * C + c) + id * s.s_id;
    return s.base + id * s.s_id + l * s.s_l + c * s.s_c;
}

// This CTA's share of one descriptor: its warps take the op's 4 KiB segments
// by grid stride (ids from shared memory).  kMode 0: same head order on both
// sides; 1: backup that changes head order (walks the host tier's pieces in
// order: contiguous stores over the link); 2: restore that changes it (walks
// the host tier's pieces in order: contiguous loads over the link).
template <int kMode>
__device__ __forceinline__ void move_loop(const Side src, const Side dst, const RingPoolK &p,
                                          uint32_t n, uint32_t nl, uint32_t l0,
                                          const FastDiv &div_lc, const int32_t *s_a,
                                          const int32_t *s_b) {
    const uint32_t total = n * nl * p.C * p.segs;   // < 2^32: checked when the server starts
    const uint32_t lane = threadIdx.x & 31u;
    // the mover CTAs 1 .. gridDim.x - 1 (CTA 0 is the leader)
    const uint32_t nwarps = ((gridDim.x - 1) * blockDim.x) >> 5;
    const uint32_t hnd = kMode == 1 ? dst.hnd : src.hnd;   // head order of the walked side
    for (uint32_t w = ((blockIdx.x - 1) * blockDim.x + threadIdx.x) >> 5; w < total; w += nwarps) {
        const uint32_t chunk = fdiv(w, p.div_segs);
        const uint32_t seg = w - chunk * p.segs;
        const uint32_t item = fdiv(chunk, div_lc);
        const uint32_t lc = chunk - item * (nl * p.C);
        const uint32_t lr = fdiv(lc, p.div_c);
        const uint32_t c = lc - lr * p.C;
        const uint32_t ia = (uint32_t)s_a[item], ib = (uint32_t)s_b[item];
        if (ia >= src.id_limit || ib >= dst.id_limit) continue;   // validated; never touch memory
        const uint64_t l = (uint64_t)l0 + lr;
        const char *sp = reinterpret_cast<const char *>(chunk_addr(src, ia, l, c, p.C));
        char *dp = reinterpret_cast<char *>(chunk_addr(dst, ib, l, c, p.C));
        const uint32_t q0 = seg * (uint32_t)kSegPieces;
        const uint32_t qn = min((uint32_t)kSegPieces, p.cb16 - q0);
        // the walked side's pieces: lane, lane + 32, ... from one base address
        const char *sl = sp + ((uint64_t)q0 + lane) * 16u;
        char *dl = dp + ((uint64_t)q0 + lane) * 16u;
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t q = u * 32u + lane;
            if (q < qn)
                v[u] = kMode == 1 ? load16(sp + (uint64_t)permute_piece(q0 + q, hnd, p) * 16u)
                                  : load16(sl + u * 512);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t q = u * 32u + lane;
            if (q < qn) {
                if (kMode == 2)
                    store16(dp + (uint64_t)permute_piece(q0 + q, hnd, p) * 16u, v[u]);
                else
                    store16(dl + u * 512, v[u]);
            }
        }
    }
}

__device__ __forceinline__ void move_share(const RingKDesc &k, const RingPoolK &p, uint32_t kind,
                                        uint32_t n, int32_t layer, const int32_t *s_a,
                                        const int32_t *s_b) {
    const bool backup = kind == KV_RING_OP_BACKUP;
    const Side pool = p.pool, host = k.host;   // by value: selected field by field in registers
    const Side src = backup ? pool : host;
    const Side dst = backup ? host : pool;
    const uint32_t nl = layer < 0 ? p.L : 1u;
    const uint32_t l0 = layer < 0 ? 0u : (uint32_t)layer;
    const FastDiv &div_lc = layer < 0 ? p.div_lc_all : p.div_lc_one;
    if (!p.transpose)
        move_loop<0>(src, dst, p, n, nl, l0, div_lc, s_a, s_b);
    else if (backup)
        move_loop<1>(src, dst, p, n, nl, l0, div_lc, s_a, s_b);
    else
        move_loop<2>(src, dst, p, n, nl, l0, div_lc, s_a, s_b);
}

// A mover CTA's arrival at the end of released descriptor number `rel`
// (1-based): its stores are ordered device-wide, then counted (acq_rel at
// device scope); the last of the movers' arrivals stores the ticket into the
// completion record with a system-scope release, which is cumulative over
// every mover's bytes, so the process that acquires the record sees them.
__device__ __forceinline__ void arrive(const RingKDesc &k, uint32_t rel, uint64_t ticket) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(&k.ctl->arrived)
                     : "memory");
        if (prev + 1 == (gridDim.x - 1) * rel)
            st_release_sys((unsigned long long *)&k.comp[(ticket - 1) % k.slots].done, ticket);
    }
}

// Leader, thread 0: completes ticket t from the GPU with an error status.
__device__ __forceinline__ void complete_failed(const RingKDesc &k, uint64_t t, int32_t status) {
    CompRec &c = k.comp[(t - 1) % k.slots];
    st_relaxed_sys32((uint32_t *)&c.err, (uint32_t)status);
    st_relaxed_sys64((unsigned long long *)&c.err_ticket, t);
    __threadfence_system();
    st_release_sys((unsigned long long *)&c.done, t);
}

// Leader, thread 0: waits (bounded) until the movers' arrivals reach `want`.
// Both count modulo 2^32 (movers x descriptors passes 2^32 after 2^32 / movers
// descriptors); the count trails `want` by at most one descriptor's arrivals,
// so the comparison is made on the signed difference.
__device__ __forceinline__ int wait_arrivals(const RingKDesc &k, uint32_t want) {
    const unsigned long long deadline = now_ns() + kSlackNs;
    for (unsigned long long polls = 0;; ++polls) {
        if ((int32_t)(ld_acquire_gpu(&k.ctl->arrived) - want) >= 0) return 1;
        if (ld_acquire_gpu(&k.ctl->gave_up) != 0 || polls >= kSlackNs / 16ull ||
            ((polls & 63u) == 63u && now_ns() > deadline))
            return 0;
        if (polls >= 4096) __nanosleep(64);
    }
}

// Checks a descriptor exactly as the host engine would, in its order: kind,
// n, pool index and a backup's layer (INVALID_ARG), the layer (OUT_OF_RANGE),
// then the ids -- any source id out of range, else whichever comes first in
// index order of a write target out of range (OUT_OF_RANGE) and a write
// target repeated from an earlier one (DUPLICATE).  Called by every thread of
// the leader CTA with the ids it holds (thread i: ids i, i + kThreads, ...);
// leaves ids [0, n) in s_a / s_b.  The three shared words start as
// "none" (0xffffffff, 0xffffffff, 0).
__device__ int32_t check_descriptor(const RingKDesc &k, uint32_t kind, uint32_t n, uint32_t pool,
                                    int32_t layer, const int32_t (&a_r)[kIdsPerThread],
                                    const int32_t (&b_r)[kIdsPerThread], int32_t *s_a,
                                    int32_t *s_b, unsigned long long *s_key,
                                    uint32_t *s_first_bad, uint32_t *s_first_dup,
                                    uint32_t *s_any_bad_a) {
    if (kind > KV_RING_OP_RESTORE || n > kMaxIds || pool >= k.npools) return KV_ERR_INVALID_ARG;
    if (kind == KV_RING_OP_BACKUP && layer != -1) return KV_ERR_INVALID_ARG;
    if (layer < -1 || (layer >= 0 && (uint32_t)layer >= k.pools[pool].L)) return KV_ERR_OUT_OF_RANGE;
    if (n == 0) return KV_OK;
    const uint32_t tid = threadIdx.x;
    const bool backup = kind == KV_RING_OP_BACKUP;
    const uint32_t lim_a = backup ? k.pools[pool].P : k.num_slots;
    const uint32_t lim_b = backup ? k.num_slots : k.pools[pool].P;
#pragma unroll
    for (int h = 0; h < kIdsPerThread; ++h) {
        const uint32_t i = tid + h * kThreads;
        if (i < n) {
            s_a[i] = a_r[h];
            s_b[i] = b_r[h];
        }
    }
    if (n <= 32) {
        // one warp, no block barrier: lane i holds id i; a repeat is a lane whose
        // write target equals a lower lane's
        if (tid < 32) {
            const bool in = tid < n;
            const int32_t a = a_r[0], b = b_r[0];
            bool dup = false;
            for (uint32_t j = 0; j < n; ++j) {
                const int32_t bj = __shfl_sync(0xffffffffu, b, j);
                dup |= in && j < tid && bj == b;
            }
            const unsigned bad_a = __ballot_sync(0xffffffffu, in && (a < 0 || (uint32_t)a >= lim_a));
            const unsigned bad_b = __ballot_sync(0xffffffffu, in && (b < 0 || (uint32_t)b >= lim_b));
            const unsigned dups = __ballot_sync(0xffffffffu, dup);
            if (tid == 0) {
                *s_any_bad_a = bad_a != 0u;
                if (bad_b) *s_first_bad = (uint32_t)__ffs(bad_b) - 1u;
                if (dups) *s_first_dup = (uint32_t)__ffs(dups) - 1u;
            }
        }
    } else {
        // sort (b, index) keys; the first repeat of a value in index order is the
        // later of two equal neighbours; pads (index >= n) sort last, never counted
        uint32_t m = 2;
        while (m < n) m <<= 1;
#pragma unroll
        for (int h = 0; h < kIdsPerThread; ++h) {
            const uint32_t i = tid + h * kThreads;
            if (i < n) {
                if (a_r[h] < 0 || (uint32_t)a_r[h] >= lim_a) *s_any_bad_a = 1u;
                if (b_r[h] < 0 || (uint32_t)b_r[h] >= lim_b) atomicMin(s_first_bad, i);
            }
            if (i < m)
                s_key[i] = i < n ? ((unsigned long long)(uint32_t)b_r[h] << 32) | i
                                 : (0xffffffffull << 32) | i;
        }
        for (uint32_t size = 2; size <= m; size <<= 1)
            for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
                __syncthreads();
                for (uint32_t i = tid; i < m; i += kThreads) {
                    const uint32_t j = i ^ stride;
                    if (j > i) {
                        const unsigned long long x = s_key[i], y = s_key[j];
                        if ((x > y) == ((i & size) == 0)) {
                            s_key[i] = y;
                            s_key[j] = x;
                        }
                    }
                }
            }
        __syncthreads();
        for (uint32_t i = tid + 1; i < m; i += kThreads) {
            const unsigned long long x = s_key[i], y = s_key[i - 1];
            const uint32_t idx = (uint32_t)x;
            if (idx < n && (x >> 32) == (y >> 32)) atomicMin(s_first_dup, idx);
        }
    }
    __syncthreads();
    if (*s_any_bad_a) return KV_ERR_OUT_OF_RANGE;
    if (*s_first_bad < *s_first_dup) return KV_ERR_OUT_OF_RANGE;
    if (*s_first_dup != 0xffffffffu) return KV_ERR_DUPLICATE;
    return KV_OK;
}

__global__ void __launch_bounds__(kThreads, 1) kv_ring_server_kernel(const __grid_constant__ RingKDesc k) {
    __shared__ int32_t s_a[kMaxIds], s_b[kMaxIds];
    __shared__ unsigned long long s_key[kMaxIds];   // leader: (b[i] << 32) | i, sorted
    __shared__ uint32_t s_hdr[6];   // kind, n, pool, layer, ready index, ready timeout (ms)
    __shared__ unsigned long long s_ready;          // ready value (0: not gated)
    __shared__ uint32_t s_first_bad, s_first_dup, s_any_bad_a;
    __shared__ int s_flag, s_done;   // descriptor wait / arrival wait results
    RingCtl *ctl = k.ctl;
    const uint32_t tid = threadIdx.x;

    if (blockIdx.x != 0) {
        // ----------------------------------------------------- mover CTAs
        for (uint32_t r = 0;; ++r) {
            if (tid == 0) {
                int go = 0;   // 1: descriptor r released; 0: stopped; -1: gave up
                const unsigned long long deadline = now_ns() + k.idle_ns + kSlackNs;
                // the poll count is capped too (a poll is an L2 round trip, far
                // above 16 ns), so the wait ends even without a running timer
                const unsigned long long max_polls = (k.idle_ns + kSlackNs) / 16ull;
                for (unsigned long long polls = 0;; ++polls) {
                    if (ld_acquire_gpu(&ctl->gen) > r) { go = 1; break; }
                    if (ld_acquire_gpu(&ctl->stop) != 0) break;
                    if (polls >= max_polls || ((polls & 63u) == 63u && now_ns() > deadline)) {
                        go = -1;
                        break;
                    }
                    if (polls >= 4096) __nanosleep(128);   // spin first: descriptors stream in
                }
                if (go < 0) atomicExch(&ctl->gave_up, 1u);
                s_flag = go;
            }
            __syncthreads();
            if (s_flag <= 0) return;
            const uint32_t kind = *(volatile uint32_t *)&ctl->kind;
            const uint32_t n = *(volatile uint32_t *)&ctl->n;
            const uint32_t pool = *(volatile uint32_t *)&ctl->pool;
            const int32_t layer = *(volatile int32_t *)&ctl->layer;
            const uint64_t ticket = *(volatile unsigned long long *)&ctl->ticket;
            for (uint32_t i = tid; i < n; i += kThreads) {
                s_a[i] = ld_relaxed_gpu(k.ids + i);
                s_b[i] = ld_relaxed_gpu(k.ids + kMaxIds + i);
            }
            __syncthreads();
            move_share(k, k.pools[pool], kind, n, layer, s_a, s_b);
            arrive(k, r + 1, ticket);
            __syncthreads();   // s_a / s_b are rewritten for the next descriptor
        }
    }

    // -------------------------------------------------------- leader CTA
    // Control only: it takes and checks descriptor t + 1 while the movers move
    // descriptor t, and releases t + 1 once every mover has arrived at t's end.
    if (tid == 0) asm volatile("st.relaxed.sys.global.s64 [%0], %1;" ::"l"(k.server_pid), "l"(k.pid)
                               : "memory");
    const uint32_t movers = gridDim.x - 1;
    uint32_t taken = 0, released = 0;
    int32_t server_status = KV_OK;
    for (;;) {
        if (taken >= k.max_ops) break;
        const uint64_t t = k.first_ticket + taken;
        const uint32_t slot = (uint32_t)((t - 1) % k.slots);
        // wait for the descriptor (idle bound) unless the host asked the server
        // to stop; the stop word is loaded first so both loads are in flight
        if (tid == 0) {
            int go = 0;
            const unsigned long long deadline = now_ns() + k.idle_ns;
            const unsigned long long max_polls = k.idle_ns / 64ull + 4096ull;
            for (unsigned long long polls = 0;; ++polls) {
                const uint32_t stop = ld_relaxed_sys_u32(k.result + 2);
                const unsigned long long tail = ld_acquire_sys(k.tail);
                if (stop != 0) break;
                if (tail >= t) { go = 1; break; }
                if (polls >= max_polls || now_ns() > deadline) break;
            }
            s_flag = go;
        }
        __syncthreads();
        if (!s_flag) break;
        // take it: header and (speculatively) every id slot, in one round trip;
        // thread i holds ids i, i + kThreads, ...
        const kv_ring_op &e = k.ops[slot];
        int32_t a_r[kIdsPerThread], b_r[kIdsPerThread];
#pragma unroll
        for (int h = 0; h < kIdsPerThread; ++h) {
            a_r[h] = ld_relaxed_sys(e.a + tid + h * kThreads);
            b_r[h] = ld_relaxed_sys(e.b + tid + h * kThreads);
        }
        if (tid == 0) {
            s_hdr[0] = (uint32_t)ld_relaxed_sys((const int32_t *)&e.kind);
            s_hdr[1] = (uint32_t)ld_relaxed_sys((const int32_t *)&e.n);
            s_hdr[2] = (uint32_t)ld_relaxed_sys((const int32_t *)&e.pool_index);
            s_hdr[3] = (uint32_t)ld_relaxed_sys(&e.layer);
            s_hdr[4] = (uint32_t)ld_relaxed_sys((const int32_t *)&e.ready_index);
            s_hdr[5] = (uint32_t)ld_relaxed_sys((const int32_t *)&e.ready_timeout_ms);
            s_ready = ld_relaxed_sys_u64((const unsigned long long *)&e.ready_value);
            s_first_bad = s_first_dup = 0xffffffffu;
            s_any_bad_a = 0u;
        }
        __syncthreads();
        ++taken;
        const uint32_t kind = s_hdr[0], n = s_hdr[1], pool = s_hdr[2];
        const int32_t layer = (int32_t)s_hdr[3];
        const uint32_t ready_index = s_hdr[4], ready_ms = s_hdr[5];
        const unsigned long long ready_value = s_ready;
        // a gate naming no ready word, or a wait above 60 s, is refused like a
        // malformed descriptor (the host server's pop does the same)
        const bool bad_gate =
            ready_value != 0 && (ready_index >= KV_RING_READY_WORDS || ready_ms > 60000u);
        const int32_t status =
            bad_gate ? (int32_t)KV_ERR_INVALID_ARG
                     : check_descriptor(k, kind, n, pool, layer, a_r, b_r, s_a, s_b, s_key,
                                        &s_first_bad, &s_first_dup, &s_any_bad_a);
        if (status != KV_OK) {   // rejected: completed at once, nothing moves
            if (tid == 0) {
                st_relaxed_sys64(k.head, t);
                complete_failed(k, t, status);
            }
            __syncthreads();
            continue;
        }
        // gated: wait (bounded) for its ready word; on time-out -- or a stop
        // request meanwhile -- it moves nothing and completes with ABORTED
        if (ready_value != 0) {
            if (tid == 0) {
                const unsigned long long limit_ns =
                    (unsigned long long)(ready_ms ? ready_ms : 10000u) * 1000000ull;
                const unsigned long long deadline = now_ns() + limit_ns;
                const unsigned long long max_polls = limit_ns / 16ull + 4096ull;
                int open = 0;
                for (unsigned long long polls = 0;; ++polls) {
                    if (ld_acquire_sys(k.ready + ready_index) >= ready_value) {
                        open = 1;
                        break;
                    }
                    if (ld_relaxed_sys_u32(k.result + 2) != 0) break;
                    if (polls >= max_polls || ((polls & 63u) == 63u && now_ns() > deadline)) break;
                    if (polls >= 4096) __nanosleep(256);
                }
                s_flag = open;
            }
            __syncthreads();
            if (!s_flag) {
                if (tid == 0) {
                    st_relaxed_sys64(k.head, t);
                    complete_failed(k, t, KV_ERR_ABORTED);
                }
                __syncthreads();
                continue;
            }
        }
        // accepted: it runs after the one released before it has ended
        if (tid == 0) {
            st_relaxed_sys64(k.head, t);
            s_done = released == 0 ? 1 : wait_arrivals(k, movers * released);
        }
        __syncthreads();
        if (!s_done) {
            server_status = KV_ERR_TIMEOUT;
            break;
        }
        if (n == 0) {   // empty: complete once everything before it is
            if (tid == 0) {
                __threadfence_system();
                st_release_sys((unsigned long long *)&k.comp[slot].done, t);
            }
            __syncthreads();
            continue;
        }
        // release it to the movers
        for (uint32_t i = tid; i < n; i += kThreads) {
            k.ids[i] = s_a[i];
            k.ids[kMaxIds + i] = s_b[i];
        }
        __threadfence();
        __syncthreads();
        ++released;
        if (tid == 0) {
            ctl->kind = kind;
            ctl->n = n;
            ctl->pool = pool;
            ctl->layer = layer;
            ctl->ticket = t;
            __threadfence();
            st_release_gpu(&ctl->gen, released);
        }
        __syncthreads();   // s_hdr, s_a and s_b are rewritten by the next take
    }
    // every released descriptor ends before the movers are told to stop
    if (tid == 0) {
        if (released > 0 && !wait_arrivals(k, movers * released)) server_status = KV_ERR_TIMEOUT;
        if (ld_acquire_gpu(&ctl->gave_up) != 0) server_status = KV_ERR_TIMEOUT;
        st_relaxed_sys32(k.result, taken);
        st_relaxed_sys32(k.result + 1, (uint32_t)server_status);
        __threadfence_system();
        st_release_gpu(&ctl->stop, 1u);
    }
}

}  // namespace

namespace {

__global__ void kv_ring_mark_kernel(unsigned long long *done, unsigned long long *err_ticket,
                                    int32_t *err, unsigned long long ticket,
                                    const unsigned long long *status, unsigned long long tag) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    if (status != nullptr && ld_relaxed_sys_u64(status) == tag) {
        asm volatile("st.relaxed.sys.global.s32 [%0], %1;" ::"l"(err), "r"((int32_t)KV_ERR_ABORTED)
                     : "memory");
        st_relaxed_sys64(err_ticket, ticket);
    }
    st_release_sys(done, ticket);   // release: the error fields are visible first
}

}  // namespace

cudaError_t preload_ring_kernels() {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, (const void *)kv_ring_server_kernel);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, (const void *)kv_ring_mark_kernel);
    return e;
}

cudaError_t launch_ring_mark(unsigned long long *done, unsigned long long *err_ticket, int32_t *err,
                             unsigned long long ticket, const unsigned long long *status,
                             unsigned long long tag, cudaStream_t stream) {
    kv_ring_mark_kernel<<<1, 32, 0, stream>>>(done, err_ticket, err, ticket, status, tag);
    return cudaGetLastError();
}

cudaError_t launch_ring_server(const RingKDesc &k, int ctas, cudaStream_t stream) {
    (void)cudaGetLastError();
    if (ctas < 2) return cudaErrorInvalidValue;   // a leader and at least one mover
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_ring_server_kernel, k);
}

}  // namespace kvb
