// kvb_kernels.cu -- sm_103a kernels of the KV backup / restore engine.
//
// The data movement of BACKUP / RESTORE in "[RFC][HiCache] Out-of-process
// HiCache data plane with device-memory IPC" (§Device IPC data path), with the
// layer restriction of "[PP + HiCache] Add PP Prefetch Tickets" (§PP Prefetch
// Ticket Path, layer-wise H2D) and the HND pool of "LMCache
// RawCudaIPCWrapper深度解析" (§在项目中的实际接入方式).  Payload moves as raw
// 16-byte integer vectors or bulk copies: no float type touches it
// (§uint8字节往返).  Every kernel copies whole KV "chunks" (the T*H*B bytes of
// one page-or-slot, layer and component) from a source side to a destination
// side described by strides or a per-(layer, component) table
// (kvb_internal.h), optionally permuting the head order inside each chunk.
//
//   kv_move_kernel  registers as staging; host-link moves (zero-copy backup /
//                   restore over mapped pinned memory) and the fallback for
//                   HBM-only moves.  The op is a flat list of 4 KiB warp
//                   segments; warps take them by grid stride (or, for a
//                   progressive layer restore, from a ticket counter in layer
//                   order).  Per segment one id lookup and address decode,
//                   then eight independent 16-byte loads per lane (4 KiB in
//                   flight per warp) and eight stores: each warp-wide access
//                   covers 512 contiguous bytes, or B-byte runs when a head
//                   permutation is fused in.
//   kv_bulk_kernel  HBM-only identity moves through cp.async.bulk and an
//                   8-stage shared-memory ring (one warp per CTA).
//   kv_tsp_kernel   HBM-only moves that change head order: whole chunks
//                   bulk-loaded into shared memory, written in destination
//                   order by 256 threads.
//   kv_gate_kernel  bounded wait for a ready fence before a gated backup.
//   kv_mark_kernel  stores a fence word after copy-engine work.
// The move kernels complete their op's fence from their last CTA (and, for a
// ring descriptor, its completion record right after); an overlapped restore
// (KV_CFG_OVERLAP_RESTORES) skips griddepcontrol.wait and publishes its fence
// only after its predecessor's.  All waits inside kernels are bounded and
// nothing traps.
#include "kvb_internal.h"

namespace kvb {

namespace {

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    const uint32_t t = __umulhi(n, f.m);
    return (uint32_t)(((uint64_t)t + n) >> f.s);
}

// 16-byte load that bypasses L1 (each byte is read exactly once).
__device__ __forceinline__ uint4 load16(const char *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte streaming store (evict-first: the data is not read again soon).
__device__ __forceinline__ void store16(char *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Piece index on the other side of a head-order permutation.  q is a 16-byte
// piece of a chunk laid out with head order `from_hnd`; returns the index of
// the same piece in the other order.
__device__ __forceinline__ uint32_t permute_piece(uint32_t q, uint32_t from_hnd,
                                                  const MoveDesc &d) {
    const uint32_t j = fdiv(q, d.div_b16);      // head vector within the chunk
    const uint32_t r = q - j * d.B16;           // piece within the head vector
    uint32_t h, t;
    if (from_hnd) {                              // j = h*T + t
        h = fdiv(j, d.div_T);
        t = j - h * d.T;
        return (t * d.H + h) * d.B16 + r;        // -> NHD
    }
    t = fdiv(j, d.div_H);                        // j = t*H + h
    h = j - t * d.H;
    return (h * d.T + t) * d.B16 + r;            // -> HND
}

constexpr int kUnroll = kSegPieces / 32;  // 16-byte pieces per lane per segment

// Address of chunk (id, layer l, component c) on one side: strided, or from
// the split pool's per-(layer, component) buffer table.
__device__ __forceinline__ uint64_t chunk_base(const Side &s, uint32_t id, uint64_t l, uint32_t c,
                                               uint32_t C) {
    if (s.lc_base != nullptr) return __ldg(s.lc_base + l * C + c) + id * s.s_id;
    return s.base + id * s.s_id + l * s.s_l + c * s.s_c;
}

// GPU time in nanoseconds (the global timer), for bounded waits.
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Overlapped restores: the last CTA waits until the previous op's fence word
// holds chain_seq or more before it publishes its own, so fences complete in
// call order.  The previous kernel let this one launch only once each of its
// CTAs was running its last segments, so it is resident and finishes without
// waiting for anything here: the wait ends.  It is bounded all the same
// (2 s of GPU time, and a poll cap in case the timer stalls); on giving up it
// sets the sticky error word (3), which the host reports with the fence.
__device__ __forceinline__ void chain_wait(const MoveDesc &d) {
    const unsigned long long t0 = global_ns();
    unsigned int sleep_ns = 32;
    for (uint32_t polls = 0; polls < (1u << 24); ++polls) {
        unsigned long long v;
        asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(d.chain_word)
                     : "memory");
        if (v >= d.chain_seq) return;
        if (global_ns() - t0 > 2000000000ull) break;
        __nanosleep(sleep_ns);
        if (sleep_ns < 1024) sleep_ns <<= 1;
    }
    if (d.err != nullptr) *(volatile uint32_t *)d.err = 3u;
}

// Completion of a grid, fused into its last CTA: every CTA's stores are
// ordered device-wide, the CTA counts itself done (acq_rel at device scope: the
// counting CTAs and the publisher all run on this GPU), and the CTA that
// finishes last publishes the sequence number with a system-scope release
// store (and resets the counter for the fence slot's next use).  A release is
// cumulative in the PTX memory model: it orders everything that precedes it in
// causality order, here every CTA's bytes through the chain of device-scope
// arrivals, so a host thread or another device that acquires the fence word
// sees them all.  No system-scope fence is taken: on GB300 each one cost ~0.6
// us at the end of every call (one-layer MLA restores: 50.7 us per call with
// one per CTA and one more in the publisher, 49.4 us with none).  An
// overlapped restore first waits for its predecessor's fence (chain_wait).  A
// ring descriptor's completion record (ext_word), when given, is stored right
// after the fence.
//
// arrive_and_publish: one thread of the CTA, once the CTA's stores are ordered
// (its own fence, or a barrier after every thread's fence).
__device__ __forceinline__ void arrive_and_publish(const MoveDesc &d) {
    unsigned int done;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(done)
                 : "l"(d.fence_count)
                 : "memory");
    if (done == gridDim.x - 1) {
        *d.fence_count = 0u;
        if (d.chain_word != nullptr) chain_wait(d);
        asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(d.fence_word),
                     "l"(d.fence_seq)
                     : "memory");
        if (d.ext_word != nullptr)
            asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(d.ext_word),
                         "l"(d.ext_value)
                         : "memory");
    }
}

// Every thread of the CTA stored: each fences, the CTA meets, one arrives.
__device__ __forceinline__ void complete_grid(const MoveDesc &d) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) arrive_and_publish(d);
}

// Progressive layers: called by lane 0 of a warp once its `count` segments of
// layer `lr` are visible device-wide.  The warp that completes a layer tries
// to become the publisher (a lock that is tried, never waited on): the
// publisher stores the fence word of every complete layer of the prefix in
// layer order, so layer j's word is never visible before layer j-1's.  After
// releasing, it looks again for a layer that completed while it held the lock
// (that layer's completer gave up when it found the lock taken); the sequential
// fences on both sides guarantee one of the two sees the other.  No loop
// waits: each round publishes at least one layer or returns.  The data is
// ordered at device scope (each warp's fence, the acq_rel counters); the fence
// words are system-scope release stores, cumulative over those bytes, so the
// host or another device that acquires a word sees its layers.
__device__ __forceinline__ void publish_layers(const MoveDesc &d, uint32_t lr, uint32_t count) {
    const uint32_t slot = (uint32_t)((d.lay_seq0 + lr) % d.lay_ring);
    unsigned int prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(prev)
                 : "l"(d.lay_done + slot), "r"(count)
                 : "memory");
    if (prev + count != d.per_layer_segs) return;
    __threadfence();
    for (;;) {
        if (atomicCAS(d.lay_lock, 0u, 1u) != 0u) return;   // the holder will look again
        __threadfence();
        uint32_t p = *(volatile uint32_t *)d.lay_published;
        while (p < d.nl) {
            const uint32_t sp = (uint32_t)((d.lay_seq0 + p) % d.lay_ring);
            unsigned int dn;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(dn) : "l"(d.lay_done + sp)
                         : "memory");
            if (dn != d.per_layer_segs) break;
            asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(d.lay_words + sp),
                         "l"(d.lay_seq0 + p)
                         : "memory");
            ++p;
        }
        *(volatile uint32_t *)d.lay_published = p;
        __threadfence();
        atomicExch(d.lay_lock, 0u);
        __threadfence();
        if (p >= d.nl) return;
        const uint32_t sp = (uint32_t)((d.lay_seq0 + p) % d.lay_ring);
        unsigned int dn;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(dn) : "l"(d.lay_done + sp)
                     : "memory");
        if (dn != d.per_layer_segs) return;   // its completer will publish it
    }
}

// kThreads = kMoveThreads (4 CTAs per SM, for HBM-only moves) or kWideThreads
// (one 32-warp CTA per SM: host-link moves packed onto as few SMs as possible,
// leaving whole SMs to whatever computes beside them).
template <bool kTranspose, int kCap, int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads == kWideThreads ? 1 : 4)
    kv_move_kernel(const __grid_constant__ MoveDesc d, const __grid_constant__ IdsT<kCap> ids) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const uint32_t lc_per_item = d.nl * d.C;

    if (d.pdl && !d.overlap) {
        // Wait for the previous kernel on this stream (and its memory) before
        // any access here; a no-op when it was not launched as a dependent.
        // An overlapped restore skips it: the host proved the two kernels'
        // bytes disjoint, and its fence is chained on the previous op's.
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    uint32_t cur_layer = 0xffffffffu, cur_count = 0;   // progressive: this warp's tally
    bool skip = false;
    if (d.skip_word != nullptr) {   // gated op: the gate decided once, before this launch
        __shared__ int s_skip;
        if (threadIdx.x == 0) {
            unsigned long long v;
            asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(d.skip_word));
            s_skip = (v == d.skip_tag);
        }
        __syncthreads();
        skip = s_skip != 0;
    }

    // Progressive layers take segments from a ticket counter in order, so a warp
    // slowed by whatever else shares its SM does less of the work instead of
    // holding back every later layer's publication; other moves use a static
    // grid stride.
    uint32_t w = skip ? d.total_segs : warp;
    if (d.layer_major) {
        uint32_t t = 0;
        if (lane == 0) t = atomicAdd(d.lay_work, 1u);
        w = __shfl_sync(0xffffffffu, t, 0);
    }
    for (; w < d.total_segs;) {
        if (d.early_trigger && w + nwarps >= d.total_segs) {
            // this warp's last segment (grid stride): the next kernel may launch
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        }
        uint32_t seg, item, lr, c;
        if (d.layer_major) {   // layer, then item, component, segment
            lr = fdiv(w, d.div_pls);
            const uint32_t rem = w - lr * d.per_layer_segs;
            item = fdiv(rem, d.div_cs);
            const uint32_t rem2 = rem - item * (d.C * d.segs);
            c = fdiv(rem2, d.div_segs);
            seg = rem2 - c * d.segs;
        } else {               // item, then layer, component, segment
            const uint32_t chunk = fdiv(w, d.div_segs);
            seg = w - chunk * d.segs;
            item = fdiv(chunk, d.div_lc);
            const uint32_t lc = chunk - item * lc_per_item;
            lr = fdiv(lc, d.div_c);
            c = lc - lr * d.C;
        }
        if (d.layer_major && lr != cur_layer) {
            // a warp walks layers in increasing order: flush the previous layer's tally
            if (cur_count != 0) {
                __threadfence();
                __syncwarp();
                if (lane == 0) publish_layers(d, cur_layer, cur_count);
            }
            cur_layer = lr;
            cur_count = 0;
        }
        ++cur_count;
        const uint64_t l = d.l0 + lr;
        const uint32_t ia = d.gid_a ? (uint32_t)__ldg(d.gid_a + item) : (uint32_t)ids.a[item];
        const uint32_t ib = d.gid_a ? (uint32_t)__ldg(d.gid_b + item) : (uint32_t)ids.b[item];
        if (ia >= d.src.id_limit || ib >= d.dst.id_limit) {
            // Host validation makes this unreachable; never touch memory for a bad id.
            if (lane == 0 && d.err != nullptr) *(volatile uint32_t *)d.err = 1u;
        } else {
        const char *sp = reinterpret_cast<const char *>(chunk_base(d.src, ia, l, c, d.C));
        char *dp = reinterpret_cast<char *>(chunk_base(d.dst, ib, l, c, d.C));
        const uint32_t q0 = seg * (uint32_t)kSegPieces;
        const uint32_t qn = min((uint32_t)kSegPieces, d.cb16 - q0);

        uint4 v[kUnroll];
        if (!kTranspose) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t k = u * 32u + lane;
                if (k < qn) v[u] = load16(sp + (uint64_t)(q0 + k) * 16u);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t k = u * 32u + lane;
                if (k < qn) store16(dp + (uint64_t)(q0 + k) * 16u, v[u]);
            }
        } else if (d.iter_dst) {
            // walk destination pieces in order: contiguous stores, B-byte-run loads
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t k = u * 32u + lane;
                if (k < qn) {
                    const uint32_t qs = permute_piece(q0 + k, d.dst.hnd, d);
                    v[u] = load16(sp + (uint64_t)qs * 16u);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t k = u * 32u + lane;
                if (k < qn) store16(dp + (uint64_t)(q0 + k) * 16u, v[u]);
            }
        } else {
            // walk source pieces in order: contiguous loads, B-byte-run stores
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t k = u * 32u + lane;
                if (k < qn) v[u] = load16(sp + (uint64_t)(q0 + k) * 16u);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t k = u * 32u + lane;
                if (k < qn) {
                    const uint32_t qd = permute_piece(q0 + k, d.src.hnd, d);
                    store16(dp + (uint64_t)qd * 16u, v[u]);
                }
            }
        }
        }   // valid ids
        if (d.layer_major) {
            uint32_t t = 0;
            if (lane == 0) t = atomicAdd(d.lay_work, 1u);
            w = __shfl_sync(0xffffffffu, t, 0);
        } else {
            w += nwarps;
        }
    }
    if (d.pdl) {
        // This CTA has issued all its copies: the next kernel on the stream may
        // start launching (it still waits for this grid to complete), which
        // hides its launch behind this grid's drain without parking its CTAs
        // on SMs for the whole of this one.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (d.layer_major && cur_count != 0) {
        __threadfence();   // this lane's stores are visible device-wide before they are counted
        __syncwarp();
        if (lane == 0) publish_layers(d, cur_layer, cur_count);
    }
    if (d.fence_word != nullptr) complete_grid(d);
}

// ----------------------------------------------------------- bulk (TMA) path


__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Bounded wait for an mbarrier phase: gives up after ~2 s of GPU time.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    for (uint32_t polls = 0; polls < (1u << 30); ++polls) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((polls & 255u) == 255u && global_ns() - t0 > 2000000000ull) return false;
    }
    return false;
}

struct BulkSeg {
    const char *src;
    char *dst;
    uint32_t bytes;
    bool ok;
};

__device__ __forceinline__ BulkSeg bulk_segment(const MoveDesc &d, const int32_t *ia_arr,
                                                const int32_t *ib_arr, uint32_t w) {
    const uint32_t chunk = fdiv(w, d.div_segs);
    const uint32_t seg = w - chunk * d.segs;
    const uint32_t item = fdiv(chunk, d.div_lc);
    const uint32_t lc = chunk - item * (d.nl * d.C);
    const uint32_t lr = fdiv(lc, d.div_c);
    const uint32_t c = lc - lr * d.C;
    const uint64_t l = d.l0 + lr;
    const uint32_t ia = (uint32_t)ia_arr[item];
    const uint32_t ib = (uint32_t)ib_arr[item];
    BulkSeg r;
    r.ok = ia < d.src.id_limit && ib < d.dst.id_limit;
    const uint64_t off = (uint64_t)seg * kBulkBytes;
    const uint64_t cb = (uint64_t)d.cb16 * 16u;
    r.bytes = (uint32_t)min((uint64_t)kBulkBytes, cb - off);
    r.src = reinterpret_cast<const char *>(chunk_base(d.src, ia, l, c, d.C) + off);
    r.dst = reinterpret_cast<char *>(chunk_base(d.dst, ib, l, c, d.C) + off);
    return r;
}

template <int kCap>
__global__ void __launch_bounds__(kBulkThreads)
    kv_bulk_kernel(const __grid_constant__ MoveDesc d, const __grid_constant__ IdsT<kCap> ids) {
    extern __shared__ __align__(128) unsigned char ring[];   // kBulkStages x kBulkBytes
    __shared__ __align__(8) unsigned long long bar[kBulkStages];
    if (d.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");   // previous kernel done
    if (threadIdx.x == 0) {
        for (int s = 0; s < kBulkStages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar[s])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

        const uint32_t first = blockIdx.x, step = gridDim.x;
        uint32_t parity = 0;          // bit s: phase parity expected next on stage s
        bool failed = false;
        // prologue: fill every stage
        for (int s = 0; s < kBulkStages; ++s) {
            const uint32_t w = first + s * step;
            if (w >= d.total_segs) break;
            const BulkSeg g = bulk_segment(d, ids.a, ids.b, w);
            const uint32_t b = smem_addr(&bar[s]);
            const uint32_t buf = smem_addr(ring + s * kBulkBytes);
            const uint32_t bytes = g.ok ? g.bytes : 0u;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b),
                         "r"(bytes) : "memory");
            if (bytes)
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                    "[%0], [%1], %2, [%3];" ::"r"(buf), "l"(g.src), "r"(bytes), "r"(b)
                    : "memory");
        }
        for (uint32_t i = 0;; ++i) {
            const uint32_t w = first + i * step;
            if (w >= d.total_segs) break;
            const int s = (int)(i % kBulkStages);
            const uint32_t b = smem_addr(&bar[s]);
            const uint32_t buf = smem_addr(ring + s * kBulkBytes);
            if (!mbar_wait(b, (parity >> s) & 1u)) {
                failed = true;
                break;
            }
            parity ^= 1u << s;
            const BulkSeg g = bulk_segment(d, ids.a, ids.b, w);
            if (g.ok) {
                asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                                 g.dst), "r"(buf), "r"(g.bytes)
                             : "memory");
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            } else if (d.err != nullptr) {
                *(volatile uint32_t *)d.err = 1u;   // unreachable after host validation
            }
            const uint32_t wn = w + kBulkStages * step;   // refill this stage
            if (wn < d.total_segs) {
                // the store must have finished reading this stage first
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                const BulkSeg gn = bulk_segment(d, ids.a, ids.b, wn);
                const uint32_t bytes = gn.ok ? gn.bytes : 0u;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b),
                             "r"(bytes) : "memory");
                if (bytes)
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                        "[%0], [%1], %2, [%3];" ::"r"(buf), "l"(gn.src), "r"(bytes), "r"(b)
                        : "memory");
            }
        }
        // every segment of this CTA is issued: the next kernel may start launching
        if (d.pdl) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (failed) {
            // Never leave while a load may still be writing this CTA's shared
            // memory: wait (bounded) for every stage, then report.
            for (int s = 0; s < kBulkStages; ++s)
                mbar_wait(smem_addr(&bar[s]), (parity >> s) & 1u);
            if (d.err != nullptr) *(volatile uint32_t *)d.err = 2u;
        }
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // every store complete
        asm volatile("fence.proxy.async.global;" ::: "memory");
        // Lane 0 issued every copy of this CTA, so it completes alone; the other
        // lanes have left already.  Parked at a barrier while lane 0 ran the
        // pipeline, they slowed it: back-to-back 1 GiB gathers ran at 6,363-6,370
        // GB/s that way and at 6,402-6,419 with lane 0 completing alone.
        if (d.fence_word != nullptr) {
            __threadfence();
            arrive_and_publish(d);
        }
    }
}

// ------------------------------------------------- transposing bulk path

// One chunk per work item: lane 0 of warp 0 bulk-loads whole chunks (T*H*B
// bytes, contiguous on the source side) into a ring of `stages` shared-memory
// buffers; every thread waits on the chunk's mbarrier, then the CTA writes the
// chunk in destination order -- consecutive threads store consecutive 16-byte
// pieces (fully coalesced) and read the matching pieces of the source order
// from shared memory (B-byte runs, conflict-free).  Waits are bounded; a CTA
// that gives up waits (bounded) for its loads in flight and sets the error word.
template <int kCap>
__global__ void __launch_bounds__(kTspThreads, 1)
    kv_tsp_kernel(const __grid_constant__ MoveDesc d, const __grid_constant__ IdsT<kCap> ids,
                  uint32_t stage_bytes, uint32_t stages) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) unsigned long long bar[kTspSmem / 4096];
    if (d.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t cb = d.cb16 * 16u;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < stages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar[s])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    auto issue = [&](uint32_t w, uint32_t s) {   // thread 0 only
        const BulkSeg g = bulk_segment(d, ids.a, ids.b, w);
        const uint32_t b = smem_addr(&bar[s]);
        const uint32_t bytes = g.ok ? cb : 0u;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes)
                     : "memory");
        if (bytes)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                "[%0], [%1], %2, [%3];" ::"r"(smem_addr(ring + s * stage_bytes)), "l"(g.src),
                "r"(bytes), "r"(b)
                : "memory");
    };
    const uint32_t first = blockIdx.x, step = gridDim.x;
    if (threadIdx.x == 0)
        for (uint32_t s = 0; s < stages; ++s) {
            const uint64_t w = first + (uint64_t)s * step;
            if (w >= d.total_segs) break;
            issue((uint32_t)w, s);
        }
    uint32_t parity = 0;
    bool failed = false;
    for (uint32_t i = 0;; ++i) {
        const uint64_t w = first + (uint64_t)i * step;
        if (w >= d.total_segs) break;
        const uint32_t s = i % stages;
        const bool ok = mbar_wait(smem_addr(&bar[s]), (parity >> s) & 1u);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        parity ^= 1u << s;
        const BulkSeg g = bulk_segment(d, ids.a, ids.b, (uint32_t)w);
        if (g.ok) {
            const uint4 *src = reinterpret_cast<const uint4 *>(ring + s * stage_bytes);
            char *dst = g.dst;
            for (uint32_t q = threadIdx.x; q < d.cb16; q += kTspThreads) {
                const uint32_t qs = permute_piece(q, d.dst.hnd, d);
                store16(dst + (uint64_t)q * 16u, src[qs]);
            }
        } else if (threadIdx.x == 0 && d.err != nullptr) {
            *(volatile uint32_t *)d.err = 1u;   // unreachable after host validation
        }
        __syncthreads();   // every read of this stage is done
        const uint64_t wn = w + (uint64_t)stages * step;
        if (threadIdx.x == 0 && wn < d.total_segs) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue((uint32_t)wn, s);
        }
    }
    if (d.pdl) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0 && failed) {
        // loads may still be landing in this CTA's shared memory: wait for all
        for (uint32_t s = 0; s < stages; ++s) mbar_wait(smem_addr(&bar[s]), (parity >> s) & 1u);
        if (d.err != nullptr) *(volatile uint32_t *)d.err = 2u;
    }
    if (d.fence_word != nullptr) complete_grid(d);
}

// Runs after copy-engine work on its stream, which is complete (and visible
// to the host) before the kernel starts; the release store orders the rest.
__global__ void kv_mark_kernel(unsigned long long *word, unsigned long long seq) {
    if (threadIdx.x == 0) {
        asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(word), "l"(seq) : "memory");
    }
}

// Ready-fence gate: bounded wait, never a trap.  The poll count is capped too,
// so the wait ends even if the global timer were not advancing.
__global__ void kv_gate_kernel(const unsigned long long *word, unsigned long long value,
                               unsigned long long timeout_ns, unsigned long long *status,
                               unsigned long long tag) {
    if (threadIdx.x != 0) return;
    const unsigned long long t0 = global_ns();
    const unsigned long long max_polls = timeout_ns / 32ull + 4096ull;
    unsigned int sleep_ns = 32;
    for (unsigned long long polls = 0;; ++polls) {
        unsigned long long v;
        asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(word) : "memory");
        if (v >= value) return;
        if (global_ns() - t0 >= timeout_ns || polls >= max_polls) {
            asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(status), "l"(tag) : "memory");
            __threadfence_system();
            return;
        }
        __nanosleep(sleep_ns);
        if (sleep_ns < 4096) sleep_ns <<= 1;
    }
}

}  // namespace

FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{d, 0u, 0u, 0u};
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    const uint64_t two32 = 1ull << 32;
    f.m = (uint32_t)((two32 * ((1ull << l) - d)) / d + 1ull);
    f.s = l;
    return f;
}

template <int kCap, int kThreads>
static cudaError_t launch_cap(const MoveDesc &d, const MoveIds &ids, int ctas, cudaStream_t stream) {
    IdsT<kCap> p;
    const uint32_t in_block = d.gid_a ? 0u : d.n;   // ids in device memory: none in the block
    for (uint32_t i = 0; i < in_block; ++i) {
        p.a[i] = ids.a[i];
        p.b[i] = ids.b[i];
    }
    if (d.pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas);
        cfg.blockDim = dim3((unsigned)kThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (d.transpose)
            return cudaLaunchKernelEx(&cfg, kv_move_kernel<true, kCap, kThreads>, d, p);
        return cudaLaunchKernelEx(&cfg, kv_move_kernel<false, kCap, kThreads>, d, p);
    }
    if (d.transpose)
        kv_move_kernel<true, kCap, kThreads><<<ctas, kThreads, 0, stream>>>(d, p);
    else
        kv_move_kernel<false, kCap, kThreads><<<ctas, kThreads, 0, stream>>>(d, p);
    return cudaGetLastError();
}

template <int kThreads>
static cudaError_t launch_threads(const MoveDesc &d, const MoveIds &ids, int ctas,
                                  cudaStream_t stream) {
    if (d.gid_a != nullptr || d.n <= 64) return launch_cap<64, kThreads>(d, ids, ctas, stream);
    if (d.n <= 512) return launch_cap<512, kThreads>(d, ids, ctas, stream);
    return launch_cap<kMaxItems, kThreads>(d, ids, ctas, stream);
}

template <int kCap>
static cudaError_t launch_bulk_cap(const MoveDesc &d, const MoveIds &ids, int ctas,
                                   cudaStream_t stream) {
    static bool attr_set = false;   // per instantiation; set once (host calls are serialised)
    const int smem = kBulkStages * (int)kBulkBytes;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kv_bulk_kernel<kCap>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    IdsT<kCap> p;
    for (uint32_t i = 0; i < d.n; ++i) {
        p.a[i] = ids.a[i];
        p.b[i] = ids.b[i];
    }
    if (d.pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas);
        cfg.blockDim = dim3((unsigned)kBulkThreads);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kv_bulk_kernel<kCap>, d, p);
    }
    kv_bulk_kernel<kCap><<<ctas, kBulkThreads, smem, stream>>>(d, p);
    return cudaGetLastError();
}

cudaError_t launch_bulk(const MoveDesc &d, const MoveIds &ids, int ctas, cudaStream_t stream) {
    (void)cudaGetLastError();
    if (d.n > (uint32_t)kMaxItems || d.transpose || d.gid_a != nullptr) return cudaErrorInvalidValue;
    if (d.n <= 64) return launch_bulk_cap<64>(d, ids, ctas, stream);
    if (d.n <= 512) return launch_bulk_cap<512>(d, ids, ctas, stream);
    return launch_bulk_cap<kMaxItems>(d, ids, ctas, stream);
}

template <int kCap>
static cudaError_t launch_tsp_cap(const MoveDesc &d, const MoveIds &ids, int ctas,
                                  cudaStream_t stream) {
    static bool attr_set = false;   // per instantiation; host calls are serialised
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kv_tsp_kernel<kCap>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kTspSmem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const uint32_t cb = d.cb16 * 16u;
    const uint32_t stage = (cb + 127u) / 128u * 128u;
    uint32_t stages = kTspSmem / stage;
    if (stages > 4) stages = 4;
    if (stages < 2) return cudaErrorInvalidValue;
    IdsT<kCap> p;
    for (uint32_t i = 0; i < d.n; ++i) {
        p.a[i] = ids.a[i];
        p.b[i] = ids.b[i];
    }
    const size_t smem = (size_t)stages * stage;
    if (d.pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ctas);
        cfg.blockDim = dim3((unsigned)kTspThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kv_tsp_kernel<kCap>, d, p, stage, stages);
    }
    kv_tsp_kernel<kCap><<<ctas, kTspThreads, smem, stream>>>(d, p, stage, stages);
    return cudaGetLastError();
}

cudaError_t launch_tsp(const MoveDesc &d, const MoveIds &ids, int ctas, cudaStream_t stream) {
    (void)cudaGetLastError();
    if (d.n > (uint32_t)kMaxItems || !d.transpose || d.segs != 1 || d.cb16 * 16u > kTspMaxChunk ||
        d.gid_a != nullptr)
        return cudaErrorInvalidValue;
    if (d.n <= 64) return launch_tsp_cap<64>(d, ids, ctas, stream);
    if (d.n <= 512) return launch_tsp_cap<512>(d, ids, ctas, stream);
    return launch_tsp_cap<kMaxItems>(d, ids, ctas, stream);
}

// Lazy loading (the CUDA default) loads a kernel's code at its first launch,
// and the load waits for the device to go idle: a first launch queued behind a
// kernel that waits -- a ready-fence gate, a resident ring server -- would
// stall until that wait ends.  Every kernel here is loaded once, up front.
cudaError_t preload_kernels() {
    cudaFuncAttributes a;
    const void *const fns[] = {
        (const void *)kv_move_kernel<false, 64, kMoveThreads>,
        (const void *)kv_move_kernel<false, 512, kMoveThreads>,
        (const void *)kv_move_kernel<false, kMaxItems, kMoveThreads>,
        (const void *)kv_move_kernel<true, 64, kMoveThreads>,
        (const void *)kv_move_kernel<true, 512, kMoveThreads>,
        (const void *)kv_move_kernel<true, kMaxItems, kMoveThreads>,
        (const void *)kv_move_kernel<false, 64, kWideThreads>,
        (const void *)kv_move_kernel<false, 512, kWideThreads>,
        (const void *)kv_move_kernel<false, kMaxItems, kWideThreads>,
        (const void *)kv_move_kernel<true, 64, kWideThreads>,
        (const void *)kv_move_kernel<true, 512, kWideThreads>,
        (const void *)kv_move_kernel<true, kMaxItems, kWideThreads>,
        (const void *)kv_bulk_kernel<64>,
        (const void *)kv_bulk_kernel<512>,
        (const void *)kv_bulk_kernel<kMaxItems>,
        (const void *)kv_tsp_kernel<64>,
        (const void *)kv_tsp_kernel<512>,
        (const void *)kv_tsp_kernel<kMaxItems>,
        (const void *)kv_mark_kernel,
        (const void *)kv_gate_kernel,
    };
    for (const void *f : fns) {
        const cudaError_t e = cudaFuncGetAttributes(&a, f);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_move(const MoveDesc &d, const MoveIds &ids, int ctas, int threads,
                        cudaStream_t stream) {
    (void)cudaGetLastError();   // report this launch's error, not an earlier call's
    if (d.n > (uint32_t)kMaxItems && d.gid_a == nullptr) return cudaErrorInvalidValue;
    if ((d.gid_a == nullptr) != (d.gid_b == nullptr)) return cudaErrorInvalidValue;
    if (threads == kWideThreads) return launch_threads<kWideThreads>(d, ids, ctas, stream);
    if (threads == kMoveThreads) return launch_threads<kMoveThreads>(d, ids, ctas, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_mark(unsigned long long *word, unsigned long long seq, cudaStream_t stream) {
    (void)cudaGetLastError();
    kv_mark_kernel<<<1, 32, 0, stream>>>(word, seq);
    return cudaGetLastError();
}

cudaError_t launch_gate(const unsigned long long *word, unsigned long long value,
                        unsigned long long timeout_ns, unsigned long long *status,
                        unsigned long long tag, cudaStream_t stream) {
    (void)cudaGetLastError();
    kv_gate_kernel<<<1, 32, 0, stream>>>(word, value, timeout_ns, status, tag);
    return cudaGetLastError();
}

}  // namespace kvb
