// kvb_ring_internal.h -- declarations shared by the descriptor ring
// (kvb_ring.cpp), its GPU-resident server kernel (kvb_ring_kernels.cu) and the
// engine (kvb_api.cpp).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvb.h"
#include "kvb_internal.h"

namespace kvb {

// Completion record of one ring slot, in the shared segment.  `done` is the
// last completed ticket of the slot; `err_ticket` / `err` are written before
// `done` when that ticket failed.
struct CompRec {
    uint64_t done;
    uint64_t err_ticket;
    int32_t err;
    int32_t pad;
    uint64_t pad2;
};
static_assert(sizeof(CompRec) == 32, "completion record size");

// One pool of a GPU-resident server's table: its device side and the geometry
// the kernel needs to decode a descriptor's work into 4 KiB warp segments.
struct RingPoolK {
    Side pool;                 // device side (strides, or a split pool's table)
    uint32_t L, C, P;          // layers, components, pages
    uint32_t H, T, B16;        // heads, tokens, 16-byte pieces per head vector
    uint32_t cb16;             // 16-byte pieces per (page, layer, component) chunk
    uint32_t segs;             // warp segments per chunk: ceil(cb16 / kSegPieces)
    uint32_t transpose;        // the pool's and the host tier's head orders differ (H, T > 1)
    uint32_t pad;
    FastDiv div_segs, div_lc_all, div_lc_one, div_c, div_b16, div_T, div_H;
};

// Control block of a resident server (device memory, zeroed before launch).
struct RingCtl {
    uint32_t gen;              // descriptors released to every CTA so far
    uint32_t stop;             // set by the leader once no more will be released
    uint32_t arrived;          // CTA arrivals at descriptor ends, cumulative mod 2^32
    uint32_t gave_up;          // a CTA's bounded wait ran out
    // the released descriptor
    uint32_t kind, n, pool;
    int32_t layer;
    uint64_t ticket;
};

// Everything the resident server kernel reads, by value.
struct RingKDesc {
    // the shared segment, device views
    const unsigned long long *tail;   // last published ticket
    const unsigned long long *ready;  // KV_RING_READY_WORDS ready words of gated descriptors
    unsigned long long *head;         // last taken ticket
    long long *server_pid;
    const kv_ring_op *ops;            // entries
    CompRec *comp;                    // completion records
    uint32_t slots;
    uint32_t max_ops;
    uint64_t first_ticket;            // head + 1 when the server starts
    uint64_t idle_ns;                 // give up after this long without a descriptor
    long long pid;                    // the serving process
    // the host tier (slot side, device-visible)
    Side host;
    uint32_t num_slots;
    uint32_t npools;
    const RingPoolK *pools;           // device array of npools
    // device scratch
    RingCtl *ctl;
    int32_t *ids;                     // 2 * KV_RING_MAX_IDS: a then b of the released descriptor
    uint32_t *result;                 // mapped pinned: [0] served, [1] kv_status of the server,
                                      // [2] set by the host: stop before the next descriptor
};

// Shape of the resident server: one leader CTA (takes, checks and releases
// descriptors) and 32 mover CTAs, all of 256 threads (on GB300 the move kernel
// reaches the D2H peak with 16 such CTAs and the H2D peak with 32); a
// 256-thread CTA leaves each thread the registers of every move variant.  The
// server holds 33 SMs while it runs, idle or not.
constexpr int kRingMovers = 32;
constexpr int kRingThreads = 256;

// Loads the resident server kernel on the current device (see preload_kernels).
cudaError_t preload_ring_kernels();

// Launches the resident server as a cooperative grid of `ctas` CTAs of
// kRingThreads threads on `stream` (every CTA resident at once): CTA 0 leads,
// the other ctas - 1 (at least one) move.
cudaError_t launch_ring_server(const RingKDesc &k, int ctas, cudaStream_t stream);

// ---- engine support for the resident server (kvb_api.cpp) ----------------
// Validates a server's pool table and host tier (live handles, one device, the
// host tier's slot geometry, no retired generation) and fills `table` (npools
// entries), the host side and slot count.  Returns a kv_status.
int ring_server_view(const kv_pool *pools, uint32_t npools, kv_host host, RingPoolK *table,
                     Side *host_side, uint32_t *num_slots, int *device);
// Launches the resident server (launch_ring_server) on `stream` and a library
// fence after it; the fence's slot is reserved before the launch, so nothing
// that might wait for the device runs while the server is resident.
int ring_launch_server(int device, const RingKDesc &k, int ctas, cudaStream_t stream,
                       kv_fence *fence);
// For a fence issued by a gated operation (kv_backup_when_ready /
// kv_restore_when_ready): the device address of its gate-status word and the
// tag the gate stores there when it gives up.  Returns a kv_status.
int fence_gate_word(kv_fence f, const unsigned long long **word, unsigned long long *tag);

// ---- host server support (kvb_ring.cpp) -----------------------------------
// Completes ring ticket `ticket` on `stream` after the work before it: when
// `status` is set and holds `tag` (the gate of the ticket's operation gave
// up), first stores ABORTED into `err` and the ticket into `err_ticket`; then
// stores the ticket into `done` (system scope, release).
cudaError_t launch_ring_mark(unsigned long long *done, unsigned long long *err_ticket,
                             int32_t *err, unsigned long long ticket,
                             const unsigned long long *status, unsigned long long tag,
                             cudaStream_t stream);

}  // namespace kvb
