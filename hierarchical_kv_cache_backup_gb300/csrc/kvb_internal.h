// kvb_internal.h -- declarations shared by the host engine (kvb_api.cpp) and
// the sm_103a kernels (kvb_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kvb {

// Invariant-divisor division by multiply-high and shift (Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication", PLDI
// 1994, unsigned case with N = 32): for d >= 1, l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1, and n / d = (umulhi(n, m) + n) >> l,
// with the addition done in 64 bits.  Exact for every 32-bit n.
struct FastDiv {
    uint32_t d, m, s, pad;
};
FastDiv make_fastdiv(uint32_t d);   // host; d >= 1

// One side of a move: where unit vectors of chunk (id, layer, comp) live.
// A "chunk" is the T*H*B bytes of one (page or slot, layer, component).
//   chunk address = base + id*s_id + layer*s_l + comp*s_c
//   inside a chunk: NHD [T][H] or HND [H][T] vectors of B bytes.
struct Side {
    uint64_t base;      // device-visible address of the side's byte 0
    uint64_t s_id;      // bytes between consecutive ids (pages or slots)
    uint64_t s_l;       // bytes between consecutive layers
    uint64_t s_c;       // bytes between components
    uint32_t hnd;       // head order inside a chunk: 0 = NHD, 1 = HND
    uint32_t id_limit;  // ids must be below this (checked again on the GPU)
    // Split pools: when set, chunk address = lc_base[layer * C + comp] + id * s_id
    // (one device buffer per layer and component; base, s_l, s_c unused).
    const unsigned long long *lc_base;
};

// Kernel-parameter budget: the ids of one launch travel inside the launch
// itself (sm_70+ accepts up to 32,764 bytes of parameters), so no device
// buffer, copy or ring is needed for them.
constexpr int kMaxItems = 2048;     // (a, b) id pairs per launch
constexpr int kSegPieces = 256;     // 16-byte pieces a warp moves per segment (4 KiB)
constexpr int kMoveThreads = 256;   // threads per CTA of the move kernel (HBM-only moves)
constexpr int kWideThreads = 1024;  // wide CTAs: host-link moves packed onto few SMs
// Bulk-copy (TMA) variant for HBM-only moves whose two sides share a head
// order: one warp per CTA, lane 0 streams each chunk through a ring of
// kBulkStages shared-memory buffers of kBulkBytes with cp.async.bulk.
// 8 x 8 KiB (64 KiB per CTA, 3 CTAs per SM) measured best on GB300 for a
// gather of random 32 KiB chunks: 6.8 TB/s, against 6.4 TB/s for 4 x 16 KiB.
constexpr int kBulkStages = 8;
constexpr uint32_t kBulkBytes = 8192;
constexpr int kBulkThreads = 32;
// Transposing variant for HBM-only moves whose sides differ in head order:
// whole chunks are bulk-loaded into a ring of shared-memory stages and 256
// threads write them out in destination order.  Chunks up to kTspMaxChunk.
constexpr int kTspThreads = 256;
constexpr uint32_t kTspSmem = 196608;        // ring bytes per CTA (1 CTA per SM)
constexpr uint32_t kTspMaxChunk = kTspSmem / 2;

struct MoveDesc {
    Side src, dst;
    uint32_t n;          // items in this launch
    uint32_t nl;         // layers per item
    uint32_t l0;         // first layer
    uint32_t C;          // components
    uint32_t cb16;       // 16-byte pieces per chunk (T*H*B/16)
    uint32_t segs;       // segments per chunk
    uint32_t total_segs; // n * nl * C * segs (< 2^32)
    uint32_t H, T, B16;  // heads, tokens, 16-byte pieces per head vector
    uint32_t transpose;  // 1 when the two sides' head orders differ (H, T > 1)
    uint32_t iter_dst;   // transpose only: 1 = walk destination order
    FastDiv div_segs, div_lc, div_c, div_b16, div_T, div_H;
    uint32_t *err;       // device-visible sticky word: 1 a kernel met a bad id, 2 a bulk
                         // copy's wait gave up, 3 a chained fence's wait gave up
    // Completion, fused: when fence_word is set, the last CTA to finish stores
    // fence_seq there (system scope, release) once every CTA's bytes are
    // visible; fence_count is a zeroed device counter that CTA resets.
    unsigned long long *fence_word;
    unsigned long long fence_seq;
    uint32_t *fence_count;
    // Gating: when skip_word is set and *skip_word == skip_tag (written by the
    // ready-fence gate that ran before this kernel), no byte is moved.
    const unsigned long long *skip_word;
    unsigned long long skip_tag;
    // Progressive layers (layer_major = 1): segments run layer by layer and
    // layer j's fence (sequence seq0 + j, ring slot (seq0 + j) % ring) is
    // published as soon as layers 0..j are all in place.
    uint32_t layer_major;
    uint32_t per_layer_segs;        // n * C * segs
    FastDiv div_pls, div_cs;        // per_layer_segs, C * segs
    unsigned long long *lay_words;  // fence words (device view of the ring)
    unsigned long long lay_seq0;
    uint32_t lay_ring;
    uint32_t *lay_done;             // per-slot finished-segment counters (zeroed before launch)
    uint32_t *lay_published;        // layers published so far (zeroed before launch)
    uint32_t *lay_work;             // next segment ticket (zeroed before launch)
    uint32_t *lay_lock;             // publisher lock (zeroed before launch)
    // Programmatic dependent launch: launched so that it may start while the
    // previous kernel on its stream finishes; it waits (griddepcontrol.wait)
    // for that kernel's completion before touching memory.
    uint32_t pdl;
    // Overlapped restores (KV_CFG_OVERLAP_RESTORES).  early_trigger: each warp
    // lets the next kernel on the stream launch when it takes its last segment
    // rather than after it, so a successor that starts moving at once finds the
    // link still busy with this kernel's last bytes.  overlap: the host proved
    // that this restore and the previous kernel on the stream (a restore of
    // the same pool) write disjoint bytes and neither writes what the other
    // reads, so this kernel skips griddepcontrol.wait; its last CTA publishes
    // the fence only once the previous op's fence word (chain_word) holds
    // chain_seq or more, so fences still complete in call order.
    uint32_t early_trigger;
    uint32_t overlap;
    const unsigned long long *chain_word;
    unsigned long long chain_seq;
    // Ids in device memory (item i: gid_a[i], gid_b[i]) instead of the launch's
    // parameter block, for one move kernel over more items than a parameter
    // block holds (progressive restores of more than kMaxItems pages).
    const int32_t *gid_a, *gid_b;
    // A second completion word (a ring descriptor's completion record): the
    // CTA that publishes the fence then stores ext_value to ext_word too.
    unsigned long long *ext_word;
    unsigned long long ext_value;
};

// Ids of one launch, inside the kernel's parameter block.  Launches use the
// smallest capacity that holds their items (64, 512 or kMaxItems), so small
// operations do not ship 16 KiB of parameters.
template <int kCap>
struct IdsT {
    int32_t a[kCap];   // source ids (pages for backup, slots for restore)
    int32_t b[kCap];   // destination ids
};
using MoveIds = IdsT<kMaxItems>;

// Loads every kernel of this file on the current device (lazy loading would
// load each at its first launch, waiting for the device to go idle).
cudaError_t preload_kernels();
// Launch the gather/scatter kernel on `stream` with `ctas` CTAs of `threads`
// threads (kMoveThreads or kWideThreads).
cudaError_t launch_move(const MoveDesc &d, const MoveIds &ids, int ctas, int threads,
                        cudaStream_t stream);
// Launch the bulk-copy variant (identity chunks only; d.segs / d.div_segs /
// d.total_segs count kBulkBytes segments).  `ctas` CTAs of kBulkThreads.
cudaError_t launch_bulk(const MoveDesc &d, const MoveIds &ids, int ctas, cudaStream_t stream);
// Launch the transposing variant (d.segs = 1: one work item per chunk; chunk
// bytes <= kTspMaxChunk).  `ctas` CTAs of kTspThreads.
cudaError_t launch_tsp(const MoveDesc &d, const MoveIds &ids, int ctas, cudaStream_t stream);
// Launch the completion marker: stores `seq` to `word` (system scope, release)
// once everything before it on `stream` has finished.
cudaError_t launch_mark(unsigned long long *word, unsigned long long seq, cudaStream_t stream);
// Launch the ready-fence gate: one thread waits until *word >= value or until
// timeout_ns has passed on the GPU's global timer (and at most a bounded
// number of polls); on time-out it stores `tag` to *status, which makes the
// gated kernels that follow on `stream` skip their work.
cudaError_t launch_gate(const unsigned long long *word, unsigned long long value,
                        unsigned long long timeout_ns, unsigned long long *status,
                        unsigned long long tag, cudaStream_t stream);

// ---- support for kv_backup_staged_noalloc (kvb_noalloc.cu) ----------------
// Records `msg` as this thread's last error and returns `status`.
int set_last_error(int status, const char *msg);
// Device of a live pool handle, or an error status.
int pool_device_of(const void *pool_handle, int *device);
// Validates a staged backup into a caller-supplied device staging area of
// `staging_bytes` and enqueues it on `stream`: the gather kernel (pool ->
// staging, host layout) and copy-engine copies (staging -> host tier).  Uses
// no heap, no CUDA allocation and no library fence; returns a kv_status.
// Issues a ring descriptor's backup (kind 0) or restore (kind 1) like
// kv_backup / kv_restore, and asks for `done_word` (device view of the ticket's
// completion record) to be set to `ticket` by the move kernel itself once the
// bytes are in place.  *fused = 1 when that was possible (a zero-copy op with
// pages to move); otherwise the caller completes the ticket itself.
int ring_issue(const void *pool_handle, const void *host_handle, int kind, const int32_t *a,
               const int32_t *b, uint32_t n, int32_t layer, void *stream,
               unsigned long long *done_word, unsigned long long ticket, uint64_t *fence,
               int *fused);
int enqueue_staged_backup_noalloc(const void *pool_handle, const void *host_handle,
                                  const int32_t *src_pages, const int32_t *host_slots, uint32_t n,
                                  void *staging, uint64_t staging_bytes, cudaStream_t stream);

}  // namespace kvb
