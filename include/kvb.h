/*
 * kvb.h -- C ABI of the GB300 paged KV-cache backup / restore engine.
 *
 * The engine moves KV-cache pages between a GPU KV pool (device memory) and a
 * pinned host KV tier, in both directions, converting between the pool's
 * layout and the host tier's page-contiguous layout on the way.  Payload is
 * opaque bytes: fp16, bf16 and fp8_e4m3 KV all take the same path.
 *
 * Pages this interface restates (cited by title and section):
 *   [RFC] "[Feature] [RFC] [HiCache] Out-of-process HiCache data plane with
 *         device-memory IPC": §Device IPC data path (REGISTER_KV_POOL, BACKUP,
 *         RESTORE descriptors; export / import / close of device memory;
 *         export / import / wait of fences), §Ownership, §Failure and
 *         lifecycle handling.
 *   [PR]  "[PP + HiCache] Add PP Prefetch Tickets for eager cross-stage
 *         storage prefetch": §PP Prefetch Ticket Path (layer-wise H2D ahead
 *         of each layer's forward).
 *   [LMC] "LMCacheRawCudaIPCWrapper深度解析：基于驱动级 CUDA IPC 共享 PyTorch
 *         之外的 KV Cache": §共享与重建的完整链路 (allocation base + byte
 *         offset), §uint8字节往返 (dtype-neutral bytes), §发送端校验 (reject,
 *         never silently copy), §重建生命周期与引用计数 (refcounted mappings,
 *         close logs but never throws), §在项目中的实际接入方式 (TRT-LLM pool
 *         [NB, NL, 2, NH*BS*HS], kv_layout = HND).
 *
 * Conventions for every call:
 *   - Status codes only.  Nothing aborts, throws or traps across this ABI.
 *     A call rejected by validation (INVALID_ARG, OUT_OF_RANGE, DUPLICATE,
 *     ALIGNMENT, LAYOUT, STALE, CLOSED) has had no side effect: validation
 *     runs before anything is enqueued ([LMC] §发送端校验).  A CUDA call that
 *     fails part-way through an op (CUDA) may leave the part already
 *     enqueued to complete, inside the op's own targets.  kv_last_error()
 *     gives a readable message (thread-local) for the last failing call.
 *   - Device pointers are plain CUDA device addresses; host pointers are
 *     plain host addresses.  Streams are cudaStream_t values passed as void*
 *     (NULL = the legacy default stream).
 *   - Page IDs and host slots are int32 arrays in HOST memory.  The call
 *     copies them before returning, so the caller may reuse them at once.
 *   - Ownership ([RFC] §Ownership): the caller owns the device pool
 *     allocation, its page allocator and page lifetimes, the pinned host
 *     memory and the streams.  The library owns IPC mappings, staging
 *     buffers, fence words and events.  Pool and host bytes named by an
 *     operation must not be touched by the caller until its fence completes.
 *
 * Unit and layouts.  A unit is the B-byte head vector of (page p, layer l,
 * component c, token t, head h); B = head_dim x element bytes.  With L layers,
 * C components (2 = K,V; 1 = MLA latent), P pages, T tokens per page and H
 * heads, the pool and the host tier are these row-major arrays of units:
 *     KV_LAYER_FIRST + KV_NHD : [L][C][P][T][H]
 *     KV_LAYER_FIRST + KV_HND : [L][C][P][H][T]
 *     KV_PAGE_FIRST  + KV_NHD : [P][L][C][T][H]
 *     KV_PAGE_FIRST  + KV_HND : [P][L][C][H][T]   (the TRT-LLM 6-D view
 *                                [NB, NL, 2, NH, BS, HS] of [LMC])
 *     host tier, NHD / HND    : [S][L][C][T][H] / [S][L][C][H][T]
 * so one host slot holds one whole page contiguously (L*C*T*H*B bytes).
 */
#ifndef KVB_H
#define KVB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVB_ABI_VERSION 2u   /* 2: gated ring descriptors (kv_ring_op grew), split-pool IPC */

#if defined(__GNUC__)
#define KVB_API __attribute__((visibility("default")))
#else
#define KVB_API
#endif

typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,   /* null handle/pointer, bad enum, bad size     */
    KV_ERR_OUT_OF_RANGE = 2,  /* page / slot / layer outside the pool / tier */
    KV_ERR_DUPLICATE = 3,     /* one call writes one page or slot twice      */
    KV_ERR_ALIGNMENT = 4,     /* B or the pool / host start not 16-B aligned */
    KV_ERR_LAYOUT = 5,        /* layout invalid, or pool and tier disagree   */
    KV_ERR_STALE = 6,         /* pool generation retired ([RFC] lifecycle)   */
    KV_ERR_TIMEOUT = 7,       /* fence not complete (query) / not in time    */
    KV_ERR_CUDA = 8,          /* a CUDA call failed; see kv_last_error()     */
    KV_ERR_NO_MEMORY = 9,     /* library could not allocate its resources    */
    KV_ERR_CLOSED = 10,       /* handle already closed                       */
    KV_ERR_ABORTED = 11,      /* op gave up: its ready fence never arrived   */
    KV_ERR_IO = 12            /* a file read / write failed (L3 record store) */
} kv_status;

typedef enum { KV_LAYER_FIRST = 0, KV_PAGE_FIRST = 1 } kv_order;
typedef enum { KV_NHD = 0, KV_HND = 1 } kv_heads;

/* Pool geometry (the `layout` argument of REGISTER_KV_POOL, [RFC] §Device IPC
 * data path).  Fixed-size POD. */
typedef struct {
    uint32_t num_layers;   /* L                                               */
    uint32_t num_comps;    /* C: 2 = K and V, 1 = MLA latent                  */
    uint32_t num_pages;    /* P                                               */
    uint32_t page_tokens;  /* T                                               */
    uint32_t num_heads;    /* H                                               */
    uint32_t head_bytes;   /* B = head_dim x element bytes; multiple of 16    */
    uint32_t order;        /* kv_order of the device pool                     */
    uint32_t heads;        /* kv_heads of the device pool                     */
    uint32_t elem_bytes;   /* informational only: payload is opaque bytes     */
    uint32_t reserved;     /* must be 0                                       */
} kv_layout;

typedef struct kv_pool_s *kv_pool;
typedef struct kv_host_s *kv_host;
typedef uint64_t kv_fence;   /* 0 is never a valid fence */

/* IPC descriptor of a pool ([RFC] §Device IPC data path REGISTER_KV_POOL with
 * instance_id / generation / device identity; [LMC] §共享与重建的完整链路
 * sender step 5: handle of the allocation base, byte offset, size, device
 * UUID).  Fixed-size POD: send its bytes over any channel. */
typedef struct {
    uint32_t magic;            /* KVB_IPC_MAGIC                                */
    uint32_t version;          /* KVB_ABI_VERSION                              */
    uint8_t handle[64];        /* cudaIpcMemHandle_t of the allocation base    */
    uint64_t alloc_offset;     /* pool start minus allocation base, in bytes   */
    uint64_t nbytes;           /* pool bytes: P x L x C x T x H x B            */
    uint64_t instance_id;      /* exporter instance identity                   */
    uint64_t generation;       /* pool generation                              */
    int64_t exporter_pid;      /* exporter process identity                    */
    uint8_t device_uuid[16];   /* device identity (resolved to an ordinal)     */
    kv_layout layout;
} kv_ipc_desc;
#define KVB_IPC_MAGIC 0x4B564231u /* "KVB1" */

/* One buffer of a split pool over IPC: the handle of the allocation that holds
 * it and the buffer's byte offset from that allocation's base.  Fixed-size
 * POD.  A split pool's kv_ipc_desc carries KVB_IPC_MAGIC_SPLIT. */
typedef struct {
    uint8_t handle[64];        /* cudaIpcMemHandle_t of the allocation base    */
    uint64_t alloc_offset;     /* buffer start minus allocation base, in bytes */
} kv_ipc_buffer;
#define KVB_IPC_MAGIC_SPLIT 0x4B564253u /* "KVBS" */

/* Transfer modes.  ZERO_COPY: one kernel moves every byte between HBM and the
 * mapped pinned host tier over the host link.  STAGED: a kernel gathers /
 * scatters between the pool and a device staging buffer in host layout, and
 * the copy engine moves the staging buffer to / from the host tier.
 * COPY_ENGINE: no kernel moves data; every contiguous run goes straight
 * between the pool and the pinned host tier as cudaMemcpyAsync /
 * cudaMemcpy2DAsync copies (one pitched copy per page when the head orders
 * agree, merged across pages whose ids and slots both step by one; a head-order
 * change costs min(H, T) pitched copies per page, layer and component, so it
 * is slow to issue).  The fence completes through a marker kernel after the
 * copies.  kv_restore_layers and ready-gated backups / restores run zero-copy
 * in every mode. */
typedef enum { KV_MODE_ZERO_COPY = 0, KV_MODE_STAGED = 1, KV_MODE_COPY_ENGINE = 2 } kv_mode;

/* kv_config.flags */
#define KV_CFG_NO_BULK 1u   /* HBM-only moves use the register kernel, not bulk copies */
#define KV_CFG_NO_PDL 2u    /* zero-copy moves and device gathers / scatters launch plainly:
                               no programmatic dependent launch overlapping a kernel's
                               launch with the previous kernel's end */
/* KV_CFG_OVERLAP_RESTORES (opt-in; needs programmatic dependent launch, so it
 * has no effect together with KV_CFG_NO_PDL).  A zero-copy kv_restore may start
 * moving bytes while the previous kernel on its stream is still finishing,
 * instead of after it, when the library can prove them independent.  Per
 * stream (a created stream: never the legacy default stream, cudaStreamLegacy
 * or cudaStreamPerThread) it keeps the run of restores of one pool handle
 * issued there since the last call that waited for its predecessor; any other
 * call of this library on that stream ends the run.  A new restore of the same
 * pool overlaps when it writes no byte that a restore of the run whose fence is
 * not yet complete writes: another layer (both one-layer restores), or no
 * destination page in common.  Restores only read the host tier, so nothing
 * else can conflict.  This is the layer-by-layer restore of the PP prefetch PR
 * (§PP Prefetch Ticket Path, "Layer-wise H2D + forward"): consecutive one-layer
 * restores keep the host link busy across the boundary between calls instead
 * of draining it.  The overlapping restore must fit one launch (n <= 2,048
 * pages).  Fences still complete in call order: a restore publishes its fence
 * only after its predecessor's (a wait on the GPU, bounded at 2 s; if it ever
 * gave up, every later fence query reports KV_ERR_TIMEOUT).  Under this flag
 * zero-copy restores run, unless max_ctas / cta_threads say otherwise, on 6
 * CTAs of 1,024 threads (6 whole SMs): overlapped, that reaches ~99% of the H2D
 * link and leaves the rest of the GPU to the forward pass.  Contract: the
 * library cannot see work that the caller itself puts on the stream between
 * two of its calls; under this flag such work must not write the host slots or
 * pages a later restore reads or writes, nor read the pages it writes. */
#define KV_CFG_OVERLAP_RESTORES 4u
/* KV_CFG_OVERLAP_BACKUPS (opt-in, same mechanism and contract): zero-copy
 * kv_backup calls take part in a stream's run of overlapped ops too.  A new op
 * (backup or restore, same pool handle, same stream) may overlap the ops of
 * the run whose fences are not yet complete when no byte that one of the two
 * writes is touched by the other: a backup reads its source pages (every
 * layer) and writes its host slots; a restore reads its host slots and writes
 * its destination pages (its layer, or every layer).  So consecutive backups
 * into disjoint slots overlap, and a backup of pages a restore is still
 * writing does not.  Useful for streams of small ops, whose time is mostly
 * latency; fences still complete in call order. */
#define KV_CFG_OVERLAP_BACKUPS 8u

/* Defaults: host-link moves (zero-copy backup / restore) run 16 CTAs of 1024
 * threads when pool and tier share a head order and 64 CTAs of 256 when the
 * move changes it (the shapes with which a backup and a restore running at
 * once come closest to the bidirectional link peak; either reaches the solo
 * peak); kv_restore_layers, made to run beside compute, runs 8 CTAs of 1024
 * threads (8 whole SMs); HBM-only moves run 4 CTAs of 256 threads per SM
 * (bulk-copy kernel: 3 per SM).  cta_threads = 256 or 1024 forces that CTA
 * size on every host-link move (64 CTAs of 256, 16 of 1024).  Sizing the SM
 * budget of moves that run beside compute: with cta_threads = 1024 each CTA
 * holds one whole SM, and on GB300 one SM moves ~42-49 GB/s from the host
 * tier and ~47 GB/s to it, so max_ctas = 6 reaches ~99% of the D2H link and
 * ~96% of H2D, 8 reaches ~99% of both. */
typedef struct {
    uint32_t mode;           /* kv_mode                                         */
    uint32_t max_ctas;       /* CTA cap of the transfer kernels, and the mover
                                CTAs of a resident ring server; 0 = default    */
    uint64_t staging_bytes;  /* STAGED: device staging bytes; 0 = default       */
    uint32_t flags;          /* KV_CFG_* bits                                   */
    uint32_t cta_threads;    /* host-link CTA size: 0 = default, 256, 1024      */
} kv_config;

/* ------------------------------------------------------------------ pools */

/* REGISTER_KV_POOL ([RFC] §Device IPC data path).  Registers a pool the
 * caller allocated: it starts `offset` bytes after device pointer `base`.
 * Checks: layout valid (dims >= 1, B % 16 == 0, enums known, sizes fit in
 * 64 bits), base+offset 16-B aligned, and the whole pool inside one device
 * allocation of the current device.  The library does not own the memory.
 * `instance_id` and `generation` identify the registering process and pool
 * version ([RFC] §Failure and lifecycle handling).
 * Errors: INVALID_ARG, LAYOUT, ALIGNMENT, OUT_OF_RANGE, CUDA, NO_MEMORY. */
KVB_API kv_status kv_pool_register(const kv_layout *layout, void *base, uint64_t offset,
                           uint64_t instance_id, uint64_t generation, kv_pool *out);

/* A layer-first pool held in separate device buffers, one per layer and
 * component -- the per-layer K and V buffers of a serving engine's pool.
 * `bases` holds L x C device pointers (entry l * C + c); each buffer holds the
 * P pages of that layer and component, page p at byte p x T x H x B, heads
 * in the layout's order ([P][T][H][B] for NHD, [P][H][T][B] for HND).  Same
 * bytes as one layer-first pool [L][C][P][T][H][B] cut at every (l, c).
 * layout->order must be KV_LAYER_FIRST.  Each buffer: 16-B aligned, device
 * memory of one device, P x T x H x B bytes inside its allocation.  The
 * library keeps a device copy of the table (freed by kv_pool_close).  Split
 * pools travel over IPC with kv_pool_export_split / kv_pool_import_split.
 * Errors: INVALID_ARG, LAYOUT, ALIGNMENT, OUT_OF_RANGE, CUDA, NO_MEMORY. */
KVB_API kv_status kv_pool_register_split(const kv_layout *layout, void *const *bases,
                                         uint64_t instance_id, uint64_t generation, kv_pool *out);

/* Export ([RFC] DeviceMemoryIPC "export allocation"; [LMC] §共享与重建的完整链路
 * sender steps 3-5): finds the allocation base of the pool start, takes the
 * IPC handle of that base and records the pool's byte offset from it.  Fails
 * (CUDA) for memory CUDA IPC cannot share; there is no alternate path
 * ([LMC] §为什么不做_share_cuda_回退).  Errors: INVALID_ARG, CLOSED, CUDA. */
KVB_API kv_status kv_pool_export(kv_pool pool, kv_ipc_desc *out);

/* Import ([RFC] DeviceMemoryIPC "import allocation"; [LMC] §共享与重建的完整链路
 * receiver steps 1-3): device UUID -> ordinal; one mapping per (process,
 * allocation), refcounted by handle bytes; cudaIpcOpenMemHandle with lazy
 * peer access when the allocation is not yet mapped; pool = mapped base +
 * alloc_offset.  Must run in a process other than the exporter.  A
 * descriptor whose generation is below the retired floor of its instance is
 * refused with STALE; one whose extent (alloc_offset + nbytes) overruns the
 * mapped allocation, with OUT_OF_RANGE (a mapping opened for it is closed
 * again).  Errors: INVALID_ARG, LAYOUT, ALIGNMENT, OUT_OF_RANGE, STALE, CUDA,
 * NO_MEMORY. */
KVB_API kv_status kv_pool_import(const kv_ipc_desc *desc, kv_pool *out);

/* Export of a split pool ([RFC] §Device IPC data path: REGISTER_KV_POOL
 * carries the memory IPC handles of the scheduler's KV allocations, and the
 * daemon imports those allocations once).  Writes the pool's descriptor to
 * `out` (magic KVB_IPC_MAGIC_SPLIT; handle and alloc_offset of buffer 0;
 * nbytes of all buffers; identity, device and layout as kv_pool_export) and
 * to `bufs` (nbufs = L x C entries, entry l * C + c) the allocation handle and
 * offset of every buffer; buffers that share an allocation carry the same
 * handle.  Errors: INVALID_ARG (NULL, nbufs != L x C), CLOSED, LAYOUT (not a
 * split pool: kv_pool_export), CUDA. */
KVB_API kv_status kv_pool_export_split(kv_pool pool, kv_ipc_desc *out, kv_ipc_buffer *bufs,
                                       uint32_t nbufs);

/* Import of a split pool: maps every distinct allocation once per process (the
 * registry kv_pool_import uses; the pool holds one reference per distinct
 * allocation, dropped by kv_pool_close), checks each buffer's extent
 * (alloc_offset + P x T x H x B) against its allocation, and builds the
 * device table of buffer addresses.  Same identity checks as kv_pool_import
 * (device UUID, retired generations: STALE); must run in a process other than
 * the exporter.  On any error every mapping this call opened is closed again.
 * Errors: INVALID_ARG, LAYOUT, ALIGNMENT, OUT_OF_RANGE, STALE, CUDA, NO_MEMORY. */
KVB_API kv_status kv_pool_import_split(const kv_ipc_desc *desc, const kv_ipc_buffer *bufs,
                                       uint32_t nbufs, kv_pool *out);

/* Close ([RFC] DeviceMemoryIPC "close mapping"; [LMC] §重建生命周期与引用计数):
 * releases the handle; for an imported pool, drops one reference of its
 * mapping and unmaps on the last one.  Teardown always completes: an unmap
 * failure is reported (CUDA) after the handle is gone.  Closing twice gives
 * CLOSED.  Operations still in flight on the pool must have completed. */
KVB_API kv_status kv_pool_close(kv_pool pool);

/* Retire every generation below `min_generation` of `instance_id` ([RFC]
 * §Failure and lifecycle handling: a restarted scheduler's older generation
 * must not be used).  Later backup / restore on such pools, and imports of
 * such descriptors, fail with STALE.  Floors only rise. */
KVB_API kv_status kv_pool_retire(uint64_t instance_id, uint64_t min_generation);

/* Device address of the pool's first byte (base + offset, or mapped base +
 * alloc_offset; a split pool's first buffer) and its byte size (all buffers
 * of a split pool).  Either output may be NULL. */
KVB_API kv_status kv_pool_info(kv_pool pool, kv_layout *layout, void **dev_ptr, uint64_t *nbytes);

/* ------------------------------------------------------------- host tier */

/* Registers the pinned host KV tier ([RFC] §Ownership: host KV physical
 * allocation).  `host` must be page-locked host memory mapped into the
 * device address space (cudaHostAlloc / torch pin_memory), 16-B aligned,
 * holding `num_slots` slots of one page each (bytes >= num_slots x page
 * bytes).  Slot geometry (L, C, T, H, B) comes from `pool_layout`; the
 * tier's head order is `host_heads` (kv_heads).  Not owned by the library.
 * Errors: INVALID_ARG, LAYOUT, ALIGNMENT, OUT_OF_RANGE, CUDA, NO_MEMORY. */
KVB_API kv_status kv_host_register(void *host, uint64_t bytes, uint32_t num_slots, uint32_t host_heads,
                           const kv_layout *pool_layout, kv_host *out);
KVB_API kv_status kv_host_close(kv_host host);

/* ------------------------------------------------------------ operations */

/* BACKUP ([RFC] §Device IPC data path): for every i < n, every layer,
 * component, token and head, host slot host_slots[i] receives the unit of
 * page src_pages[i]; no other byte changes.  Enqueued on `stream` after
 * earlier work on it; returns at once with a fence.  Checks, before
 * enqueueing: handles live and not retired (CLOSED / STALE), pool and tier
 * geometry equal (LAYOUT), ids in range (OUT_OF_RANGE), no slot written
 * twice (DUPLICATE; repeated source pages are fine), arrays non-null when
 * n > 0 (INVALID_ARG).  n = 0 enqueues only the fence.  Errors as listed and
 * CUDA, NO_MEMORY. */
KVB_API kv_status kv_backup(kv_pool pool, kv_host host, const int32_t *src_pages,
                    const int32_t *host_slots, uint32_t n, void *stream, kv_fence *fence);

/* BACKUP with its ready_fence ([RFC] §Device IPC data path: BACKUP(operation_id,
 * source_pages, cache_keys, ready_fence); §Ownership: the scheduler publishes
 * which source pages are safe to back up).  As kv_backup, but on the GPU the
 * copy waits until the 64-bit word `ready_word` holds a value >= ready_value
 * -- a word the scheduler, another process or the host sets when the pages
 * are ready.  `ready_word` must be 8-B aligned device memory or page-locked
 * host memory mapped into the device.  The wait is bounded: after
 * ready_timeout_ns (<= 60 s, GPU global timer) it gives up, the operation moves
 * no byte and its fence completes with KV_ERR_ABORTED (fail closed); nothing
 * traps or hangs.  Always the zero-copy path.  Errors: as kv_backup, plus
 * INVALID_ARG / ALIGNMENT for the ready word or timeout. */
KVB_API kv_status kv_backup_when_ready(kv_pool pool, kv_host host, const int32_t *src_pages,
                                       const int32_t *host_slots, uint32_t n,
                                       const uint64_t *ready_word, uint64_t ready_value,
                                       uint64_t ready_timeout_ns, void *stream, kv_fence *fence);

/* RESTORE gated on its data being in the host tier ([PR] §PP Prefetch Ticket
 * Path: the storage GET lands in host memory before the layer-wise H2D).  As
 * kv_restore, but on the GPU the copy waits until the 64-bit `ready_word`
 * holds a value >= ready_value (set by whoever fills the host slots: a
 * storage client, another process, the host); same rules for the word and the
 * bounded wait as kv_backup_when_ready.  On time-out no pool byte is written
 * and the fence completes with KV_ERR_ABORTED.  Always the zero-copy path. */
KVB_API kv_status kv_restore_when_ready(kv_pool pool, kv_host host, const int32_t *host_slots,
                                        const int32_t *dst_pages, uint32_t n, int32_t layer,
                                        const uint64_t *ready_word, uint64_t ready_value,
                                        uint64_t ready_timeout_ns, void *stream, kv_fence *fence);

/* RESTORE ([RFC] §Device IPC data path; layer-wise per [PR] §PP Prefetch
 * Ticket Path): for every i < n, page dst_pages[i] receives the units of
 * host slot host_slots[i] for every layer (layer = -1) or for that one layer
 * (0 <= layer < L); no other byte changes.  Checks as kv_backup, with
 * DUPLICATE for a destination page written twice and OUT_OF_RANGE for a
 * layer outside [-1, L). */
KVB_API kv_status kv_restore(kv_pool pool, kv_host host, const int32_t *host_slots,
                     const int32_t *dst_pages, uint32_t n, int32_t layer, void *stream,
                     kv_fence *fence);

/* Layer-wise restore of many layers in one call, with progressive per-layer
 * fences ([PR] §PP Prefetch Ticket Path: "Layer-wise H2D + forward" and the
 * progressive publication of the globally safe prefix).  Same bytes as
 * num_layers calls kv_restore(..., first_layer + j, ...), j = 0..num_layers-1,
 * but one kernel streams every layer back to back through the host link.
 * fences[j] (num_layers outputs) completes once layers first_layer ..
 * first_layer + j are all in place, so layer j's fence implies every earlier
 * one; a compute stream waits for one layer with kv_fence_stream_wait, which
 * waits on the GPU for that fence word while later layers are still moving.
 * Limits: 1 <= num_layers <= 2048, first_layer + num_layers <= L, and
 * n x num_layers x components x (page-layer chunk / 4 KiB) below 2^31.  Up to
 * 2048 pages the ids travel in the launch; above, the call copies them into a
 * library device buffer (through a library pinned buffer, on `stream`) and
 * still runs one kernel; the next such call waits for that kernel on the GPU
 * before reusing the buffer.
 * Errors: as kv_restore. */
KVB_API kv_status kv_restore_layers(kv_pool pool, kv_host host, const int32_t *host_slots,
                                    const int32_t *dst_pages, uint32_t n, uint32_t first_layer,
                                    uint32_t num_layers, void *stream, kv_fence *fences);

/* Device-side gather / scatter in host-tier layout (the first half of a
 * STAGED transfer, exposed on its own for callers that move the result with
 * their own engine: a NIC, storage, another process).  `buf` is DEVICE
 * memory of the pool's device holding n items in the host tier's form with
 * head order `buf_heads`: item i at byte i x (nl x C x T x H x B), where
 * nl = L for a gather or a whole-page scatter and nl = 1 for a one-layer
 * scatter.  kv_device_gather: item i <- page src_pages[i] (every layer).
 * kv_device_scatter: page dst_pages[i] <- item i (every layer, or only
 * `layer`).  Checks as kv_backup / kv_restore; buf must be 16-B aligned and
 * buf_bytes >= n x item bytes (OUT_OF_RANGE); DUPLICATE for a page written
 * twice by a scatter.  HBM-bound: one read and one write of every byte.
 * `fence` may be NULL: the op is then ordered only by `stream` (no fence is
 * reserved and the kernel skips its fused completion, ~2% faster); with a
 * fence it completes like a backup's. */
KVB_API kv_status kv_device_gather(kv_pool pool, void *buf, uint64_t buf_bytes, uint32_t buf_heads,
                                   const int32_t *src_pages, uint32_t n, void *stream,
                                   kv_fence *fence);
KVB_API kv_status kv_device_scatter(kv_pool pool, const void *buf, uint64_t buf_bytes,
                                    uint32_t buf_heads, const int32_t *dst_pages, uint32_t n,
                                    int32_t layer, void *stream, kv_fence *fence);

/* Staged backup that allocates nothing.  No counterpart on the pages: this
 * entry point exists for callers that cannot allocate GPU memory when they
 * back pages up (an engine whose allocator owns all of HBM, an out-of-memory
 * or teardown path, a runtime that forbids allocation calls while it records
 * work).  Same result as kv_backup: host slot host_slots[i] receives page
 * src_pages[i].  It stages through one static device array of
 * KVB_NOALLOC_STAGING_BYTES that is part of the library (every GPU that loads
 * the library's device code holds it until the process exits), so the call
 * makes no cudaMalloc, cudaFree, pinned or event allocation and returns no
 * fence: the work is ordered on `stream`, and the caller waits on that stream
 * (or an event of its own) before reading the host slots.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array.  Nothing in it needs to
 *     start at zero (each call writes every byte it later reads), but calls
 *     whose work overlaps on the GPU (different streams, not ordered) race on
 *     it and corrupt each other's output: order them on one stream.
 *   - Limits: n <= 2048 and n x page bytes <= KVB_NOALLOC_STAGING_BYTES, else
 *     OUT_OF_RANGE with a message naming the limit.  Other checks and codes
 *     as kv_backup. */
#define KVB_NOALLOC_STAGING_BYTES (32ull << 20)
KVB_API kv_status kv_backup_staged_noalloc(kv_pool pool, kv_host host, const int32_t *src_pages,
                                           const int32_t *host_slots, uint32_t n, void *stream);

/* Host-side validation of an operation without a GPU (kind 0 = backup with
 * a = src pages, b = slots; kind 1 = restore with a = slots, b = dst pages).
 * Same checks and codes as kv_backup / kv_restore minus handle state. */
KVB_API kv_status kv_op_validate(const kv_layout *layout, uint32_t num_slots, int kind,
                         const int32_t *a, const int32_t *b, uint32_t n, int32_t layer);

/* ------------------------------------------------- descriptor ring (IPC) */

/* A shared-memory submission / completion ring between a submitting process
 * (the scheduler) and a serving process (the data plane) on one node ([RFC]
 * §Device IPC data path: operations carry page IDs and fences, not tensors;
 * control and completion through shared-memory submission/completion rings,
 * NVMe-style).  One submitter and one server per ring.  Tickets are 1, 2, 3...
 * in submission order.  The server registers the ring's completion records
 * with CUDA, so the GPU itself stores a ticket into shared memory when that
 * operation's bytes are in place; the submitter polls it with no help from
 * the server's CPU (cross-process completion, [RFC] DeviceSyncIPC).  A server
 * that dies leaves the submitter's waits to time out (fail closed). */
typedef struct kv_ring_s *kv_ring;

#define KV_RING_MAX_IDS 1024
#define KV_RING_OP_BACKUP 0u
#define KV_RING_OP_RESTORE 1u

#define KV_RING_READY_WORDS 64

/* One BACKUP / RESTORE descriptor ([RFC] §Device IPC data path).  POD.
 * Ready fence ([RFC] BACKUP(..., ready_fence)): with ready_value != 0 the
 * operation starts only once the ring's ready word ready_index (one of
 * KV_RING_READY_WORDS 64-bit words in the shared segment, set with
 * kv_ring_ready_set or kv_ring_ready_stream_set) holds a value >= ready_value.
 * The server waits for it on the GPU, at most ready_timeout_ms (1..60000;
 * 0 = 10000); on time-out the operation moves no byte and its ticket completes
 * with ABORTED (fail closed).  ready_value = 0: no gate. */
typedef struct {
    uint32_t kind;           /* KV_RING_OP_BACKUP or KV_RING_OP_RESTORE              */
    uint32_t pool_index;     /* index into the server's pool table                 */
    uint32_t n;              /* ids in a[] and b[] (<= KV_RING_MAX_IDS)            */
    int32_t layer;           /* restore: -1 = all layers, else one; backup: -1     */
    uint64_t operation_id;   /* the submitter's operation_id, returned by pop      */
    uint32_t ready_index;    /* ready word gating the operation (< KV_RING_READY_WORDS) */
    uint32_t ready_timeout_ms;    /* bound on the wait for it; 0 = 10 s            */
    uint64_t ready_value;    /* start once the word >= this; 0 = not gated        */
    int32_t a[KV_RING_MAX_IDS];   /* backup: source pages; restore: host slots     */
    int32_t b[KV_RING_MAX_IDS];   /* backup: host slots; restore: destination pages */
} kv_ring_op;

/* Creates POSIX shared memory `name` ("/name", no other '/') holding a ring of
 * `slots` (2..4096) descriptors and completion records, and attaches to it.
 * The creator unlinks the name when it closes.  Errors: INVALID_ARG (name,
 * slots, name exists), NO_MEMORY. */
KVB_API kv_status kv_ring_create(const char *name, uint32_t slots, kv_ring *out);
/* Attaches to an existing ring.  Errors: INVALID_ARG (no such ring, wrong
 * magic or version, or a header whose regions do not fit the segment). */
KVB_API kv_status kv_ring_attach(const char *name, kv_ring *out);
/* Detaches (and unlinks, for the creator).  Any process that registered the
 * segment with CUDA -- a server, or a submitter that called
 * kv_ring_ready_stream_set -- unregisters it here, so every store into the
 * segment that this process queued on a stream (ready words set from a
 * stream, the host server's completion marks) must run first: close waits up
 * to 2 s for them, and if one has not run it returns TIMEOUT and the ring
 * stays open (the handle stays valid: close it again once that stream's work
 * has finished).  A resident server still running on this handle is asked to
 * stop and waited for (bounded); if it has not ended, TIMEOUT, the handle is
 * closed and the memory stays mapped.  Errors: CLOSED, TIMEOUT. */
KVB_API kv_status kv_ring_close(kv_ring ring);

/* Submitter: copies `op` into the next slot and publishes it; waits up to
 * timeout_ns for a free slot (TIMEOUT: ring full -- the server is behind or
 * gone).  Returns the ticket.  Errors: INVALID_ARG (kind, n, ready_index or
 * ready_timeout_ms of a gated op), TIMEOUT. */
KVB_API kv_status kv_ring_submit(kv_ring ring, const kv_ring_op *op, uint64_t timeout_ns,
                                 uint64_t *ticket);
/* Submitter: waits up to timeout_ns for `ticket` to complete and returns the
 * operation's own status in *op_status (OK, or the error the server met, e.g.
 * OUT_OF_RANGE).  TIMEOUT if not complete in time, INVALID_ARG for a ticket
 * never submitted. */
KVB_API kv_status kv_ring_wait(kv_ring ring, uint64_t ticket, uint64_t timeout_ns,
                               kv_status *op_status);

/* Sets ready word `index` (< KV_RING_READY_WORDS) of the ring to `value` from
 * the CPU (a release store into the shared segment); either process may call
 * it.  Words start at 0 and are the caller's to sequence: a gate opens once
 * its word is >= its ready_value.  Errors: CLOSED, INVALID_ARG (index). */
KVB_API kv_status kv_ring_ready_set(kv_ring ring, uint32_t index, uint64_t value);
/* Sets ready word `index` to `value` from the GPU, once the work enqueued
 * before it on `stream` has finished (a stream memory write): a scheduler's
 * forward stream releases the data plane's gated backup with no CPU wait in
 * either process.  The first call registers the shared segment with CUDA in
 * this process.  Launch once, beforehand, any kernel of this process that
 * precedes the word on `stream`: under lazy module loading a kernel's first
 * launch waits for the device to go idle, and a gate (or a resident server)
 * waiting in the same process keeps it busy until its bound.  Errors: CLOSED,
 * INVALID_ARG (index), CUDA. */
KVB_API kv_status kv_ring_ready_stream_set(kv_ring ring, uint32_t index, uint64_t value,
                                           void *stream);

/* Server: takes up to max_ops descriptors, waiting up to idle_timeout_ns for
 * the first, and enqueues each on `stream` as kv_backup / kv_restore on
 * pools[op.pool_index] and `host` (a gated one as kv_backup_when_ready /
 * kv_restore_when_ready on its ready word); the GPU completes each ticket in
 * shared memory after its bytes (ABORTED for a gate that timed out).  A
 * descriptor the engine rejects is completed at once with that error.
 * *served = descriptors taken.  Errors: INVALID_ARG, CUDA (registering the
 * completion page). */
KVB_API kv_status kv_ring_serve(kv_ring ring, const kv_pool *pools, uint32_t npools, kv_host host,
                                void *stream, uint32_t max_ops, uint64_t idle_timeout_ns,
                                uint32_t *served);
/* Server without a GPU (tests, or a server that moves bytes some other way):
 * takes the next descriptor (waiting up to timeout_ns; TIMEOUT if none) ...
 * A descriptor that kv_ring_submit would refuse (unknown kind, n above
 * KV_RING_MAX_IDS, or a bad gate: ready_index >= KV_RING_READY_WORDS or
 * ready_timeout_ms above 60000 on a gated op -- written into the shared
 * segment some other way) is taken, completed with INVALID_ARG and reported as
 * INVALID_ARG with *ticket set and op->n = 0; kv_ring_serve counts it as
 * served and moves on. */
KVB_API kv_status kv_ring_pop(kv_ring ring, uint64_t timeout_ns, kv_ring_op *op,
                              uint64_t *ticket);
/* ... and completes a ticket from the CPU with the given status. */
KVB_API kv_status kv_ring_complete(kv_ring ring, uint64_t ticket, kv_status op_status);

/* Server on the GPU ([RFC] §Device IPC data path: a high-frequency path as an
 * NVMe-style submission / completion queue).  Enqueues on `stream` one
 * resident kernel (a cooperative grid of CTAs of 256 threads -- a leader and
 * 32 movers, or kv_config.max_ctas movers when that is set -- holding that
 * many SMs for as long as it runs) that takes
 * descriptors from the ring itself -- polling the tail in the shared segment,
 * which is mapped into the GPU -- checks each exactly as kv_ring_serve would
 * (the same status for every rejected descriptor: INVALID_ARG for a kind, n,
 * pool index or backup layer it refuses, then OUT_OF_RANGE / DUPLICATE for
 * layers and ids in the host engine's order), moves the accepted ones
 * zero-copy in ticket order -- a gated one once its ready word allows, or
 * completed with ABORTED after its ready_timeout_ms -- and completes every
 * ticket from the GPU.  No host thread and no launch per descriptor.  The
 * server ends after max_ops
 * descriptors, or once idle_timeout_ns (<= 60 s) pass without a new one;
 * every other wait inside it is bounded too.  Returns at once; *fence
 * completes when the kernel has ended (then kv_ring_device_result).  The
 * table (<= 64 pools, one device) and host tier are checked when it starts:
 * live handles, no retired generation, the host tier's slot geometry; a
 * generation retired while it runs is not seen.  One server per ring at a
 * time (host or device); INVALID_ARG while this ring's previous resident
 * server is still running.  The pool table and host tier must stay open, and
 * the caller's stream is busy, until the fence completes.  While it runs, a
 * CUDA call that synchronizes the device (cudaDeviceSynchronize, cudaFree,
 * pinned allocations, ...) waits for the server to end.  Errors: CLOSED,
 * INVALID_ARG, STALE, LAYOUT, CUDA. */
KVB_API kv_status kv_ring_serve_device(kv_ring ring, const kv_pool *pools, uint32_t npools,
                                       kv_host host, void *stream, uint32_t max_ops,
                                       uint64_t idle_timeout_ns, kv_fence *fence);
/* After the resident server's fence: descriptors it took (*served) and its
 * own status (OK, or TIMEOUT if one of its bounded internal waits ran out).
 * Errors: CLOSED, INVALID_ARG (no server started), TIMEOUT (still running). */
KVB_API kv_status kv_ring_device_result(kv_ring ring, uint32_t *served, kv_status *status);
/* Asks the ring's resident server to end before it takes another descriptor
 * (the one it is moving completes); returns at once, and the server's fence
 * completes when it has ended.  kv_ring_close does this itself and never
 * unmaps the segment under a running server.  Errors: CLOSED, INVALID_ARG
 * (no server started). */
KVB_API kv_status kv_ring_device_stop(kv_ring ring);

/* ------------------------------------------------ L3 record store (files) */

/* The tier below the host tier ([RFC] §Summary: the daemon's host tier with
 * external L3 storage below it; §Relationship to existing SGLang work: the
 * standalone L3 StorageServer keeps its bulk bytes in shared memfd host
 * memory).  A store is `num_records` fixed-size records of a file descriptor:
 * record r is bytes [base_offset + r * record_bytes, + record_bytes).  Puts and
 * gets move whole host-tier pages: slot s of a host tier is bytes
 * [s * record_bytes, + record_bytes) of `host` (the page-contiguous host tier
 * registered with kv_host_register, whose page bytes equal record_bytes, or
 * any host buffer of that shape).  The bytes are never interpreted. */
typedef struct kv_l3_s *kv_l3;

/* Opens a store over `fd` (a regular file, a memfd or a block device; the
 * caller keeps ownership and closes it after kv_l3_close).  `threads` worker
 * threads move the bytes (0 = 8, at most 64).  The file is not resized: a put
 * past its end grows it, a get past its end fails with KV_ERR_IO.  If the
 * caller opened fd with O_DIRECT, buffers, offsets and record_bytes must meet
 * its alignment or calls fail with KV_ERR_IO.  A regular file or memfd opened
 * read-write without O_DIRECT is mapped once and calls copy through the
 * mapping; other descriptors take one pwritev / preadv per run of records.
 * While the store is open nobody else may shrink the file below a record in
 * use: a mapped store touching a page past the end would take SIGBUS.
 * Errors: INVALID_ARG (fd not open / not a file or block device, zero sizes,
 * threads > 64), OUT_OF_RANGE (num_records > 2^31 or offsets overflow),
 * NO_MEMORY. */
KVB_API kv_status kv_l3_open(int fd, uint64_t base_offset, uint64_t record_bytes,
                             uint64_t num_records, uint32_t threads, kv_l3 *out);
/* Stops the workers (a call in flight on another thread finishes first). */
KVB_API kv_status kv_l3_close(kv_l3 store);

/* PUT: record records[i] <- host slot slots[i], for i < n.  Synchronous:
 * returns once every byte is written to the descriptor (no fsync).  Runs of
 * consecutive records go out as one copy (or one pwritev) each, spread over
 * the workers.
 * Checks before any write: ids in range (slots < host_slots, records <
 * num_records), no record named twice.  The host slots must not be written
 * meanwhile (wait for the backup's fence first).
 * Errors: CLOSED, INVALID_ARG, OUT_OF_RANGE, DUPLICATE (nothing written);
 * IO (a write failed: the named records are then undefined). */
KVB_API kv_status kv_l3_put(kv_l3 store, const void *host, uint64_t host_slots,
                            const int32_t *slots, const int32_t *records, uint32_t n);
/* GET: host slot slots[i] <- record records[i], for i < n.  Synchronous; runs
 * of consecutive records come in as one copy (or one preadv) each.  Checks as for PUT, with
 * no slot named twice.  Restore from the slots only after this returns (or
 * gate the restore with kv_restore_when_ready on a word set afterwards).
 * Errors: CLOSED, INVALID_ARG, OUT_OF_RANGE, DUPLICATE (nothing read);
 * IO (a read failed or a record lies past the end of the file: the named
 * slots are then undefined). */
KVB_API kv_status kv_l3_get(kv_l3 store, void *host, uint64_t host_slots,
                            const int32_t *records, const int32_t *slots, uint32_t n);

/* --------------------------------------------------------------- fences */

/* DeviceSyncIPC wait/query ([RFC] §Device IPC data path).  A fence completes
 * when every byte of its operation is in place.  Completion is a sequence
 * number the GPU stores into a mapped pinned word after the operation, so
 * the host learns of it without a CUDA call.  The word is stored with a
 * system-scope release that orders every byte of the operation: a host
 * thread that sees the fence complete may read a backup's host slots at once,
 * and work on a stream that waited with kv_fence_stream_wait sees a restore's
 * pages.
 * kv_fence_query: OK when complete, TIMEOUT when not yet, ABORTED when the
 * operation completed by giving up (kv_backup_when_ready whose ready fence
 * never arrived), INVALID_ARG for a fence never issued.  kv_fence_wait: polls
 * until complete or until timeout_ns has passed (TIMEOUT): spinning for the
 * first 50 us, then yielding the core between polls up to 20 ms (the calling
 * thread stays runnable, so it sees the fence within microseconds), then
 * sleeping between polls.  kv_fence_stream_wait: makes `stream` wait
 * for the fence on the GPU (the compute stream of a layer-wise restore): the
 * stream waits for the fence's word itself (a 64-bit stream wait-value) where
 * the driver supports it, else for the fence's event. */
KVB_API kv_status kv_fence_query(kv_fence fence);
KVB_API kv_status kv_fence_wait(kv_fence fence, uint64_t timeout_ns);
KVB_API kv_status kv_fence_stream_wait(kv_fence fence, void *stream);

/* ------------------------------------------------------------ utilities */

KVB_API kv_status kv_config_get(kv_config *out);
/* Process-wide; applies to operations issued afterwards.  Errors: INVALID_ARG. */
KVB_API kv_status kv_config_set(const kv_config *cfg);
/* Bytes of one page (= one host slot) of a valid layout. */
KVB_API kv_status kv_layout_page_bytes(const kv_layout *layout, uint64_t *out);
/* Number of kernels this library has launched in this process. */
KVB_API uint64_t kv_launch_count(void);
/* Number of ops this process issued overlapped with the previous one on their
 * stream (KV_CFG_OVERLAP_RESTORES / KV_CFG_OVERLAP_BACKUPS): a way to check
 * that the flags apply to a caller's pattern of calls. */
KVB_API uint64_t kv_overlap_count(void);
/* Message of the last failing call on this thread ("" if none). */
KVB_API const char *kv_last_error(void);
KVB_API uint32_t kv_abi_version(void);

/* Host-side failure drills ([PR] §Targeted fault-injection validation: an
 * injected allocation failure must fall back and leave the service running).
 * The next `count` passes through `point` fail as if the CUDA call there had
 * failed -- "staging_alloc" (NO_MEMORY), "fence_reserve" (NO_MEMORY),
 * "launch" (CUDA, at an op's first kernel launch), "ipc_open" (CUDA),
 * "host_register" (CUDA), "launch_nth" (CUDA: only the count-th move-kernel
 * launch from now fails, possibly in the middle of an op -- what the op had
 * enqueued before it still runs, and later ops wait for it); count 0 disarms.
 * One drill reaches a kernel without faulting it: "chain_stall" makes the next
 * overlapped restore (KV_CFG_OVERLAP_RESTORES) chain its fence on a sequence
 * number that never arrives, so its bounded GPU wait runs out after 2 s, its
 * bytes still land, and from then on every fence query of this process on
 * that device reports TIMEOUT (the kernel error word is sticky: drill it in a
 * process of its own).  The environment variable
 * KVB_FAULT="point:count[,point:count]" arms points at first use.  Errors:
 * INVALID_ARG for an unknown point. */
KVB_API kv_status kv_fault_inject(const char *point, uint32_t count);

#ifdef __cplusplus
}
#endif
#endif /* KVB_H */
