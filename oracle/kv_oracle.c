/*
 * kv_oracle.c -- plain CPU oracle for paged KV-cache backup / restore.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference leg use it.  It shares no source, header, table or
 * helper with the CUDA library and is deliberately slow and obvious.
 *
 * Sources (web pages this restates; cited by title and section):
 *   [RFC]   "[Feature] [RFC] [HiCache] Out-of-process HiCache data plane with
 *           device-memory IPC" -- §Device IPC data path: BACKUP(operation_id,
 *           source_pages, cache_keys, ready_fence) copies the named GPU pages
 *           to the host tier; RESTORE(operation_id, cache_keys,
 *           destination_pages, completion_fence) copies host-tier data back
 *           into destination pages chosen by the scheduler.
 *   [PR]    "[PP + HiCache] Add PP Prefetch Tickets for eager cross-stage
 *           storage prefetch" -- §PP Prefetch Ticket Path (sequence diagram):
 *           "Layer-wise H2D + forward", i.e. a restore may be limited to one
 *           layer at a time.
 *   [LMC]   "LMCache RawCudaIPCWrapper深度解析" -- §uint8字节往返: the transfer
 *           only sees bytes, dtype is irrelevant; §在项目中的实际接入方式: the
 *           TRT-LLM pool [NB, NL, 2, NH*BS*HS] with kv_layout="HND" is viewed
 *           as the 6-D array [NB, NL, 2, NH, BS, HS].
 *
 * What is computed (the plain definition; no blocking, fusion or reordering):
 *   A "unit" is the B-byte head vector at coordinate (page p, layer l,
 *   component c, token t, head h).  With Doff the device-pool byte offset and
 *   Hoff the host-tier byte offset of a unit,
 *     backup : for all i,l,c,t,h   host[Hoff(slot[i],l,c,t,h) .. +B)
 *                                    = pool[Doff(src[i],l,c,t,h) .. +B)
 *     restore: for all i, l in (layer < 0 ? every layer : {layer}), c,t,h
 *              pool[Doff(dst[i],l,c,t,h) .. +B) = host[Hoff(slot[i],l,c,t,h) .. +B)
 *   Every byte not named above is left unchanged.  Bytes are copied as bytes
 *   (no float type ever touches the payload), per [LMC] §uint8字节往返.
 *
 * Readings taken where the pages are silent (all row-major):
 *   layer-first NHD : pool viewed as [L][C][P][T][H][B]
 *   layer-first HND : pool viewed as [L][C][P][H][T][B]
 *   page-first  NHD : pool viewed as [P][L][C][T][H][B]
 *   page-first  HND : pool viewed as [P][L][C][H][T][B]
 *                     (= the TRT-LLM 6-D view [NB, NL, 2, NH, BS, HS] of [LMC])
 *   host tier       : slot-major and page-contiguous, [S][L][C][T][H][B]
 *                     (NHD) or [S][L][C][H][T][B] (HND).
 *
 * Parity pins: every function here is pinned by tests (coordinate tags
 * against numpy row-major views, the TRT-LLM 4-D/6-D reshape statement,
 * round-trip and untouched-bytes invariants, brute force over tiny pools, and
 * planted-mistake checks); none is "parity unpinned".
 */
#include <stdint.h>
#include <string.h>
#include <pthread.h>

typedef struct {
    int64_t L;          /* layers                                         */
    int64_t C;          /* KV components: 2 = K and V, 1 = MLA latent      */
    int64_t P;          /* pages in the device pool                        */
    int64_t T;          /* tokens per page                                 */
    int64_t H;          /* KV heads                                        */
    int64_t B;          /* bytes per head vector (head_dim x element size) */
    int32_t page_first; /* 0 = layer-first pool, 1 = page-first pool       */
    int32_t dev_hnd;    /* device pool: 0 = NHD, 1 = HND                   */
    int32_t host_hnd;   /* host tier:   0 = NHD, 1 = HND                   */
    int32_t pad_;
} kvo_geom;

/* Byte offset of unit (p,l,c,t,h) inside the device pool. */
int64_t kvo_dev_offset(const kvo_geom *g, int64_t p, int64_t l, int64_t c,
                       int64_t t, int64_t h)
{
    /* the (page, layer, component) prefix of the index, per pool order */
    int64_t outer;
    if (g->page_first)
        outer = (p * g->L + l) * g->C + c;   /* [P][L][C] */
    else
        outer = (l * g->C + c) * g->P + p;   /* [L][C][P] */
    /* the (token, head) suffix, per head order */
    int64_t inner;
    if (g->dev_hnd)
        inner = h * g->T + t;                /* [H][T] */
    else
        inner = t * g->H + h;                /* [T][H] */
    return (outer * (g->T * g->H) + inner) * g->B;
}

/* Byte offset of unit (slot s, l, c, t, h) inside the host tier. */
int64_t kvo_host_offset(const kvo_geom *g, int64_t s, int64_t l, int64_t c,
                        int64_t t, int64_t h)
{
    int64_t outer = (s * g->L + l) * g->C + c;   /* [S][L][C] */
    int64_t inner;
    if (g->host_hnd)
        inner = h * g->T + t;
    else
        inner = t * g->H + h;
    return (outer * (g->T * g->H) + inner) * g->B;
}

/* Bytes of one page (= one host slot): L*C*T*H*B. */
int64_t kvo_page_bytes(const kvo_geom *g)
{
    return g->L * g->C * g->T * g->H * g->B;
}

/* backup of items [i0, i1): host[slot[i]] <- pool[src[i]], all layers. */
static void backup_range(const kvo_geom *g, const uint8_t *pool, uint8_t *host,
                         const int32_t *src, const int32_t *slot,
                         int64_t i0, int64_t i1)
{
    for (int64_t i = i0; i < i1; ++i)
        for (int64_t l = 0; l < g->L; ++l)
            for (int64_t c = 0; c < g->C; ++c)
                for (int64_t t = 0; t < g->T; ++t)
                    for (int64_t h = 0; h < g->H; ++h)
                        memcpy(host + kvo_host_offset(g, slot[i], l, c, t, h),
                               pool + kvo_dev_offset(g, src[i], l, c, t, h),
                               (size_t)g->B);
}

/* restore of items [i0, i1): pool[dst[i]] <- host[slot[i]] for the chosen layers. */
static void restore_range(const kvo_geom *g, uint8_t *pool, const uint8_t *host,
                          const int32_t *slot, const int32_t *dst, int32_t layer,
                          int64_t i0, int64_t i1)
{
    int64_t l_lo = layer < 0 ? 0 : layer;
    int64_t l_hi = layer < 0 ? g->L : (int64_t)layer + 1;
    for (int64_t i = i0; i < i1; ++i)
        for (int64_t l = l_lo; l < l_hi; ++l)
            for (int64_t c = 0; c < g->C; ++c)
                for (int64_t t = 0; t < g->T; ++t)
                    for (int64_t h = 0; h < g->H; ++h)
                        memcpy(pool + kvo_dev_offset(g, dst[i], l, c, t, h),
                               host + kvo_host_offset(g, slot[i], l, c, t, h),
                               (size_t)g->B);
}

/*
 * BACKUP ([RFC] §Device IPC data path).  The pool starts `pool_offset` bytes
 * after `pool_base` (the allocation-base + byte-offset addressing of [LMC]
 * §共享与重建的完整链路).  Caller guarantees ids are in range.
 */
void kvo_backup(const kvo_geom *g, const uint8_t *pool_base, int64_t pool_offset,
                uint8_t *host, const int32_t *src, const int32_t *slot, int64_t n)
{
    backup_range(g, pool_base + pool_offset, host, src, slot, 0, n);
}

/*
 * RESTORE ([RFC] §Device IPC data path); `layer` < 0 restores every layer,
 * otherwise only that layer ([PR] §PP Prefetch Ticket Path, layer-wise H2D).
 */
void kvo_restore(const kvo_geom *g, uint8_t *pool_base, int64_t pool_offset,
                 const uint8_t *host, const int32_t *slot, const int32_t *dst,
                 int64_t n, int32_t layer)
{
    restore_range(g, pool_base + pool_offset, host, slot, dst, layer, 0, n);
}

/* ---- the same definitions, items split evenly over host threads ---- */

typedef struct {
    const kvo_geom *g;
    uint8_t *pool;
    uint8_t *host;
    const int32_t *a;
    const int32_t *b;
    int32_t layer;
    int32_t is_backup;
    int64_t i0, i1;
} kvo_job;

static void *run_job(void *arg)
{
    kvo_job *j = (kvo_job *)arg;
    if (j->is_backup)
        backup_range(j->g, j->pool, j->host, j->a, j->b, j->i0, j->i1);
    else
        restore_range(j->g, j->pool, j->host, j->a, j->b, j->layer, j->i0, j->i1);
    return 0;
}

static int run_threads(const kvo_geom *g, uint8_t *pool, uint8_t *host,
                       const int32_t *a, const int32_t *b, int64_t n,
                       int32_t layer, int32_t is_backup, int threads)
{
    enum { MAXT = 256 };
    pthread_t tid[MAXT];
    int joined[MAXT];
    kvo_job job[MAXT];
    if (threads < 1) threads = 1;
    if (threads > MAXT) threads = MAXT;
    if (threads > n) threads = n > 0 ? (int)n : 1;
    int started = 0;
    for (int k = 0; k < threads; ++k) {
        job[k].g = g; job[k].pool = pool; job[k].host = host;
        job[k].a = a; job[k].b = b; job[k].layer = layer;
        job[k].is_backup = is_backup;
        job[k].i0 = n * k / threads;
        job[k].i1 = n * (k + 1) / threads;
        joined[k] = pthread_create(&tid[k], 0, run_job, &job[k]) == 0;
        if (joined[k])
            ++started;
        else
            run_job(&job[k]);          /* no thread: do the share inline */
    }
    for (int k = 0; k < threads; ++k)
        if (joined[k]) pthread_join(tid[k], 0);
    return started;
}

/* Multi-threaded BACKUP; writes to distinct slots never overlap.  Returns the
 * number of threads actually started. */
int kvo_backup_mt(const kvo_geom *g, const uint8_t *pool_base, int64_t pool_offset,
                  uint8_t *host, const int32_t *src, const int32_t *slot, int64_t n,
                  int threads)
{
    return run_threads(g, (uint8_t *)(pool_base + pool_offset), host, src, slot,
                       n, -1, 1, threads);
}

/* Multi-threaded RESTORE; writes to distinct destination pages never overlap. */
int kvo_restore_mt(const kvo_geom *g, uint8_t *pool_base, int64_t pool_offset,
                   const uint8_t *host, const int32_t *slot, const int32_t *dst,
                   int64_t n, int32_t layer, int threads)
{
    return run_threads(g, pool_base + pool_offset, (uint8_t *)host, slot, dst,
                       n, layer, 0, threads);
}

/* ------------------------------------------------------ L3 record store
 * The tier below the host tier ("[Feature] [RFC] [HiCache] Out-of-process
 * HiCache data plane with device-memory IPC", §Summary: host tier and L3
 * storage under the daemon; §Relationship to existing SGLang work: the L3
 * StorageServer's bulk bytes live in shared memfd memory).  Reading taken: a
 * store is fixed-size records of a file, record r at byte base + r * rb, one
 * host-tier page per record; host slot s is bytes [s * rb, (s + 1) * rb) of the
 * host tier.  The file is modelled by its byte image.
 *   put: for all i, b < rb:  file[base + records[i] * rb + b] = host[slots[i] * rb + b]
 *   get: for all i, b < rb:  host[slots[i] * rb + b] = file[base + records[i] * rb + b]
 * Every other byte is left unchanged. */
void kvo_l3_put(const uint8_t *host, int64_t rb, const int32_t *slots,
                const int32_t *records, int64_t n, uint8_t *file, int64_t base)
{
    for (int64_t i = 0; i < n; ++i)
        for (int64_t b = 0; b < rb; ++b)
            file[base + (int64_t)records[i] * rb + b] = host[(int64_t)slots[i] * rb + b];
}

void kvo_l3_get(const uint8_t *file, int64_t base, int64_t rb, const int32_t *records,
                const int32_t *slots, int64_t n, uint8_t *host)
{
    for (int64_t i = 0; i < n; ++i)
        for (int64_t b = 0; b < rb; ++b)
            host[(int64_t)slots[i] * rb + b] = file[base + (int64_t)records[i] * rb + b];
}
