// kvb_noalloc.cu -- a staged backup that allocates nothing.
//
// Who this is for: callers that cannot allocate GPU memory at the time they
// back pages up -- code running under an allocator that owns all device memory
// (a serving engine that reserved HBM up front), code in a teardown or
// out-of-memory path where cudaMalloc may fail or stall, or a runtime that
// forbids allocation calls while it records work.  The regular STAGED mode
// cudaMallocs its staging buffer on first use; this entry point instead stages
// through one fixed device array that is part of the library's module.
//
// The array holds KVB_NOALLOC_STAGING_BYTES (32 MiB).  It exists on every GPU
// where this library's device code is loaded, and stays until the process
// exits.  In host code its name is only a host-side stand-in, so its device
// address is looked up once per device with cudaGetSymbolAddress and passed to
// the kernel.
#include "kvb.h"
#include "kvb_internal.h"

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_noalloc_staging[KVB_NOALLOC_STAGING_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_staging_ptr[kMaxDevices] = {};   // device address of the array, per device

}  // namespace

extern "C" KVB_API kv_status kv_backup_staged_noalloc(kv_pool pool, kv_host host,
                                                      const int32_t *src_pages,
                                                      const int32_t *host_slots, uint32_t n,
                                                      void *stream) {
    int device = -1;
    int st = kvb::pool_device_of(pool, &device);
    if (st != KV_OK) return (kv_status)st;
    if (device < 0 || device >= kMaxDevices)
        return (kv_status)kvb::set_last_error(KV_ERR_INVALID_ARG, "pool device out of range");
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != device && cudaSetDevice(device) != cudaSuccess)
        return (kv_status)kvb::set_last_error(KV_ERR_CUDA, "cudaSetDevice(pool device) failed");
    void *staging = nullptr;
    {
        // Set-up, once per device, with that device current: the array's device address.
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_staging_ptr[device] == nullptr) {
            void *ptr = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_staging);
            if (e != cudaSuccess || ptr == nullptr) {
                if (prev >= 0 && prev != device) cudaSetDevice(prev);
                return (kv_status)kvb::set_last_error(
                    KV_ERR_CUDA, "cudaGetSymbolAddress(static staging array) failed");
            }
            g_staging_ptr[device] = ptr;
        }
        staging = g_staging_ptr[device];
    }
    st = kvb::enqueue_staged_backup_noalloc(pool, host, src_pages, host_slots, n, staging,
                                            KVB_NOALLOC_STAGING_BYTES, (cudaStream_t)stream);
    if (prev >= 0 && prev != device) cudaSetDevice(prev);
    return (kv_status)st;
}
