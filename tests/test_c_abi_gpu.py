"""The C ABI end to end from a C program on the GPU: the program allocates
with the CUDA runtime, registers a page-first HND pool at a byte offset and a
mapped pinned NHD host tier, backs pages up, restores one layer into other
pages and then every layer one per call with overlapped restores through
kvb.h, and compares every byte of the host tier and of the pool allocation
with the oracle's C functions (linked into the test program only;
the library never links the oracle)."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from hierarchical_kv_cache_backup_gb300 import build as kbuild  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include "kvb.h"
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

/* the oracle (test infrastructure), compiled into this test program */
typedef struct { int64_t L, C, P, T, H, B; int32_t page_first, dev_hnd, host_hnd, pad_; } kvo_geom;
void kvo_backup(const kvo_geom *g, const uint8_t *pool_base, int64_t pool_offset, uint8_t *host,
                const int32_t *src, const int32_t *slot, int64_t n);
void kvo_restore(const kvo_geom *g, uint8_t *pool_base, int64_t pool_offset,
                 const uint8_t *host, const int32_t *slot, const int32_t *dst, int64_t n,
                 int32_t layer);

#define CK(x) do { if ((x) != cudaSuccess) { printf("cuda fail line %d\n", __LINE__); return 2; } } while (0)
#define KV(x) do { kv_status s_ = (x); if (s_ != KV_OK) { printf("kv %d line %d: %s\n", (int)s_, __LINE__, kv_last_error()); return 3; } } while (0)

static void fill(uint8_t *p, size_t n, uint64_t seed) {
    uint64_t x = seed;
    for (size_t i = 0; i < n; ++i) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        p[i] = (uint8_t)(x >> 56);
    }
}

int main(void) {
    const uint32_t L = 4, C = 2, P = 64, T = 16, H = 4, B = 128, S = 12, n = 8;
    const uint64_t off = 4096 + 48;
    const uint64_t pb = (uint64_t)L * C * T * H * B, pool_bytes = (uint64_t)P * pb;
    kv_layout lay = {L, C, P, T, H, B, KV_PAGE_FIRST, KV_HND, 2, 0};
    kvo_geom g = {L, C, P, T, H, B, 1, 1, 0, 0};
    int32_t src[8] = {3, 17, 42, 5, 63, 0, 8, 33}, slots[8] = {7, 0, 3, 5, 1, 2, 4, 11};
    int32_t dst[8] = {10, 11, 12, 13, 14, 15, 16, 18};
    uint8_t *alloc_d = NULL, *host = NULL;
    uint8_t *img = malloc(off + pool_bytes), *want_host = malloc(S * pb), *got = malloc(off + pool_bytes);
    kv_pool pool;
    kv_host tier;
    kv_fence f;
    if (!img || !want_host || !got) return 4;
    CK(cudaMalloc((void **)&alloc_d, off + pool_bytes));
    CK(cudaHostAlloc((void **)&host, S * pb, cudaHostAllocMapped | cudaHostAllocPortable));
    fill(img, off + pool_bytes, 11);
    fill(host, S * pb, 12);
    memcpy(want_host, host, S * pb);
    CK(cudaMemcpy(alloc_d, img, off + pool_bytes, cudaMemcpyHostToDevice));
    KV(kv_pool_register(&lay, alloc_d, off, 1, 1, &pool));
    KV(kv_host_register(host, S * pb, S, KV_NHD, &lay, &tier));

    KV(kv_backup(pool, tier, src, slots, n, NULL, &f));
    KV(kv_fence_wait(f, 20000000000ull));
    kvo_backup(&g, img, (int64_t)off, want_host, src, slots, n);
    if (memcmp(host, want_host, S * pb) != 0) { printf("host tier differs\n"); return 5; }

    KV(kv_restore(pool, tier, slots, dst, n, 2, NULL, &f));     /* layer 2 only */
    KV(kv_fence_wait(f, 20000000000ull));
    kvo_restore(&g, img, (int64_t)off, want_host, slots, dst, n, 2);
    CK(cudaMemcpy(got, alloc_d, off + pool_bytes, cudaMemcpyDeviceToHost));
    if (memcmp(got, img, off + pool_bytes) != 0) { printf("pool differs\n"); return 6; }

    /* every layer restored one per call on a created stream, overlapped */
    {
        kv_config cfg;
        cudaStream_t st;
        int32_t dst2[8] = {20, 21, 22, 23, 24, 25, 26, 27};
        kv_fence fl[4];
        uint64_t c0 = kv_overlap_count();
        KV(kv_config_get(&cfg));
        cfg.flags |= KV_CFG_OVERLAP_RESTORES;
        KV(kv_config_set(&cfg));
        CK(cudaStreamCreate(&st));
        for (uint32_t l = 0; l < L; ++l) KV(kv_restore(pool, tier, slots, dst2, n, (int32_t)l, st, &fl[l]));
        if (kv_overlap_count() - c0 != L - 1) { printf("overlap count %llu\n", (unsigned long long)(kv_overlap_count() - c0)); return 7; }
        KV(kv_fence_wait(fl[L - 1], 20000000000ull));
        for (uint32_t l = 0; l < L; ++l) {
            KV(kv_fence_query(fl[l]));
            kvo_restore(&g, img, (int64_t)off, want_host, slots, dst2, n, (int32_t)l);
        }
        CK(cudaMemcpy(got, alloc_d, off + pool_bytes, cudaMemcpyDeviceToHost));
        if (memcmp(got, img, off + pool_bytes) != 0) { printf("pool differs (overlapped)\n"); return 8; }
        cfg.flags &= ~KV_CFG_OVERLAP_RESTORES;
        KV(kv_config_set(&cfg));
        CK(cudaStreamDestroy(st));
    }

    KV(kv_pool_close(pool));
    KV(kv_host_close(tier));
    CK(cudaFreeHost(host));
    CK(cudaFree(alloc_d));
    free(img); free(want_host); free(got);
    printf("c-abi gpu ok\n");
    return 0;
}
"""


def cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_c_program_backup_restore_against_the_oracle(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    lib = kbuild.build_library()
    libdir = os.path.dirname(lib)
    home = cuda_home()
    cudalib = next((d for d in (os.path.join(home, "lib64"), os.path.join(home, "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so"))), None)
    if cudalib is None:
        pytest.skip("libcudart.so not found")
    src = tmp_path / "t.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    subprocess.run([gcc, "-std=c11", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(home, "include"), str(src),
                    os.path.join(ROOT, "oracle", "kv_oracle.c"), "-L", libdir, "-lkvb",
                    "-L", cudalib, "-lcudart", "-lpthread",
                    f"-Wl,-rpath,{libdir}:{cudalib}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "c-abi gpu ok" in out.stdout
