"""Seeded synthetic workloads: pool geometries, page-ID lists and random payload.

This module feeds both the CUDA library (tests, benchmark) and the CPU oracle
(tests), so it deliberately holds none of the method's arithmetic: no layout
offsets, no copy logic.  It only names the five workload shapes, sizes buffers
(pages x bytes per page) and draws seeded IDs and bytes.

Workload shapes follow the HiCache / LMCache pages: page size 256 with fp8 KV
and 16,384-token prefixes ("[PP + HiCache] Add PP Prefetch Tickets..." --
§Benchmark setup), the TRT-LLM pool [NB, NL, 2, NH*BS*HS] with HND heads
("LMCache RawCudaIPCWrapper深度解析" -- §在项目中的实际接入方式), and
Llama-8B-shaped and tiny pools.  Payload is random bytes: fp16 / bf16 /
fp8_e4m3 values are opaque bytes on this path, so random bit patterns
(NaN and Inf included) are the hardest honest input.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

LAYER_FIRST, PAGE_FIRST = 0, 1
NHD, HND = 0, 1


@dataclass(frozen=True)
class Geometry:
    """Pool geometry.  ``B`` is bytes per head vector (head_dim x element bytes)."""

    L: int            # layers
    C: int            # components: 2 = K,V ; 1 = MLA latent
    P: int            # pages in the device pool
    T: int            # tokens per page
    H: int            # KV heads
    B: int            # bytes per head vector
    order: int = LAYER_FIRST
    dev_heads: int = NHD
    host_heads: int = NHD
    elem_bytes: int = 2

    @property
    def page_bytes(self) -> int:
        """Bytes one page occupies (= one host slot)."""
        return self.L * self.C * self.T * self.H * self.B

    @property
    def layer_page_bytes(self) -> int:
        """Bytes of one layer of one page."""
        return self.C * self.T * self.H * self.B

    @property
    def pool_bytes(self) -> int:
        return self.P * self.page_bytes

    def with_(self, **kw) -> "Geometry":
        return replace(self, **kw)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                 # 0-based position in the list of five workloads
    geom: Geometry
    n: int                     # pages per backup / restore call
    host_slots: int            # slots in the host tier
    pool_offset: int = 0       # byte offset of the pool inside its allocation
    layerwise: bool = False    # restore one layer per call
    concurrent: bool = False   # backup and restore in flight together
    notes: str = field(default="", compare=False)

    @property
    def seed(self) -> int:
        return 1000 + self.index


# 1. tiny pool: 2 layers x {K,V} x 2 heads x page 16 x head_dim 64, 16-bit elements.
TINY = Workload("tiny", 0, Geometry(L=2, C=2, P=64, T=16, H=2, B=128), n=8, host_slots=16,
                notes="8 random pages to 8 random slots of 16; restore into 8 other free pages")
# 2. Llama-8B-shaped: 32 layers x {K,V} x 8 heads x head_dim 128 bf16, page 16, 4096 pages, layer-first NHD.
LLAMA8B = Workload("llama8b", 1, Geometry(L=32, C=2, P=4096, T=16, H=8, B=256), n=512,
                   host_slots=512,
                   notes="backup 512 random pages to slots 0..511, restore all 512 into 512 other pages")
# 3. MLA fp8: 61 layers, one 576-byte latent per token, page 256, 2048 pages; layer-wise restore.
MLA_FP8 = Workload("mla_fp8", 2, Geometry(L=61, C=1, P=2048, T=256, H=1, B=576, elem_bytes=1),
                   n=64, host_slots=64, layerwise=True,
                   notes="16,384-token prefix = 64 pages restored one layer per call")
# 4. TRT-LLM pool [2048, 40, 2, 8*32*128] bf16, page-first HND, at a nonzero offset in one allocation.
TRTLLM = Workload("trtllm_ipc", 3, Geometry(L=40, C=2, P=2048, T=32, H=8, B=256,
                                            order=PAGE_FIRST, dev_heads=HND, host_heads=NHD),
                  n=512, host_slots=1024, pool_offset=2 * 1024 * 1024 + 48, concurrent=True,
                  notes="backup 25% of pages (slots 0..511) while restoring another 25% (slots 512..1023)")
# 5. bandwidth sweep: one opaque run per page (L=C=T=H=1, B = page bytes), 8192 pages.
SWEEP_PAGE_BYTES = [4096 << k for k in range(9)]          # 4 KiB .. 1 MiB
SWEEP_BATCHES = [1 << k for k in range(13)]               # 1 .. 4096


def sweep(page_bytes: int, n: int, pages: int = 8192) -> Workload:
    return Workload(f"sweep_{page_bytes}_{n}", 4,
                    Geometry(L=1, C=1, P=pages, T=1, H=1, B=page_bytes, elem_bytes=1),
                    n=n, host_slots=2 * n, concurrent=True)


WORKLOADS = [TINY, LLAMA8B, MLA_FP8, TRTLLM, sweep(65536, 512)]


# ---------------------------------------------------------------- seeded draws

def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def distinct_pages(g: np.random.Generator, P: int, n: int, exclude=()) -> np.ndarray:
    """n distinct page IDs drawn uniformly from [0, P) minus ``exclude`` (int32)."""
    if len(exclude):
        pool = np.setdiff1d(np.arange(P, dtype=np.int64), np.asarray(exclude, dtype=np.int64))
    else:
        pool = np.arange(P, dtype=np.int64)
    if n > pool.size:
        raise ValueError(f"cannot draw {n} distinct pages from {pool.size}")
    return pool[g.permutation(pool.size)[:n]].astype(np.int32)


def random_bytes(g: np.random.Generator, nbytes: int) -> np.ndarray:
    return g.integers(0, 256, size=nbytes, dtype=np.uint8)


@dataclass
class OpIds:
    """Page / slot lists of one workload: a backup and a restore."""

    backup_src: np.ndarray
    backup_slots: np.ndarray
    restore_slots: np.ndarray
    restore_dst: np.ndarray


def op_ids(w: Workload, seed: int | None = None) -> OpIds:
    """The IDs each workload's statement asks for, drawn from its seed."""
    g = rng(w.seed if seed is None else seed)
    P, n = w.geom.P, w.n
    if w.index == 0:      # tiny: random slots of a 16-slot tier; restore into other free pages
        src = distinct_pages(g, P, n)
        slots = distinct_pages(g, w.host_slots, n)
        dst = distinct_pages(g, P, n, exclude=src)
        return OpIds(src, slots, slots.copy(), dst)
    if w.layerwise:       # MLA: the prefix sits in slots 0..n-1; restore into random pages
        slots = np.arange(n, dtype=np.int32)
        dst = distinct_pages(g, P, n)
        src = distinct_pages(g, P, n)
        return OpIds(src, slots, slots.copy(), dst)
    if w.concurrent:      # backup one set while restoring another (disjoint pages, disjoint slots)
        src = distinct_pages(g, P, n)
        dst = distinct_pages(g, P, n, exclude=src)
        return OpIds(src, np.arange(n, dtype=np.int32), np.arange(n, 2 * n, dtype=np.int32), dst)
    src = distinct_pages(g, P, n)                  # Llama-8B: backup, then restore elsewhere
    dst = distinct_pages(g, P, n, exclude=src)
    slots = np.arange(n, dtype=np.int32)
    return OpIds(src, slots, slots.copy(), dst)


def sequential_ids(n: int, start: int = 0) -> np.ndarray:
    return np.arange(start, start + n, dtype=np.int32)


def fill_random_(t, seed: int):
    """Fill a uint8 torch tensor (any device) with seeded random bytes, in place."""
    import torch

    gen = torch.Generator(device=t.device)
    gen.manual_seed(int(seed))
    flat = t.view(-1)
    step = 1 << 30
    for lo in range(0, flat.numel(), step):
        hi = min(flat.numel(), lo + step)
        flat[lo:hi] = torch.randint(0, 256, (hi - lo,), dtype=torch.uint8, device=t.device,
                                    generator=gen)
    return t
