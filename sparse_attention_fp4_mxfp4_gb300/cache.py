"""Paged FP4 KV store and FP8 sliding-window rings, allocated with torch.

The store layout is the library's (include/csa2.h): 128-entry pages of the main
plane (36864 B) and of the indexer plane (9216 B) sharing one int32 block
table [B, max_pages], and rings [n_rings, 128, 512] of E4M3 bytes. This module
only allocates and maps pages; the kernels write them.
"""
from __future__ import annotations

import torch

from . import PAGE_TOKENS, PLANE_INDEX, PLANE_MAIN, csa2_page_bytes, csa2_ring_bytes


class PagedCache:
    def __init__(self, B: int, max_ctx: int, n_rings: int = 0, device="cuda", shuffle_seed: int | None = None,
                 spare_pages: int = 0):
        """B sequences of up to max_ctx entries each. Physical pages are handed
        out contiguously per sequence, or in a seeded random order when
        shuffle_seed is given (exercises the block table)."""
        self.B, self.max_ctx = B, max_ctx
        self.max_pages = (max_ctx + PAGE_TOKENS - 1) // PAGE_TOKENS
        self.n_pages = B * self.max_pages + spare_pages
        self.main_pages = torch.zeros(self.n_pages, csa2_page_bytes(PLANE_MAIN), dtype=torch.uint8, device=device)
        self.idx_pages = torch.zeros(self.n_pages, csa2_page_bytes(PLANE_INDEX), dtype=torch.uint8, device=device)
        order = torch.arange(self.n_pages, dtype=torch.int32)
        if shuffle_seed is not None:
            g = torch.Generator().manual_seed(shuffle_seed)
            order = order[torch.randperm(self.n_pages, generator=g)]
        self.block_table = order[: B * self.max_pages].reshape(B, self.max_pages).contiguous().to(device)
        self.n_rings = n_rings
        self.rings = torch.zeros(max(1, n_rings), csa2_ring_bytes() // 512, 512, dtype=torch.uint8, device=device)

    def nbytes(self) -> int:
        return self.main_pages.numel() + self.idx_pages.numel() + self.rings.numel()
