"""One decode (or chunked-prefill) step of a materialised workload: the
launch sequence that the benchmark times and the full-size tests check."""
from __future__ import annotations

import torch

from .workload import Setup, append_main


def append_layers(S: Setup, swa=None, q_idx=None):
    """csa2_decode_appends' per-layer arguments of a decode step: every
    layer's window entries and, for FULL and REINDEX layers, its indexer
    query (swa / q_idx: per-layer replacements of the step's own tensors)."""
    out = []
    for li, L in enumerate(S.layers):
        d = {"swa": S.step_swa[li] if swa is None else swa[li], "ring_idx": S.step_ring_idx[li],
             "rings": S.cache.rings}
        if L.kind in ("full", "reindex"):
            d.update(q_idx=L.q_idx if q_idx is None else q_idx[li], q_codes=L.q_codes, q_scales=L.q_scales)
        out.append(d)
    return out


class Runner:
    """One decode step of a materialised workload, as bench.py times it: the
    step's appends (A1, A2) and indexer-query quantisations (one launch at
    one token per entry), then every layer in order. A FULL layer scans,
    selects the pool and the top-512; a REINDEX layer rescores its pool;
    every layer then runs sparse attention with the latest top-k, its own
    query and its own ring.

    prefill=True runs the step's n_q tokens as one prefill chunk instead: each
    layer's window entries of the chunk are encoded to E4M3 into a chunk
    buffer (not the ring), the attention takes every token's exact causal
    window from that buffer and the ring, and each layer's ring is refilled
    with the chunk's last 128 entries after its attention."""

    def __init__(self, S: Setup, out_dtype=torch.bfloat16, prefill=False):
        import sparse_attention_fp4_mxfp4_gb300 as csa2
        self.csa2 = csa2
        self.S = S
        dev = S.seq_len.device
        B, n_q, N = S.B, S.n_q, S.N
        Q = B * n_q
        self.max_blocks = (N // S.m + 7) // 8
        self.ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_DECODE_LAYER, B, n_q, N), dtype=torch.uint8,
                              device=dev)
        bm_bytes = Q * self.max_blocks * 4
        self.bm = self.ws[:bm_bytes].view(torch.float32).view(B, n_q, self.max_blocks)
        self.rws = self.ws[((bm_bytes + 255) // 256) * 256:]
        self.pool = torch.empty(B, n_q, 2048, dtype=torch.int32, device=dev)
        self.topk = S.topk if S.layers[0].kind == "reuse" else torch.empty(B, n_q, 512, dtype=torch.int32,
                                                                            device=dev)
        self.out = [torch.empty(B, n_q, 64, 512, dtype=out_dtype, device=dev) for _ in S.layers]
        self.lse = [torch.empty(B, n_q, 64, dtype=torch.float32, device=dev) for _ in S.layers]
        self.launches = 0
        # The attention splits a token's five key chunks over several work
        # items of two CTAs each (plus a merge kernel) only while there are
        # fewer than half as many tokens as SMs.
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.attn_launches = 1 if Q >= 256 or min(5, max(1, sms // (2 * Q))) == 1 else 2
        self.prefill = prefill
        # One launch for the step's stores and query quantisations (decode at
        # one token per entry); otherwise one call each.
        self.fused_appends = S.m == 1 and not prefill and len(S.layers) <= 16
        self.append_args = append_layers(S) if self.fused_appends else None
        self.chunk = [torch.empty(B, n_q, 512, dtype=torch.uint8, device=dev) for _ in S.layers] if prefill else None

    def step(self, mark=None):
        """All launches on the current stream, in the order of the public-call
        path (csa2_decode_group after the appends and quantisations), so that
        every kernel overlaps its predecessor's tail through programmatic
        dependent launch; side streams would join through events, which
        this overlap does not cross."""
        csa2, S, c = self.csa2, self.S, self.S.cache
        mark = mark or (lambda name: None)
        n = 0
        if self.fused_appends:
            csa2.csa2_decode_appends(S.step_latent, S.step_idx_key, S.step_seq, S.step_pos, c.block_table,
                                     c.main_pages, c.idx_pages, self.append_args)
            n += 1
        else:
            append_main(S)
            n += 1 if S.m == 1 else 2
            for li, L in enumerate(S.layers):
                if self.prefill:
                    csa2.csa2_quant_fp8_entries(S.step_swa[li], self.chunk[li])
                else:
                    csa2.csa2_append_swa(S.step_swa[li], S.step_ring_idx[li], S.step_pos, c.rings)
                n += 1
                if L.kind in ("full", "reindex"):
                    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)
                    n += 1
        for li, L in enumerate(S.layers):
            if L.kind == "full":
                mark("scan0")
                csa2.csa2_indexer_scan(L.q_codes, L.q_scales, L.w, S.seq_len, S.N, c.block_table, c.n_pages,
                                       c.idx_pages, self.bm, m=S.m)
                mark("scan1")
                mark("blocktopk0")
                csa2.csa2_block_topk(self.bm, S.seq_len, self.pool, m=S.m)
                mark("blocktopk1")
                n += 2
            if L.kind in ("full", "reindex"):
                pool = self.pool if L.kind == "full" else L.pool
                mark("rescore0")
                csa2.csa2_indexer_reindex(L.q_codes, L.q_scales, L.w, S.seq_len, c.block_table, c.n_pages,
                                          c.idx_pages, pool, self.topk, self.rws, m=S.m)
                mark("rescore1")
                n += 2
            mark("attn0")
            if self.prefill:
                csa2.csa2_sparse_attn_prefill(L.q, self.topk, S.seq_len, c.block_table, c.n_pages, c.main_pages,
                                              c.rings, L.ring_idx, self.chunk[li], self.out[li], self.lse[li],
                                              self.ws, m=S.m)
            else:
                csa2.csa2_sparse_attn(L.q, self.topk, S.seq_len, c.block_table, c.n_pages, c.main_pages, c.rings,
                                      L.ring_idx, self.out[li], self.lse[li], self.ws, m=S.m)
            mark("attn1")
            n += self.attn_launches
            if self.prefill:
                csa2.csa2_ring_refill(self.chunk[li], S.seq_len, L.ring_idx, c.rings)
                n += 1
        self.launches = n
