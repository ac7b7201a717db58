"""A synthetic CSA2 workload materialised on the device.

Inputs come from the seeded generator (synth), are copied to the device and
written into the paged store through the library's own append calls; nothing
here computes any of the method's arithmetic. The benchmark and the tests
build their workloads with build(); the decode step that runs on them is
sparse_attention_fp4_mxfp4_gb300.step.Runner.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from synth.workloads import Workload


def u16_to_bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_to_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class Layer:
    kind: str
    q: torch.Tensor            # bf16 [B, n_q, 64, 512]
    q_u16: np.ndarray
    q_idx: torch.Tensor | None = None   # bf16 [B, n_q, 32, 128]
    q_idx_u16: np.ndarray | None = None
    w: torch.Tensor | None = None       # fp32 [B, n_q, 32]
    w_np: np.ndarray | None = None
    q_codes: torch.Tensor | None = None
    q_scales: torch.Tensor | None = None
    pool: torch.Tensor | None = None    # int32 [B, n_q, 2048]
    ring_idx: torch.Tensor | None = None


@dataclass
class Setup:
    wl: Workload
    N: int
    cache: object
    seq_len: torch.Tensor
    layers: list = field(default_factory=list)
    topk: torch.Tensor | None = None       # int32 [B, n_q, 512]
    step_latent: torch.Tensor | None = None
    step_idx_key: torch.Tensor | None = None
    step_seq: torch.Tensor | None = None
    step_pos: torch.Tensor | None = None
    step_swa: list = field(default_factory=list)     # per layer bf16 [B*n_q, 512]
    step_ring_idx: list = field(default_factory=list)
    step_kv_gate: torch.Tensor | None = None         # m > 1: compression logits of the step's tokens
    step_idx_gate: torch.Tensor | None = None
    tail: torch.Tensor | None = None                 # m > 1: bf16 [B, m-1, 1280] compressor state

    @property
    def B(self):
        return self.wl.B

    @property
    def n_q(self):
        return self.wl.n_q

    @property
    def m(self):
        return self.wl.m

    def t(self, j: int) -> int:
        return self.N - self.n_q + j


def n_blocks(t: int) -> int:
    return (t + 8) // 8


def build(wl: Workload, device="cuda", *, N=None, B=None, n_q=None, shuffle_seed=None, prefill_step=False,
          chunk=65536):
    """Materialise a workload on the device.

    Positions 0 .. N-n_q-1 of every sequence are appended at set-up; the step's
    n_q tokens (positions N-n_q .. N-1) are prepared in step_* tensors and are
    appended by append_step() (or here too when prefill_step is set).
    """
    import sparse_attention_fp4_mxfp4_gb300 as csa2
    from .cache import PagedCache

    if N is not None or B is not None or n_q is not None:
        wl = Workload(wl.index, wl.name, wl.mode, B=B or wl.B, N=N or wl.N, n_q=n_q or wl.n_q, layers=wl.layers,
                      prefill=wl.prefill, m=wl.m)
    N, Bq, nq, seed, m = wl.N, wl.B, wl.n_q, wl.seed, wl.m
    n_layers = len(wl.layers)
    # The store holds entries: one per token (m = 1) or per m tokens.
    cache = PagedCache(Bq, (N + m - 1) // m, n_rings=Bq * n_layers, device=device, shuffle_seed=shuffle_seed)
    S = Setup(wl=wl, N=N, cache=cache, seq_len=torch.full((Bq,), N, dtype=torch.int64, device=device))
    if m > 1:
        S.tail = torch.zeros(Bq, m - 1, 1280, dtype=torch.bfloat16, device=device)
    pre = N - nq
    for b in range(Bq):
        for p0 in range(0, pre, chunk):
            n = min(chunk, pre - p0)
            lat = u16_to_bf16(synth.latent(seed, b, p0, n), device)
            key = u16_to_bf16(synth.normal(seed, synth.IDXKEY, b, p0, n, 128), device)
            seq = torch.full((n,), b, dtype=torch.int32, device=device)
            pos = torch.arange(p0, p0 + n, dtype=torch.int64, device=device)
            if m == 1:
                csa2.csa2_append_kv(lat, key, seq, pos, cache.block_table, cache.main_pages, cache.idx_pages)
            else:
                lg = u16_to_bf16(synth.normal(seed, synth.KVGATE, b, p0, n, 512), device)
                kg = u16_to_bf16(synth.normal(seed, synth.IDXGATE, b, p0, n, 128), device)
                csa2.csa2_compress_append(lat, lg, key, kg, seq, pos, m, S.tail, cache.block_table, cache.main_pages,
                                          cache.idx_pages)
    # Window entries of the 128 positions before the step's tokens, one ring per
    # (layer, sequence): the ring state a prefill chunk starts from; a decode
    # step's appends then leave positions N-128 .. N-1.
    lo = max(0, pre - 128)
    for li in range(n_layers):
        for b in range(Bq):
            if pre > lo:
                x = u16_to_bf16(synth.latent(seed, b, lo, pre - lo, tensor=synth.SWA + li), device)
                ridx = torch.full((pre - lo,), li * Bq + b, dtype=torch.int32, device=device)
                pos = torch.arange(lo, pre, dtype=torch.int64, device=device)
                csa2.csa2_append_swa(x, ridx, pos, cache.rings)
    # The step's new tokens.
    lat = np.concatenate([synth.latent(seed, b, pre, nq) for b in range(Bq)])
    key = np.concatenate([synth.normal(seed, synth.IDXKEY, b, pre, nq, 128) for b in range(Bq)])
    S.step_latent = u16_to_bf16(lat, device)
    S.step_idx_key = u16_to_bf16(key, device)
    if m > 1:
        S.step_kv_gate = u16_to_bf16(np.concatenate([synth.normal(seed, synth.KVGATE, b, pre, nq, 512)
                                                     for b in range(Bq)]), device)
        S.step_idx_gate = u16_to_bf16(np.concatenate([synth.normal(seed, synth.IDXGATE, b, pre, nq, 128)
                                                      for b in range(Bq)]), device)
    S.step_seq = torch.arange(Bq, dtype=torch.int32, device=device).repeat_interleave(nq)
    S.step_pos = torch.arange(pre, N, dtype=torch.int64, device=device).repeat(Bq)
    for li in range(n_layers):
        x = np.concatenate([synth.latent(seed, b, pre, nq, tensor=synth.SWA + li) for b in range(Bq)])
        S.step_swa.append(u16_to_bf16(x, device))
        S.step_ring_idx.append((li * Bq + torch.arange(Bq, dtype=torch.int32, device=device)).repeat_interleave(nq))
    # Per-layer queries.
    for li, kind in enumerate(wl.layers):
        qn = np.stack([synth.normal(seed, synth.Q + li, b, pre, nq, 64 * 512) for b in range(Bq)])
        qn = qn.reshape(Bq, nq, 64, 512)
        L = Layer(kind=kind, q=u16_to_bf16(qn, device), q_u16=qn,
                  ring_idx=(li * Bq + torch.arange(Bq, dtype=torch.int32, device=device)))
        if kind in ("full", "reindex"):
            qi = np.stack([synth.normal(seed, synth.IDXQ + li, b, pre, nq, 32 * 128) for b in range(Bq)])
            L.q_idx_u16 = qi.reshape(Bq, nq, 32, 128)
            L.q_idx = u16_to_bf16(L.q_idx_u16, device)
            L.w_np = np.stack([synth.uniform(seed, synth.W + li, b, pre, nq, 32) for b in range(Bq)])
            L.w = torch.from_numpy(L.w_np).to(device)
            L.q_codes = torch.empty(Bq, nq, 32, 64, dtype=torch.uint8, device=device)
            L.q_scales = torch.empty(Bq, nq, 32, 8, dtype=torch.uint8, device=device)
        if kind == "reindex":
            pools = np.full((Bq, nq, 2048), -1, np.int32)
            for b in range(Bq):
                for j in range(nq):
                    t = N - nq + j
                    te = (t + 1) // m - 1  # the token's last visible entry
                    if te >= 0:
                        s = synth.sample_sorted(seed, synth.POOL + li, b, t, n_blocks(te), 2048)
                        pools[b, j, : s.size] = s
            L.pool = torch.from_numpy(pools).to(device)
        S.layers.append(L)
    if wl.layers[0] == "reuse":
        tk = np.full((Bq, nq, 512), -1, np.int32)
        for b in range(Bq):
            for j in range(nq):
                t = N - nq + j
                te = (t + 1) // m - 1
                if te >= 0:
                    s = synth.sample_sorted(seed, synth.TOPK, b, t, te + 1, 512)
                    tk[b, j, : s.size] = s
        S.topk = torch.from_numpy(tk).to(device)
    else:
        S.topk = torch.full((Bq, nq, 512), -1, dtype=torch.int32, device=device)
    if prefill_step:
        append_step(S)
    return S


def append_main(S: Setup, latent=None, idx_key=None, kv_gate=None, idx_gate=None):
    """A1 of the step: the n_q new tokens of every sequence into the store
    (compressed m tokens per entry when m > 1)."""
    import sparse_attention_fp4_mxfp4_gb300 as csa2
    c = S.cache
    lat = S.step_latent if latent is None else latent
    key = S.step_idx_key if idx_key is None else idx_key
    if S.m == 1:
        csa2.csa2_append_kv(lat, key, S.step_seq, S.step_pos, c.block_table, c.main_pages, c.idx_pages)
    else:
        csa2.csa2_compress_append(lat, S.step_kv_gate if kv_gate is None else kv_gate, key,
                                  S.step_idx_gate if idx_gate is None else idx_gate, S.step_seq, S.step_pos, S.m,
                                  S.tail, c.block_table, c.main_pages, c.idx_pages)


def append_step(S: Setup):
    """A1 + A2 of one decode step: the n_q new entries of every sequence."""
    import sparse_attention_fp4_mxfp4_gb300 as csa2
    c = S.cache
    append_main(S)
    for li in range(len(S.layers)):
        csa2.csa2_append_swa(S.step_swa[li], S.step_ring_idx[li], S.step_pos, c.rings)
