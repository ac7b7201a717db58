"""Workload construction and oracle references shared by the GPU tests and the
benchmark.

Inputs come from the seeded generator (synth), are copied to the device and
written into the paged store through the library's own append call; the CPU
oracle receives the very same generator arrays. Nothing here computes any of
the method's arithmetic itself: it wires inputs to the library and to the
oracle, and compares their outputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from synth.workloads import WORKLOADS, Workload

TAU = 1.0 / math.sqrt(512)
TOL_ATTN_F32 = 2e-3    # max over channels |o - r| / max |r|, per (query, head)
# A bf16 output adds its rounding: half an ulp is at most 2^-8 of the value
# (reached just above a power of two), and |o| <= (1 + 2e-3) max |r|.
TOL_ATTN_BF16 = TOL_ATTN_F32 + 2.0 ** -8 * (1 + TOL_ATTN_F32)
TOPK_TIE_RTOL = 1e-5   # selections may differ only among scores this close to the k-th
# Log-sum-exp (natural log), absolute: the kernel rounds every p = 2^(l - m) to
# f16 and its normaliser sums exactly those rounded values, so the sum carries
# a relative error of at most 2^-11 (half an f16 ulp; p >= 2^-14 stays normal
# except for negligible keys, which add at most 640 * 2^-25), plus fp32
# accumulation (the relative 1e-5 the tests add covers the logits' fp32 dot
# products). With few keys the roundings do not average out.
TOL_LSE = 2.0 ** -11 + 640 * 2.0 ** -25 + 1e-5


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
    from sparse_attention_fp4_mxfp4_gb300.cache import PagedCache

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


class Runner:
    """One decode step of a materialised workload, as bench.py times it: the
    step's appends (A1, A2), then every layer in order. A FULL layer quantises
    its indexer query, scans, selects the pool and the top-512; a REINDEX
    layer quantises its query and rescores its pool; every layer then runs
    sparse attention with the latest top-k, its own query and its own ring.

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
        # The attention launch splits a token's five key chunks over several
        # CTAs (plus a merge kernel) only while there are fewer tokens than SMs.
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        self.attn_launches = 1 if Q >= 256 or min(5, max(1, sms // Q)) == 1 else 2
        self.side = None
        self.prefill = prefill
        self.chunk = [torch.empty(B, n_q, 512, dtype=torch.uint8, device=dev) for _ in S.layers] if prefill else None

    def step(self, mark=None):
        """The window-ring appends and the indexer-query quantisations do not
        depend on the main append, so they run on two side streams forked from
        the current one and joined before their first consumer."""
        csa2, S, c = self.csa2, self.S, self.S.cache
        mark = mark or (lambda name: None)
        n = 0
        main = torch.cuda.current_stream()
        if self.side is None:
            self.side = (torch.cuda.Stream(device=main.device), torch.cuda.Stream(device=main.device))
        s_swa, s_q = self.side
        s_swa.wait_stream(main)
        s_q.wait_stream(main)
        with torch.cuda.stream(s_swa):
            for li in range(len(S.layers)):
                if self.prefill:
                    csa2.csa2_quant_fp8_entries(S.step_swa[li], self.chunk[li])
                else:
                    csa2.csa2_append_swa(S.step_swa[li], S.step_ring_idx[li], S.step_pos, c.rings)
        with torch.cuda.stream(s_q):
            for L in S.layers:
                if L.kind in ("full", "reindex"):
                    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)
                    n += 1
        append_main(S)
        n += (1 if S.m == 1 else 2) + len(S.layers)
        main.wait_stream(s_q)
        swa_joined = False
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
            if not swa_joined:
                main.wait_stream(s_swa)
                swa_joined = True
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


# ---- oracle references ------------------------------------------------------------

def entries_seen(S: Setup, t: int) -> int:
    """Complete entries visible to the token at position t."""
    return (t + 1) // S.m


def oracle_entry_rows(S: Setup, b: int, entries, key=False) -> np.ndarray:
    """bf16 rows of the given entries: the tokens' own values (m = 1) or the
    oracle's compression of each entry's m tokens."""
    import oracle
    seed, m = S.wl.seed, S.m
    e = np.asarray(entries, np.int64)
    if m == 1:
        if key:
            return synth.normal_rows(seed, synth.IDXKEY, np.full(e.size, b), e, 128)
        return synth.latent_rows(seed, np.full(e.size, b), e)
    toks = (e[:, None] * m + np.arange(m)).reshape(-1)
    bs = np.full(toks.size, b)
    if key:
        x = synth.normal_rows(seed, synth.IDXKEY, bs, toks, 128)
        z = synth.normal_rows(seed, synth.IDXGATE, bs, toks, 128)
    else:
        x = synth.latent_rows(seed, bs, toks)
        z = synth.normal_rows(seed, synth.KVGATE, bs, toks, 512)
    d = x.shape[-1]
    return oracle.compress(x.reshape(e.size, m, d), z.reshape(e.size, m, d))


def oracle_keys(S: Setup, b: int, t: int) -> np.ndarray:
    """Indexer keys (bf16) of every entry visible at token position t."""
    if S.m == 1:
        return synth.normal(S.wl.seed, synth.IDXKEY, b, 0, t + 1, 128)
    import oracle
    n = entries_seen(S, t)
    x = synth.normal(S.wl.seed, synth.IDXKEY, b, 0, n * S.m, 128).reshape(n, S.m, 128)
    z = synth.normal(S.wl.seed, synth.IDXGATE, b, 0, n * S.m, 128).reshape(n, S.m, 128)
    return oracle.compress(x, z)


def oracle_full(S: Setup, b: int, j: int, li: int = 0, keys=None):
    import oracle
    L = S.layers[li]
    t = S.t(j)
    keys = oracle_keys(S, b, t) if keys is None else keys
    return oracle.full_indexer(L.q_idx_u16[b, j], L.w_np[b, j], keys, entries_seen(S, t) - 1)


def oracle_reindex(S: Setup, b: int, j: int, li: int, pool_row, keys=None):
    import oracle
    L = S.layers[li]
    t = S.t(j)
    keys = oracle_keys(S, b, t) if keys is None else keys
    return oracle.reindex(L.q_idx_u16[b, j], L.w_np[b, j], keys, entries_seen(S, t) - 1,
                          np.asarray(pool_row, np.int32))


def oracle_attention(S: Setup, b: int, j: int, li: int, topk_row, exact_window=False):
    """exact_window: the prefill window (all of max(0, t-127) .. t), which is
    the decode window of a context that ends at t."""
    import oracle
    seed = S.wl.seed
    t = S.t(j)
    sel = np.asarray(topk_row)
    sel = sel[sel >= 0].astype(np.int64)
    main = oracle_entry_rows(S, b, sel)
    win = oracle.window_positions(t, t + 1 if exact_window else S.N, 128)
    wrows = synth.latent_rows(seed, np.full(win.size, b), win, tensor=synth.SWA + li)
    return oracle.sparse_attention(S.layers[li].q_u16[b, j], main, wrows, TAU)


# ---- comparisons -------------------------------------------------------------------

def check_selection(got, want, score_of, k, what=""):
    """Selections equal except for elements whose oracle score lies within
    TOPK_TIE_RTOL (relative) of the oracle's k-th score."""
    got = np.asarray(got)
    want = np.asarray(want)
    g = set(got[got >= 0].tolist())
    w = set(want[want >= 0].tolist())
    assert len(g) == (got >= 0).sum(), f"{what}: duplicate selections"
    assert len(g) == len(w), f"{what}: {len(g)} selected, oracle {len(w)}"
    if g == w:
        return 0
    wl = sorted(w, key=lambda i: -score_of(i))
    kth = score_of(wl[min(k, len(wl)) - 1])
    tol = TOPK_TIE_RTOL * max(abs(kth), 1e-30)
    for i in g ^ w:
        assert abs(score_of(i) - kth) <= tol, (
            f"{what}: element {i} (score {score_of(i)!r}) differs from the oracle's selection "
            f"and is not tied with the k-th score {kth!r}")
    return len(g ^ w)


def check_attention(out, ref, tol):
    """Per (head) row: max_c |o - r| / max_c |r| <= tol."""
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(out - ref).max(-1) / np.maximum(np.abs(ref).max(-1), 1e-30)
    assert (err <= tol).all(), f"attention max-relative error {err.max():.3e} > {tol} (head {int(err.argmax())})"
    return float(err.max())


# ---- page unpacking (test-side view of the documented layout) ---------------------------

def unpack_main(cache, b: int, positions) -> tuple[np.ndarray, np.ndarray]:
    """codes uint8 [n, 256] and scales uint8 [n, 32] of the main entries at positions."""
    bt = cache.block_table.cpu().numpy()
    pages = cache.main_pages
    out_c, out_s = [], []
    pos = np.asarray(positions, np.int64)
    rows = torch.from_numpy(bt[b, pos // 128].astype(np.int64)).to(pages.device)
    slots = torch.from_numpy(pos % 128).to(pages.device)
    ent = pages.view(pages.shape[0], 128, 288)[rows, slots].cpu().numpy()
    return ent[:, :256], ent[:, 256:]


def unpack_idx(cache, b: int, positions) -> tuple[np.ndarray, np.ndarray]:
    """codes uint8 [n, 64] (channel order) and scales uint8 [n, 8] of indexer keys."""
    bt = cache.block_table.cpu().numpy()
    pages = cache.idx_pages
    pos = np.asarray(positions, np.int64)
    pg = pages.view(pages.shape[0], 16, 576)
    rows = torch.from_numpy(bt[b, pos // 128].astype(np.int64)).to(pages.device)
    grp = torch.from_numpy((pos % 128) // 8).to(pages.device)
    g = pg[rows, grp].cpu().numpy()  # [n, 576]
    r = pos % 8
    codes = g[:, :512].reshape(-1, 4, 8, 16)[np.arange(pos.size), :, r, :].reshape(-1, 64)
    scales = g[:, 512:].reshape(-1, 8, 8)[np.arange(pos.size), r, :]
    return codes, scales
