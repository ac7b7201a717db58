"""Oracle references and comparisons of the GPU tests.

Workloads are built on the device by sparse_attention_fp4_mxfp4_gb300.workload
(seeded generator inputs written through the library's own append calls); the
CPU oracle receives the very same generator arrays. Nothing here computes any
of the method's arithmetic itself: it wires inputs to the oracle and compares
the library's outputs with the oracle's.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import synth

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


# The workload builder and the timed step live in the package (bench.py uses
# them too); the tests reach them through this module.
from sparse_attention_fp4_mxfp4_gb300.workload import (  # noqa: E402,F401
    Layer, Setup, append_main, append_step, bf16_to_u16, build, n_blocks, u16_to_bf16)
from sparse_attention_fp4_mxfp4_gb300.step import Runner  # noqa: E402,F401


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
