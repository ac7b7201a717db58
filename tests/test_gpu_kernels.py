"""Parity of every CUDA kernel with the CPU oracle at sizes the oracle finishes
in seconds: several tiles, ragged tails, n_q > 1, shuffled page tables, and
the degenerate cases (a single position, contexts shorter than a page, than
512 positions and than 2048 blocks).

Criteria: FP4 / FP8 codes and scales bit-exact; top-k sets equal except for
ties within 1e-5 relative of the k-th score; attention within 2e-3
max-relative per (query, head) row (fp32 output) or that plus bf16 rounding,
2^-8 (1 + 2e-3), for bf16 output.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.workloads import WORKLOADS, Workload
from tests import harness as H

pytestmark = pytest.mark.gpu

import sparse_attention_fp4_mxfp4_gb300 as csa2  # noqa: E402  (fails loudly without the library)

DEV = "cuda"


def _status_ok():
    st = csa2.csa2_check_device_status()
    assert st == csa2.OK, csa2.device_status_message()


# ---- codecs --------------------------------------------------------------------------

def _finite_bf16():
    u = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_to_f32(u)
    return u[np.isfinite(f)]


def test_mxfp4_quant_every_bf16_against_every_scale():
    """Every finite bf16 value is quantised against every positive E4M3 scale
    that keeps it within range: each block holds 6 * scale (which fixes the
    scale) and 15 swept values."""
    vals = _finite_bf16()
    fv = synth.bf16_to_f32(vals)
    blocks = []
    for sb in range(1, 0x7F):
        sf = oracle.e4m3_value(sb)
        anchor = np.float32(6.0 * sf)
        a16 = (np.array([anchor], np.float32).view(np.uint32) >> 16).astype(np.uint16)
        assert synth.bf16_to_f32(a16)[0] == anchor
        sel = vals[np.abs(fv) <= anchor]
        pad = (-sel.size) % 15
        sel = np.concatenate([sel, np.zeros(pad, np.uint16)]).reshape(-1, 15)
        blocks.append(np.concatenate([np.full((sel.shape[0], 1), a16[0], np.uint16), sel], 1))
    x = np.concatenate(blocks).reshape(-1)
    codes, scales = csa2.csa2_quant_mxfp4(H.u16_to_bf16(x, DEV))
    rc, rs = oracle.mxfp4_quant(synth.bf16_to_f32(x))
    assert np.array_equal(scales.cpu().numpy().reshape(-1), rs.reshape(-1))
    assert np.array_equal(codes.cpu().numpy().reshape(-1), rc.reshape(-1))


def test_mxfp4_quant_random_blocks_and_special_values():
    rng = np.random.default_rng(1)
    parts = [synth.latent(5, 0, 0, 4000).reshape(-1), synth.normal(5, synth.IDXKEY, 0, 0, 4000, 128).reshape(-1)]
    mags = (rng.standard_normal((20000, 16)) * 2.0 ** rng.integers(-20, 12, (20000, 1))).astype(np.float32)
    parts.append((mags.view(np.uint32) >> 16).astype(np.uint16).reshape(-1))
    special = np.array([0.0, -0.0, 2688, -2688, 3008, 1e30, -1e30, 2.0 ** -130, 448 * 6.5], np.float32)
    sp = np.resize((special.view(np.uint32) >> 16).astype(np.uint16), 16 * 40)
    parts.append(sp)
    x = np.concatenate(parts)
    codes, scales = csa2.csa2_quant_mxfp4(H.u16_to_bf16(x, DEV))
    rc, rs = oracle.mxfp4_quant(synth.bf16_to_f32(x))
    assert np.array_equal(scales.cpu().numpy().reshape(-1), rs.reshape(-1))
    assert np.array_equal(codes.cpu().numpy().reshape(-1), rc.reshape(-1))
    deq = csa2.csa2_dequant_mxfp4(codes, scales).cpu().numpy().reshape(-1).astype(np.float64)
    assert np.array_equal(deq, oracle.mxfp4_dequant(rc, rs).reshape(-1))


def test_fp8_every_fp32_bit_pattern():
    """fp32 -> E4M3 (RNE, saturating) for all 2^32 bit patterns except NaNs."""
    chunk = 1 << 27
    for lo in range(0, 1 << 32, chunk):
        bits = np.arange(lo, lo + chunk, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        x = x[~np.isnan(x)]
        if x.size == 0:
            continue
        got = csa2.csa2_quant_fp8(torch.from_numpy(x).to(DEV)).cpu().numpy()
        want = oracle.e4m3_encode(x)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (hex(lo), x[bad[:4]], got[bad[:4]], want[bad[:4]])


# ---- append ----------------------------------------------------------------------------

@pytest.mark.parametrize("N,n_q", [(1, 1), (130, 1), (1000, 3), (3000, 6)])
def test_append_pages_and_rings_bit_exact(N, n_q):
    wl = Workload(90, "t", "group", B=3, N=N, n_q=n_q, layers=("reindex", "reuse"))
    S = H.build(wl, DEV, shuffle_seed=7, prefill_step=True)
    torch.cuda.synchronize()
    _status_ok()
    for b in range(3):
        pos = np.arange(N)
        mc, ms = H.unpack_main(S.cache, b, pos)
        rc, rs = oracle.mxfp4_quant(synth.bf16_to_f32(synth.latent(wl.seed, b, 0, N)))
        assert np.array_equal(mc, rc) and np.array_equal(ms, rs)
        ic, is_ = H.unpack_idx(S.cache, b, pos)
        kc, ks = oracle.mxfp4_quant(synth.bf16_to_f32(synth.normal(wl.seed, synth.IDXKEY, b, 0, N, 128)))
        assert np.array_equal(ic, kc) and np.array_equal(is_, ks)
        for li in range(2):
            lo = max(0, N - 128)
            ring = S.cache.rings[li * 3 + b].cpu().numpy()
            want = oracle.fp8_quant(synth.bf16_to_f32(synth.latent(wl.seed, b, lo, N - lo, tensor=synth.SWA + li)))
            assert np.array_equal(ring[np.arange(lo, N) % 128], want)


@pytest.mark.parametrize("N,n_q,layers", [(1, 1, ("full",)), (1000, 3, ("reindex", "reuse", "full")),
                                         (3000, 6, ("full", "reuse"))])
def test_decode_appends_one_launch_bit_exact(N, n_q, layers):
    """csa2_decode_appends (the step's stores and query quantisations in one
    launch) writes the oracle's bytes: pages, every layer's ring, every
    indexed layer's query codes."""
    from sparse_attention_fp4_mxfp4_gb300.step import append_layers
    wl = Workload(91, "t", "group", B=3, N=N, n_q=n_q, layers=layers)
    S = H.build(wl, DEV, shuffle_seed=7, prefill_step=False)
    c = S.cache
    csa2.csa2_decode_appends(S.step_latent, S.step_idx_key, S.step_seq, S.step_pos, c.block_table, c.main_pages,
                             c.idx_pages, append_layers(S))
    torch.cuda.synchronize()
    _status_ok()
    for b in range(3):
        pos = np.arange(N)
        mc, ms = H.unpack_main(c, b, pos)
        rc, rs = oracle.mxfp4_quant(synth.bf16_to_f32(synth.latent(wl.seed, b, 0, N)))
        assert np.array_equal(mc, rc) and np.array_equal(ms, rs)
        ic, is_ = H.unpack_idx(c, b, pos)
        kc, ks = oracle.mxfp4_quant(synth.bf16_to_f32(synth.normal(wl.seed, synth.IDXKEY, b, 0, N, 128)))
        assert np.array_equal(ic, kc) and np.array_equal(is_, ks)
        for li in range(len(layers)):
            lo = max(0, N - 128)
            ring = c.rings[li * 3 + b].cpu().numpy()
            want = oracle.fp8_quant(synth.bf16_to_f32(synth.latent(wl.seed, b, lo, N - lo, tensor=synth.SWA + li)))
            assert np.array_equal(ring[np.arange(lo, N) % 128], want)
    for L in S.layers:
        if L.kind in ("full", "reindex"):
            qc, qs = oracle.mxfp4_quant(synth.bf16_to_f32(L.q_idx_u16))
            assert np.array_equal(L.q_codes.cpu().numpy(), qc) and np.array_equal(L.q_scales.cpu().numpy(), qs)


def test_decode_appends_without_entries_quantises_only():
    """T = 0: no page or window store, every indexed layer's query codes still written."""
    wl = Workload(98, "t", "group", B=2, N=700, n_q=2, layers=("full", "reuse", "reindex"))
    S = H.build(wl, DEV, shuffle_seed=2, prefill_step=True)
    c = S.cache
    pages_before = (c.main_pages.clone(), c.idx_pages.clone(), c.rings.clone())
    layers = [{"q_idx": L.q_idx, "q_codes": L.q_codes, "q_scales": L.q_scales} if L.kind != "reuse" else {}
              for L in S.layers]
    empty_bf16 = torch.empty(0, 512, dtype=torch.bfloat16, device=DEV)
    csa2.csa2_decode_appends(empty_bf16, torch.empty(0, 128, dtype=torch.bfloat16, device=DEV),
                             torch.empty(0, dtype=torch.int32, device=DEV), torch.empty(0, dtype=torch.int64, device=DEV),
                             c.block_table, c.main_pages, c.idx_pages, layers)
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(c.main_pages, pages_before[0]) and torch.equal(c.idx_pages, pages_before[1])
    assert torch.equal(c.rings, pages_before[2])
    for L in S.layers:
        if L.kind != "reuse":
            qc, qs = oracle.mxfp4_quant(synth.bf16_to_f32(L.q_idx_u16))
            assert np.array_equal(L.q_codes.cpu().numpy(), qc) and np.array_equal(L.q_scales.cpu().numpy(), qs)


def test_decode_appends_unmapped_page_sets_the_bounds_status():
    """An entry whose page is unmapped is skipped and reported; the other entries and parts are stored."""
    from sparse_attention_fp4_mxfp4_gb300.step import append_layers
    wl = Workload(99, "t", "full", B=2, N=300, n_q=1)
    S = H.build(wl, DEV, shuffle_seed=2, prefill_step=False)
    c = S.cache
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK
    bt = c.block_table.clone()
    bt[0, 299 // 128] = -1  # sequence 0's new entry (position 299) has no page
    csa2.csa2_decode_appends(S.step_latent, S.step_idx_key, S.step_seq, S.step_pos, bt, c.main_pages, c.idx_pages,
                             append_layers(S))
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.ERR_DEVICE_BOUNDS
    assert csa2.csa2_check_device_status() == csa2.OK  # cleared by the read
    # Sequence 1's entry, both window entries and the query codes are stored.
    mc, ms = H.unpack_main(c, 1, np.arange(300))
    rc, rs = oracle.mxfp4_quant(synth.bf16_to_f32(synth.latent(wl.seed, 1, 0, 300)))
    assert np.array_equal(mc, rc) and np.array_equal(ms, rs)
    for b in range(2):
        ring = c.rings[b].cpu().numpy()
        want = oracle.fp8_quant(synth.bf16_to_f32(synth.latent(wl.seed, b, 299, 1, tensor=synth.SWA)))
        assert np.array_equal(ring[299 % 128], want[0])
    L = S.layers[0]
    qc, qs = oracle.mxfp4_quant(synth.bf16_to_f32(L.q_idx_u16))
    assert np.array_equal(L.q_codes.cpu().numpy(), qc) and np.array_equal(L.q_scales.cpu().numpy(), qs)


# ---- indexer ---------------------------------------------------------------------------

def _quant_q(S, L):
    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)


@pytest.mark.parametrize("N,n_q,B", [(1, 1, 1), (9, 1, 2), (129, 2, 2), (1000, 1, 2), (5003, 3, 2), (20000, 1, 2),
                                     (20001, 6, 1)])
def test_indexer_scan_block_max(N, n_q, B):
    wl = Workload(91, "t", "full", B=B, N=N, n_q=n_q)
    S = H.build(wl, DEV, shuffle_seed=3, prefill_step=True)
    L = S.layers[0]
    _quant_q(S, L)
    mb = (N + 7) // 8 + 5
    bm = torch.full((B, n_q, mb), 12345.0, device=DEV)
    csa2.csa2_indexer_scan(L.q_codes, L.q_scales, L.w, S.seq_len, N, S.cache.block_table, S.cache.n_pages,
                           S.cache.idx_pages, bm)
    got = bm.cpu().numpy()
    _status_ok()
    for b in range(B):
        for j in range(n_q):
            ref = H.oracle_full(S, b, j)["blockmax"]
            nb = ref.size
            np.testing.assert_allclose(got[b, j, :nb], ref, rtol=2e-6, atol=1e-6 * max(1.0, np.abs(ref).max()))
            assert (got[b, j, nb:] == 12345.0).all(), "scan wrote past the causal blocks"


# (6000, 8, 20): 160 tokens, more than the SMs: the selections run in two waves of CTAs.
@pytest.mark.parametrize("N,n_q,B", [(1, 1, 1), (600, 1, 2), (4097, 2, 2), (20000, 1, 2), (40000, 3, 1),
                                     (9000, 8, 2), (6000, 8, 20)])
def test_indexer_full_pool_and_topk(N, n_q, B):
    wl = Workload(92, "t", "full", B=B, N=N, n_q=n_q)
    S = H.build(wl, DEV, shuffle_seed=5, prefill_step=True)
    L = S.layers[0]
    _quant_q(S, L)
    pool = torch.empty(B, n_q, 2048, dtype=torch.int32, device=DEV)
    topk = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_FULL, B, n_q, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_indexer_full(L.q_codes, L.q_scales, L.w, S.seq_len, N, S.cache.block_table, S.cache.n_pages,
                           S.cache.idx_pages, pool, topk, ws)
    gp, gt = pool.cpu().numpy(), topk.cpu().numpy()
    _status_ok()
    for b in range(B):
        for j in range(n_q):
            ref = H.oracle_full(S, b, j)
            H.check_selection(gp[b, j], ref["pool"], lambda i: ref["blockmax"][i], 2048, "pool")
            H.check_selection(gt[b, j], ref["topk"], lambda i: ref["scores"][i], 512, "topk")
            assert (np.diff(gp[b, j][gp[b, j] >= 0]) > 0).all() and (np.diff(gt[b, j][gt[b, j] >= 0]) > 0).all()
            pool_pos = set((gp[b, j][gp[b, j] >= 0][:, None] * 8 + np.arange(8)).reshape(-1).tolist())
            assert set(gt[b, j][gt[b, j] >= 0].tolist()) <= pool_pos


@pytest.mark.parametrize("N,n_q,B", [(700, 1, 2), (20000, 1, 3), (50000, 6, 1), (20000, 8, 20)])
def test_indexer_reindex(N, n_q, B):
    wl = Workload(93, "t", "reindex", B=B, N=N, n_q=n_q, layers=("reindex",))
    S = H.build(wl, DEV, shuffle_seed=9, prefill_step=True)
    L = S.layers[0]
    _quant_q(S, L)
    topk = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_REINDEX, B, n_q, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_indexer_reindex(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table, S.cache.n_pages,
                              S.cache.idx_pages, L.pool, topk, ws)
    gt = topk.cpu().numpy()
    pools = L.pool.cpu().numpy()
    _status_ok()
    for b in range(B):
        for j in range(n_q):
            ref = H.oracle_reindex(S, b, j, 0, pools[b, j])
            ps = ref["pos_scores"]
            slot = {int(pools[b, j][i // 8]) * 8 + i % 8: ps[i] for i in range(ps.size) if pools[b, j][i // 8] >= 0}
            H.check_selection(gt[b, j], ref["topk"], lambda p: slot[p], 512, "reindex topk")


# ---- attention ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,n_q,B,out", [(1, 1, 1, "f32"), (5, 1, 2, "f32"), (100, 3, 2, "f32"), (600, 1, 2, "f32"),
                                         (5000, 1, 3, "f32"), (5000, 6, 2, "f32"), (5000, 2, 2, "bf16"),
                                         (3000, 8, 2, "f32")])
def test_sparse_attention(N, n_q, B, out):
    wl = Workload(94, "t", "reuse", B=B, N=N, n_q=n_q, layers=("reuse",))
    S = H.build(wl, DEV, shuffle_seed=11, prefill_step=True)
    L = S.layers[0]
    dt = torch.float32 if out == "f32" else torch.bfloat16
    o = torch.empty(B, n_q, 64, 512, dtype=dt, device=DEV)
    lse = torch.empty(B, n_q, 64, dtype=torch.float32, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_SPARSE_ATTN, B, n_q, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_sparse_attn(L.q, S.topk, S.seq_len, S.cache.block_table, S.cache.n_pages, S.cache.main_pages,
                          S.cache.rings, L.ring_idx, o, lse, ws)
    go, gl = o.float().cpu().numpy(), lse.cpu().numpy()
    tk = S.topk.cpu().numpy()
    _status_ok()
    for b in range(B):
        for j in range(n_q):
            ro, rl = H.oracle_attention(S, b, j, 0, tk[b, j])
            H.check_attention(go[b, j], ro, H.TOL_ATTN_F32 if out == "f32" else H.TOL_ATTN_BF16)
            np.testing.assert_allclose(gl[b, j], rl, rtol=1e-5, atol=H.TOL_LSE)


@pytest.mark.parametrize("B,n_q,out", [(2, 3, "f32"), (40, 4, "f32"), (3, 2, "bf16")])
def test_sparse_attention_derotated(B, n_q, out):
    """CSA2_OUT_DEROTATE: the output's rotary channels rotated back by the token
    position, against the oracle's attention followed by its de-rotation. 160
    tokens take the one-CTA-per-token path, 6 the split-and-merge path."""
    N = 5000
    wl = Workload(93, "t", "reuse", B=B, N=N, n_q=n_q, layers=("reuse",))
    S = H.build(wl, DEV, shuffle_seed=12, prefill_step=True)
    L = S.layers[0]
    dt = torch.float32 if out == "f32" else torch.bfloat16
    o = torch.empty(B, n_q, 64, 512, dtype=dt, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_SPARSE_ATTN, B, n_q, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_sparse_attn(L.q, S.topk, S.seq_len, S.cache.block_table, S.cache.n_pages, S.cache.main_pages,
                          S.cache.rings, L.ring_idx, o, None, ws, derotate=True)
    go = o.float().cpu().numpy()
    tk = S.topk.cpu().numpy()
    _status_ok()
    rng = np.random.default_rng(5)
    pairs = {(int(rng.integers(B)), int(rng.integers(n_q))) for _ in range(12)}
    for b, j in sorted(pairs)[:6]:
        ro, _ = H.oracle_attention(S, b, j, 0, tk[b, j])
        ro = oracle.output_derotate(ro, S.t(j))
        H.check_attention(go[b, j], ro, H.TOL_ATTN_F32 if out == "f32" else H.TOL_ATTN_BF16)


def test_sparse_attention_with_padded_topk():
    """Fewer than 512 selected positions (-1 padding), e.g. a short context."""
    wl = Workload(95, "t", "reuse", B=2, N=3000, n_q=1, layers=("reuse",))
    S = H.build(wl, DEV, prefill_step=True)
    tk = S.topk.clone()
    tk[0, 0, 100:] = -1
    tk[1, 0, :] = -1  # window only
    L = S.layers[0]
    o = torch.empty(2, 1, 64, 512, device=DEV)
    lse = torch.empty(2, 1, 64, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_SPARSE_ATTN, 2, 1, 3000), dtype=torch.uint8, device=DEV)
    csa2.csa2_sparse_attn(L.q, tk, S.seq_len, S.cache.block_table, S.cache.n_pages, S.cache.main_pages,
                          S.cache.rings, L.ring_idx, o, lse, ws)
    _status_ok()
    tkn = tk.cpu().numpy()
    for b in range(2):
        ro, _ = H.oracle_attention(S, b, 0, 0, tkn[b, 0])
        H.check_attention(o[b, 0].cpu().numpy(), ro, H.TOL_ATTN_F32)


@pytest.mark.parametrize("B", [3, 300])
def test_sparse_attention_query_out_of_f16_range_sets_the_range_status(B):
    """A query element at 7e4 does not fit f16 (the tensor cores' operand
    type): the call records CSA2_ERR_DEVICE_RANGE; the other tokens' outputs
    stay right. B = 3 takes the split-and-merge path, 300 one CTA per token."""
    N = 3000
    wl = Workload(92, "t", "reuse", B=B, N=N, n_q=1, layers=("reuse",))
    S = H.build(wl, DEV, shuffle_seed=13, prefill_step=True)
    L = S.layers[0]
    q = L.q.clone()
    q[1, 0, 5, 17] = 7e4
    o = torch.empty(B, 1, 64, 512, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_SPARSE_ATTN, B, 1, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_sparse_attn(q, S.topk, S.seq_len, S.cache.block_table, S.cache.n_pages, S.cache.main_pages,
                          S.cache.rings, L.ring_idx, o, None, ws)
    assert csa2.csa2_check_device_status() == csa2.ERR_DEVICE_RANGE
    tk = S.topk.cpu().numpy()
    go = o.cpu().numpy()
    for b in (0, 2, B - 1):
        ro, _ = H.oracle_attention(S, b, 0, 0, tk[b, 0])
        H.check_attention(go[b, 0], ro, H.TOL_ATTN_F32)
    # The largest finite f16-representable bf16 below the limit is accepted.
    q[1, 0, 5, 17] = 65280.0
    csa2.csa2_sparse_attn(q, S.topk, S.seq_len, S.cache.block_table, S.cache.n_pages, S.cache.main_pages,
                          S.cache.rings, L.ring_idx, o, None, ws)
    _status_ok()


# ---- dispatcher ------------------------------------------------------------------------------

def test_decode_group_full_then_reuse_and_reindex_inheritance():
    """FULL -> REUSE (inherits FULL's top-k) -> REINDEX (inherits FULL's pool)
    -> REUSE (inherits REINDEX's top-k). Each layer has its own query and ring.
    A REUSE layer with FULL's top-k equals FULL's own attention when given the
    same query and ring (Reuse reproduces Full)."""
    wl = Workload(96, "t", "group", B=2, N=20000, n_q=2, layers=("full", "reuse", "reindex", "reuse"))
    S = H.build(wl, DEV, shuffle_seed=13, prefill_step=True)
    B, n_q, N = 2, 2, 20000
    for L in S.layers:
        if L.q_idx is not None:
            _quant_q(S, L)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_DECODE_LAYER, B, n_q, N), dtype=torch.uint8, device=DEV)
    pool = torch.empty(B, n_q, 2048, dtype=torch.int32, device=DEV)
    tk_full = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    tk_re = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    outs = [torch.empty(B, n_q, 64, 512, device=DEV) for _ in range(4)]
    c = S.cache
    common = dict(B=B, n_q=n_q, max_ctx=N, seq_len=S.seq_len, block_table=c.block_table, n_pages=c.n_pages,
                  main_pages=c.main_pages, idx_pages=c.idx_pages, rings=c.rings, ws=ws)
    L0, L1, L2, L3 = S.layers
    args = [
        csa2.layer_args(csa2.MODE_FULL, ring_idx=L0.ring_idx, q=L0.q, out=outs[0], q_idx_codes=L0.q_codes,
                        q_idx_scales=L0.q_scales, w=L0.w, pool=pool, topk=tk_full, **common),
        csa2.layer_args(csa2.MODE_REUSE, ring_idx=L1.ring_idx, q=L1.q, out=outs[1], **common),
        csa2.layer_args(csa2.MODE_REINDEX, ring_idx=L2.ring_idx, q=L2.q, out=outs[2], q_idx_codes=L2.q_codes,
                        q_idx_scales=L2.q_scales, w=L2.w, topk=tk_re, **common),
        csa2.layer_args(csa2.MODE_REUSE, ring_idx=L3.ring_idx, q=L3.q, out=outs[3], **common),
    ]
    csa2.csa2_decode_group(args)
    _status_ok()
    pl, tf, tr = pool.cpu().numpy(), tk_full.cpu().numpy(), tk_re.cpu().numpy()
    for b in range(B):
        for j in range(n_q):
            ref = H.oracle_full(S, b, j, 0)
            H.check_selection(tf[b, j], ref["topk"], lambda i: ref["scores"][i], 512, "full topk")
            rr = H.oracle_reindex(S, b, j, 2, pl[b, j])
            slot = {int(pl[b, j][i // 8]) * 8 + i % 8: rr["pos_scores"][i] for i in range(16384) if pl[b, j][i // 8] >= 0}
            H.check_selection(tr[b, j], rr["topk"], lambda p: slot[p], 512, "reindex topk")
            for li, tk in ((0, tf), (1, tf), (2, tr), (3, tr)):
                ro, _ = H.oracle_attention(S, b, j, li, tk[b, j])
                H.check_attention(outs[li][b, j].cpu().numpy(), ro, H.TOL_ATTN_F32)


# ---- device-side checks and host validation ------------------------------------------------

def test_unmapped_pages_set_the_bounds_status_without_faulting():
    wl = Workload(97, "t", "full", B=1, N=1000, n_q=1)
    S = H.build(wl, DEV, prefill_step=True)
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK
    bt = S.cache.block_table.clone()
    bt[0, 3] = -1
    L = S.layers[0]
    _quant_q(S, L)
    bm = torch.zeros(1, 1, 125, device=DEV)
    csa2.csa2_indexer_scan(L.q_codes, L.q_scales, L.w, S.seq_len, 1000, bt, S.cache.n_pages, S.cache.idx_pages, bm)
    assert csa2.csa2_check_device_status() == csa2.ERR_DEVICE_BOUNDS
    assert csa2.csa2_check_device_status() == csa2.OK  # cleared by the read
    tk = torch.full((1, 1, 512), -1, dtype=torch.int32, device=DEV)
    tk[0, 0, 0] = 5000  # a position past the query
    o = torch.empty(1, 1, 64, 512, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_SPARSE_ATTN, 1, 1, 1000), dtype=torch.uint8, device=DEV)
    csa2.csa2_sparse_attn(L.q, tk, S.seq_len, S.cache.block_table, S.cache.n_pages, S.cache.main_pages,
                          S.cache.rings, L.ring_idx, o, None, ws)
    assert csa2.csa2_check_device_status() == csa2.ERR_DEVICE_BOUNDS
    assert torch.isfinite(o).all()


def test_host_validation_errors():
    x = torch.zeros(16, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_quant_mxfp4(x[:, :8].contiguous().view(-1)[:8])
    assert e.value.status == csa2.ERR_INVALID_ARG
    wl = Workload(98, "t", "reuse", B=1, N=300, n_q=1, layers=("reuse",))
    S = H.build(wl, DEV, prefill_step=True)
    L = S.layers[0]
    o = torch.empty(1, 1, 64, 512, device=DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_sparse_attn(L.q, S.topk, S.seq_len, S.cache.block_table, S.cache.n_pages, S.cache.main_pages,
                              S.cache.rings, L.ring_idx, o, None, small)
    assert e.value.status == csa2.ERR_WORKSPACE


@pytest.mark.parametrize("N", [100000, 140000])
@pytest.mark.parametrize("weights", ["zero", "mixed_sign"])
def test_indexer_full_ties_and_mixed_sign_scores(weights, N):
    """All scores tied (zero head weights: the lowest blocks and positions win)
    and scores of both signs (negative head weights), at a context whose
    12,500 block maxima fit one CTA of the block selection and at one whose
    17,500 span several CTAs of a cluster."""
    B = 2
    wl = Workload(99, "t", "full", B=B, N=N, n_q=1)
    S = H.build(wl, DEV, shuffle_seed=17, prefill_step=True)
    L = S.layers[0]
    if weights == "zero":
        L.w.zero_()
        L.w_np[:] = 0
    else:
        L.w.mul_(2.0).sub_(1.0)
        L.w_np[:] = L.w.cpu().numpy()
    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)
    pool = torch.empty(B, 1, 2048, dtype=torch.int32, device=DEV)
    topk = torch.empty(B, 1, 512, dtype=torch.int32, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_FULL, B, 1, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_indexer_full(L.q_codes, L.q_scales, L.w, S.seq_len, N, S.cache.block_table, S.cache.n_pages,
                           S.cache.idx_pages, pool, topk, ws)
    gp, gt = pool.cpu().numpy(), topk.cpu().numpy()
    _status_ok()
    for b in range(B):
        if weights == "zero":
            assert gp[b, 0].tolist() == list(range(2048))
            assert gt[b, 0].tolist() == list(range(512))
        else:
            ref = H.oracle_full(S, b, 0)
            H.check_selection(gp[b, 0], ref["pool"], lambda i: ref["blockmax"][i], 2048, "pool")
            H.check_selection(gt[b, 0], ref["topk"], lambda i: ref["scores"][i], 512, "topk")
