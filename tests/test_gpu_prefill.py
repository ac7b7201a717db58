"""Parity of the prefill (chunked prefill) path with the CPU oracle: n_q new
tokens per sequence in one call, each attending causally ("DeepSeek V4.1:
model architecture and system design, a close reading" section 2.2 and
"DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" section 3.3:
the same indexer and attention over a run of query tokens).

What differs from decode: the Full scan serves the chunk in groups of 8 tokens
(ragged last group), every token keeps its own causal limit, and a token's
window is exactly positions max(0, t-127) .. t, taken from the chunk's own
E4M3 entries and from the ring state before the chunk. Afterwards the ring is
refilled with the chunk's last 128 entries ("SWA Bounded Replay", section 2.4
of the first page: the window state rebuilt from the last n_win tokens).

Criteria as for decode: block maxima rtol 2e-6; selections equal up to ties
within 1e-5 of the k-th score; attention within 2e-3 max-relative per (token,
head) (fp32) or that plus bf16 rounding; ring bytes bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth.workloads import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu

import sparse_attention_fp4_mxfp4_gb300 as csa2  # noqa: E402  (fails loudly without the library)

DEV = "cuda"


def _status_ok():
    st = csa2.csa2_check_device_status()
    assert st == csa2.OK, csa2.device_status_message()


def _tokens(n_q):
    """Sampled chunk tokens: both ends, group edges, the window's 128 boundary."""
    return sorted({j for j in (0, 1, 7, 8, 9, 126, 127, 128, 129, n_q // 2, n_q - 9, n_q - 2, n_q - 1)
                   if 0 <= j < n_q})


@pytest.mark.parametrize("N,n_q,B", [(200, 200, 1), (5003, 37, 2), (20000, 64, 1)])
def test_prefill_scan_block_max_every_token(N, n_q, B):
    wl = Workload(95, "t", "full", B=B, N=N, n_q=n_q)
    S = H.build(wl, DEV, shuffle_seed=17, prefill_step=True)
    L = S.layers[0]
    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)
    mb = (N + 7) // 8 + 3
    bm = torch.full((B, n_q, mb), 12345.0, device=DEV)
    csa2.csa2_indexer_scan(L.q_codes, L.q_scales, L.w, S.seq_len, N, S.cache.block_table, S.cache.n_pages,
                           S.cache.idx_pages, bm)
    got = bm.cpu().numpy()
    _status_ok()
    for b in range(B):
        keys = H.oracle_keys(S, b, N - 1)
        for j in range(n_q):
            ref = oracle.full_indexer(L.q_idx_u16[b, j], L.w_np[b, j], keys, S.t(j), want_scores=False)["blockmax"]
            nb = ref.size
            np.testing.assert_allclose(got[b, j, :nb], ref, rtol=2e-6, atol=1e-6 * max(1.0, np.abs(ref).max()),
                                       err_msg=f"token {j}")
            assert (got[b, j, nb:] == 12345.0).all(), f"token {j}: the scan wrote past its causal blocks"


def _check_ring_refilled(S, li, b):
    """Ring of (layer li, sequence b) holds the E4M3 of positions N-128 .. N-1."""
    lo = max(0, S.N - 128)
    ring = S.cache.rings[li * S.B + b].cpu().numpy()
    want = oracle.fp8_quant(synth.bf16_to_f32(synth.latent(S.wl.seed, b, lo, S.N - lo, tensor=synth.SWA + li)))
    assert np.array_equal(ring[np.arange(lo, S.N) % 128], want)


@pytest.mark.parametrize("N,n_q,B", [(300, 300, 1), (20000, 300, 2), (17000, 21, 1)])
def test_prefill_full_layer_step(N, n_q, B):
    """One Full layer over a prefill chunk, through the step bench.py times."""
    wl = Workload(96, "t", "full", B=B, N=N, n_q=n_q)
    S = H.build(wl, DEV, shuffle_seed=19)
    R = H.Runner(S, out_dtype=torch.float32, prefill=True)
    R.step()
    torch.cuda.synchronize()
    gp, gt = R.pool.cpu().numpy(), R.topk.cpu().numpy()
    go, gl = R.out[0].cpu().numpy(), R.lse[0].cpu().numpy()
    _status_ok()
    for b in range(B):
        keys = H.oracle_keys(S, b, N - 1)
        for j in _tokens(n_q):
            ref = H.oracle_full(S, b, j, keys=keys)
            H.check_selection(gp[b, j], ref["pool"], lambda i: ref["blockmax"][i], 2048, f"pool {j}")
            H.check_selection(gt[b, j], ref["topk"], lambda i: ref["scores"][i], 512, f"topk {j}")
            ro, rl = H.oracle_attention(S, b, j, 0, gt[b, j], exact_window=True)
            H.check_attention(go[b, j], ro, H.TOL_ATTN_F32)
            np.testing.assert_allclose(gl[b, j], rl, rtol=1e-5, atol=H.TOL_LSE)
        _check_ring_refilled(S, 0, b)


@pytest.mark.parametrize("N,n_q,B,out", [(3000, 260, 1, "bf16"), (900, 130, 3, "f32"), (129, 129, 2, "f32")])
def test_prefill_reuse_layer(N, n_q, B, out):
    """A Reuse layer over a prefill chunk with given top-k sets (ragged, -1
    padded for early tokens), windows that cross from the ring into the chunk."""
    wl = Workload(97, "t", "reuse", B=B, N=N, n_q=n_q, layers=("reuse",))
    S = H.build(wl, DEV, shuffle_seed=23)
    R = H.Runner(S, out_dtype=torch.float32 if out == "f32" else torch.bfloat16, prefill=True)
    R.step()
    torch.cuda.synchronize()
    go, gl = R.out[0].float().cpu().numpy(), R.lse[0].cpu().numpy()
    tk = S.topk.cpu().numpy()
    _status_ok()
    for b in range(B):
        for j in _tokens(n_q):
            ro, rl = H.oracle_attention(S, b, j, 0, tk[b, j], exact_window=True)
            H.check_attention(go[b, j], ro, H.TOL_ATTN_F32 if out == "f32" else H.TOL_ATTN_BF16)
            np.testing.assert_allclose(gl[b, j], rl, rtol=1e-5, atol=H.TOL_LSE)
        _check_ring_refilled(S, 0, b)


def test_prefill_group_through_the_dispatcher_matches_the_step():
    """csa2_decode_group with swa_chunk set (Full then Reuse) gives the same
    bytes as the step's separate calls."""
    B, N, n_q = 2, 18000, 40
    wl = Workload(98, "t", "group", B=B, N=N, n_q=n_q, layers=("full", "reuse"))
    S = H.build(wl, DEV, shuffle_seed=29)
    csa2.csa2_append_kv(S.step_latent, S.step_idx_key, S.step_seq, S.step_pos, S.cache.block_table,
                        S.cache.main_pages, S.cache.idx_pages)
    c = S.cache
    chunks = [csa2.csa2_quant_fp8_entries(S.step_swa[li]).view(B, n_q, 512) for li in range(2)]
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_DECODE_LAYER, B, n_q, N), dtype=torch.uint8, device=DEV)
    pool = torch.empty(B, n_q, 2048, dtype=torch.int32, device=DEV)
    topk = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    outs = [torch.empty(B, n_q, 64, 512, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    L0 = S.layers[0]
    csa2.csa2_quant_mxfp4(L0.q_idx, L0.q_codes, L0.q_scales)
    args = []
    for li, L in enumerate(S.layers):
        kw = dict(q_idx_codes=L0.q_codes, q_idx_scales=L0.q_scales, w=L0.w, pool=pool, topk=topk) if li == 0 else {}
        args.append(csa2.layer_args(csa2.MODE_FULL if li == 0 else csa2.MODE_REUSE, B=B, n_q=n_q, max_ctx=N,
                                    seq_len=S.seq_len, block_table=c.block_table, n_pages=c.n_pages,
                                    main_pages=c.main_pages, idx_pages=c.idx_pages, rings=c.rings,
                                    ring_idx=L.ring_idx, q=L.q, out=outs[li], ws=ws, swa_chunk=chunks[li], **kw))
    csa2.csa2_decode_group(args)
    torch.cuda.synchronize()
    _status_ok()
    got = [o.clone() for o in outs]
    R = H.Runner(S, out_dtype=torch.bfloat16, prefill=True)
    R.step()
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(R.topk, topk)
    for li in range(2):
        assert torch.equal(R.out[li].view(torch.int16), got[li].view(torch.int16)), f"layer {li}"


@pytest.mark.parametrize("n", [1, 40, 128, 200])
def test_ring_refill_from_the_last_entries(n):
    """csa2_ring_refill: the last min(n, 128) entries land in slot p % 128;
    every other slot keeps its bytes."""
    B, R = 3, 5
    g = torch.Generator().manual_seed(n)
    rings = torch.randint(0, 256, (R, 128, 512), dtype=torch.uint8, generator=g).to(DEV)
    before = rings.cpu().numpy().copy()
    seq_len = torch.tensor([n, n + 77, n + 1000], dtype=torch.int64, device=DEV)
    ring_idx = torch.tensor([4, 0, 2], dtype=torch.int32, device=DEV)
    x = torch.randn(B * n, 512, generator=g).to(torch.bfloat16).to(DEV)
    ent = csa2.csa2_quant_fp8_entries(x).view(B, n, 512)
    csa2.csa2_ring_refill(ent, seq_len, ring_idx, rings)
    got = rings.cpu().numpy()
    _status_ok()
    want_codes = oracle.fp8_quant(x.float().cpu().numpy().astype(np.float64)).reshape(B, n, 512)
    assert np.array_equal(ent.cpu().numpy(), want_codes)
    want = before.copy()
    for b, (sl, ri) in enumerate(zip(seq_len.tolist(), ring_idx.tolist())):
        for i in range(max(0, n - 128), n):
            want[ri, (sl - n + i) % 128] = want_codes[b, i]
    assert np.array_equal(got, want)


def test_ring_refill_equals_the_appended_history():
    """Bounded replay's ring rebuild from the last 128 tokens gives the ring
    that appending the whole history one token at a time leaves."""
    B, N = 2, 1000
    x = torch.randn(B, N, 512, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).to(DEV)
    inc = torch.zeros(B, 128, 512, dtype=torch.uint8, device=DEV)
    for p0 in range(0, N, 128):  # in order: later positions overwrite their slot
        n = min(128, N - p0)
        xi = x[:, p0:p0 + n].reshape(B * n, 512).contiguous()
        ridx = torch.arange(B, dtype=torch.int32, device=DEV).repeat_interleave(n)
        pos = torch.arange(p0, p0 + n, dtype=torch.int64, device=DEV).repeat(B)
        csa2.csa2_append_swa(xi, ridx, pos, inc)
    reb = torch.zeros_like(inc)
    last = csa2.csa2_quant_fp8_entries(x[:, N - 128:].reshape(B * 128, 512).contiguous()).view(B, 128, 512)
    csa2.csa2_ring_refill(last, torch.full((B,), N, dtype=torch.int64, device=DEV),
                          torch.arange(B, dtype=torch.int32, device=DEV), reb)
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(inc, reb)


@pytest.mark.parametrize("N,n_q,B", [(20000, 100, 1), (3000, 140, 2)])
def test_prefill_reindex_layer(N, n_q, B):
    """A Reindex layer over a prefill chunk: every token rescores its own pool
    (2048 blocks, fewer near the start) and attends with its exact window."""
    wl = Workload(101, "t", "reindex", B=B, N=N, n_q=n_q, layers=("reindex",))
    S = H.build(wl, DEV, shuffle_seed=41)
    R = H.Runner(S, out_dtype=torch.float32, prefill=True)
    R.step()
    torch.cuda.synchronize()
    gt = R.topk.cpu().numpy()
    go, gl = R.out[0].cpu().numpy(), R.lse[0].cpu().numpy()
    pools = S.layers[0].pool.cpu().numpy()
    _status_ok()
    for b in range(B):
        keys = H.oracle_keys(S, b, N - 1)
        for j in _tokens(n_q):
            ref = H.oracle_reindex(S, b, j, 0, pools[b, j], keys=keys)
            ps = ref["pos_scores"]
            slot = {int(pools[b, j][i // 8]) * 8 + i % 8: ps[i] for i in range(ps.size) if pools[b, j][i // 8] >= 0}
            H.check_selection(gt[b, j], ref["topk"], lambda p: slot[p], 512, f"reindex topk {j}")
            ro, rl = H.oracle_attention(S, b, j, 0, gt[b, j], exact_window=True)
            H.check_attention(go[b, j], ro, H.TOL_ATTN_F32)
            np.testing.assert_allclose(gl[b, j], rl, rtol=1e-5, atol=H.TOL_LSE)
        _check_ring_refilled(S, 0, b)
