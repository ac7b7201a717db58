"""Parity of the encoder-side CSA2 path (m = 2 tokens per entry) with the CPU
oracle ("DeepSeek V4.1: model architecture and system design, a close
reading" section 1 and "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
Compression" section 3.1: the encoder's CSA2 layers compress 2 tokens per
entry; "DeepSeek-V4 model structure (7)", KV cache of hybrid attention: an
unfinished entry's tail tokens and their compression weights are state).

The compressor's entries are built on the GPU in fp64 and rounded once to
bf16 like the oracle's, so the stored MXFP4 codes and scales must be
bit-exact. The indexer and attention then work in entry space: a token at
position t sees entries 0 .. floor((t + 1) / 2) - 1, its window stays the
last 128 tokens. Criteria as for decode.
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


def _inputs(seed, b, p0, n):
    lat = synth.latent(seed, b, p0, n)
    lg = synth.normal(seed, synth.KVGATE, b, p0, n, 512)
    key = synth.normal(seed, synth.IDXKEY, b, p0, n, 128)
    kg = synth.normal(seed, synth.IDXGATE, b, p0, n, 128)
    return lat, lg, key, kg


@pytest.mark.parametrize("N,splits", [(1, (1,)), (2, (1, 1)), (9, (3, 1, 5)), (300, (1, 2, 7, 64, 226)),
                                      (1001, (500, 1, 500))])
def test_compress_append_pages_and_tail_bit_exact(N, splits):
    """Tokens arrive in calls of the given sizes (all sequences in each call);
    every complete entry's stored bytes equal the oracle's compression +
    MXFP4, and the tail holds the pending token."""
    from sparse_attention_fp4_mxfp4_gb300.cache import PagedCache
    assert sum(splits) == N
    B, m, seed = 3, 2, 77
    cache = PagedCache(B, (N + 1) // 2, device=DEV, shuffle_seed=5)
    tail = torch.zeros(B, m - 1, 1280, dtype=torch.bfloat16, device=DEV)
    p0 = 0
    for n in splits:
        parts = [_inputs(seed, b, p0, n) for b in range(B)]
        cat = [H.u16_to_bf16(np.concatenate([pr[i] for pr in parts]), DEV) for i in range(4)]
        seq = torch.arange(B, dtype=torch.int32, device=DEV).repeat_interleave(n)
        pos = torch.arange(p0, p0 + n, dtype=torch.int64, device=DEV).repeat(B)
        csa2.csa2_compress_append(cat[0], cat[1], cat[2], cat[3], seq, pos, m, tail, cache.block_table,
                                  cache.main_pages, cache.idx_pages)
        p0 += n
    torch.cuda.synchronize()
    _status_ok()
    E = N // m
    for b in range(B):
        lat, lg, key, kg = _inputs(seed, b, 0, N)
        if E:
            ent = oracle.compress(lat[: E * m].reshape(E, m, 512), lg[: E * m].reshape(E, m, 512))
            kent = oracle.compress(key[: E * m].reshape(E, m, 128), kg[: E * m].reshape(E, m, 128))
            mc, ms = H.unpack_main(cache, b, np.arange(E))
            rc, rs = oracle.mxfp4_quant(synth.bf16_to_f32(ent))
            assert np.array_equal(mc, rc) and np.array_equal(ms, rs)
            ic, is_ = H.unpack_idx(cache, b, np.arange(E))
            kc, ks = oracle.mxfp4_quant(synth.bf16_to_f32(kent))
            assert np.array_equal(ic, kc) and np.array_equal(is_, ks)
        if N % m:
            row = H.bf16_to_u16(tail[b, 0])
            want = np.concatenate([lat[N - 1], lg[N - 1], key[N - 1], kg[N - 1]])
            assert np.array_equal(row, want), "tail does not hold the pending token"


def test_ratio_one_compress_append_equals_append_kv():
    from sparse_attention_fp4_mxfp4_gb300.cache import PagedCache
    B, N, seed = 2, 700, 78
    a = PagedCache(B, N, device=DEV, shuffle_seed=1)
    c = PagedCache(B, N, device=DEV, shuffle_seed=1)
    parts = [_inputs(seed, b, 0, N) for b in range(B)]
    cat = [H.u16_to_bf16(np.concatenate([pr[i] for pr in parts]), DEV) for i in range(4)]
    seq = torch.arange(B, dtype=torch.int32, device=DEV).repeat_interleave(N)
    pos = torch.arange(N, dtype=torch.int64, device=DEV).repeat(B)
    csa2.csa2_append_kv(cat[0], cat[2], seq, pos, a.block_table, a.main_pages, a.idx_pages)
    csa2.csa2_compress_append(cat[0], cat[1], cat[2], cat[3], seq, pos, 1, None, c.block_table, c.main_pages,
                              c.idx_pages)
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(a.main_pages, c.main_pages) and torch.equal(a.idx_pages, c.idx_pages)


def _tokens(n_q):
    return sorted({j for j in (0, 1, 2, n_q // 2, n_q - 2, n_q - 1) if 0 <= j < n_q})


@pytest.mark.parametrize("N,n_q,B,prefill", [(40001, 1, 2, False), (40000, 2, 1, False), (4000, 3, 2, False),
                                             (36000, 150, 1, True), (257, 257, 1, True)])
def test_encoder_full_layer(N, n_q, B, prefill):
    """A Full layer at m = 2 through the step bench.py times: pool, top-512
    and attention of sampled tokens against the oracle in entry space."""
    wl = Workload(99, "t", "full", B=B, N=N, n_q=n_q, m=2, prefill=prefill)
    S = H.build(wl, DEV, shuffle_seed=31)
    R = H.Runner(S, out_dtype=torch.float32, prefill=prefill)
    R.step()
    torch.cuda.synchronize()
    gp, gt = R.pool.cpu().numpy(), R.topk.cpu().numpy()
    go, gl = R.out[0].cpu().numpy(), R.lse[0].cpu().numpy()
    _status_ok()
    for b in range(B):
        keys = H.oracle_keys(S, b, N - 1)
        for j in _tokens(n_q):
            n_ent = H.entries_seen(S, S.t(j))
            if n_ent == 0:
                assert (gp[b, j] == -1).all() and (gt[b, j] == -1).all()
            else:
                ref = H.oracle_full(S, b, j, keys=keys[:n_ent])
                H.check_selection(gp[b, j], ref["pool"], lambda i: ref["blockmax"][i], 2048, f"pool {j}")
                H.check_selection(gt[b, j], ref["topk"], lambda i: ref["scores"][i], 512, f"topk {j}")
            ro, rl = H.oracle_attention(S, b, j, 0, gt[b, j], exact_window=prefill)
            H.check_attention(go[b, j], ro, H.TOL_ATTN_F32)
            np.testing.assert_allclose(gl[b, j], rl, rtol=1e-5, atol=H.TOL_LSE)


def test_encoder_group_through_the_dispatcher():
    """Full then Reuse at m = 2 via csa2_decode_group (tokens_per_entry = 2)
    gives the step's bytes; the Reuse layer's attention matches the oracle."""
    B, N, n_q = 2, 30000, 2
    wl = Workload(100, "t", "group", B=B, N=N, n_q=n_q, layers=("full", "reuse"), m=2)
    S = H.build(wl, DEV, shuffle_seed=37, prefill_step=True)
    c = S.cache
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_DECODE_LAYER, B, n_q, N), dtype=torch.uint8, device=DEV)
    pool = torch.empty(B, n_q, 2048, dtype=torch.int32, device=DEV)
    topk = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    outs = [torch.empty(B, n_q, 64, 512, dtype=torch.float32, device=DEV) for _ in range(2)]
    L0 = S.layers[0]
    csa2.csa2_quant_mxfp4(L0.q_idx, L0.q_codes, L0.q_scales)
    args = []
    for li, L in enumerate(S.layers):
        kw = dict(q_idx_codes=L0.q_codes, q_idx_scales=L0.q_scales, w=L0.w, pool=pool, topk=topk) if li == 0 else {}
        args.append(csa2.layer_args(csa2.MODE_FULL if li == 0 else csa2.MODE_REUSE, B=B, n_q=n_q, max_ctx=N,
                                    seq_len=S.seq_len, block_table=c.block_table, n_pages=c.n_pages,
                                    main_pages=c.main_pages, idx_pages=c.idx_pages, rings=c.rings,
                                    ring_idx=L.ring_idx, q=L.q, out=outs[li], ws=ws, m=2, **kw))
    csa2.csa2_decode_group(args)
    torch.cuda.synchronize()
    _status_ok()
    got = [o.clone() for o in outs]
    tk = topk.cpu().numpy()
    R = H.Runner(S, out_dtype=torch.float32)
    R.step()
    torch.cuda.synchronize()
    _status_ok()
    assert torch.equal(R.topk, topk)
    for li in range(2):
        assert torch.equal(R.out[li], got[li]), f"layer {li}"
    for b in range(B):
        for j in range(n_q):
            ro, rl = H.oracle_attention(S, b, j, 1, tk[b, j])
            H.check_attention(got[1][b, j].cpu().numpy(), ro, H.TOL_ATTN_F32)
