"""Guard regions: every workspace and output buffer of the main calls sits
between two 4 KB canary regions filled with 0xA5, and each call must leave
both untouched. This is the bounds check that compute-sanitizer would give
(closed on this pool): a kernel writing past either end of a buffer it was
handed fails here, at sizes that exercise split attention, several tiles and
ragged tails. The results are compared with the unguarded calls' as well.
"""
import pytest
import torch

from synth.workloads import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu

import sparse_attention_fp4_mxfp4_gb300 as csa2  # noqa: E402

DEV = "cuda"
GUARD = 4096
CANARY = 0xA5


class Guarded:
    """A byte buffer with canary regions on both sides; .view(dtype, shape) is the usable middle."""

    def __init__(self, nbytes):
        self.nbytes = nbytes
        self.buf = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=DEV)

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        lo, hi = self.buf[:GUARD], self.buf[GUARD + self.nbytes:]
        return bool((lo == CANARY).all()) and bool((hi == CANARY).all())


def _bytes(dtype, shape):
    n = 1
    for d in shape:
        n *= d
    return n * torch.tensor([], dtype=dtype).element_size()


def _guarded(dtype, shape):
    g = Guarded(_bytes(dtype, shape))
    return g, g.view(dtype, shape)


def _status_ok():
    st = csa2.csa2_check_device_status()
    assert st == csa2.OK, csa2.device_status_message()


@pytest.mark.parametrize("B,n_q,N", [(2, 2, 5000), (3, 1, 40000)])
def test_full_indexer_and_split_attention_stay_inside_their_buffers(B, n_q, N):
    wl = Workload(95, "guards", "full", B=B, N=N, n_q=n_q)
    S = H.build(wl, DEV, shuffle_seed=3, prefill_step=True)
    L = S.layers[0]
    c = S.cache
    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)

    g_ws, ws = _guarded(torch.uint8, (csa2.csa2_workspace_bytes(csa2.OP_INDEXER_FULL, B, n_q, N),))
    g_pool, pool = _guarded(torch.int32, (B, n_q, 2048))
    g_topk, topk = _guarded(torch.int32, (B, n_q, 512))
    csa2.csa2_indexer_full(L.q_codes, L.q_scales, L.w, S.seq_len, N, c.block_table, c.n_pages, c.idx_pages,
                           pool, topk, ws)
    torch.cuda.synchronize()
    _status_ok()
    assert g_ws.intact() and g_pool.intact() and g_topk.intact()

    # The same call on plain buffers gives the same selections.
    pool2 = torch.empty(B, n_q, 2048, dtype=torch.int32, device=DEV)
    topk2 = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    ws2 = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_FULL, B, n_q, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_indexer_full(L.q_codes, L.q_scales, L.w, S.seq_len, N, c.block_table, c.n_pages, c.idx_pages,
                           pool2, topk2, ws2)
    assert torch.equal(pool, pool2) and torch.equal(topk, topk2)

    # Attention over few tokens splits each token's key chunks over several
    # work items and merges their partial outputs through the workspace.
    g_aws, aws = _guarded(torch.uint8, (csa2.csa2_workspace_bytes(csa2.OP_SPARSE_ATTN, B, n_q, N),))
    g_out, out = _guarded(torch.float32, (B, n_q, 64, 512))
    g_lse, lse = _guarded(torch.float32, (B, n_q, 64))
    csa2.csa2_sparse_attn(L.q, topk, S.seq_len, c.block_table, c.n_pages, c.main_pages, c.rings, L.ring_idx, out,
                          lse, aws)
    torch.cuda.synchronize()
    _status_ok()
    assert g_aws.intact() and g_out.intact() and g_lse.intact()
    out2 = torch.empty(B, n_q, 64, 512, dtype=torch.float32, device=DEV)
    lse2 = torch.empty(B, n_q, 64, dtype=torch.float32, device=DEV)
    aws2 = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_SPARSE_ATTN, B, n_q, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_sparse_attn(L.q, topk, S.seq_len, c.block_table, c.n_pages, c.main_pages, c.rings, L.ring_idx, out2,
                          lse2, aws2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_reindex_and_decode_stores_stay_inside_their_buffers():
    B, n_q, N = 4, 3, 20000
    wl = Workload(96, "guards", "reindex", B=B, N=N, n_q=n_q, layers=("reindex",))
    S = H.build(wl, DEV, shuffle_seed=4, prefill_step=False)
    L = S.layers[0]
    c = S.cache
    # The step's stores and the query codes, in one launch, into guarded code buffers.
    from sparse_attention_fp4_mxfp4_gb300.step import append_layers
    g_codes, codes = _guarded(torch.uint8, tuple(L.q_codes.shape))
    g_scales, scales = _guarded(torch.uint8, tuple(L.q_scales.shape))
    layers = append_layers(S)
    layers[0].update(q_codes=codes, q_scales=scales)
    csa2.csa2_decode_appends(S.step_latent, S.step_idx_key, S.step_seq, S.step_pos, c.block_table, c.main_pages,
                             c.idx_pages, layers)
    torch.cuda.synchronize()
    _status_ok()
    assert g_codes.intact() and g_scales.intact()
    ref_codes, ref_scales = csa2.csa2_quant_mxfp4(L.q_idx)
    assert torch.equal(codes, ref_codes) and torch.equal(scales, ref_scales)

    g_ws, ws = _guarded(torch.uint8, (csa2.csa2_workspace_bytes(csa2.OP_INDEXER_REINDEX, B, n_q, N),))
    g_topk, topk = _guarded(torch.int32, (B, n_q, 512))
    csa2.csa2_indexer_reindex(codes, scales, L.w, S.seq_len, c.block_table, c.n_pages, c.idx_pages, L.pool, topk,
                              ws)
    torch.cuda.synchronize()
    _status_ok()
    assert g_ws.intact() and g_topk.intact()
    topk2 = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    ws2 = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_REINDEX, B, n_q, N), dtype=torch.uint8, device=DEV)
    csa2.csa2_indexer_reindex(codes, scales, L.w, S.seq_len, c.block_table, c.n_pages, c.idx_pages, L.pool, topk2,
                              ws2)
    assert torch.equal(topk, topk2)
