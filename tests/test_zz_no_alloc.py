"""csa2_indexer_reindex_noalloc: the Reindex indexer for callers that cannot
allocate device memory (inside graph capture, under a framework that owns all
allocations, on an allocation-free decode path). It keeps its scores in the
library's fixed device array instead of a caller workspace, so its results must
equal those of csa2_indexer_reindex on the same inputs, call after call, even
though every call reuses the same array.

Collected last on purpose (file name): if it fails, a run that stops at the
first failure has already run every other test.
"""
import pytest
import torch

from synth.workloads import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu

import sparse_attention_fp4_mxfp4_gb300 as csa2  # noqa: E402

DEV = "cuda"


def _setup(index, B, n_q, N):
    wl = Workload(index, "noalloc", "reindex", B=B, N=N, n_q=n_q, layers=("reindex",))
    S = H.build(wl, DEV, shuffle_seed=index, prefill_step=True)
    L = S.layers[0]
    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)
    return S, L


def _with_workspace(S, L):
    B, n_q = S.B, S.n_q
    topk = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_REINDEX, B, n_q, S.N), dtype=torch.uint8, device=DEV)
    csa2.csa2_indexer_reindex(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table, S.cache.n_pages,
                              S.cache.idx_pages, L.pool, topk, ws)
    return topk


def _no_alloc(S, L):
    topk = torch.full((S.B, S.n_q, 512), -7, dtype=torch.int32, device=DEV)
    csa2.csa2_indexer_reindex_noalloc(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table,
                                      S.cache.n_pages, S.cache.idx_pages, L.pool, topk)
    return topk


def test_no_alloc_reindex_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    # Two different problems back to back: the second call finds the first
    # call's scores in the shared array and must not be affected by them.
    S1, L1 = _setup(201, B=4, n_q=2, N=30000)    # 8 query tokens, full pools
    S2, L2 = _setup(202, B=16, n_q=4, N=9000)    # 64 query tokens (the maximum), partial pools
    ref1 = _with_workspace(S1, L1)
    ref2 = _with_workspace(S2, L2)
    got1 = _no_alloc(S1, L1)
    got2 = _no_alloc(S2, L2)
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK, csa2.device_status_message()
    assert torch.equal(got1, ref1)
    assert torch.equal(got2, ref2)
    # And again in the other order.
    got2b = _no_alloc(S2, L2)
    got1b = _no_alloc(S1, L1)
    torch.cuda.synchronize()
    assert torch.equal(got1b, ref1) and torch.equal(got2b, ref2)


def test_no_alloc_reindex_rejects_more_than_64_query_tokens():
    S, L = _setup(203, B=13, n_q=5, N=2000)  # 65 query tokens
    topk = torch.zeros(13, 5, 512, dtype=torch.int32, device=DEV)
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_indexer_reindex_noalloc(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table,
                                          S.cache.n_pages, S.cache.idx_pages, L.pool, topk)
    assert e.value.status == csa2.ERR_UNSUPPORTED
    assert "64" in str(e.value)
    assert int(topk.abs().sum()) == 0  # nothing was launched
