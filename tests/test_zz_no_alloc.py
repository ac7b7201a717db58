"""csa2_indexer_reindex_noalloc: the Reindex indexer for callers that cannot
allocate device memory (a plug-in under a framework that owns every
allocation, a decode loop that must not allocate mid-step). It keeps its
scores in the library's fixed device array instead of a caller workspace, so
its results must equal those of csa2_indexer_reindex on the same inputs, call
after call, even though every call reuses the same array.

Collected last on purpose (file name): if it fails, a run that stops at the
first failure has already run every other test.
"""
import pytest
import torch

from synth.workloads import Workload
from sparse_attention_fp4_mxfp4_gb300.workload import build

pytestmark = pytest.mark.gpu

import sparse_attention_fp4_mxfp4_gb300 as csa2  # noqa: E402

DEV = "cuda"


def _setup(index, B, n_q, N, m=1):
    wl = Workload(index, "noalloc", "reindex", B=B, N=N, n_q=n_q, layers=("reindex",), m=m)
    S = build(wl, DEV, shuffle_seed=index, prefill_step=True)
    L = S.layers[0]
    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)
    return S, L


def _with_workspace(S, L):
    B, n_q = S.B, S.n_q
    topk = torch.empty(B, n_q, 512, dtype=torch.int32, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_REINDEX, B, n_q, S.N), dtype=torch.uint8, device=DEV)
    csa2.csa2_indexer_reindex(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table, S.cache.n_pages,
                              S.cache.idx_pages, L.pool, topk, ws, m=S.m)
    return topk


def _no_alloc(S, L, topk=None):
    if topk is None:
        topk = torch.full((S.B, S.n_q, 512), -7, dtype=torch.int32, device=DEV)
    csa2.csa2_indexer_reindex_noalloc(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table,
                                      S.cache.n_pages, S.cache.idx_pages, L.pool, topk, m=S.m)
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


def test_no_alloc_reindex_at_two_tokens_per_entry():
    # The encoder side (m = 2): pools and top-k count entries, the causal
    # limit of a token is floor((t + 1) / 2) - 1.
    S, L = _setup(204, B=3, n_q=3, N=20001, m=2)
    ref = _with_workspace(S, L)
    got = _no_alloc(S, L)
    got_again = _no_alloc(S, L)
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK, csa2.device_status_message()
    assert torch.equal(got, ref) and torch.equal(got_again, ref)


def test_no_alloc_reindex_leaves_free_device_memory_unchanged():
    S, L = _setup(205, B=2, n_q=1, N=5000)
    topk = torch.empty(2, 1, 512, dtype=torch.int32, device=DEV)
    _no_alloc(S, L, topk)  # the first call on the device does the one-time set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _no_alloc(S, L, topk)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.equal(topk, _with_workspace(S, L))


def test_no_alloc_reindex_rejects_more_than_64_query_tokens():
    S, L = _setup(203, B=13, n_q=5, N=2000)  # 65 query tokens
    topk = torch.zeros(13, 5, 512, dtype=torch.int32, device=DEV)
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_indexer_reindex_noalloc(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table,
                                          S.cache.n_pages, S.cache.idx_pages, L.pool, topk)
    assert e.value.status == csa2.ERR_UNSUPPORTED
    assert "64" in str(e.value)
    # The same shape check as the workspace entry point: a ratio it rejects,
    # it rejects too, with the same status.
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_indexer_reindex_noalloc(L.q_codes, L.q_scales, L.w, S.seq_len, S.cache.block_table,
                                          S.cache.n_pages, S.cache.idx_pages, L.pool, topk, m=3)
    assert e.value.status == csa2.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(topk.abs().sum()) == 0  # nothing was launched
