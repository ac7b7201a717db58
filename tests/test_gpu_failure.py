"""Failure detection on the GPU without a fault: a bounded wait inside a kernel
that runs out records CSA2_ERR_DEVICE_TIMEOUT, the kernel still returns (its
copies and tensor-core work drained, its tensor memory released), and the
next call on the same stream computes the right result.

csa2_debug_force_wait_timeout makes the waits at one internal site give up at
once, exactly as if their time limit had passed; nothing is left waiting for
a flag that no one sets, and no GPU fault is involved.
"""
import pytest
import torch

from synth.workloads import Workload
from tests import harness as H

pytestmark = pytest.mark.gpu

import sparse_attention_fp4_mxfp4_gb300 as csa2  # noqa: E402

DEV = "cuda"
SITE_INDEXER_MMA_WAIT = 210  # the indexer's tensor-core issuer waiting for a tile's copy


@pytest.fixture()
def full_setup():
    wl = Workload(0, "timeout", "full", B=3, N=20000, n_q=1)
    S = H.build(wl, DEV, shuffle_seed=7, prefill_step=True)
    L = S.layers[0]
    csa2.csa2_quant_mxfp4(L.q_idx, L.q_codes, L.q_scales)
    assert csa2.csa2_check_device_status() == csa2.OK
    yield S, L
    csa2.csa2_debug_force_wait_timeout(0)


def _scan(S, L, fill=-7.0):
    c = S.cache
    mb = (S.N + 7) // 8
    bm = torch.full((S.B, S.n_q, mb), fill, dtype=torch.float32, device=DEV)
    csa2.csa2_indexer_scan(L.q_codes, L.q_scales, L.w, S.seq_len, S.N, c.block_table, c.n_pages, c.idx_pages, bm)
    return bm


def _reindex(S, L, pool):
    c = S.cache
    topk = torch.full((S.B, S.n_q, 512), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(csa2.csa2_workspace_bytes(csa2.OP_INDEXER_REINDEX, S.B, S.n_q, S.N), dtype=torch.uint8,
                     device=DEV)
    csa2.csa2_indexer_reindex(L.q_codes, L.q_scales, L.w, S.seq_len, c.block_table, c.n_pages, c.idx_pages, pool,
                              topk, ws)
    return topk


def test_scan_wait_timeout_is_reported_and_the_next_call_is_right(full_setup):
    S, L = full_setup
    ref = _scan(S, L)
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK
    csa2.csa2_debug_force_wait_timeout(SITE_INDEXER_MMA_WAIT)
    try:
        aborted = _scan(S, L)
        torch.cuda.synchronize()  # returns: the kernel did not hang
        st = csa2.csa2_check_device_status()
    finally:
        csa2.csa2_debug_force_wait_timeout(0)
    assert st == csa2.ERR_DEVICE_TIMEOUT
    msg = csa2.device_status_message()
    assert "indexer" in msg and str(SITE_INDEXER_MMA_WAIT) in msg
    # No tile was scored: every block maximum keeps its fill value.
    assert bool((aborted == -7.0).all())
    # The status was cleared by the read; the same call on the same stream is right again.
    again = _scan(S, L)
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK
    assert torch.equal(again, ref)


def test_pool_rescore_wait_timeout_is_reported_and_the_next_call_is_right(full_setup):
    S, L = full_setup
    pool = torch.empty(S.B, S.n_q, 2048, dtype=torch.int32, device=DEV)
    csa2.csa2_block_topk(_scan(S, L), S.seq_len, pool)
    ref = _reindex(S, L, pool)
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK
    csa2.csa2_debug_force_wait_timeout(SITE_INDEXER_MMA_WAIT)
    try:
        _reindex(S, L, pool)
        torch.cuda.synchronize()
        st = csa2.csa2_check_device_status()
    finally:
        csa2.csa2_debug_force_wait_timeout(0)
    assert st == csa2.ERR_DEVICE_TIMEOUT
    again = _reindex(S, L, pool)
    torch.cuda.synchronize()
    assert csa2.csa2_check_device_status() == csa2.OK
    assert torch.equal(again, ref)
    # And the selection is the oracle's (up to ties).
    tk = again.cpu().numpy()
    for b in range(S.B):
        r = H.oracle_full(S, b, 0)
        H.check_selection(tk[b, 0], r["topk"], lambda i: r["scores"][i], 512, f"topk {b}")


def test_forced_timeout_site_rejects_negative():
    with pytest.raises(csa2.Csa2Error) as e:
        csa2.csa2_debug_force_wait_timeout(-1)
    assert e.value.status == csa2.ERR_INVALID_ARG
