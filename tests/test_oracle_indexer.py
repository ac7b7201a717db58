"""Pins of the oracle's hierarchical sparse indexer.

Inputs are built on the E2M1 grid with a +-6 in every 16-channel block, so the
MXFP4 round trip is exact (scale 1.0) and every score has a closed form in
exact rational arithmetic. The score definition is sum_h w_h * ReLU(q_h . k)
over 32 heads x 128 dims (head/dim counts from "DeepSeek V4.1: model
architecture and system design, a close reading" section 1; block size 8 and
2048 pool blocks from the same section and from "DeepSeek-V4.1-Flash: Pushing
the Limits of KV Cache Compression" section 3.4).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

H, D = 32, 128
GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])


def grid_rows(rng, n, dim=D):
    """Rows whose MXFP4 round trip is exact: grid values, a +-6 in every block."""
    v = rng.choice(GRID, size=(n, dim)) * rng.choice([-1, 1], size=(n, dim))
    v[:, ::16] = 6 * rng.choice([-1, 1], size=(n, dim // 16))
    return v


def to_bf16_bits(v):
    a = np.asarray(v, np.float32)
    u = a.view(np.uint32)
    assert (u & 0xFFFF == 0).all()
    return (u >> 16).astype(np.uint16)


def exact_scores(q, w, keys):
    """Exact rational scores (grid values times 2 are integers)."""
    qi = (q * 2).astype(np.int64)
    ki = (keys * 2).astype(np.int64)
    dots = ki @ qi.T  # [n, H], in units of 1/4
    out = []
    for row in dots:
        s = sum((Fraction(float(w[h])) * Fraction(int(d), 4) for h, d in enumerate(row) if d > 0),
                Fraction(0))
        out.append(s)
    return out


def make_case(seed, n):
    rng = np.random.default_rng(seed)
    q = grid_rows(rng, H)
    keys = grid_rows(rng, n)
    w = (2.0 ** rng.integers(-4, 3, size=H)).astype(np.float32)  # exact, distinct per head
    return q, w, keys


def lex_topk(scores, k):
    """Brute force: sort by (-score, index), take k, return ascending."""
    idx = sorted(range(len(scores)), key=lambda i: (-scores[i], i))[:k]
    return sorted(idx)


def test_scores_closed_form():
    q, w, keys = make_case(1, 700)
    r = oracle.full_indexer(to_bf16_bits(q), w, to_bf16_bits(keys), t=699)
    ex = exact_scores(q, w, keys)
    assert [Fraction(float(s)) for s in r["scores"]] == ex
    # The ReLU matters on this input: some head dot products are negative.
    assert ((keys * 2).astype(np.int64) @ (q * 2).astype(np.int64).T < 0).any()


def test_block_max_partial_block_and_causality():
    q, w, keys = make_case(2, 64)
    # Plant strong matches (k = q of the heaviest head) around block edges and past t.
    hb = int(np.argmax(w))
    for p in (7, 8, 23, 40):
        keys[p] = np.abs(q[hb]) * np.sign(q[hb])
    t = 37  # position 40 is in the future
    r = oracle.full_indexer(to_bf16_bits(q), w, to_bf16_bits(keys), t=t)
    ex = exact_scores(q, w, keys[: t + 1])
    assert len(r["scores"]) == t + 1
    want_bm = [max(ex[b * 8: min(t + 1, b * 8 + 8)]) for b in range((t + 8) // 8)]
    assert [Fraction(float(x)) for x in r["blockmax"]] == want_bm
    assert len(r["blockmax"]) == 5  # 38 causal positions -> 4 full blocks + 1 partial
    assert 40 not in set(r["topk"].tolist())


def test_topk_and_pool_brute_force_with_ties():
    q, w, keys = make_case(3, 20000)
    keys[5000:5100] = keys[100:200]  # exact duplicates -> tied scores
    t = 19999
    r = oracle.full_indexer(to_bf16_bits(q), w, to_bf16_bits(keys), t=t, n_pool=2048, k=512)
    ex = exact_scores(q, w, keys)
    assert r["topk"].tolist() == lex_topk(ex, 512)
    nb = (t + 8) // 8
    bm = [max(ex[b * 8:(b + 1) * 8]) for b in range(nb)]
    assert r["pool"].tolist() == lex_topk(bm, 2048)
    # The final top-512 lies inside the pool (the pages' candidate restriction).
    pool_pos = {b * 8 + j for b in r["pool"].tolist() for j in range(8)}
    assert set(r["topk"].tolist()) <= pool_pos


def test_small_context_takes_everything_and_pads():
    q, w, keys = make_case(4, 101)
    r = oracle.full_indexer(to_bf16_bits(q), w, to_bf16_bits(keys), t=100)
    assert r["topk"].tolist() == list(range(101)) + [-1] * (512 - 101)
    assert r["pool"].tolist() == list(range(13)) + [-1] * (2048 - 13)


def test_zero_weights_tie_everything_to_lowest_positions():
    q, w, keys = make_case(5, 30000)
    r = oracle.full_indexer(to_bf16_bits(q), np.zeros(H, np.float32), to_bf16_bits(keys), t=29999)
    assert r["topk"].tolist() == list(range(512))
    assert r["pool"].tolist() == list(range(2048))


def test_reindex_with_full_pool_reproduces_full_topk():
    """Full's top-512 over all causal positions equals the top-512 of its own
    pool (every block ranked above a global top-512 member holds a position
    that beats it), so Reindex with Full's query and pool gives Full's answer."""
    seed, t = 77, 40000
    keys = synth.normal(seed, synth.IDXKEY, 0, 0, t + 1, D)
    q = synth.normal(seed, synth.IDXQ, 0, t, 1, H * D).reshape(H, D)
    w = synth.uniform(seed, synth.W, 0, t, 1, H)[0]
    full = oracle.full_indexer(q, w, keys, t=t)
    re = oracle.reindex(q, w, keys, t=t, pool=full["pool"])
    assert re["topk"].tolist() == full["topk"].tolist()
    # Reindex's scores of pool slots equal Full's scores of those positions.
    ps = re["pos_scores"].reshape(-1, 8)
    for i, b in enumerate(full["pool"][:50]):
        np.testing.assert_array_equal(ps[i], full["scores"][b * 8: b * 8 + 8])


def test_reindex_scores_only_pool_positions_and_respects_causality():
    q, w, keys = make_case(6, 4000)
    t = 3990
    pool = np.full(2048, -1, np.int32)
    pool[:3] = [10, 100, 498]  # block 498 = positions 3984..3991, 3991 is in the future
    re = oracle.reindex(to_bf16_bits(q), w, to_bf16_bits(keys), t=t, pool=pool, k=512)
    cand = [p for b in (10, 100, 498) for p in range(8 * b, 8 * b + 8) if p <= t]
    assert re["topk"].tolist() == cand + [-1] * (512 - len(cand))
    assert np.isneginf(re["pos_scores"][2 * 8 + 7])
    assert np.isneginf(re["pos_scores"][3 * 8:]).all()
