"""Pins of the oracle's sparse attention.

When the context has at most 512 entries the top-k is every position, so the
method reduces to plain dense softmax attention over all main entries plus the
window entries; torch's scaled_dot_product_attention (fp64, CPU) is the
independent reference there. K = V = the 512-channel latent with 64 query
heads ("DeepSeek V4.1: model architecture and system design, a close reading"
section 1; "DeepSeek-V4 model structure (7): structure decides the system",
closing summary on K = V single-head MQA over top-k plus 128 window entries).
"""
import math

import numpy as np
import torch

import oracle
import synth

HQ, D = 64, 512
TAU = 1.0 / math.sqrt(512)


def _dense_case(seed, n_ctx, t):
    main = synth.latent(seed, 0, 0, n_ctx)
    win_pos = oracle.window_positions(t, n_ctx, 128)
    win = synth.latent(seed, 0, 0, n_ctx, tensor=synth.SWA)[win_pos]
    q = synth.normal(seed, synth.Q, 0, t, 1, HQ * D).reshape(HQ, D)
    return q, main[: t + 1], win


def test_dense_case_equals_torch_sdpa():
    q, main, win = _dense_case(5, 300, 299)
    out, lse = oracle.sparse_attention(q, main, win, TAU)
    # Dequantised keys: MXFP4 via the (separately pinned) oracle codec; FP8 via torch.
    c, s = oracle.mxfp4_quant(synth.bf16_to_f32(main))
    k_main = oracle.mxfp4_dequant(c, s)
    k_win = torch.from_numpy(synth.bf16_to_f32(win)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    K = torch.from_numpy(np.concatenate([k_main, k_win]))
    Q = torch.from_numpy(synth.bf16_to_f32(q).astype(np.float64))
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q[:, None, :], K[None].expand(HQ, -1, -1), K[None].expand(HQ, -1, -1), scale=TAU)[:, 0]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp(TAU * Q @ K.T, dim=1).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)
    assert K.shape[0] == 300 + 128


def test_single_key_returns_that_key():
    q, main, _ = _dense_case(6, 10, 9)
    out, lse = oracle.sparse_attention(q, main[3:4], np.zeros((0, D), np.uint16), TAU)
    c, s = oracle.mxfp4_quant(synth.bf16_to_f32(main[3:4]))
    k = oracle.mxfp4_dequant(c, s)[0]
    np.testing.assert_array_equal(out, np.broadcast_to(k, (HQ, D)))
    np.testing.assert_allclose(lse, TAU * synth.bf16_to_f32(q).astype(np.float64) @ k, rtol=1e-13)


def test_duplicated_keys_count_twice():
    # A position that is both in the top-k and in the window is attended twice
    # (once as FP4, once as FP8): duplicates are kept, which shifts the LSE by ln 2
    # when every key appears twice.
    q, main, _ = _dense_case(7, 40, 39)
    o1, l1 = oracle.sparse_attention(q, main, np.zeros((0, D), np.uint16), TAU)
    o2, l2 = oracle.sparse_attention(q, np.concatenate([main, main]), np.zeros((0, D), np.uint16), TAU)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2 - l1, math.log(2), rtol=1e-12)


def test_output_is_convex_combination_of_keys():
    q, main, win = _dense_case(8, 200, 199)
    out, _ = oracle.sparse_attention(q, main, win, TAU)
    c, s = oracle.mxfp4_quant(synth.bf16_to_f32(main))
    K = np.concatenate([oracle.mxfp4_dequant(c, s), oracle.fp8_dequant(oracle.fp8_quant(synth.bf16_to_f32(win)))])
    assert (out <= K.max(0) + 1e-12).all() and (out >= K.min(0) - 1e-12).all()


def test_window_positions_rule():
    # Ring of the last 128 positions of a sequence of N entries; query t sees
    # positions max(0, t-127, N-128) .. t.
    N = 1000
    assert oracle.window_positions(N - 1, N).tolist() == list(range(N - 128, N))
    assert oracle.window_positions(N - 6, N).tolist() == list(range(N - 128, N - 5))  # 123 entries
    assert oracle.window_positions(5, 6).tolist() == list(range(0, 6))
    assert len(oracle.window_positions(N - 6, N)) == 123
