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
import pytest
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


# ---- output de-rotation ---------------------------------------------------------------

def _rotary_as_complex(rows):
    r = np.asarray(rows, np.float64)[..., 448:]
    return r[..., 0::2] + 1j * r[..., 1::2]


def test_derotation_is_complex_multiplication_by_the_inverse_phase():
    """Pairs (448+2i, 449+2i) as complex numbers x0 + i x1: rotating back by
    position t multiplies pair i by exp(-i t theta_i), theta_i = 10000^(-2i/64)
    (numpy's complex exponential, not the oracle's cos/sin)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 512))
    for t in (1, 7, 4095, 1 << 20):
        got = oracle.output_derotate(x, t)
        theta = 10000.0 ** (-2.0 * np.arange(32) / 64.0)
        want = _rotary_as_complex(x) * np.exp(-1j * t * theta)
        # t * theta reaches 1e6 rad, whose double has an ulp of 1.2e-10: the two
        # routes may round the angle differently by that much (|x| < 5 here).
        np.testing.assert_allclose(_rotary_as_complex(got), want, rtol=0, atol=1e-9)
        assert np.array_equal(got[:, :448], x[:, :448])  # the other channels are untouched


def test_derotation_worked_values_and_group_laws():
    x = np.zeros((1, 512))
    x[0, 448] = 1.0  # pair 0, theta_0 = 1
    y = oracle.output_derotate(x, 1)
    assert y[0, 448] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert y[0, 449] == pytest.approx(-math.sin(1.0), abs=1e-15)
    rng = np.random.default_rng(4)
    r = rng.standard_normal((3, 512))
    assert np.array_equal(oracle.output_derotate(r, 0), r)  # position 0: identity
    a = oracle.output_derotate(oracle.output_derotate(r, 300), 700)
    b = oracle.output_derotate(r, 1000)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)  # rotations compose
    pr = r[:, 448:].reshape(3, 32, 2)
    pd = oracle.output_derotate(r, 12345)[:, 448:].reshape(3, 32, 2)
    np.testing.assert_allclose(np.hypot(pd[..., 0], pd[..., 1]), np.hypot(pr[..., 0], pr[..., 1]), rtol=1e-13)
