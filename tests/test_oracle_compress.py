"""Pins of the oracle's compressed entries (encoder-side CSA2 at m = 2 tokens
per entry; the pages give the ratio, the state of an unfinished entry's tail
tokens and their compression weights, but no formula: per channel, the softmax
of the m tokens' compression logits weights their candidates, rounded once to
bf16). Checked against closed forms, special cases and invariants, with a
bf16 rounding written here from its definition (nearest, ties to even, from
the exact binary value)."""
import math
import struct

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def bf16_bits(v: float) -> int:
    """Round a double to bf16 (8 significant bits), nearest, ties to even,
    straight from its 52-bit mantissa; normal range only."""
    if v == 0.0:
        return 0x8000 if math.copysign(1.0, v) < 0 else 0
    u = struct.unpack("<Q", struct.pack("<d", v))[0]
    sign, exp, man = u >> 63, (u >> 52) & 0x7FF, u & ((1 << 52) - 1)
    m = man | (1 << 52)                     # 53 significant bits
    q, rem = divmod(m, 1 << 45)             # keep 8
    half = 1 << 44
    if rem > half or (rem == half and (q & 1)):
        q += 1
    if q == 1 << 8:
        q >>= 1
        exp += 1
    e8 = exp - 1023 + 127
    assert 1 <= e8 <= 254, "outside the normal bf16 range"
    return (sign << 15) | (e8 << 7) | (q & 0x7F)


def value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def rand_bf16(rng, shape, lo=2.0 ** -6, hi=8.0):
    mag = np.exp(rng.uniform(math.log(lo), math.log(hi), shape))
    sgn = np.where(rng.random(shape) < 0.5, -1.0, 1.0)
    return np.array([bf16_bits(float(v)) for v in (sgn * mag).ravel()], np.uint16).reshape(shape)


def test_rounding_helper_on_known_values():
    assert bf16_bits(1.0) == 0x3F80 and bf16_bits(-2.0) == 0xC000
    assert bf16_bits(1.0 + 2.0 ** -8) == 0x3F80          # tie -> even (down)
    assert bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (up)
    assert bf16_bits(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81


def test_equal_logits_give_the_rounded_mean():
    rng = np.random.default_rng(1)
    x = rand_bf16(rng, (200, 2, 64))
    z = np.tile(rand_bf16(rng, (200, 1, 64)), (1, 2, 1))  # both tokens share each channel's logit
    got = oracle.compress(x, z)
    for e in range(200):
        for c in range(64):
            mean = (value(x[e, 0, c]) + value(x[e, 1, c])) / 2.0   # exact in double
            assert got[e, c] == bf16_bits(mean) if mean != 0 else value(got[e, c]) == 0.0


def test_two_token_closed_form_is_a_logistic_weight():
    """x = (1, 0): the entry is exp(z0) / (exp(z0) + exp(z1)) = 1 / (1 + e^(z1 - z0))."""
    zs = [-6.0, -2.5, -1.0, -0.125, 0.0, 0.5, 1.0, 3.0, 7.0]
    x = np.array([[[bf16_bits(1.0)], [0]]] * len(zs), np.uint16)
    z = np.array([[[0], [bf16_bits(d) if d else 0]] for d in zs], np.uint16)
    got = oracle.compress(x, z)[:, 0]
    for d, g in zip(zs, got):
        assert g == bf16_bits(1.0 / (1.0 + math.exp(d))), d


def test_a_dominant_logit_selects_its_token():
    rng = np.random.default_rng(2)
    x = rand_bf16(rng, (50, 2, 32))
    z = np.zeros((50, 2, 32), np.uint16)
    z[:, 1, :] = bf16_bits(-300.0)
    assert np.array_equal(oracle.compress(x, z), x[:, 0, :])
    z[:, 1, :] = bf16_bits(300.0)
    assert np.array_equal(oracle.compress(x, z), x[:, 1, :])


def test_invariances_and_convex_hull():
    rng = np.random.default_rng(3)
    x = rand_bf16(rng, (100, 2, 48))
    # logits on a quarter grid in [-4, 4], so that a shift by 2 stays exact in bf16
    zq = rng.integers(-16, 17, (100, 2, 48)) / 4.0
    z = np.vectorize(bf16_bits)(zq).astype(np.uint16)
    base = oracle.compress(x, z)
    # the order of an entry's tokens does not matter
    assert np.array_equal(oracle.compress(x[:, ::-1].copy(), z[:, ::-1].copy()), base)
    # softmax is invariant to a common shift of the logits
    zs = np.vectorize(bf16_bits)(zq + 2.0).astype(np.uint16)
    assert np.array_equal(oracle.compress(x, zs), base)
    # every entry lies between its tokens' values
    lo = np.minimum(np.vectorize(value)(x[:, 0]), np.vectorize(value)(x[:, 1]))
    hi = np.maximum(np.vectorize(value)(x[:, 0]), np.vectorize(value)(x[:, 1]))
    v = np.vectorize(value)(base)
    assert ((v >= lo) & (v <= hi)).all()


def test_ratio_one_is_the_identity_and_entry_limits():
    rng = np.random.default_rng(4)
    x = rand_bf16(rng, (30, 1, 16))
    z = rand_bf16(rng, (30, 1, 16))
    assert np.array_equal(oracle.compress(x, z), x[:, 0, :])
    assert [oracle.entry_limit(t, 2) for t in range(6)] == [0, 1, 1, 2, 2, 3]
    assert [oracle.entry_limit(t, 1) for t in range(4)] == [1, 2, 3, 4]
