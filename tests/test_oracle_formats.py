"""Pins of the oracle's number formats against things other than itself.

* hand-computed worked examples (tests/golden/*.txt, each citing the pages),
* torch's float8_e4m3fn conversion (round-to-nearest-even, no saturation) as an
  independent library routine for E4M3,
* an exact-rational brute force (fractions.Fraction) of "nearest E2M1 grid
  value, ties to the even code" for the block quantiser,
* the format range the pages print (448 x 6 = 2688).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _records(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [x.strip() for x in line.split("|")]


def test_e2m1_grid_definition():
    # E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit.
    want = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert [oracle.e2m1_value(c) for c in range(8)] == want
    assert [oracle.e2m1_value(c + 8) for c in range(8)] == [-x for x in want]


def test_e4m3_decode_matches_torch_all_bytes():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(i) for i in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2
    assert (got[~nan] == ref[~nan]).all()
    assert oracle.e4m3_value(0x7E) == 448.0


def test_e4m3_worked_examples():
    for x, byte in _records("e4m3_worked.txt"):
        assert oracle.e4m3_encode([float(x)])[0] == int(byte, 16), x


def _e4m3_boundary_inputs():
    """Every E4M3 value, every midpoint between neighbours, and 1 ulp around each."""
    vals = np.array(sorted({oracle.e4m3_value(i) for i in range(0x7F)}), np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    pts = np.concatenate([vals, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(-np.inf))
    allp = np.concatenate([pts, up, dn])
    return np.concatenate([allp, -allp]).astype(np.float32)


def test_e4m3_encode_matches_torch_rne_near_every_boundary():
    x = _e4m3_boundary_inputs()
    x = x[np.abs(x) < 464]  # torch does not saturate; beyond 464 it gives NaN
    got = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_matches_torch_on_random_bit_patterns():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 464)]
    got = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (got == ref).all()


def test_e4m3_saturates_at_format_max():
    x = np.array([464.0, 464.1, 500, 1e6, np.inf, -np.inf, 3.4e38], np.float32)
    got = oracle.e4m3_encode(x)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E]


def _bf16_exact(vals):
    a = np.asarray(vals, np.float32)
    u = a.view(np.uint32)
    assert (u & 0xFFFF == 0).all(), "golden inputs must be exact in bf16"
    return a


def test_mxfp4_worked_examples():
    for name, vin, scale, codes, deq in _records("mxfp4_worked.txt"):
        x = _bf16_exact([float(v) for v in vin.split()])
        c, s = oracle.mxfp4_quant(x)
        assert s[0] == int(scale, 16), name
        assert list(c) == [int(b, 16) for b in codes.split()], name
        d = oracle.mxfp4_dequant(c, s)
        assert list(d) == [float(v) for v in deq.split()], name


def test_mxfp4_format_range_2688():
    # The pages: the format represents magnitudes up to 448 x 6 = 2688.
    x = np.zeros(16, np.float32)
    x[3] = 2688.0
    c, s = oracle.mxfp4_quant(x)
    assert s[0] == 0x7E and oracle.e4m3_value(int(s[0])) == 448.0
    assert (c[1] >> 4) == 7
    assert oracle.mxfp4_dequant(c, s)[3] == 2688.0
    # Larger magnitudes saturate to the same 2688.
    x[3] = 1e5
    c, s = oracle.mxfp4_quant(x)
    assert oracle.mxfp4_dequant(c, s)[3] == 2688.0


E2M1_GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
             Fraction(4), Fraction(6)]


def _brute_block(v):
    """Exact-rational reference of one block: torch RNE for the scale, brute
    nearest-grid search (ties to the even code) for the elements."""
    amax = np.float32(np.max(np.abs(v)))
    s32 = np.float32(amax / np.float32(6.0))
    if s32 >= 448:
        sb = 0x7E
    else:
        sb = int(torch.tensor([float(s32)], dtype=torch.float32).to(torch.float8_e4m3fn)
                 .view(torch.uint8)[0])
    sf = Fraction(oracle.e4m3_value(sb))
    codes = []
    for x in v:
        if sf == 0:
            codes.append(0)
            continue
        r = Fraction(float(abs(x))) / sf
        d = [abs(r - g) for g in E2M1_GRID]
        best = min(d)
        cands = [k for k in range(8) if d[k] == best]
        k = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        if k and x < 0:
            k |= 8
        codes.append(k)
    packed = [codes[2 * i] | (codes[2 * i + 1] << 4) for i in range(8)]
    return sb, packed


def _random_blocks(rng, n):
    out = []
    for i in range(n):
        kind = i % 4
        mag = 2.0 ** rng.integers(-12, 14)
        v = rng.standard_normal(16) * mag
        if kind == 1:  # put exact grid midpoints of a power-of-two scale in the block
            sf = 2.0 ** rng.integers(-8, 8)
            v = rng.choice([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, 6, -5, -0.25], 16) * sf
            v[0] = 6 * sf
        elif kind == 2:  # heavy outlier
            v[rng.integers(16)] *= 40
        v = v.astype(np.float32)
        v = (v.view(np.uint32) & 0xFFFF0000).view(np.float32)  # bf16-exact like real inputs
        out.append(v)
    return out


def test_mxfp4_quant_matches_exact_rational_brute_force():
    rng = np.random.default_rng(11)
    blocks = _random_blocks(rng, 3000)
    x = np.concatenate(blocks)
    c, s = oracle.mxfp4_quant(x)
    for i, v in enumerate(blocks):
        sb, packed = _brute_block(v)
        assert s[i] == sb, (i, v)
        assert list(c[8 * i: 8 * i + 8]) == packed, (i, v)


def test_fp8_roundtrip_is_torch_rne_for_latent_magnitudes():
    # Sliding-window entries are RMSNormed latents, |x| <= 22.6, far below 448:
    # FP8 quantisation is plain RNE there.
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(200000) * 4).astype(np.float32)
    got = oracle.fp8_dequant(oracle.fp8_quant(x))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert (got == ref).all()


@pytest.mark.parametrize("plant", ["sign_dropped", "tie_up"])
def test_planted_quantiser_mistakes_are_caught(plant):
    """Mistakes of the kind a quantiser plausibly has change at least one
    worked-example byte, so the goldens above would fail."""
    recs = list(_records("mxfp4_worked.txt"))
    name, vin, scale, codes, deq = [r for r in recs if r[0] == "ties"][0]
    x = _bf16_exact([float(v) for v in vin.split()])
    c, _ = oracle.mxfp4_quant(x)
    if plant == "sign_dropped":
        c = c & 0x77
    else:  # round ties up instead of to even
        c = c.copy()
        c[1] = (c[1] & 0xF0) | 3  # 0.75 -> code 1 ... use an off-by-one code
    assert list(c) != [int(b, 16) for b in codes.split()]
