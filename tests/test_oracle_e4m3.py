"""Pins for the oracle's E4M3 decoder and encoder (CPU only).

What pins them, besides the oracle itself:
  * torch's own float8_e4m3fn dtype (a library routine) decodes all 256 codes
    and rounds fp32 to the nearest E4M3 value in the range where the pages'
    rules and OCP E4M3FN coincide;
  * fixed points the pages state (448 <-> 0x7E, zero, saturation of NaN/Inf,
    flush below 2^-6), stored in tests/golden/e4m3_encode_specials.txt;
  * exhaustive round trip over all codes, RNE ties, carries and overflow;
  * a brute-force nearest-value search written with exact rationals.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "e4m3_encode_specials.txt")


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_float8_all_codes(orc):
    ours = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = torch_decode_all()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_page_facts(orc):
    # bias 7, 448 the largest finite value, 2^-6 the smallest normal
    assert orc.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert orc.e4m3_decode(np.uint8(0xFE)) == -448.0
    assert orc.e4m3_decode(np.uint8(0x38)) == 1.0
    assert orc.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6
    assert orc.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9
    assert orc.e4m3_decode(np.uint8(0x00)) == 0.0
    vals = orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(vals) > 0), "positive codes must increase"


def test_encode_golden_specials(orc):
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            bits_s, byte_s = line.split()[:2]
            got = orc.e4m3_encode_bits(np.array([int(bits_s, 16)],
                                                dtype=np.uint32))[0]
            assert got == int(byte_s, 16), line
            n += 1
    assert n >= 30


def test_encode_exhaustive_round_trip(orc):
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.e4m3_decode(codes)
    finite = ~np.isnan(vals)
    enc = orc.e4m3_encode(vals[finite].astype(np.float32))
    c = codes[finite]
    normal = ((c & 0x78) != 0)  # exponent field 1..15
    assert np.array_equal(enc[normal], c[normal])
    assert normal.sum() == 238  # 0x08..0x7E and 0x88..0xFE
    # +-0 -> 0x00; E4M3 subnormals (exponent field 0) are flushed to 0x00
    assert np.all(enc[~normal] == 0)
    # 0x7F / 0xFF (NaN codes) never come out of the encoder
    big = np.float32(480.0)
    assert orc.e4m3_encode(big) == 0x7E
    assert orc.e4m3_encode(-big) == 0xFE


def test_encode_never_emits_nan_codes(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64)
    enc = orc.e4m3_encode_bits(bits.astype(np.uint32))
    assert not np.any(enc == 0x7F)
    assert not np.any(enc == 0xFF)


def test_encode_all_midpoints_round_to_even(orc):
    vals = orc.e4m3_decode(np.arange(0x08, 0x7F, dtype=np.uint8))
    for i in range(len(vals) - 1):
        mid = np.float32((vals[i] + vals[i + 1]) / 2)
        assert float(mid) == (vals[i] + vals[i + 1]) / 2  # exact in fp32
        lo_code = 0x08 + i
        want = lo_code if lo_code % 2 == 0 else lo_code + 1
        assert orc.e4m3_encode(mid) == want, (i, float(mid))
        assert orc.e4m3_encode(-mid) == want | 0x80


def test_encode_overflow_band(orc):
    for v in list(range(447, 481)) + [463.99, 464.0, 464.01, 479.9, 495.9,
                                       496.0, 1e30, 3.4e38]:
        assert orc.e4m3_encode(np.float32(v)) == 0x7E, v
        assert orc.e4m3_encode(np.float32(-v)) == 0xFE, v


def test_encode_matches_torch_rne_in_normal_range(orc):
    """In [2^-6, 464) the pages' rules are plain RNE to the nearest finite
    E4M3FN value, which is what torch's fp32 -> float8_e4m3fn cast does."""
    rng = np.random.default_rng(11)
    lo = np.float32(2.0 ** -6).view(np.uint32)
    hi = np.float32(464.0).view(np.uint32)
    bits = rng.integers(int(lo), int(hi), size=1_000_000, dtype=np.int64)
    bits = bits.astype(np.uint32)
    sign = (rng.integers(0, 2, size=bits.size) << 31).astype(np.uint32)
    bits = bits | sign
    x = bits.view(np.float32)
    ours = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_monotone_on_positive_bit_patterns(orc):
    # every 997th positive fp32 bit pattern (finite and non-finite), in order
    bits = np.arange(0, 0x7F800001, 997, dtype=np.uint64).astype(np.uint32)
    enc = orc.e4m3_encode_bits(bits).astype(np.int32)
    assert np.all(np.diff(enc) >= 0)


def test_encode_nearest_brute_force(orc):
    """dec(enc(v)) is a nearest E4M3 value, ties to the even code, for v in
    [2^-6, 448]; checked with exact rationals against the decoded table."""
    table = [(Fraction(float(orc.e4m3_decode(np.uint8(c)))), c)
             for c in range(0x08, 0x7F)]
    rng = np.random.default_rng(3)
    xs = rng.uniform(2.0 ** -6, 448.0, size=3000).astype(np.float32)
    for x in xs:
        fx = Fraction(float(x))
        best = min(abs(fx - v) for v, _ in table)
        cands = [c for v, c in table if abs(fx - v) == best]
        want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        assert orc.e4m3_encode(x) == want


def test_encode_sign_symmetry(orc):
    rng = np.random.default_rng(5)
    x = rng.standard_normal(100_000).astype(np.float32) * 100
    a = orc.e4m3_encode(np.abs(x))
    b = orc.e4m3_encode(-np.abs(x))
    nz = a != 0
    assert np.array_equal(b[nz], a[nz] | 0x80)
    assert np.all(b[~nz] == 0)
