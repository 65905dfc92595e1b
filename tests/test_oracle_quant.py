"""Pins for the oracle's absmax and scaled E4M3 quantization (CPU only)."""
import numpy as np

import synthetic


def f32_bits(v):
    return int(np.float32(v).view(np.uint32))


def test_absmax_matches_numpy_and_planted_max(orc):
    x = synthetic.normal_f32(1, 100_003)
    x[777] = np.float32(-123.5)
    assert orc.absmax_bits(x) == f32_bits(123.5)
    assert orc.absmax_bits(x) == f32_bits(np.max(np.abs(x)))


def test_absmax_special_values(orc):
    assert orc.absmax_bits(np.zeros(0, np.float32)) == 0
    assert orc.absmax_bits(np.array([-0.0], np.float32)) == 0
    assert orc.absmax_bits(np.array([np.nan, -2.0, np.nan], np.float32)) == f32_bits(2.0)
    assert orc.absmax_bits(np.array([np.nan], np.float32)) == 0
    assert orc.absmax_bits(np.array([1.0, -np.inf], np.float32)) == f32_bits(np.inf)
    sub = np.array([0x00000001, 0x80000003], np.uint32).view(np.float32)
    assert orc.absmax_bits(sub) == 3
    # NaN payloads with the sign bit set are still skipped
    neg_nan = np.array([0xFFC00001, 0x3F800000], np.uint32).view(np.float32)
    assert orc.absmax_bits(neg_nan) == f32_bits(1.0)


def test_absmax_nan_skipping_equals_numpy_nanmax():
    import oracle
    rng = np.random.default_rng(2)
    x = rng.standard_normal(50_000).astype(np.float32)
    x[rng.integers(0, x.size, 100)] = np.nan
    assert oracle.absmax_bits(x) == f32_bits(np.nanmax(np.abs(x)))


def test_scales_zero_absmax_uses_one(orc):
    q, d = orc.scales(0)
    assert q == np.float32(448.0) and d == np.float32(1.0) / np.float32(448.0)
    q, d = orc.scales(f32_bits(448.0))
    assert q == np.float32(1.0) and d == np.float32(1.0)
    # correctly rounded fp32 division (numpy float32 division is IEEE RN)
    # (448 / 2^-140 overflows to +Inf in fp32, as it does on the device)
    for a in [3.7, 1e-30, 12345.678, 2.0 ** -140]:
        q, d = orc.scales(f32_bits(a))
        with np.errstate(over="ignore"):
            assert q == np.float32(448.0) / np.float32(a)
        assert d == np.float32(a) / np.float32(448.0)


def test_quant_with_unit_scale_is_the_unscaled_encoder(orc):
    x = synthetic.normal_f32(9, 50_000) * np.float32(100.0)
    b, deq = orc.quant_e4m3(x, f32_bits(448.0))
    assert deq == np.float32(1.0)
    assert np.array_equal(b, orc.e4m3_encode(x))


def test_quant_scaled_value_rounding(orc):
    """b = enc(fl32(x * s)): one fp32 multiply, no double rounding."""
    x = synthetic.normal_f32(4, 200_000)
    a = orc.absmax_bits(x)
    s, deq = orc.scales(a)
    b, deq2 = orc.quant_e4m3(x, a)
    assert deq == deq2
    assert np.array_equal(b, orc.e4m3_encode(x * s))  # numpy f32 multiply is RN
    # the absmax element lands on +-448
    i = int(np.argmax(np.abs(x)))
    assert b[i] in (0x7E, 0xFE)
    # dequantized bytes stay within half an E4M3 ulp (2^-4 relative) of x
    v = orc.e4m3_decode(b) * float(deq)
    big = np.abs(x) >= 2.0 ** -6 * float(deq)
    rel = np.abs(v[big] - x[big]) / np.abs(x[big])
    assert rel.max() <= 2.0 ** -4 + 1e-6


def test_quant_non_finite_and_zero_inputs(orc):
    x = np.array([0x7FC00000, 0xFFC00000, 0x7F800000, 0xFF800000, 0x00000000,
                  0x80000000], np.uint32).view(np.float32)
    for a in [f32_bits(1.0), f32_bits(448.0), f32_bits(np.inf), 1]:
        b, _ = orc.quant_e4m3(x, a)
        assert list(b) == [0x7E, 0xFE, 0x7E, 0xFE, 0x00, 0x00], hex(a)


def test_quant_infinite_absmax_flushes_finite_values(orc):
    x = np.array([1.0, -3.0, 448.0, np.inf, -np.inf], np.float32)
    a = orc.absmax_bits(x)
    assert a == f32_bits(np.inf)
    b, deq = orc.quant_e4m3(x, a)
    assert list(b) == [0, 0, 0, 0x7E, 0xFE]
    assert np.isinf(deq)


def test_quant_subnormal_absmax_overflowing_scale(orc):
    x = np.array([0x00000002, 0x80000001, 0], np.uint32).view(np.float32)
    a = orc.absmax_bits(x)
    s, _ = orc.scales(a)
    assert np.isinf(s)
    b, _ = orc.quant_e4m3(x, a)
    assert list(b) == [0x7E, 0xFE, 0x00]


def test_route_and_padding(orc):
    assert [orc.route_is_gemm(m, 4) for m in range(1, 7)] == [
        False, False, False, True, True, True]
    assert [orc.pad_m(m) for m in (1, 15, 16, 17, 512, 2047)] == [
        16, 16, 16, 32, 512, 2048]
