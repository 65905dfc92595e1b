"""Pins for the oracle's fp64 GEMV, FP8 GEMM and FP8 weight cache (CPU)."""
import numpy as np
import pytest

import synthetic

Q4K, Q6K = 12, 14


@pytest.mark.parametrize("qtype", [Q4K, Q6K])
def test_gemv_unit_vectors_pick_columns(orc, qtype):
    N, K = 4, 256
    W = synthetic.weight_matrix(3, qtype, N, K)
    exact = np.stack([orc.decode_block(qtype, W[n], exact=True) for n in range(N)])
    for k in [0, 1, 31, 32, 63, 64, 127, 128, 200, 255]:
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        y, a = orc.gemv(qtype, W, x, N, K)
        assert np.array_equal(y[0], exact[:, k])
        assert np.array_equal(a[0], np.abs(exact[:, k]))


@pytest.mark.parametrize("qtype", [Q4K, Q6K])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_brute_force_vs_numpy(orc, qtype, M):
    N, K = 4, 512
    W = synthetic.weight_matrix(11 + M, qtype, N, K)
    x = synthetic.activation(5, M, K)
    exact = np.concatenate(
        [np.stack([orc.decode_block(qtype, W[n, s * (144 if qtype == Q4K else 210):
                                               (s + 1) * (144 if qtype == Q4K else 210)],
                                    exact=True) for s in range(K // 256)]).ravel()[None]
         for n in range(N)])
    ref = x.astype(np.float64) @ exact.T
    y, a = orc.gemv(qtype, W, x, N, K)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(x.astype(np.float64)) @ np.abs(exact.T), rtol=1e-12)


def test_gemv_rows_matches_full(orc):
    N, K = 9, 768
    W = synthetic.q4k_matrix(2, N, K)
    x = synthetic.activation(2, 2, K)
    y, a = orc.gemv(Q4K, W, x, N, K)
    rows = np.array([8, 0, 3])
    yr, ar = orc.gemv_rows(Q4K, W, x, N, K, rows)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(ar, a[:, rows])


def test_gemv_linearity(orc):
    N, K = 5, 1024
    W = synthetic.q4k_matrix(8, N, K)
    x1 = synthetic.activation(1, 1, K)
    x2 = synthetic.activation(2, 1, K)
    y1, _ = orc.gemv(Q4K, W, x1, N, K)
    y2, _ = orc.gemv(Q4K, W, x2, N, K)
    y12, _ = orc.gemv(Q4K, W, (x1 + x2).astype(np.float32), N, K)
    ref = y1 + y2
    # x1+x2 rounds once in fp32; allow that rounding only
    assert np.allclose(y12, ref, rtol=1e-6, atol=1e-5)


def test_fp8_gemm_integer_valued_exact(orc):
    """Bytes whose values are small integers give exactly integer sums."""
    rng = np.random.default_rng(0)
    ints = {v: int(orc.e4m3_encode(np.float32(v))) for v in range(-8, 9)}
    M, N, K = 5, 7, 384
    xv = rng.integers(-8, 9, (M, K))
    wv = rng.integers(-8, 9, (N, K))
    Xb = np.vectorize(ints.get)(xv).astype(np.uint8)
    Wb = np.vectorize(ints.get)(wv).astype(np.uint8)
    Y = orc.fp8_gemm(Xb, 1.0, Wb, 1.0)
    assert np.array_equal(Y, (xv @ wv.T).astype(np.float64))
    Y2 = orc.fp8_gemm(Xb, 0.5, Wb, 0.25)
    assert np.array_equal(Y2, (xv @ wv.T) * 0.125)


def test_fp8_gemm_identity_weight(orc):
    K = 128
    one = int(orc.e4m3_encode(np.float32(1.0)))
    Wb = np.where(np.eye(K, dtype=bool), one, 0).astype(np.uint8)
    Xb = synthetic.random_bytes(4, 3 * K).reshape(3, K)
    Xb[(Xb & 0x7F) == 0x7F] = 0  # drop NaN codes
    Y = orc.fp8_gemm(Xb, 2.0, Wb, 3.0)
    assert np.array_equal(Y, orc.e4m3_decode(Xb) * 6.0)


def test_fp8_gemm_random_vs_numpy_and_pairs(orc):
    M, N, K = 6, 9, 1024
    Xb = synthetic.random_bytes(1, M * K).reshape(M, K)
    Wb = synthetic.random_bytes(2, N * K).reshape(N, K)
    Xb[(Xb & 0x7F) == 0x7F] = 0x7E
    Wb[(Wb & 0x7F) == 0x7F] = 0x7E
    xd, wd = np.float32(0.013), np.float32(0.0071)
    Y = orc.fp8_gemm(Xb, xd, Wb, wd)
    ref = (orc.e4m3_decode(Xb) @ orc.e4m3_decode(Wb).T) * float(xd) * float(wd)
    assert np.allclose(Y, ref, rtol=1e-13, atol=0)
    ms, ns = np.array([0, 5, 3]), np.array([8, 0, 4])
    assert np.array_equal(orc.fp8_gemm_pairs(Xb, xd, Wb, wd, ms, ns), Y[ms, ns])


@pytest.mark.parametrize("qtype", [Q4K, Q6K])
def test_fp8_weight_cache_composition(orc, qtype):
    N, K = 6, 512
    W = synthetic.weight_matrix(21, qtype, N, K)
    b, deq = orc.fp8_weight_cache(qtype, W, N, K)
    w = orc.dequant(qtype, W, N, K)
    a = orc.absmax_bits(w)
    b2, deq2 = orc.quant_e4m3(w, a)
    assert np.array_equal(b, b2) and deq == deq2
    assert deq == np.float32(np.float32(np.max(np.abs(w))) / np.float32(448.0))
    i = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert b[i] in (0x7E, 0xFE)
    v = orc.e4m3_decode(b) * float(deq)
    big = np.abs(w) >= 2.0 ** -6 * float(deq)
    assert np.max(np.abs(v[big] - w[big]) / np.abs(w[big])) <= 2.0 ** -4 + 1e-6
