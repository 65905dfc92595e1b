"""GPU parity: FP8 weight cache (bit-exact bytes and scale) and the tcgen05
FP8 GEMM (|gpu - ref| <= 2e-3*|ref| + 1e-3*rms(ref row))."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import device_view, empty, gemm_ok, random_e4m3, to_dev, u32

pytestmark = pytest.mark.gpu

Q4K, Q6K = 12, 14


@pytest.fixture(scope="module")
def rq():
    import quantized_linear_layers_gb300 as rq
    return rq


def scalar(v):
    return to_dev(np.array([v], np.float32))


def gpu_gemm(rq, Xb, xdeq, Wb, wdeq, M, pad_fill=0):
    """Xb holds M rows; it is padded to M_pad rows filled with pad_fill."""
    K = Xb.shape[1]
    N = Wb.shape[0]
    m_pad = (M + 15) // 16 * 16
    xp = np.full((m_pad, K), pad_fill, np.uint8)
    xp[:M] = Xb
    y = empty(M * N + 256, torch.float32)
    y.fill_(float("nan"))
    rq.rq_fp8_gemm(to_dev(xp), scalar(xdeq), to_dev(Wb), scalar(wdeq), y, M, N, K)
    assert rq.rq_get_device_status() == 0
    out = y.cpu().numpy()
    assert np.all(np.isnan(out[M * N:])), "wrote past y"
    return out[:M * N].reshape(M, N)


def check_full(got, ref):
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    ok, worst = gemm_ok(got, ref, rms)
    assert ok, "worst error / bound = %.3g" % worst


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (15, 128, 256), (16, 256, 128),
                                   (17, 200, 512), (100, 384, 1024), (256, 128, 384),
                                   (300, 130, 256), (513, 64, 128), (40, 1000, 640)])
def test_small_random_bytes(rq, M, N, K):
    Xb = random_e4m3(M * 7 + K, (M, K))
    Wb = random_e4m3(N * 5 + K + 1, (N, K))
    xdeq, wdeq = np.float32(0.0123), np.float32(0.0071)
    got = gpu_gemm(rq, Xb, xdeq, Wb, wdeq, M)
    ref = oracle.fp8_gemm(Xb, xdeq, Wb, wdeq)
    check_full(got, ref)


def test_integer_valued_products_are_exact(rq):
    """Codes of small integers with unit scales: every partial sum is an
    integer below 2^24, so the fp32 accumulator must be exact."""
    vals = np.arange(-8, 9)
    code = {v: int(oracle.e4m3_encode(np.float32(v))) for v in vals}
    M, N, K = 48, 256, 1024
    rng = np.random.default_rng(0)
    xv = rng.integers(-8, 9, (M, K))
    wv = rng.integers(-8, 9, (N, K))
    Xb = np.vectorize(code.get)(xv).astype(np.uint8)
    Wb = np.vectorize(code.get)(wv).astype(np.uint8)
    got = gpu_gemm(rq, Xb, 1.0, Wb, 1.0, M)
    assert np.array_equal(got, (xv @ wv.T).astype(np.float32))


def test_pad_rows_do_not_leak(rq):
    """Pad rows full of NaN codes must not affect rows < M."""
    M, N, K = 21, 256, 256
    Xb = random_e4m3(9, (M, K))
    Wb = random_e4m3(10, (N, K))
    got = gpu_gemm(rq, Xb, 0.5, Wb, 0.25, M, pad_fill=0x7F)
    check_full(got, oracle.fp8_gemm(Xb, 0.5, Wb, 0.25))


@pytest.mark.parametrize("qtype,N,K", [(Q4K, 37, 512), (Q6K, 45, 768), (Q4K, 3584, 3584),
                                       (Q6K, 512, 3584), (Q4K, 18944, 3584)])
def test_weight_cache_bit_exact(rq, qtype, N, K):
    W = synthetic.weight_matrix(55 + N, qtype, N, K)
    ctx = rq.Context()
    Wd = to_dev(W)
    wq, wd = ctx.rq_fp8_weight_cache(qtype, Wd, N, K)
    wq2, wd2 = ctx.rq_fp8_weight_cache(qtype, Wd, N, K)
    assert (wq, wd) == (wq2, wd2) and ctx.stats()["weights"] == 1
    torch.cuda.synchronize()
    gb = device_view(wq, N * K, torch.uint8)
    gd = device_view(wd, 1, torch.float32)
    ob, od = oracle.fp8_weight_cache(qtype, W, N, K)
    assert np.float32(gd.item()) == od
    assert np.array_equal(gb.cpu().numpy(), ob.ravel())
    ctx.close()


@pytest.mark.parametrize("N,K", [(3584, 3584), (512, 3584), (18944, 3584), (3584, 18944)])
@pytest.mark.parametrize("M", [512, 2048])
def test_full_size_prefill_shapes(rq, N, K, M):
    """Prefill shapes at full size: device-built weight cache and activation
    quantization (both bit-exact with the oracle), then the GEMM checked on
    one full row in every band of 64 tokens (every token tile of the launch
    holds at least one checked row) and the last row, against the exact
    oracle."""
    W = synthetic.q4k_matrix(900 + N + K, N, K)
    x = synthetic.activation(901 + M, M, K, outlier_frac=1e-3)
    ctx = rq.Context()
    wq, wd = ctx.rq_fp8_weight_cache(Q4K, to_dev(W), N, K)
    xd = to_dev(x)
    m_pad = (M + 15) // 16 * 16
    bits = empty(1, torch.int32)
    xq = empty(m_pad * K, torch.uint8)
    xq.zero_()
    xdq = empty(1, torch.float32)
    rq.rq_absmax(xd, M * K, bits)
    rq.rq_quant_e4m3(xd, M * K, bits, xq, xdq)
    y = empty((M, N), torch.float32)
    rq.rq_fp8_gemm(xq, xdq, wq, wd, y, M, N, K)
    assert rq.rq_get_device_status() == 0
    # oracle side: its own bytes, checked equal to the device's
    ob_w, od_w = oracle.fp8_weight_cache(Q4K, W, N, K)
    a = oracle.absmax_bits(x)
    ob_x, od_x = oracle.quant_e4m3(x, a)
    assert u32(bits) == a
    assert np.array_equal(xq.cpu().numpy()[:M * K], ob_x.ravel())
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    rows = [64 * b + (37 * b) % 64 for b in range(M // 64)] + [M - 1]
    for m in rows:
        ref = oracle.fp8_gemm_pairs(ob_x, od_x, ob_w, od_w, np.full(N, m), np.arange(N))
        rms = np.sqrt(np.mean(ref ** 2))
        ok, worst = gemm_ok(got[m], ref, rms)
        assert ok, (m, worst)
    ctx.close()


@pytest.mark.parametrize("bn", [16, 48, 112, 208, 256])
def test_forced_tile_widths(rq, bn, monkeypatch):
    """Every tile width the shape heuristic can pick gives the same result."""
    monkeypatch.setenv("RQ_GEMM_BN", str(bn))
    M, N, K = 300, 200, 384
    Xb = random_e4m3(77, (M, K))
    Wb = random_e4m3(78, (N, K))
    got = gpu_gemm(rq, Xb, 0.01, Wb, 0.02, M)
    check_full(got, oracle.fp8_gemm(Xb, 0.01, Wb, 0.02))


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("M,N,K,bn", [(17, 256, 256, 0), (300, 384, 512, 0), (64, 1000, 384, 0),
                                      (512, 640, 1024, 128), (2048, 512, 3584, 0),
                                      (700, 3584, 256, 224)])
def test_single_and_pair_kernels(rq, monkeypatch, pair, M, N, K, bn):
    """The one-CTA and the CTA-pair (cta_group::2) kernels agree with the
    oracle on ragged shapes, including weight-row tiles that straddle N."""
    monkeypatch.setenv("RQ_GEMM_PAIR", pair)
    if bn:
        monkeypatch.setenv("RQ_GEMM_BN", str(bn))
    Xb = random_e4m3(M + 3 * N, (M, K))
    Wb = random_e4m3(N + 5 * K, (N, K))
    got = gpu_gemm(rq, Xb, 0.01, Wb, 0.02, M)
    check_full(got, oracle.fp8_gemm(Xb, 0.01, Wb, 0.02))


@pytest.mark.parametrize("S", ["2", "3", "5", "8"])
@pytest.mark.parametrize("M,N,K", [(300, 200, 4096), (5, 384, 2048), (2048, 512, 3584)])
def test_split_k_cluster_kernel(rq, monkeypatch, S, M, N, K):
    """The split-K kernel (a cluster of S CTAs per output tile, partials
    summed through distributed shared memory) agrees with the oracle for
    every split count, ragged M and N included."""
    monkeypatch.setenv("RQ_GEMM_SPLIT", S)
    Xb = random_e4m3(M + N + int(S), (M, K))
    Wb = random_e4m3(N + K + int(S), (N, K))
    got = gpu_gemm(rq, Xb, 0.01, Wb, 0.02, M)
    check_full(got, oracle.fp8_gemm(Xb, 0.01, Wb, 0.02))


def test_split_k_integer_sums_are_exact(rq, monkeypatch):
    """Integer-valued codes: every partial and the rank-ordered sum of the
    partials are exact integers, so the split result is exact."""
    monkeypatch.setenv("RQ_GEMM_SPLIT", "4")
    vals = np.arange(-8, 9)
    code = {v: int(oracle.e4m3_encode(np.float32(v))) for v in vals}
    M, N, K = 64, 384, 2048
    rng = np.random.default_rng(5)
    xv = rng.integers(-8, 9, (M, K))
    wv = rng.integers(-8, 9, (N, K))
    Xb = np.vectorize(code.get)(xv).astype(np.uint8)
    Wb = np.vectorize(code.get)(wv).astype(np.uint8)
    got = gpu_gemm(rq, Xb, 1.0, Wb, 1.0, M)
    assert np.array_equal(got, (xv @ wv.T).astype(np.float32))
