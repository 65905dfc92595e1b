"""rq_fp8_linear_noalloc: the FP8 linear layer for callers that cannot
allocate device memory while serving (code inside a host framework that owns
all device memory, or a process under a fixed memory budget).  It must give
the FP8 route's result -- the oracle's absmax, E4M3 bytes and exact FP8 dot
products -- while keeping its activation scratch in a fixed array inside the
library, and it must take no device memory.

This file is named so that pytest collects it last."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_util import empty, gemm_ok, to_dev

Q4K = 12
GUARD = 4096
SENTINEL = 0x7FC0DEAD


@pytest.fixture(scope="module")
def rq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_linear_layers_gb300 as rq
    return rq


def test_noalloc_rejects_bad_arguments_before_launch(rq):
    """Host-side validation only (no GPU work): nulls, shapes, alignment and
    an activation larger than the fixed array."""
    lib = rq.lib()
    a = 0x10000
    assert lib.rq_fp8_linear_noalloc(None, a, a, a, 16, 128, 128, None) == 1
    assert lib.rq_fp8_linear_noalloc(a, None, a, a, 16, 128, 128, None) == 1
    assert lib.rq_fp8_linear_noalloc(a, a, a, a, 0, 128, 128, None) == 2
    assert lib.rq_fp8_linear_noalloc(a, a, a, a, 16, 0, 128, None) == 2
    assert lib.rq_fp8_linear_noalloc(a, a, a, a, 16, 128, 64, None) == 2
    assert lib.rq_fp8_linear_noalloc(a + 4, a, a, a, 16, 128, 128, None) == 2
    # (M rounded up to 16) * K above the array: 2048 x 4224 bytes > 8 MiB
    assert rq.NOALLOC_MAX_ACT_BYTES == 8 * 1024 * 1024
    assert lib.rq_fp8_linear_noalloc(a, a, a, a, 2048, 128, 4224, None) == 2


def oracle_rows(W, N, K, x, rows):
    """The oracle's FP8 route for token rows `rows`: its weight cache, the
    activation's absmax and E4M3 bytes, exact FP8 dot products."""
    wb, wd = oracle.fp8_weight_cache(Q4K, W, N, K)
    xb, xd = oracle.quant_e4m3(x, oracle.absmax_bits(x))
    ms = np.repeat(np.asarray(rows), N)
    ns = np.tile(np.arange(N), len(rows))
    return oracle.fp8_gemm_pairs(xb, xd, wb, wd, ms, ns).reshape(len(rows), N)


def check_rows(got, ref):
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    ok, worst = gemm_ok(got, ref, rms)
    assert ok, worst


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_calls_in_a_row_without_allocating(rq):
    """Three calls in a row against the oracle.  The first has an outlier
    1e4 times its other entries, the next ones are 1e-3 times smaller: an
    absmax word or scale left over from an earlier call would push most of
    their codes to zero.  After the first call (which may load the library's
    module and look up the array), the device's free memory does not change
    across a call."""
    import torch
    N, K = 384, 1024
    W = synthetic.q4k_matrix(2024, N, K)
    ctx = rq.Context()
    wq, wd = ctx.rq_fp8_weight_cache(Q4K, to_dev(W), N, K)
    calls = []
    for M, seed, scale in ((40, 11, 1.0), (21, 12, 1e-3), (33, 13, 1e-3)):
        x = (synthetic.activation(seed, M, K) * np.float32(scale)).astype(np.float32)
        if seed == 11:
            x[3, 17] = np.float32(1e4)
        calls.append((M, x, to_dev(x), empty((M, N), torch.float32)))
    torch.cuda.synchronize()
    for i, (M, x, xd, y) in enumerate(calls):
        free0 = torch.cuda.mem_get_info()[0]
        rq.rq_fp8_linear_noalloc(xd, wq, wd, y, M, N, K)
        assert rq.rq_get_device_status() == 0
        if i > 0:
            assert torch.cuda.mem_get_info()[0] == free0
        check_rows(y.cpu().numpy(), oracle_rows(W, N, K, x, np.arange(M)))
    ctx.close()


@pytest.mark.gpu
def test_noalloc_at_the_array_limit_writes_only_y(rq):
    """An activation that fills the array exactly (M = 2033 rounds up to
    2048 rows; 2048 x 4096 bytes = 8 MiB) with a ragged last tile: sampled
    rows against the oracle, and the words around y keep their sentinel."""
    import torch
    M, N, K = 2033, 256, 4096
    assert (M + 15) // 16 * 16 * K == rq.NOALLOC_MAX_ACT_BYTES
    W = synthetic.q4k_matrix(2025, N, K)
    x = synthetic.activation(2026, M, K, outlier_frac=1e-3)
    ctx = rq.Context()
    wq, wd = ctx.rq_fp8_weight_cache(Q4K, to_dev(W), N, K)
    buf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int32, device="cuda")
    y = buf[GUARD:GUARD + M * N].view(torch.float32).view(M, N)
    rq.rq_fp8_linear_noalloc(to_dev(x), wq, wd, y, M, N, K)
    assert rq.rq_get_device_status() == 0
    b = buf.cpu().numpy().view(np.uint32)
    assert np.all(b[:GUARD] == SENTINEL) and np.all(b[GUARD + M * N:] == SENTINEL)
    rows = np.array([0, 1, 1023, 2015, 2016, 2031, 2032])
    got = y.cpu().numpy()[rows]
    check_rows(got, oracle_rows(W, N, K, x, rows))
    ctx.close()
