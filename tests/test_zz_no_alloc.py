"""rq_fp8_linear_noalloc: the FP8 linear layer for callers that cannot
allocate device memory while serving (code inside a host framework that owns
all device memory, or a process under a fixed memory budget).  It must give
the same result as the FP8 route of rq_linear while keeping its activation
scratch in a fixed array inside the library.

This file is named so that pytest collects it last."""
import numpy as np
import pytest

import synthetic
from gpu_util import empty, gemm_ok, to_dev

Q4K = 12


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


@pytest.mark.gpu
def test_noalloc_matches_rq_linear_on_two_calls(rq):
    """Two calls in a row (the second smaller, so stale bytes from the first
    would show), each compared with rq_linear's FP8 route on the same input
    and weight, within the FP8 GEMM tolerance used by the other tests."""
    import torch
    N, K = 384, 1024
    W = synthetic.q4k_matrix(2024, N, K)
    Wd = to_dev(W)
    ctx = rq.Context()
    wq, wd = ctx.rq_fp8_weight_cache(Q4K, Wd, N, K)
    for M, seed in ((40, 11), (21, 12)):
        x = synthetic.activation(seed, M, K, outlier_frac=1e-3)
        xd = to_dev(x)
        want = empty((M, N), torch.float32)
        ctx.rq_act_cache_invalidate()
        ctx.rq_linear(Q4K, Wd, xd, want, M, N, K)
        got = empty((M, N), torch.float32)
        rq.rq_fp8_linear_noalloc(xd, wq, wd, got, M, N, K)
        assert rq.rq_get_device_status() == 0
        ref = want.cpu().numpy().astype(np.float64)
        rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
        ok, worst = gemm_ok(got.cpu().numpy(), ref, rms)
        assert ok, (M, worst)
    ctx.close()
