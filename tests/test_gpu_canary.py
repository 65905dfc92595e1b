"""GPU: no kernel writes outside its output.  Each y is a window in the
middle of a larger buffer filled with a NaN sentinel; after the call the
words before and after the window still hold the sentinel, bit for bit
(masked stores at ragged M and N edges, the rows between M and the padded
M of the FP8 route, the member boundaries of grouped calls), and the window
holds what the oracle gives."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import gemm_ok, gemv_ok, to_dev

pytestmark = pytest.mark.gpu

Q4K, Q6K = 12, 14
GUARD = 4096                # words on each side of the window
SENTINEL = 0x7FC0DEAD       # a quiet NaN no kernel produces


@pytest.fixture(scope="module")
def rq():
    import quantized_linear_layers_gb300 as rq
    return rq


def guarded(M, N):
    """(buffer, y): y is an [M x N] fp32 view GUARD words into the buffer."""
    buf = torch.full((M * N + 2 * GUARD,), SENTINEL, dtype=torch.int32, device="cuda")
    y = buf[GUARD:GUARD + M * N].view(torch.float32).view(M, N)
    return buf, y


def check_guards(buf, M, N):
    b = buf.cpu().numpy().view(np.uint32)
    before, after = b[:GUARD], b[GUARD + M * N:]
    assert np.all(before == SENTINEL), np.flatnonzero(before != SENTINEL)[:8]
    assert np.all(after == SENTINEL), np.flatnonzero(after != SENTINEL)[:8]


def check_result(qtype, W, x, N, K, got):
    M = x.shape[0]
    if oracle.route_is_gemm(M, 4):
        wb, wd = oracle.fp8_weight_cache(qtype, W, N, K)
        xb, xd = oracle.quant_e4m3(x, oracle.absmax_bits(x))
        ref = oracle.fp8_gemm(xb, xd, wb, wd)
        rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
        ok, worst = gemm_ok(got, ref, rms)
    else:
        ref, absdot = oracle.gemv(qtype, W, x, N, K)
        ok, worst = gemv_ok(got, ref, absdot)
    assert ok, worst


@pytest.mark.parametrize("qtype,M,N,K", [
    (Q4K, 1, 300, 512),      # one-token kernel, a few rows per CTA
    (Q4K, 1, 300, 18944),    # one-token kernel, rows split between two CTAs
    (Q4K, 3, 1000, 1024),    # three tokens: one launch of the one-token kernel each
    (Q6K, 1, 301, 512),      # one-token Q6_K kernel, odd row count
    (Q6K, 3, 300, 1024),     # few-token Q6_K kernel
    (Q4K, 4, 300, 512),      # FP8 route at the threshold
    (Q6K, 37, 300, 512),     # ragged M and N on the FP8 route
    (Q4K, 300, 2000, 2048),  # several token and weight tiles
])
def test_linear_writes_only_y(rq, qtype, M, N, K):
    W = synthetic.weight_matrix(900 + M + N, qtype, N, K)
    x = synthetic.activation(910 + M + K, M, K, outlier_frac=1e-3)
    buf, y = guarded(M, N)
    ctx = rq.Context()
    ctx.rq_linear(qtype, to_dev(W), to_dev(x), y, M, N, K)
    torch.cuda.synchronize()
    assert rq.rq_get_device_status() == 0
    check_guards(buf, M, N)
    check_result(qtype, W, x, N, K, y.cpu().numpy())
    ctx.close()


@pytest.mark.parametrize("M", [1, 3, 37])
def test_group_writes_only_its_members(rq, M):
    K = 1024
    members = [(Q4K, 300), (Q4K, 72), (Q6K, 136)]
    Ws = [synthetic.weight_matrix(950 + i, qt, N, K) for i, (qt, N) in enumerate(members)]
    x = synthetic.activation(960 + M, M, K, outlier_frac=1e-3)
    bufs = [guarded(M, N) for _, N in members]
    ctx = rq.Context()
    ctx.rq_linear_group([qt for qt, _ in members], [to_dev(W) for W in Ws], to_dev(x),
                        [y for _, y in bufs], [N for _, N in members], M, K)
    torch.cuda.synchronize()
    assert rq.rq_get_device_status() == 0
    for (qt, N), W, (buf, y) in zip(members, Ws, bufs):
        check_guards(buf, M, N)
        check_result(qt, W, x, N, K, y.cpu().numpy())
    ctx.close()
