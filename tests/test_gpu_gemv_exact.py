"""GPU parity of the decode GEMVs on inputs built to defeat their fast paths.

Every GEMV kernel must meet |gpu - oracle| <= 1e-4 * sum_k |x_k w_k| on
every finite input.  The fast paths keep x as fixed-point planes per
sub-block and factor Q4_K as d*sc*sum(q x) - dmin*m*sum(x), so they lose
accuracy when a sub-block's largest |x| sits on a zero weight, when x spans
many orders of magnitude inside a sub-block, or when a weight's two terms
cancel.  The kernels carry a per-output error certificate and recompute the
outputs it does not cover exactly; these tests build each of those inputs,
check every output against the fp64 oracle, and check through
rq_gemv_exact_outputs that the exact path ran (and that it does not run on
the decoder's ordinary data)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gguf_pack import pack_q4k_matrix, pack_q6k_matrix
from gpu_util import empty, gemv_ok, to_dev

pytestmark = pytest.mark.gpu

Q4K, Q6K = 12, 14


@pytest.fixture(scope="module")
def rq():
    import quantized_linear_layers_gb300 as rq
    return rq


@pytest.fixture
def ctx(rq):
    c = rq.Context()
    yield c
    c.close()


def gpu_gemv(rq, qtype, W, x, N, K):
    M = x.shape[0]
    y = empty((M, N), torch.float32)
    y.fill_(float("nan"))
    fn = rq.rq_q4k_gemv if qtype == Q4K else rq.rq_q6k_gemv
    fn(to_dev(W), to_dev(x), y, M, N, K)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def exact_count(rq):
    return rq.rq_gemv_exact_outputs()


# ------------------------------------------------------------ inputs ----

def q4k_zero_weights(seed, N, K, zero_k):
    """Q4_K weights with every min 0 and the quant at positions zero_k of
    every row 0, so w(n, k) = 0 there for all rows; elsewhere q in 1..15."""
    rng = np.random.default_rng(seed)
    nsb = K // 256
    d = rng.uniform(1e-3, 1e-2, (N, nsb))
    dmin = rng.uniform(1e-3, 1e-2, (N, nsb))
    sc = rng.integers(1, 64, (N, nsb, 8))
    mn = np.zeros((N, nsb, 8), np.int64)
    q = rng.integers(1, 16, (N, nsb, 256))
    qf = q.reshape(N, K)
    qf[:, zero_k] = 0
    return pack_q4k_matrix(d, dmin, sc, mn, qf.reshape(N, nsb, 256))


def q4k_cancelling_weights(seed, N, K, cancel_k):
    """Q4_K weights with d = dmin and sc_j = m_j, so w = d sc (q - 1): the
    quant 1 placed at positions cancel_k makes those weights exactly zero
    through cancellation of the two terms."""
    rng = np.random.default_rng(seed)
    nsb = K // 256
    d = rng.uniform(1e-3, 1e-2, (N, nsb))
    sc = rng.integers(1, 64, (N, nsb, 8))
    q = rng.integers(0, 16, (N, nsb, 256)).reshape(N, K)
    q[:, cancel_k] = 1
    return pack_q4k_matrix(d, d, sc, sc, q.reshape(N, nsb, 256))


def q6k_zero_weights(seed, N, K, zero_k):
    """Q6_K weights with the quant 32 (weight 0) at positions zero_k."""
    rng = np.random.default_rng(seed)
    nsb = K // 256
    d = rng.uniform(1e-3, 1e-2, (N, nsb))
    scales = rng.integers(-32, 32, (N, nsb, 16))
    scales[scales == 0] = 1
    q = rng.integers(0, 64, (N, nsb, 256)).reshape(N, K)
    q[q == 32] = 33
    q[:, zero_k] = 32
    return pack_q6k_matrix(d, scales, q.reshape(N, nsb, 256))


def big_on_positions(seed, M, K, big_k, ratio):
    """x whose entries at big_k are +-1 and all others ratio * N(0,1)."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((M, K)) * ratio).astype(np.float32)
    x[:, big_k] = np.where(rng.random((M, len(big_k))) < 0.5, -1.0, 1.0)
    return x


def check(got, W, x, qtype, N, K):
    ref, absdot = oracle.gemv(qtype, W, x, N, K)
    ok, worst = gemv_ok(got, ref, absdot)
    assert ok, "worst error / bound = %.3g" % worst


# The kernels each case runs through: (qtype, M, N, K, environment).
Q4_LAUNCHES = [
    pytest.param(1, 96, 3584, {}, id="q4k_m1"),
    pytest.param(1, 40, 18944, {}, id="q4k_m1_ksplit"),
    pytest.param(3, 64, 3584, {}, id="q4k_per_token"),
    pytest.param(1, 64, 3584, {"RQ_GEMV_GENERIC": "1"}, id="q4k_generic_m1"),
    pytest.param(5, 64, 3584, {"RQ_GEMV_GENERIC": "1"}, id="q4k_generic_m5"),
]
Q6_LAUNCHES = [
    pytest.param(1, 96, 3584, {}, id="q6k_m1"),
    pytest.param(4, 64, 3584, {}, id="q6k_mt"),
    pytest.param(8, 32, 3584, {}, id="q6k_mt_ksplit"),
    pytest.param(1, 64, 3584, {"RQ_GEMV_Q6_GENERIC": "1"}, id="q6k_generic_m1"),
    pytest.param(5, 64, 3584, {"RQ_GEMV_Q6_GENERIC": "1"}, id="q6k_generic_m5"),
]

def set_env(monkeypatch, env):
    for k, v in env.items():
        monkeypatch.setenv(k, v)


@pytest.mark.parametrize("ratio", [1e-7, 1e-3])
@pytest.mark.parametrize("M,N,K,env", Q4_LAUNCHES)
def test_q4k_sub_block_max_on_zero_weight(rq, monkeypatch, ratio, M, N, K, env):
    """In every 32-weight sub-block the largest |x| (1.0) multiplies a
    weight that is zero in every row (quant 0, min 0), and the other entries
    are `ratio` times smaller: the planes, scaled to that maximum, cannot
    hold them, so only the certificate and the exact path keep the bound."""
    set_env(monkeypatch, env)
    big_k = np.arange(5, K, 32)
    W = q4k_zero_weights(11 + M, N, K, big_k)
    x = big_on_positions(12 + M, M, K, big_k, ratio)
    exact_count(rq)
    got = gpu_gemv(rq, Q4K, W, x, N, K)
    check(got, W, x, Q4K, N, K)
    if not env and ratio == 1e-7:  # the plane kernels (the generic ones need no exact path)
        assert exact_count(rq) > 0


@pytest.mark.parametrize("M,N,K,env", Q4_LAUNCHES)
def test_q4k_weights_cancelling_under_large_x(rq, monkeypatch, M, N, K, env):
    """w = d*sc*q - dmin*m with d = dmin, sc = m and q = 1 is exactly zero;
    x is large there: the factored sum d*sc*sum(q x) - dmin*m*sum(x)
    cancels to the size of its rounding error, which the certificate
    counts against the (small) rest of the row."""
    set_env(monkeypatch, env)
    big_k = np.arange(9, K, 32)
    W = q4k_cancelling_weights(21 + M, N, K, big_k)
    x = big_on_positions(22 + M, M, K, big_k, 1e-6)
    x[:, big_k] *= np.float32(1e3)
    exact_count(rq)
    got = gpu_gemv(rq, Q4K, W, x, N, K)
    check(got, W, x, Q4K, N, K)
    if not env:
        assert exact_count(rq) > 0


@pytest.mark.parametrize("M,N,K,env", Q4_LAUNCHES)
def test_q4k_token_with_one_huge_outlier(rq, monkeypatch, M, N, K, env):
    """Random weights and N(0,1) tokens with one entry 1e7 times larger:
    rows whose weight at that position is zero (or small) keep the bound."""
    set_env(monkeypatch, env)
    W = synthetic.q4k_matrix(31 + K, N, K)
    x = synthetic.activation(32 + M, M, K)
    rng = np.random.default_rng(33)
    x[np.arange(M), rng.integers(0, K, M)] *= np.float32(1e7)
    got = gpu_gemv(rq, Q4K, W, x, N, K)
    check(got, W, x, Q4K, N, K)


@pytest.mark.parametrize("ratio", [1e-7, 1e-3])
@pytest.mark.parametrize("M,N,K,env", Q6_LAUNCHES)
def test_q6k_sub_block_max_on_zero_weight(rq, monkeypatch, ratio, M, N, K, env):
    """Q6_K: the largest |x| of every 16-weight sub-block multiplies the
    quant 32 (weight zero in every row), the rest are `ratio` times smaller."""
    set_env(monkeypatch, env)
    big_k = np.arange(3, K, 16)
    W = q6k_zero_weights(41 + M, N, K, big_k)
    x = big_on_positions(42 + M, M, K, big_k, ratio)
    exact_count(rq)
    got = gpu_gemv(rq, Q6K, W, x, N, K)
    check(got, W, x, Q6K, N, K)
    if not env and ratio == 1e-7:  # the plane kernels (the generic ones need no exact path)
        assert exact_count(rq) > 0


@pytest.mark.parametrize("M,N,K,env", Q6_LAUNCHES)
def test_q6k_token_with_one_huge_outlier(rq, monkeypatch, M, N, K, env):
    set_env(monkeypatch, env)
    W = synthetic.q6k_matrix(51 + K, N, K)
    x = synthetic.activation(52 + M, M, K)
    rng = np.random.default_rng(53)
    x[np.arange(M), rng.integers(0, K, M)] *= np.float32(1e7)
    got = gpu_gemv(rq, Q6K, W, x, N, K)
    check(got, W, x, Q6K, N, K)


def magnitude_mix(seed, M, K):
    """N(0,1) x with each 32-value sub-block scaled by 10^e, e in -30..30,
    and one sub-block per token pushed below fp32's normal range."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K))
    e = rng.integers(-30, 31, (M, K // 32))
    x = x * np.repeat(10.0 ** e, 32, axis=1)
    x[:, 64:96] = rng.standard_normal((M, 32)) * 1e-39
    return x.astype(np.float32)


@pytest.mark.parametrize("qtype", [Q4K, Q6K])
@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("generic", [False, True])
def test_magnitudes_across_sixty_decades(rq, monkeypatch, qtype, M, generic):
    """Sub-blocks of x from 1e-30 to 1e30 and one of fp32 subnormals (whose
    planes would not be valid): every output within the bound."""
    if generic:
        monkeypatch.setenv("RQ_GEMV_GENERIC" if qtype == Q4K else "RQ_GEMV_Q6_GENERIC", "1")
    N, K = 80, 3584
    W = synthetic.weight_matrix(61 + qtype, qtype, N, K)
    x = magnitude_mix(62 + M, M, K)
    got = gpu_gemv(rq, qtype, W, x, N, K)
    check(got, W, x, qtype, N, K)


@pytest.mark.parametrize("qtype", [Q4K, Q6K])
@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("generic", [False, True])
def test_non_finite_x_propagates_as_in_ieee(rq, monkeypatch, qtype, M, generic):
    """A NaN in a token makes all its outputs NaN; +Inf gives +-Inf, or NaN
    where the weight is zero, exactly as the fp64 oracle does."""
    if generic:
        monkeypatch.setenv("RQ_GEMV_GENERIC" if qtype == Q4K else "RQ_GEMV_Q6_GENERIC", "1")
    N, K = 48, 1024
    W = synthetic.weight_matrix(71 + qtype, qtype, N, K)
    x = synthetic.activation(72, M, K)
    x[0, 100] = np.nan
    if M > 1:
        x[1, 700] = np.inf
    got = gpu_gemv(rq, qtype, W, x, N, K)
    ref, _ = oracle.gemv(qtype, W, x, N, K)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin].astype(np.float32))


def test_decoder_layer_groups_on_adversarial_weights(rq, ctx):
    """The grouped launches (q/k/v as one Q4_K + Q6_K launch, gate/up as one
    Q4_K launch) at one and two tokens, on weights that are zero under the
    sub-block maxima of x: every member's outputs within the bound."""
    K = 3584
    big = np.arange(7, K, 16)
    Wq = q4k_zero_weights(81, 160, K, big)
    Wk = q4k_zero_weights(82, 64, K, big)
    Wv = q6k_zero_weights(83, 64, K, big)
    for M in (1, 2):
        x = big_on_positions(84 + M, M, K, big, 1e-7)
        xs = to_dev(x)
        ys = [empty((M, n), torch.float32) for n in (160, 64, 64)]
        ctx.rq_linear_group([Q4K, Q4K, Q6K], [to_dev(Wq), to_dev(Wk), to_dev(Wv)], xs, ys,
                            [160, 64, 64], M, K)
        torch.cuda.synchronize()
        for (W, qt, n), y in zip(((Wq, Q4K, 160), (Wk, Q4K, 64), (Wv, Q6K, 64)), ys):
            check(y.cpu().numpy(), W, x, qt, n, K)
        ys2 = [empty((M, n), torch.float32) for n in (160, 64)]
        ctx.rq_linear_group([Q4K, Q4K], [to_dev(Wq), to_dev(Wk)], xs, ys2, [160, 64], M, K)
        torch.cuda.synchronize()
        check(ys2[0].cpu().numpy(), Wq, x, Q4K, 160, K)
        check(ys2[1].cpu().numpy(), Wk, x, Q4K, 64, K)


@pytest.mark.parametrize("qtype,N,K", [(Q4K, 18944, 3584), (Q4K, 3584, 18944),
                                       (Q4K, 3584, 3584), (Q6K, 512, 3584)])
@pytest.mark.parametrize("outliers", [0.0, 1e-3, 1e-2])
def test_certificate_holds_on_decoder_data(rq, qtype, N, K, outliers):
    """On the decoder's shapes and data (x N(0,1), 0.1 % / 1 % of entries
    x50) the certificate covers every output: the exact path never runs."""
    W = synthetic.weight_matrix(91 + N + K, qtype, N, K)
    x = synthetic.activation(92 + N, 1, K, outlier_frac=outliers)
    exact_count(rq)
    got = gpu_gemv(rq, qtype, W, x, N, K)
    assert exact_count(rq) == 0
    rows = np.unique(np.linspace(0, N - 1, 64).astype(np.int64))
    ref, absdot = oracle.gemv_rows(qtype, W, x, N, K, rows)
    assert gemv_ok(got[:, rows], ref, absdot)[0]
