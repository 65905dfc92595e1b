"""GPU parity: Q4_K / Q6_K decode GEMV against the fp64 oracle, within
|gpu - oracle| <= 1e-4 * sum_k |x_k w_k| per element."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import empty, gemv_ok, to_dev

pytestmark = pytest.mark.gpu

Q4K, Q6K = 12, 14


@pytest.fixture(scope="module")
def rq():
    import quantized_linear_layers_gb300 as rq
    return rq


def gpu_gemv(rq, qtype, W, x, N, K):
    M = x.shape[0]
    y = empty((M, N), torch.float32)
    y.fill_(float("nan"))
    fn = rq.rq_q4k_gemv if qtype == Q4K else rq.rq_q6k_gemv
    fn(to_dev(W), to_dev(x), y, M, N, K)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("qtype", [Q4K, Q6K])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(1, 256), (67, 768), (130, 2560), (33, 8448)])
def test_small_shapes_all_m(rq, qtype, M, N, K):
    W = synthetic.weight_matrix(1000 + N + K, qtype, N, K)
    x = synthetic.activation(M + K, M, K)
    got = gpu_gemv(rq, qtype, W, x, N, K)
    ref, absdot = oracle.gemv(qtype, W, x, N, K)
    ok, worst = gemv_ok(got, ref, absdot)
    assert ok, "worst error / bound = %.3g" % worst


def test_c1_q4k_gemv_full(rq):
    """Single Q4_K GEMV, M=1, N=512, K=1024, every output checked."""
    N, K = 512, 1024
    W = synthetic.q4k_matrix(1, N, K)
    x = synthetic.activation(2, 1, K)
    got = gpu_gemv(rq, Q4K, W, x, N, K)
    ref, absdot = oracle.gemv(Q4K, W, x, N, K)
    ok, worst = gemv_ok(got, ref, absdot)
    assert ok, worst


C3_SHAPES = [(Q4K, 3584, 3584), (Q4K, 512, 3584), (Q6K, 512, 3584),
             (Q4K, 18944, 3584), (Q4K, 3584, 18944)]


@pytest.mark.parametrize("qtype,N,K", C3_SHAPES)
@pytest.mark.parametrize("M", [1, 4, 8])
def test_c3_full_size_sampled_rows(rq, qtype, N, K, M):
    """Decoder shapes at full size, in the launch the benchmark times: the
    oracle checks two rows in each of 304 equal row bands (so every CTA's
    contiguous block of rows, on up to 152 CTAs, has checked rows) plus the
    first and last rows."""
    W = synthetic.weight_matrix(31 * N + K, qtype, N, K)
    x = synthetic.activation(7 + M, M, K)
    got = gpu_gemv(rq, qtype, W, x, N, K)
    assert np.all(np.isfinite(got))
    bands = np.linspace(0, N, 305).astype(np.int64)
    rows = np.unique(np.concatenate([[0, N - 1], bands[:-1], (bands[:-1] + bands[1:]) // 2]))
    rows = rows[rows < N]
    ref, absdot = oracle.gemv_rows(qtype, W, x, N, K, rows)
    ok, worst = gemv_ok(got[:, rows], ref, absdot)
    assert ok, worst


def test_gemv_writes_only_its_outputs(rq):
    N, K, M = 37, 512, 3
    W = synthetic.q4k_matrix(3, N, K)
    x = synthetic.activation(3, M, K)
    buf = empty(M * N + 64, torch.float32)
    buf.fill_(12345.0)
    rq.rq_q4k_gemv(to_dev(W), to_dev(x), buf, M, N, K)
    torch.cuda.synchronize()
    tail = buf[M * N:].cpu().numpy()
    assert np.all(tail == 12345.0)


@pytest.mark.parametrize("M", [2, 4, 8])
def test_one_token_and_generic_kernels_agree(rq, monkeypatch, M):
    """Several Q4_K tokens run one launch of the one-token kernel each; the
    generic kernel (switched on by RQ_GEMV_GENERIC) takes all tokens in one
    launch; both meet the bound on the same input."""
    N, K = 512, 3584
    W = synthetic.q4k_matrix(40 + M, N, K)
    x = synthetic.activation(41 + M, M, K, outlier_frac=1e-3)
    ref, absdot = oracle.gemv(Q4K, W, x, N, K)
    got = gpu_gemv(rq, Q4K, W, x, N, K)
    assert gemv_ok(got, ref, absdot)[0]
    monkeypatch.setenv("RQ_GEMV_GENERIC", "1")
    got2 = gpu_gemv(rq, Q4K, W, x, N, K)
    assert gemv_ok(got2, ref, absdot)[0]


@pytest.mark.parametrize("N,K", [(157, 768), (1001, 2560), (3001, 18944), (512, 3584)])
def test_q6k_one_token_rows_and_alignment_groups(rq, N, K):
    """One-token Q6_K kernel: 210-byte super-blocks make rows 16-byte
    aligned only in groups of 2, 4 or 8; row blocks, stages and the last
    partial stage (bytes past the final 16-byte boundary) all meet the bound."""
    W = synthetic.q6k_matrix(600 + N, N, K)
    x = synthetic.activation(601 + K, 1, K, outlier_frac=1e-3)
    got = gpu_gemv(rq, Q6K, W, x, N, K)
    ref, absdot = oracle.gemv(Q6K, W, x, N, K)
    ok, worst = gemv_ok(got, ref, absdot)
    assert ok, worst


@pytest.mark.parametrize("M", [1, 3])
def test_q6k_weight_only_4_byte_aligned(rq, M):
    """A Q6_K weight at a 4-byte (not 16-byte) aligned address takes the
    generic kernel and gives the same bound."""
    N, K = 200, 1024
    W = synthetic.q6k_matrix(9, N, K)
    buf = torch.zeros(W.size + 16, dtype=torch.uint8, device="cuda")
    buf[4:4 + W.size] = to_dev(W.ravel())
    x = synthetic.activation(10, M, K)
    y = empty((M, N), torch.float32)
    rq.rq_q6k_gemv(buf[4:], to_dev(x), y, M, N, K)
    torch.cuda.synchronize()
    ref, absdot = oracle.gemv(Q6K, W, x, N, K)
    assert gemv_ok(y.cpu().numpy(), ref, absdot)[0]


@pytest.mark.parametrize("force", ["", "1", "0"])
@pytest.mark.parametrize("N,K", [(1, 512), (67, 768), (300, 8704), (151, 18944), (37, 40960),
                                 (3, 65536)])
def test_one_token_q4k_rows_split_between_two_ctas(rq, monkeypatch, force, N, K):
    """One token, rows whose super-blocks are split between the two CTAs of
    a cluster (automatic for rows longer than 8 warps' worth, forced on or
    off otherwise; K = 40960 needs it): every output against the oracle."""
    if force:
        monkeypatch.setenv("RQ_GEMV_KSPLIT", force)
    W = synthetic.q4k_matrix(2000 + N + K, N, K)
    x = synthetic.activation(2001 + K, 1, K, outlier_frac=1e-3)
    got = gpu_gemv(rq, Q4K, W, x, N, K)
    ref, absdot = oracle.gemv(Q4K, W, x, N, K)
    ok, worst = gemv_ok(got, ref, absdot)
    assert ok, "worst error / bound = %.3g" % worst


@pytest.mark.parametrize("env", [{}, {"RQ_GEMV_ONE_KERNEL": "0"},
                                 {"RQ_GEMV_ONE_KERNEL": "0", "RQ_GEMV_W16": "0"},
                                 {"RQ_GEMV_TEAM_CAP": "0"}, {"RQ_GEMV_EVICT_FIRST": "0"}])
@pytest.mark.parametrize("N,K", [(3584, 3584), (512, 3584), (3584, 18944), (1001, 2560)])
def test_one_token_q4k_launch_variants(rq, monkeypatch, capfd, env, N, K):
    """One-token Q4_K launches run the kernel of the mixed q/k/v launch with
    every CTA on its Q4_K side by default (the log says so), their own
    kernel instances with RQ_GEMV_ONE_KERNEL=0 (those compiled for 512
    threads unless RQ_GEMV_W16=0), every team with RQ_GEMV_TEAM_CAP=0 and
    weight copies without the L2 hint with RQ_GEMV_EVICT_FIRST=0: every
    output of each against the oracle (1001 x 2560: few rows a CTA, two rows
    per team and stage)."""
    monkeypatch.setenv("RQ_GEMV_LOG", "1")
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    W = synthetic.q4k_matrix(4000 + N + K, N, K)
    x = synthetic.activation(4001 + K, 1, K, outlier_frac=1e-3)
    capfd.readouterr()
    got = gpu_gemv(rq, Q4K, W, x, N, K)
    lines = [l for l in capfd.readouterr().err.splitlines() if l.startswith("rq_gemv:")]
    ref, absdot = oracle.gemv(Q4K, W, x, N, K)
    ok, worst = gemv_ok(got, ref, absdot)
    assert ok, "worst error / bound = %.3g" % worst
    assert len(lines) == 1, lines
    assert ("(mixed kernel)" in lines[0]) == (env.get("RQ_GEMV_ONE_KERNEL") != "0"), lines


@pytest.mark.parametrize("qtype,N,K,M,kernel", [
    (Q4K, 3584, 3584, 1, "q4k_m1"), (Q4K, 18944, 3584, 1, "q4k_m1"),
    (Q4K, 3584, 18944, 1, "q4k_m1_ksplit"), (Q6K, 512, 3584, 1, "q6k_m1"),
    (Q4K, 3584, 3584, 4, "q4k_m1"), (Q4K, 3584, 18944, 8, "q4k_m1_ksplit"),
    (Q6K, 512, 3584, 4, "q6k_mt"), (Q6K, 512, 3584, 8, "q6k_mt_ksplit")])
def test_decoder_shapes_take_their_kernels(rq, monkeypatch, capfd, qtype, N, K, M, kernel):
    """The decoder's shapes run on the kernels the measurements are for (a
    shape that does not fit them falls back to the generic kernel, which
    is correct but slow, so a silent fallback is a regression)."""
    monkeypatch.setenv("RQ_GEMV_LOG", "1")
    W = synthetic.weight_matrix(3000 + N + K, qtype, N, K)
    x = synthetic.activation(3001 + M, M, K)
    capfd.readouterr()
    gpu_gemv(rq, qtype, W, x, N, K)
    lines = [l for l in capfd.readouterr().err.splitlines() if l.startswith("rq_gemv:")]
    # Q4_K: one launch per token; Q6_K: one launch for all tokens
    want = M if qtype == Q4K else 1
    assert len(lines) == want and all(l.split()[1] == kernel for l in lines), lines


@pytest.mark.parametrize("force", ["", "1", "0"])
@pytest.mark.parametrize("M", [2, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 512), (37, 1024), (512, 3584), (1001, 2048), (300, 18944)])
def test_few_token_q6k_rows_split_between_two_ctas(rq, monkeypatch, force, M, N, K):
    """A few tokens on Q6_K with each row's super-blocks split between the
    two CTAs of a cluster (automatic when there are fewer row groups than
    SMs, forced on or off otherwise): every output against the oracle."""
    if force:
        monkeypatch.setenv("RQ_GEMV_Q6_KSPLIT", force)
    W = synthetic.q6k_matrix(3300 + N + K, N, K)
    x = synthetic.activation(3301 + M + K, M, K, outlier_frac=1e-3)
    got = gpu_gemv(rq, Q6K, W, x, N, K)
    ref, absdot = oracle.gemv(Q6K, W, x, N, K)
    ok, worst = gemv_ok(got, ref, absdot)
    assert ok, "worst error / bound = %.3g" % worst
