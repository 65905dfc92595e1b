"""GPU: rq_linear routing by the M threshold, FP8 activation reuse across
linears that share an input, and the bounded-wait timeout path."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import device_view, empty, gemm_ok, gemv_ok, to_dev

pytestmark = pytest.mark.gpu

Q4K, Q6K = 12, 14


@pytest.fixture(scope="module")
def rq():
    import quantized_linear_layers_gb300 as rq
    return rq


def gemm_route_ref(qtype, W, x, N, K):
    wb, wd = oracle.fp8_weight_cache(qtype, W, N, K)
    xb, xd = oracle.quant_e4m3(x, oracle.absmax_bits(x))
    return oracle.fp8_gemm(xb, xd, wb, wd)


def check_gemm(got, ref):
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    ok, worst = gemm_ok(got, ref, rms)
    assert ok, worst


@pytest.mark.parametrize("qtype", [Q4K, Q6K])
def test_routing_around_threshold(rq, qtype):
    N, K = 160, 1024
    W = synthetic.weight_matrix(4, qtype, N, K)
    Wd = to_dev(W)
    ctx = rq.Context()
    assert ctx.gemm_threshold == 4
    for M in (1, 2, 3, 4, 5):
        x = synthetic.activation(40 + M, M, K, outlier_frac=1e-3)
        y = empty((M, N), torch.float32)
        before = ctx.stats()
        ctx.rq_linear(qtype, Wd, to_dev(x), y, M, N, K)
        torch.cuda.synchronize()
        after = ctx.stats()
        got = y.cpu().numpy()
        if oracle.route_is_gemm(M, 4):
            assert after["act_misses"] == before["act_misses"] + 1
            check_gemm(got, gemm_route_ref(qtype, W, x, N, K))
        else:
            assert after == before
            ref, absdot = oracle.gemv(qtype, W, x, N, K)
            assert gemv_ok(got, ref, absdot)[0]
    ctx.close()


def test_raised_threshold_runs_gemv_in_chunks_of_8(rq):
    N, K, M = 96, 512, 13
    W = synthetic.q4k_matrix(8, N, K)
    x = synthetic.activation(8, M, K)
    ctx = rq.Context(gemm_threshold=32)
    y = empty((M, N), torch.float32)
    ctx.rq_linear(Q4K, to_dev(W), to_dev(x), y, M, N, K)
    torch.cuda.synchronize()
    ref, absdot = oracle.gemv(Q4K, W, x[:8], N, K)
    ref2, absdot2 = oracle.gemv(Q4K, W, x[8:], N, K)
    assert gemv_ok(y.cpu().numpy(), np.vstack([ref, ref2]), np.vstack([absdot, absdot2]))[0]
    assert ctx.stats()["act_misses"] == 0
    ctx.close()


def test_threshold_from_environment(rq, monkeypatch):
    monkeypatch.setenv("RQ_GEMM_THRESHOLD", "9")
    ctx = rq.Context()
    assert ctx.gemm_threshold == 9
    ctx.set_gemm_threshold(2)
    assert ctx.gemm_threshold == 2
    ctx.close()


def test_activation_reuse_counts_and_results(rq):
    """q/k/v share x and gate/up share h: 3 reuses per layer as on the pages
    (Q computes, K and V reuse; gate computes, up reuses)."""
    K, M = 512, 40
    shapes = [("q", Q4K, 256), ("k", Q4K, 128), ("v", Q6K, 128), ("o", Q4K, 256),
              ("gate", Q4K, 384), ("up", Q4K, 384)]
    host = {n: synthetic.weight_matrix(70 + i, qt, N, K) for i, (n, qt, N) in enumerate(shapes)}
    dev_w = {n: to_dev(w) for n, w in host.items()}
    acts = {"x": synthetic.activation(1, M, K, outlier_frac=1e-3),
            "a": synthetic.activation(2, M, K), "h": synthetic.activation(3, M, K)}
    dev_a = {k: to_dev(v) for k, v in acts.items()}
    src = {"q": "x", "k": "x", "v": "x", "o": "a", "gate": "h", "up": "h"}
    ctx = rq.Context()
    for layer in range(2):
        for name, qt, N in shapes:
            y = empty((M, N), torch.float32)
            ctx.rq_linear(qt, dev_w[name], dev_a[src[name]], y, M, N, K)
            torch.cuda.synchronize()
            check_gemm(y.cpu().numpy(), gemm_route_ref(qt, host[name], acts[src[name]], N, K))
    st = ctx.stats()
    # per layer: q miss, k hit, v hit, o miss, gate miss, up hit
    assert st["act_hits"] == 6 and st["act_misses"] == 6
    assert st["weights"] == 6
    # rewriting x in place requires an explicit invalidation
    new_x = synthetic.activation(9, M, K)
    dev_a["x"].copy_(to_dev(new_x))
    ctx.rq_act_cache_invalidate()
    y = empty((M, 256), torch.float32)
    ctx.rq_linear(Q4K, dev_w["q"], dev_a["x"], y, M, 256, K)
    torch.cuda.synchronize()
    assert ctx.stats()["act_misses"] == 7
    check_gemm(y.cpu().numpy(), gemm_route_ref(Q4K, host["q"], new_x, 256, K))
    ctx.close()


def act_cache_bytes(ctx, xd, M, K):
    xq, xdq = ctx.rq_fp8_act_cache(xd, M, K)
    torch.cuda.synchronize()
    m_pad = (M + 15) // 16 * 16
    b = device_view(xq, m_pad * K, torch.uint8).cpu().numpy()
    d = np.float32(device_view(xdq, 1, torch.float32).item())
    return b, d


def oracle_act_bytes(x, M, K):
    m_pad = (M + 15) // 16 * 16
    ob, od = oracle.quant_e4m3(x, oracle.absmax_bits(x))
    want = np.zeros(m_pad * K, np.uint8)
    want[:M * K] = ob.ravel()
    return want, od


def act_quant_kernels(mode, n, reg=True):
    """Kernels the activation cache launches for n elements: the one-cluster
    kernel up to 2^17 elements; the one-pass kernel from 2^20 elements on
    while x fits on chip in one wave (per SM at least 512 and at most
    512 x 24 float4 in registers plus 220 KB of shared memory; reg=False:
    RQ_QUANT_REG=0) or what does not fit one wave of shared memory (220 KB
    per SM) is at most 16 MB (128 MB for tensors of 2^24 elements or more);
    else the two kernels."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chunk = max(4096, ((n + sms - 1) // sms + 3) & ~3)
    grid = (n + chunk - 1) // chunk
    head = 4 * n - 16 * grid * min(chunk // 4, 220 * 1024 // 16)
    if mode == "cluster" or (mode == "default" and n <= 1 << 17):
        return 1
    least = {"1": 0, "0": None, "default": 1 << 20}[mode]
    if least is None or n < least:
        return 2
    n4 = n // 4
    per4 = (n4 + sms - 1) // sms
    if reg and n4 >= sms * 512 and per4 <= 512 * 24 + 220 * 1024 // 16:
        return 1
    cap = (128 << 20) if n >= 1 << 24 else (16 << 20)
    return 1 if head <= cap else 2


def set_act_quant_mode(monkeypatch, mode):
    """"cluster": the one-cluster kernel at every size; "1": the one-pass
    kernel wherever it may run (no minimum size); "0": the two kernels;
    "default": the library's own choice."""
    if mode == "cluster":
        monkeypatch.setenv("RQ_CLUSTER_QUANT_MAX", str(1 << 40))
    elif mode != "default":
        monkeypatch.setenv("RQ_CLUSTER_QUANT_MAX", "0")
        monkeypatch.setenv("RQ_ONE_PASS_QUANT", mode)
        if mode == "1":
            monkeypatch.setenv("RQ_ONE_PASS_MIN", "0")


@pytest.mark.parametrize("one_pass", ["cluster", "1", "0", "default"])
@pytest.mark.parametrize("M,K", [(2048, 3584), (611, 1024), (611, 1023), (37, 3584), (5, 256),
                                 (16, 128), (3, 4101), (2048, 18944), (1001, 18947),
                                 (512, 18944), (509, 18947), (16, 18944), (128, 3584)])
def test_activation_cache_bytes_bit_exact(rq, monkeypatch, one_pass, M, K):
    """The FP8 activation (one-cluster kernel, one-pass kernel or absmax +
    quant kernels) is the oracle's bytes, pad rows zero, over three
    successive misses with different maxima; the second x has no NaN, so
    the kernels' path for all-finite inputs is checked as well as the one
    with fix-ups."""
    set_act_quant_mode(monkeypatch, one_pass)
    ctx = rq.Context()
    x = synthetic.activation(5000 + M + K, M, K, outlier_frac=1e-3)
    x.ravel()[min(4, x.size - 1)] = np.nan
    xd = to_dev(x)
    for scale in (1.0, 0.25, 3.0):
        xs = (x * np.float32(scale)).astype(np.float32)
        if scale == 0.25:
            xs.ravel()[min(4, x.size - 1)] = np.float32(0.75)
            assert np.isfinite(xs).all()
        xd.copy_(to_dev(xs))
        ctx.rq_act_cache_invalidate()
        ctx.rq_ctx_trace_begin(8)
        got, gd = act_cache_bytes(ctx, xd, M, K)
        tr = ctx.rq_ctx_trace_end()
        assert rq.rq_get_device_status() == 0
        want, wd = oracle_act_bytes(xs, M, K)
        assert gd == wd
        assert np.array_equal(got, want), np.flatnonzero(got != want)[:8]
        # absmax and encoding are traced together as QUANT
        assert tr["absmax"][0] == 0
        assert tr["quant"][0] == act_quant_kernels(one_pass, M * K)
    # a hit returns the same bytes without launching anything
    ctx.rq_ctx_trace_begin(8)
    got2, _ = act_cache_bytes(ctx, xd, M, K)
    assert sum(c for c, _ in ctx.rq_ctx_trace_end().values()) == 0
    assert np.array_equal(got2, got)
    ctx.close()


@pytest.mark.parametrize("one_pass", ["cluster", "1", "0"])
@pytest.mark.parametrize("M,K", [(16, 3584), (37, 4101), (300, 18944)])
def test_activation_cache_infinite_max(rq, monkeypatch, one_pass, M, K):
    """With -Inf in x the maximum is +Inf, so the scale is 0: every finite
    value encodes to 0x00 and -Inf to 0xFE, in every kernel."""
    set_act_quant_mode(monkeypatch, one_pass)
    ctx = rq.Context()
    x = synthetic.activation(6000 + M + K, M, K, outlier_frac=1e-3)
    x.ravel()[x.size // 2] = -np.inf
    x.ravel()[x.size // 3] = np.float32(1e-30)
    ctx.rq_ctx_trace_begin(8)
    got, gd = act_cache_bytes(ctx, to_dev(x), M, K)
    tr = ctx.rq_ctx_trace_end()
    assert rq.rq_get_device_status() == 0
    want, wd = oracle_act_bytes(x, M, K)
    assert gd == wd and np.isinf(gd)
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:8]
    assert got[x.size // 2] == 0xFE and np.count_nonzero(got) == 1
    assert tr["quant"][0] == act_quant_kernels(one_pass, M * K)
    ctx.close()


@pytest.mark.parametrize("reg", ["1", "0"])
@pytest.mark.parametrize("M,K", [(2048, 3584), (611, 1023), (128, 3584), (300, 18944),
                                 (4096, 3584), (512, 18944), (3000, 4101)])
def test_one_pass_register_and_shared_memory_forms(rq, monkeypatch, reg, M, K):
    """Tensors that fit on chip take the register form of the one-pass
    kernel by default (all in registers, or registers plus shared memory:
    4096 x 3584, 512 x 18944, 3000 x 4101), the shared-memory form (or the
    two kernels) with RQ_QUANT_REG=0; every form gives the oracle's bytes,
    with a NaN in x (fix-up path) and without (all-finite path), n % 4 != 0
    included."""
    set_act_quant_mode(monkeypatch, "1")
    monkeypatch.setenv("RQ_QUANT_REG", reg)
    ctx = rq.Context()
    x = synthetic.activation(7300 + M + K, M, K, outlier_frac=1e-3)
    for nan in (False, True):
        xs = x.copy()
        if nan:
            xs.ravel()[xs.size // 2 + 1] = np.nan
        ctx.rq_act_cache_invalidate()
        ctx.rq_ctx_trace_begin(8)
        got, gd = act_cache_bytes(ctx, to_dev(xs), M, K)
        tr = ctx.rq_ctx_trace_end()
        assert rq.rq_get_device_status() == 0
        assert tr["quant"][0] == act_quant_kernels("1", M * K, reg=reg == "1")
        want, wd = oracle_act_bytes(xs, M, K)
        assert gd == wd
        assert np.array_equal(got, want), (nan, np.flatnonzero(got != want)[:8])
    ctx.close()


@pytest.mark.parametrize("offset", [4, 8])
def test_one_pass_head_at_16_and_32_byte_alignment(rq, monkeypatch, offset):
    """A tensor larger than the wave holds (1001 x 18947, n % 4 = 3: a
    head streamed twice by all CTAs) at an x that is 16-byte but not
    32-byte aligned (offset 4 floats) and at one that is 32-byte aligned
    (offset 8): the stash boundaries and the tail fall differently; the
    oracle's bytes either way."""
    set_act_quant_mode(monkeypatch, "1")
    M, K = 1001, 18947
    ctx = rq.Context()
    x = synthetic.activation(7400 + offset, M, K, outlier_frac=1e-3)
    buf = empty((M * K + 8,), torch.float32)
    assert buf.data_ptr() % 32 == 0
    xv = buf[offset:offset + M * K]
    xv.copy_(to_dev(x.ravel()))
    ctx.rq_ctx_trace_begin(8)
    got, gd = act_cache_bytes(ctx, xv, M, K)
    tr = ctx.rq_ctx_trace_end()
    assert rq.rq_get_device_status() == 0
    assert tr["quant"][0] == act_quant_kernels("1", M * K)
    want, wd = oracle_act_bytes(x, M, K)
    assert gd == wd
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:8]
    ctx.close()


def test_one_pass_launches_of_different_grids_on_one_context(rq, monkeypatch):
    """One-pass launches in a row on one context with 1, 152, 33, 1, 152 and
    152 CTAs: each publishes its CTAs' maxima and meets at its own grid
    barrier, whose arrival count every launch leaves at zero.  The maxima
    differ by up to 10^4 from one launch to the next, so a stale one would
    change the bytes."""
    set_act_quant_mode(monkeypatch, "1")
    ctx = rq.Context()
    shapes = [(5, 256, 1.0), (2048, 3584, 1e-3), (37, 3584, 10.0), (5, 256, 1e-2),
              (611, 1024, 1.0), (2048, 3584, 1e2)]
    for i, (M, K, scale) in enumerate(shapes):
        x = (synthetic.activation(7100 + i, M, K, outlier_frac=1e-3) *
             np.float32(scale)).astype(np.float32)
        ctx.rq_act_cache_invalidate()
        ctx.rq_ctx_trace_begin(8)
        got, gd = act_cache_bytes(ctx, to_dev(x), M, K)
        tr = ctx.rq_ctx_trace_end()
        assert rq.rq_get_device_status() == 0
        assert tr["quant"][0] == 1
        want, wd = oracle_act_bytes(x, M, K)
        assert gd == wd
        assert np.array_equal(got, want), (i, np.flatnonzero(got != want)[:8])
    ctx.close()


def test_activation_cache_rejects_unaligned_x(rq):
    """The activation cache takes x on a 16-byte boundary only: RQ_ERR_SHAPE
    before anything is launched."""
    M, K = 16, 3584
    ctx = rq.Context()
    big = to_dev(np.zeros(M * K + 4, np.float32))
    with pytest.raises(rq.RqError) as err:
        ctx.rq_fp8_act_cache(big[1:], M, K)
    assert err.value.status == 2  # RQ_ERR_SHAPE
    ctx.close()


@pytest.mark.parametrize("one_pass", ["cluster", "0"])
def test_activation_cache_all_zero_input_each_kernel(rq, monkeypatch, one_pass):
    """An all-zero x: absmax 0 is read as 1, so the scale is 1/448 and every
    byte is 0x00, with both small-activation kernels."""
    set_act_quant_mode(monkeypatch, one_pass)
    M, K = 16, 3584
    ctx = rq.Context()
    xd = to_dev(np.zeros((M, K), np.float32))
    got, gd = act_cache_bytes(ctx, xd, M, K)
    assert not got.any() and gd == np.float32(1.0) / np.float32(448.0)
    ctx.close()


def test_activation_cache_all_zero_input(rq):
    M, K = 64, 512
    ctx = rq.Context()
    xd = to_dev(np.zeros((M, K), np.float32))
    got, gd = act_cache_bytes(ctx, xd, M, K)
    assert not got.any() and gd == np.float32(1.0) / np.float32(448.0)
    ctx.close()


def test_wait_timeout_is_reported_and_cleared(rq):
    rq.rq_debug_wait_timeout(20_000_000)  # 20 ms on a barrier nobody completes
    assert rq.rq_get_device_status() == 7  # RQ_ERR_TIMEOUT
    assert rq.rq_get_device_status() == 0  # cleared
    # the context is still usable
    N, K, M = 128, 256, 16
    W = synthetic.q4k_matrix(2, N, K)
    x = synthetic.activation(2, M, K)
    ctx = rq.Context()
    y = empty((M, N), torch.float32)
    ctx.rq_linear(Q4K, to_dev(W), to_dev(x), y, M, N, K)
    assert rq.rq_get_device_status() == 0
    check_gemm(y.cpu().numpy(), gemm_route_ref(Q4K, W, x, N, K))
    ctx.close()


def test_trace_kinds_mask(rq):
    """Tracing restricted to GEMMs records only the GEMM launch; an empty
    mask is rejected; restoring all kinds traces the activation kernels."""
    N, K, M = 256, 512, 64
    W = synthetic.q4k_matrix(3, N, K)
    Wd = to_dev(W)
    xd = to_dev(synthetic.activation(4, M, K))
    y = empty((M, N), torch.float32)
    ctx = rq.Context()
    ctx.rq_ctx_trace_kinds(["gemm"])
    ctx.rq_ctx_trace_begin(16)
    ctx.rq_linear(Q4K, Wd, xd, y, M, N, K)
    tr = ctx.rq_ctx_trace_end()
    assert tr["gemm"][0] == 1 and tr["gemm"][1] > 0
    assert tr["wcache"][0] == tr["quant"][0] == tr["absmax"][0] == 0
    with pytest.raises(rq.RqError):
        ctx.rq_ctx_trace_kinds([])
    ctx.rq_ctx_trace_kinds(list(ctx.TRACE_KINDS))
    ctx.rq_act_cache_invalidate()
    ctx.rq_ctx_trace_begin(16)
    ctx.rq_linear(Q4K, Wd, xd, y, M, N, K)
    tr = ctx.rq_ctx_trace_end()
    # 64 x 512 elements: one launch of the one-cluster kernel
    assert tr["gemm"][0] == 1 and tr["quant"][0] == 1
    ctx.close()


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 64, 300])
def test_linear_group_matches_separate_linears(rq, M):
    """rq_linear_group over members that share x (ragged N, both formats,
    rows straddling 128-row tiles and GEMV stages) gives each member what
    the oracle gives for it, on the GEMV (M < 4) and FP8 routes."""
    K = 1024
    members = [(Q4K, 200), (Q4K, 77), (Q6K, 130)]
    Ws = [synthetic.weight_matrix(300 + i, qt, N, K) for i, (qt, N) in enumerate(members)]
    Wd = [to_dev(W) for W in Ws]
    x = synthetic.activation(310 + M, M, K, outlier_frac=1e-3)
    xd = to_dev(x)
    ys = [empty((M, N), torch.float32) for _, N in members]
    ctx = rq.Context()
    ctx.rq_linear_group([qt for qt, _ in members], Wd, xd, ys, [N for _, N in members], M, K)
    torch.cuda.synchronize()
    assert rq.rq_get_device_status() == 0
    for (qt, N), W, y in zip(members, Ws, ys):
        got = y.cpu().numpy()
        if oracle.route_is_gemm(M, 4):
            check_gemm(got, gemm_route_ref(qt, W, x, N, K))
        else:
            ref, absdot = oracle.gemv(qt, W, x, N, K)
            assert gemv_ok(got, ref, absdot)[0]
    st = ctx.stats()
    if oracle.route_is_gemm(M, 4):
        assert st["weights"] == 1 and st["act_misses"] == 1
        # a second call hits both caches
        ctx.rq_linear_group([qt for qt, _ in members], Wd, xd, ys, [N for _, N in members], M, K)
        assert ctx.stats()["act_hits"] == 1 and ctx.stats()["weights"] == 1
    ctx.close()


def test_linear_group_decoder_shapes_one_token(rq):
    """q + k (Q4_K, 3584 + 512 rows) and gate + up (2 x 18944) of the
    decoder as one-token groups, sampled rows against the oracle."""
    K = 3584
    for seed, Ns in ((1, (3584, 512)), (2, (18944, 18944))):
        Ws = [synthetic.q4k_matrix(400 + seed * 10 + i, N, K) for i, N in enumerate(Ns)]
        x = synthetic.activation(420 + seed, 1, K)
        ys = [empty((1, N), torch.float32) for N in Ns]
        ctx = rq.Context()
        ctx.rq_linear_group([Q4K] * len(Ns), [to_dev(W) for W in Ws], to_dev(x), ys, list(Ns), 1, K)
        torch.cuda.synchronize()
        for W, y, N in zip(Ws, ys, Ns):
            rows = np.array([0, 1, N // 2, N - 2, N - 1])
            ref, absdot = oracle.gemv_rows(Q4K, W, x, N, K, rows)
            assert gemv_ok(y.cpu().numpy()[:, rows], ref, absdot)[0]
        ctx.close()


@pytest.mark.parametrize("g6", [None, "1", "40", "151"])
def test_linear_group_mixed_formats_one_launch(rq, monkeypatch, g6):
    """One token through q + k (Q4_K) and v (Q6_K) of the decoder: one
    GEMV launch whose CTAs split between the two formats (the split forced
    to its extremes too); every member's sampled rows against the oracle."""
    if g6 is not None:
        monkeypatch.setenv("RQ_GEMV_DUAL_G6", g6)
    K = 3584
    members = [(Q4K, 3584), (Q4K, 512), (Q6K, 512)]
    Ws = [synthetic.weight_matrix(430 + i, qt, N, K) for i, (qt, N) in enumerate(members)]
    x = synthetic.activation(440, 1, K)
    ys = [empty((1, N), torch.float32) for _, N in members]
    ctx = rq.Context()
    ctx.rq_ctx_trace_kinds(list(ctx.TRACE_KINDS))
    ctx.rq_ctx_trace_begin(16)
    ctx.rq_linear_group([qt for qt, _ in members], [to_dev(W) for W in Ws], to_dev(x), ys,
                        [N for _, N in members], 1, K)
    tr = ctx.rq_ctx_trace_end()
    assert tr["gemv"][0] == 1
    assert rq.rq_get_device_status() == 0
    for (qt, N), W, y in zip(members, Ws, ys):
        rows = np.array([0, 1, 2, 3, N // 2 - 1, N // 2, N - 3, N - 2, N - 1])
        ref, absdot = oracle.gemv_rows(qt, W, x, N, K, rows)
        assert gemv_ok(y.cpu().numpy()[:, rows], ref, absdot)[0], (qt, N)
    ctx.close()


@pytest.mark.parametrize("K,N4,N6", [(256, 3, 5), (768, 1, 1), (1280, 333, 97)])
def test_linear_group_mixed_formats_ragged(rq, K, N4, N6):
    """A Q4_K and a Q6_K member sharing one token: row counts below and
    off the Q6_K row alignment, every row against the oracle."""
    members = [(Q6K, N6), (Q4K, N4)]
    Ws = [synthetic.weight_matrix(450 + i, qt, N, K) for i, (qt, N) in enumerate(members)]
    x = synthetic.activation(460, 1, K, outlier_frac=1e-3)
    ys = [empty((1, N), torch.float32) for _, N in members]
    ctx = rq.Context()
    ctx.rq_linear_group([qt for qt, _ in members], [to_dev(W) for W in Ws], to_dev(x), ys,
                        [N for _, N in members], 1, K)
    torch.cuda.synchronize()
    assert rq.rq_get_device_status() == 0
    for (qt, N), W, y in zip(members, Ws, ys):
        ref, absdot = oracle.gemv(qt, W, x, N, K)
        assert gemv_ok(y.cpu().numpy(), ref, absdot)[0], (qt, N)
    ctx.close()


@pytest.mark.parametrize("M", [4, 8])
def test_linear_group_decoder_shapes_few_tokens(rq, monkeypatch, M):
    """q + k and gate + up of the decoder at a few tokens (GEMV route, the
    threshold raised above M): each group's Q4_K members in one launch per
    token; sampled rows of every member against the oracle."""
    K = 3584
    ctx = rq.Context(gemm_threshold=9)
    for seed, Ns in ((3, (3584, 512)), (4, (18944, 18944))):
        Ws = [synthetic.q4k_matrix(460 + seed * 10 + i, N, K) for i, N in enumerate(Ns)]
        x = synthetic.activation(480 + seed + M, M, K)
        ys = [empty((M, N), torch.float32) for N in Ns]
        ctx.rq_ctx_trace_kinds(list(ctx.TRACE_KINDS))
        ctx.rq_ctx_trace_begin(16)
        ctx.rq_linear_group([Q4K] * len(Ns), [to_dev(W) for W in Ws], to_dev(x), ys, list(Ns),
                            M, K)
        assert ctx.rq_ctx_trace_end()["gemv"][0] == M
        assert rq.rq_get_device_status() == 0
        for W, y, N in zip(Ws, ys, Ns):
            rows = np.array([0, 1, 15, 16, N // 2, N - 17, N - 16, N - 1])
            ref, absdot = oracle.gemv_rows(Q4K, W, x, N, K, rows)
            assert gemv_ok(y.cpu().numpy()[:, rows], ref, absdot)[0], (N, M)
    ctx.close()


@pytest.mark.parametrize("M,kernels", [(1, ["dual_q4k_q6k_m1"]),
                                       (4, ["dual_q4k_q6k_m1"] * 4),
                                       (8, ["dual_q4k_q6k_m1"] * 8)])
def test_decoder_qkv_group_launches(rq, monkeypatch, capfd, M, kernels):
    """q/k/v of the decoder as one group call: one launch per token, which
    the Q4_K and Q6_K members share."""
    monkeypatch.setenv("RQ_GEMV_LOG", "1")
    K = 3584
    members = [(Q4K, 3584), (Q4K, 512), (Q6K, 512)]
    Ws = [to_dev(synthetic.weight_matrix(3100 + i, qt, N, K)) for i, (qt, N) in enumerate(members)]
    x = to_dev(synthetic.activation(3110 + M, M, K))
    ys = [empty((M, N), torch.float32) for _, N in members]
    ctx = rq.Context(gemm_threshold=9)
    capfd.readouterr()
    ctx.rq_linear_group([qt for qt, _ in members], Ws, x, ys, [N for _, N in members], M, K)
    torch.cuda.synchronize()
    got = [l.split()[1] for l in capfd.readouterr().err.splitlines() if l.startswith("rq_gemv:")]
    assert got == kernels
    ctx.close()


@pytest.mark.parametrize("M", [1, 3, 40])
def test_linear_group_of_four_members(rq, M):
    """RQ_MAX_GROUP members (Q4_K and Q6_K mixed, one of them twice): each
    member's output against the oracle on the route M takes."""
    K = 768
    members = [(Q4K, 48), (Q6K, 33), (Q4K, 130), (Q4K, 48)]
    Ws = [synthetic.weight_matrix(3200 + i, qt, N, K) for i, (qt, N) in enumerate(members[:3])]
    Ws.append(Ws[0])
    Wd = [to_dev(W) for W in Ws[:3]]
    Wd.append(Wd[0])
    x = synthetic.activation(3210 + M, M, K, outlier_frac=1e-3)
    ys = [empty((M, N), torch.float32) for _, N in members]
    ctx = rq.Context()
    ctx.rq_linear_group([qt for qt, _ in members], Wd, to_dev(x), ys, [N for _, N in members],
                        M, K)
    torch.cuda.synchronize()
    assert rq.rq_get_device_status() == 0
    for (qt, N), W, y in zip(members, Ws, ys):
        got = y.cpu().numpy()
        if oracle.route_is_gemm(M, 4):
            check_gemm(got, gemm_route_ref(qt, W, x, N, K))
        else:
            ref, absdot = oracle.gemv(qt, W, x, N, K)
            assert gemv_ok(got, ref, absdot)[0]
    ctx.close()


@pytest.mark.parametrize("M,N,K", [(16, 3584, 3584), (300, 640, 1024), (2048, 3584, 3584),
                                   (1000, 4608, 2048)])
def test_cached_weight_calls_match_the_oracle(rq, M, N, K):
    """Calls after the first find the FP8 weight in the cache, and the GEMM
    then starts loading its first weight tiles before the launch before it
    has completed; every call, with a new activation each time, against the
    oracle (split-K, one-CTA and CTA-pair shapes)."""
    W = synthetic.q4k_matrix(3400 + N + K, N, K)
    Wd = to_dev(W)
    wb, wd = oracle.fp8_weight_cache(Q4K, W, N, K)
    ctx = rq.Context()
    for call in range(3):
        x = synthetic.activation(3410 + call + M, M, K, outlier_frac=1e-3)
        y = empty((M, N), torch.float32)
        ctx.rq_act_cache_invalidate()
        ctx.rq_linear(Q4K, Wd, to_dev(x), y, M, N, K)
        torch.cuda.synchronize()
        assert rq.rq_get_device_status() == 0
        xb, xd = oracle.quant_e4m3(x, oracle.absmax_bits(x))
        got = y.cpu().numpy()
        for m in sorted({0, 1, M // 2, M - 1}):
            ref = oracle.fp8_gemm_pairs(xb, xd, wb, wd, np.full(N, m), np.arange(N))
            ok, worst = gemm_ok(got[m], ref, np.sqrt(np.mean(ref ** 2)))
            assert ok, (call, m, worst)
    assert ctx.stats()["weights"] == 1
    ctx.close()


def test_linear_group_rejects_bad_counts(rq):
    ctx = rq.Context()
    with pytest.raises(rq.RqError):
        ctx.rq_linear_group([], [], empty((1, 256), torch.float32), [], [], 1, 256)
    ctx.close()


# ------------------------------------------------- a full decoder layer --

LAYER_CALLS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))
LAYER_SOURCE = {"q": "x", "k": "x", "v": "x", "o": "a", "gate": "h", "up": "h", "down": "g"}


@pytest.fixture(scope="module")
def decoder_layer():
    """One decoder layer's seven weights (full shapes) and the oracle's FP8
    weight caches of them."""
    layer = {}
    for i, (name, qt, N, K) in enumerate(synthetic.LAYER_LINEARS):
        W = synthetic.weight_matrix(synthetic.layer_seed(77, 0, i), qt, N, K)
        layer[name] = (qt, N, K, W, oracle.fp8_weight_cache(qt, W, N, K))
    return layer


@pytest.mark.parametrize("M,rows", [
    (16, [0, 7, 15]),
    (128, [0, 45, 77, 109, 127]),
    (4096, [256 * b + (97 * b) % 256 for b in range(16)] + [4095])])
def test_full_decoder_layer_fp8_route(rq, decoder_layer, M, rows):
    """The prefill stack's four calls for one layer at M tokens, as the
    benchmark makes them (rq_linear_group for q/k/v and gate/up, rq_linear
    for o and down): every member's sampled token rows (full output rows,
    one in every band of M/16 tokens and the last) against the oracle's FP8
    route -- its weight caches, the activation's absmax and E4M3 bytes, exact
    FP8 dot products."""
    ctx = rq.Context()
    acts = {kind: synthetic.activation(5000 + 10 * M + j, M, K, outlier_frac=1e-3)
            for j, (kind, K) in enumerate((("x", 3584), ("a", 3584), ("h", 3584),
                                           ("g", 18944)))}
    dacts = {k: to_dev(v) for k, v in acts.items()}
    ys = {name: empty((M, N), torch.float32) for name, (_, N, _, _, _) in decoder_layer.items()}
    Wd = {name: to_dev(v[3]) for name, v in decoder_layer.items()}
    for grp in LAYER_CALLS:
        K = decoder_layer[grp[0]][2]
        x = dacts[LAYER_SOURCE[grp[0]]]
        if len(grp) == 1:
            qt, N = decoder_layer[grp[0]][:2]
            ctx.rq_linear(qt, Wd[grp[0]], x, ys[grp[0]], M, N, K)
        else:
            ctx.rq_linear_group([decoder_layer[n][0] for n in grp], [Wd[n] for n in grp], x,
                                [ys[n] for n in grp], [decoder_layer[n][1] for n in grp], M, K)
    assert rq.rq_get_device_status() == 0
    quant = {k: oracle.quant_e4m3(v, oracle.absmax_bits(v)) for k, v in acts.items()}
    for name, (qt, N, K, W, (wb, wd)) in decoder_layer.items():
        xb, xd = quant[LAYER_SOURCE[name]]
        ms = np.repeat(np.asarray(rows), N)
        ns = np.tile(np.arange(N), len(rows))
        ref = oracle.fp8_gemm_pairs(xb, xd, wb, wd, ms, ns).reshape(len(rows), N)
        got = ys[name].cpu().numpy()[rows]
        check_gemm(got, ref)
    ctx.close()


@pytest.mark.parametrize("M", [1, 512])
def test_decoder_layer_replayed_from_a_cuda_graph(rq, decoder_layer, M):
    """One layer's four calls (q/k/v and gate/up grouped, o and down alone)
    captured once in a CUDA graph and replayed twice with new activations
    copied into the captured buffers in between, at one token (GEMV route)
    and at 512 (FP8 route, the weight caches built before the capture):
    every member's sampled rows of each replay against the oracle."""
    ctx = rq.Context()
    kinds = (("x", 3584), ("a", 3584), ("h", 3584), ("g", 18944))
    bufs = {k: empty((M, K), torch.float32) for k, K in kinds}
    ys = {name: empty((M, N), torch.float32) for name, (_, N, _, _, _) in decoder_layer.items()}
    Wd = {name: to_dev(v[3]) for name, v in decoder_layer.items()}

    def layer(stream=None):
        if M >= ctx.gemm_threshold:
            ctx.rq_act_cache_invalidate()  # the activations are rewritten in place
        for grp in LAYER_CALLS:
            K = decoder_layer[grp[0]][2]
            x = bufs[LAYER_SOURCE[grp[0]]]
            if len(grp) == 1:
                qt, N = decoder_layer[grp[0]][:2]
                ctx.rq_linear(qt, Wd[grp[0]], x, ys[grp[0]], M, N, K, stream)
            else:
                ctx.rq_linear_group([decoder_layer[n][0] for n in grp], [Wd[n] for n in grp],
                                    x, [ys[n] for n in grp],
                                    [decoder_layer[n][1] for n in grp], M, K, stream)

    for k, K in kinds:  # warm call: caches and launch settings before capture
        bufs[k].copy_(to_dev(synthetic.activation(6000 + K, M, K)))
    layer()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer(s)
    torch.cuda.synchronize()
    rows = [0] if M == 1 else [0, 255, 511]
    for rep in range(2):
        acts = {k: synthetic.activation(6100 + 10 * rep + j, M, K, outlier_frac=1e-3)
                for j, (k, K) in enumerate(kinds)}
        for k, _ in kinds:
            bufs[k].copy_(to_dev(acts[k]))
        for y in ys.values():
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert rq.rq_get_device_status() == 0
        for name, (qt, N, K, W, (wb, wd)) in decoder_layer.items():
            x = acts[LAYER_SOURCE[name]]
            got = ys[name].cpu().numpy()[rows]
            if M == 1:
                ref, absdot = oracle.gemv(qt, W, x, N, K)
                assert gemv_ok(got, ref, absdot)[0], (rep, name)
            else:
                xb, xd = oracle.quant_e4m3(x, oracle.absmax_bits(x))
                ms = np.repeat(np.asarray(rows), N)
                ns = np.tile(np.arange(N), len(rows))
                check_gemm(got, oracle.fp8_gemm_pairs(xb, xd, wb, wd, ms, ns).reshape(len(rows), N))
    ctx.close()
