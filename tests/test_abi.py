"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rq.h")


@pytest.fixture(scope="module")
def rq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_linear_layers_gb300 as rq
    return rq


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(rq_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("rq_absmax", "rq_quant_e4m3", "rq_q4k_gemv", "rq_q6k_gemv",
                     "rq_fp8_weight_cache", "rq_fp8_gemm", "rq_linear",
                     "rq_ctx_create", "rq_ctx_destroy", "rq_act_cache_invalidate",
                     "rq_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(rq):
    lib = ctypes.CDLL(rq.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(rq.EXPORTED) == set(declared_functions())


def test_abi_version_and_status_strings(rq):
    lib = rq.lib()
    assert lib.rq_abi_version() == 1
    for s in range(9):
        assert lib.rq_status_string(s)


def test_library_does_not_link_the_oracle(rq):
    import subprocess
    out = subprocess.run(["ldd", rq.LIB_PATH], capture_output=True, text=True).stdout
    assert "oracle" not in out
    syms = subprocess.run(["nm", "-D", rq.LIB_PATH], capture_output=True, text=True).stdout
    assert "orc_" not in syms


NULL = None


def test_null_pointers_rejected_before_launch(rq):
    lib = rq.lib()
    fake = 0x1000  # never dereferenced: validation fails first
    assert lib.rq_absmax(NULL, 16, fake, NULL) == 1
    assert lib.rq_absmax(fake, 16, NULL, NULL) == 1
    assert lib.rq_quant_e4m3(fake, 16, NULL, fake, fake, NULL) == 1
    assert lib.rq_quant_e4m3(fake, 16, fake, fake, NULL, NULL) == 1
    assert lib.rq_q4k_gemv(NULL, fake, fake, 1, 8, 256, NULL) == 1
    assert lib.rq_q6k_gemv(NULL, fake, fake, 1, 8, 256, NULL) == 1
    assert lib.rq_fp8_gemm(fake, fake, NULL, fake, fake, 16, 128, 128, NULL) == 1
    assert lib.rq_linear(NULL, 12, fake, fake, fake, 1, 8, 256, NULL) == 1
    assert lib.rq_fp8_weight_cache(NULL, 12, fake, 8, 256, NULL, NULL, NULL) == 1
    out = ctypes.byref(ctypes.c_void_p())
    assert lib.rq_fp8_act_cache(NULL, fake, 16, 128, out, out, NULL) == 1
    assert lib.rq_fp8_act_cache(fake, NULL, 16, 128, out, out, NULL) == 1
    assert lib.rq_fp8_act_cache(fake, fake, 16, 128, NULL, out, NULL) == 1
    assert lib.rq_ctx_create(NULL) == 1
    assert lib.rq_act_cache_invalidate(NULL) == 1
    assert lib.rq_ctx_set_gemm_threshold(NULL, 4) == 1
    assert lib.rq_ctx_get_gemm_threshold(NULL) == -1
    assert lib.rq_ctx_trace_kinds(NULL, 1) == 1
    assert lib.rq_linear_group(NULL, 2, fake, fake, fake, fake, fake, 1, 256, NULL) == 1
    lib.rq_ctx_destroy(NULL)  # no-op


def test_bad_shapes_rejected_before_launch(rq):
    lib = rq.lib()
    a = 0x10000  # 64 KiB aligned fake address
    assert lib.rq_absmax(a, -1, a, NULL) == 2
    assert lib.rq_absmax(a, 8, a + 2, NULL) == 2          # misaligned word
    for M, N, K in ((0, 8, 256), (9, 8, 256), (1, 0, 256), (1, 8, 255),
                    (1, 8, 0), (1, 8, 384)):
        assert lib.rq_q4k_gemv(a, a, a, M, N, K, NULL) == 2, (M, N, K)
        assert lib.rq_q6k_gemv(a, a, a, M, N, K, NULL) == 2, (M, N, K)
    assert lib.rq_q4k_gemv(a + 4, a, a, 1, 8, 256, NULL) == 2   # Q4_K needs 16 B
    assert lib.rq_q4k_gemv(a, a + 4, a, 1, 8, 256, NULL) == 2   # x needs 16 B
    assert lib.rq_q6k_gemv(a + 2, a, a, 1, 8, 256, NULL) == 2   # Q6_K needs 4 B
    assert lib.rq_q4k_gemv(a, a, a, 8, 8, 65536, NULL) == 2     # x sums > smem
    for M, N, K in ((0, 128, 128), (16, 0, 128), (16, 128, 64), (16, 128, 200)):
        assert lib.rq_fp8_gemm(a, a, a, a, a, M, N, K, NULL) == 2, (M, N, K)
    assert lib.rq_fp8_gemm(a + 8, a, a, a, a, 16, 128, 128, NULL) == 2  # TMA: 16 B
    assert lib.rq_debug_wait_timeout(0, NULL) == 2
    out = ctypes.byref(ctypes.c_void_p())
    fake_ctx = ctypes.c_void_p(a)  # not dereferenced: shape checks come first
    assert lib.rq_fp8_act_cache(fake_ctx, a, 0, 128, out, out, NULL) == 2
    assert lib.rq_fp8_act_cache(fake_ctx, a, 16, 0, out, out, NULL) == 2
    assert lib.rq_fp8_act_cache(fake_ctx, a + 4, 16, 128, out, out, NULL) == 2


def test_bad_qtype_rejected(rq):
    lib = rq.lib()
    a = 0x10000
    fake_ctx = ctypes.c_void_p(a)  # not dereferenced: qtype check comes first
    assert lib.rq_linear(fake_ctx, 2, a, a, a, 16, 8, 256, NULL) == 3
    assert lib.rq_fp8_weight_cache(fake_ctx, 99, a, 8, 256, ctypes.byref(ctypes.c_void_p()),
                                   ctypes.byref(ctypes.c_void_p()), NULL) == 3
