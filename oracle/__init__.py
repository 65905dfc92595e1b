"""CPU oracle for the quantized linear layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product (the CUDA library
``librq.so`` and its binding) neither imports it nor shares any code with it.

The arithmetic lives in ``oracle.c`` (plain C, compiled without fast-math or
FMA contraction); this module only marshals numpy arrays into it.  Each C
function cites the passage of the source pages it follows (realizar 0.8.4,
``cublas_prefill/gemm.rs``, ``cublas_prefill/mod.rs``,
``q6k_gemv_indexed.rs``).
"""
import ctypes
import os

import numpy as np

from . import build as _build

Q4K = 12
Q6K = 14
QK = 256
BLOCK_BYTES = {Q4K: 144, Q6K: 210}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c_u8p = ctypes.POINTER(ctypes.c_uint8)
        c_fp = ctypes.POINTER(ctypes.c_float)
        c_dp = ctypes.POINTER(ctypes.c_double)
        c_i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_absmax_bits.argtypes = [c_fp, i64]
        L.orc_absmax_bits.restype = ctypes.c_uint32
        L.orc_scales.argtypes = [ctypes.c_uint32, c_fp, c_fp]
        L.orc_scales.restype = None
        L.orc_encode_scaled.argtypes = [ctypes.c_float, ctypes.c_float]
        L.orc_encode_scaled.restype = ctypes.c_uint8
        L.orc_quant_e4m3.argtypes = [c_fp, i64, ctypes.c_uint32, c_u8p, c_fp]
        L.orc_quant_e4m3.restype = None
        L.orc_half_to_float.argtypes = [ctypes.c_uint16]
        L.orc_half_to_float.restype = ctypes.c_float
        L.orc_q4k_scale_min.argtypes = [c_u8p, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(ctypes.c_int)]
        L.orc_q4k_scale_min.restype = None
        for name in ("orc_q4k_decode_block", "orc_q6k_decode_block"):
            getattr(L, name).argtypes = [c_u8p, c_fp]
            getattr(L, name).restype = None
        for name in ("orc_q4k_decode_block_f64", "orc_q6k_decode_block_f64"):
            getattr(L, name).argtypes = [c_u8p, c_dp]
            getattr(L, name).restype = None
        L.orc_dequant.argtypes = [ctypes.c_int, c_u8p, i64, i64, c_fp]
        L.orc_dequant.restype = ctypes.c_int
        L.orc_gemv_rows.argtypes = [ctypes.c_int, c_u8p, c_fp, i64, i64, i64,
                                    c_i64p, i64, c_dp, c_dp]
        L.orc_gemv_rows.restype = ctypes.c_int
        L.orc_gemv.argtypes = [ctypes.c_int, c_u8p, c_fp, i64, i64, i64,
                               c_dp, c_dp]
        L.orc_gemv.restype = ctypes.c_int
        L.orc_fp8_gemm_pairs.argtypes = [c_u8p, ctypes.c_float, c_u8p,
                                         ctypes.c_float, i64, i64, i64,
                                         c_i64p, c_i64p, i64, c_dp]
        L.orc_fp8_gemm_pairs.restype = ctypes.c_int
        L.orc_fp8_gemm.argtypes = [c_u8p, ctypes.c_float, c_u8p,
                                   ctypes.c_float, i64, i64, i64, c_dp]
        L.orc_fp8_gemm.restype = ctypes.c_int
        L.orc_fp8_weight_cache.argtypes = [ctypes.c_int, c_u8p, i64, i64,
                                           c_fp, c_u8p, c_fp]
        L.orc_fp8_weight_cache.restype = ctypes.c_int
        L.orc_e4m3_encode_array.argtypes = [c_fp, i64, c_u8p]
        L.orc_e4m3_encode_array.restype = None
        L.orc_encode_scaled_array.argtypes = [c_fp, i64, ctypes.c_float, c_u8p]
        L.orc_encode_scaled_array.restype = None
        L.orc_e4m3_decode_array.argtypes = [c_u8p, i64, c_dp]
        L.orc_e4m3_decode_array.restype = None
        L.orc_half_to_float_array.argtypes = [
            ctypes.POINTER(ctypes.c_uint16), i64, c_fp]
        L.orc_half_to_float_array.restype = None
        L.orc_route_is_gemm.argtypes = [i64, i64]
        L.orc_route_is_gemm.restype = ctypes.c_int
        L.orc_pad_m.argtypes = [i64]
        L.orc_pad_m.restype = i64
        _lib = L
    return _lib


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# ---------------------------------------------------------------- E4M3 ----

def e4m3_decode(b):
    """Value of E4M3 byte(s) as float64 (NaN for 0x7F / 0xFF)."""
    arr = np.asarray(b, dtype=np.uint8)
    flat = np.ascontiguousarray(arr.ravel())
    out = np.empty(flat.size, dtype=np.float64)
    lib().orc_e4m3_decode_array(_p(flat, ctypes.c_uint8), flat.size,
                                _p(out, ctypes.c_double))
    return out.reshape(arr.shape) if arr.shape else float(out[0])


def e4m3_encode(v):
    """Unscaled FP32 -> E4M3 encoder applied elementwise."""
    arr = np.asarray(v, dtype=np.float32)
    flat = np.ascontiguousarray(arr.ravel())
    out = np.empty(flat.size, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_p(flat, ctypes.c_float), flat.size,
                                _p(out, ctypes.c_uint8))
    return out.reshape(arr.shape) if arr.shape else int(out[0])


def e4m3_encode_bits(bits):
    """Encoder applied to fp32 bit patterns (uint32 array)."""
    f = np.asarray(bits, dtype=np.uint32).view(np.float32)
    return e4m3_encode(f)


def absmax_bits(x):
    x = _c(x, np.float32).ravel()
    return int(lib().orc_absmax_bits(_p(x, ctypes.c_float), x.size))


def scales(absmax_bits_value):
    q = ctypes.c_float()
    d = ctypes.c_float()
    lib().orc_scales(ctypes.c_uint32(absmax_bits_value), ctypes.byref(q),
                     ctypes.byref(d))
    return np.float32(q.value), np.float32(d.value)


def encode_scaled(x, s):
    arr = np.asarray(x, dtype=np.float32)
    flat = np.ascontiguousarray(arr.ravel())
    out = np.empty(flat.size, dtype=np.uint8)
    lib().orc_encode_scaled_array(_p(flat, ctypes.c_float), flat.size,
                                  float(np.float32(s)),
                                  _p(out, ctypes.c_uint8))
    return out.reshape(arr.shape)


def quant_e4m3(x, absmax_bits_value):
    """Scaled quantization of x with the given absmax bits -> (bytes, deq)."""
    x = _c(x, np.float32)
    flat = x.ravel()
    out = np.empty(flat.size, dtype=np.uint8)
    deq = ctypes.c_float()
    lib().orc_quant_e4m3(_p(flat, ctypes.c_float), flat.size,
                         ctypes.c_uint32(absmax_bits_value),
                         _p(out, ctypes.c_uint8), ctypes.byref(deq))
    return out.reshape(x.shape), np.float32(deq.value)


# ---------------------------------------------------------------- GGUF ----

def half_to_float(h):
    arr = np.asarray(h, dtype=np.uint16)
    flat = np.ascontiguousarray(arr.ravel())
    out = np.empty(flat.size, dtype=np.float32)
    lib().orc_half_to_float_array(_p(flat, ctypes.c_uint16), flat.size,
                                  _p(out, ctypes.c_float))
    return out.reshape(arr.shape)


def q4k_scale_min(scales12, j):
    s = _c(scales12, np.uint8)
    sc = ctypes.c_int()
    mn = ctypes.c_int()
    lib().orc_q4k_scale_min(_p(s, ctypes.c_uint8), j, ctypes.byref(sc),
                            ctypes.byref(mn))
    return sc.value, mn.value


def decode_block(qtype, blk, exact=False):
    blk = _c(blk, np.uint8)
    if qtype == Q4K:
        fn32, fn64 = lib().orc_q4k_decode_block, lib().orc_q4k_decode_block_f64
    elif qtype == Q6K:
        fn32, fn64 = lib().orc_q6k_decode_block, lib().orc_q6k_decode_block_f64
    else:
        raise ValueError(qtype)
    if exact:
        out = np.empty(QK, dtype=np.float64)
        fn64(_p(blk, ctypes.c_uint8), _p(out, ctypes.c_double))
    else:
        out = np.empty(QK, dtype=np.float32)
        fn32(_p(blk, ctypes.c_uint8), _p(out, ctypes.c_float))
    return out


def dequant(qtype, W, N, K):
    W = _c(W, np.uint8)
    out = np.empty((N, K), dtype=np.float32)
    rc = lib().orc_dequant(qtype, _p(W, ctypes.c_uint8), N, K,
                           _p(out, ctypes.c_float))
    if rc:
        raise ValueError("orc_dequant rc=%d" % rc)
    return out


def gemv(qtype, W, x, N, K):
    """Full fp64 GEMV -> (y [M,N] float64, absdot [M,N])."""
    W = _c(W, np.uint8)
    x = _c(x, np.float32)
    M = x.shape[0] if x.ndim == 2 else 1
    y = np.empty((M, N), dtype=np.float64)
    a = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_gemv(qtype, _p(W, ctypes.c_uint8), _p(x, ctypes.c_float),
                        M, N, K, _p(y, ctypes.c_double), _p(a, ctypes.c_double))
    if rc:
        raise ValueError("orc_gemv rc=%d" % rc)
    return y, a


def gemv_rows(qtype, W, x, N, K, rows):
    """fp64 GEMV for selected rows -> (y [M,len(rows)], absdot)."""
    W = _c(W, np.uint8)
    x = _c(x, np.float32)
    rows = _c(rows, np.int64)
    M = x.shape[0] if x.ndim == 2 else 1
    y = np.empty((M, rows.size), dtype=np.float64)
    a = np.empty((M, rows.size), dtype=np.float64)
    rc = lib().orc_gemv_rows(qtype, _p(W, ctypes.c_uint8),
                             _p(x, ctypes.c_float), M, N, K,
                             _p(rows, ctypes.c_int64), rows.size,
                             _p(y, ctypes.c_double), _p(a, ctypes.c_double))
    if rc:
        raise ValueError("orc_gemv_rows rc=%d" % rc)
    return y, a


# ---------------------------------------------------------------- GEMM ----

def fp8_gemm(Xb, x_deq, Wb, w_deq):
    Xb = _c(Xb, np.uint8)
    Wb = _c(Wb, np.uint8)
    M, K = Xb.shape
    N = Wb.shape[0]
    Y = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_fp8_gemm(_p(Xb, ctypes.c_uint8), float(x_deq),
                            _p(Wb, ctypes.c_uint8), float(w_deq), M, N, K,
                            _p(Y, ctypes.c_double))
    if rc:
        raise ValueError("orc_fp8_gemm rc=%d" % rc)
    return Y


def fp8_gemm_pairs(Xb, x_deq, Wb, w_deq, ms, ns):
    Xb = _c(Xb, np.uint8)
    Wb = _c(Wb, np.uint8)
    M, K = Xb.shape
    N = Wb.shape[0]
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    y = np.empty(ms.size, dtype=np.float64)
    rc = lib().orc_fp8_gemm_pairs(_p(Xb, ctypes.c_uint8), float(x_deq),
                                  _p(Wb, ctypes.c_uint8), float(w_deq), M, N,
                                  K, _p(ms, ctypes.c_int64),
                                  _p(ns, ctypes.c_int64), ms.size,
                                  _p(y, ctypes.c_double))
    if rc:
        raise ValueError("orc_fp8_gemm_pairs rc=%d" % rc)
    return y


def fp8_weight_cache(qtype, W, N, K):
    """-> (E4M3 bytes [N,K], w_deq float32)."""
    W = _c(W, np.uint8)
    scratch = np.empty(N * K, dtype=np.float32)
    out = np.empty((N, K), dtype=np.uint8)
    deq = ctypes.c_float()
    rc = lib().orc_fp8_weight_cache(qtype, _p(W, ctypes.c_uint8), N, K,
                                    _p(scratch, ctypes.c_float),
                                    _p(out, ctypes.c_uint8), ctypes.byref(deq))
    if rc:
        raise ValueError("orc_fp8_weight_cache rc=%d" % rc)
    return out, np.float32(deq.value)


def route_is_gemm(M, threshold):
    return bool(lib().orc_route_is_gemm(M, threshold))


def pad_m(M):
    return int(lib().orc_pad_m(M))
