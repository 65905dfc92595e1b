"""Python binding of librq.so, the GB300 quantized linear layer.

Thin ctypes marshalling over the C ABI declared in ``include/rq.h``; every
step of the computation runs in the library's CUDA kernels.  PyTorch only
supplies device memory (``tensor.data_ptr()``) and the current CUDA stream.
There is no fallback: if ``librq.so`` has not been built, importing this
package raises ImportError.

Function names are those of the C ABI (``rq_absmax``, ``rq_quant_e4m3``,
``rq_q4k_gemv``, ``rq_q6k_gemv``, ``rq_fp8_weight_cache``, ``rq_fp8_gemm``,
``rq_linear``...); ``Context`` wraps ``rq_ctx``.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librq.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "rq.h")

RQ_Q4K = 12
RQ_Q6K = 14
STATUS = {0: "RQ_OK", 1: "RQ_ERR_NULL", 2: "RQ_ERR_SHAPE", 3: "RQ_ERR_QTYPE",
          4: "RQ_ERR_NOT_CACHED", 5: "RQ_ERR_ALLOC", 6: "RQ_ERR_CUDA",
          7: "RQ_ERR_TIMEOUT", 8: "RQ_ERR_ARCH"}


class RqError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (%d)" % (where, STATUS.get(status, "?"), status))


if not os.path.exists(LIB_PATH):
    raise ImportError(
        "librq.so is not built (expected %s); run "
        "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_SIGS = {
    "rq_abi_version": ([], _i32),
    "rq_status_string": ([_i32], ctypes.c_char_p),
    "rq_ctx_create": ([ctypes.POINTER(_vp)], _i32),
    "rq_ctx_destroy": ([_vp], None),
    "rq_ctx_set_gemm_threshold": ([_vp, _i32], _i32),
    "rq_ctx_get_gemm_threshold": ([_vp], _i32),
    "rq_ctx_get_stats": ([_vp, _vp, _vp, _vp, _vp], _i32),
    "rq_absmax": ([_vp, _i64, _vp, _vp], _i32),
    "rq_quant_e4m3": ([_vp, _i64, _vp, _vp, _vp, _vp], _i32),
    "rq_q4k_gemv": ([_vp, _vp, _vp, _i32, _i32, _i32, _vp], _i32),
    "rq_q6k_gemv": ([_vp, _vp, _vp, _i32, _i32, _i32, _vp], _i32),
    "rq_fp8_weight_cache": ([_vp, _i32, _vp, _i32, _i32, ctypes.POINTER(_vp),
                             ctypes.POINTER(_vp), _vp], _i32),
    "rq_fp8_gemm": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp], _i32),
    "rq_fp8_act_cache": ([_vp, _vp, _i32, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                          _vp], _i32),
    "rq_linear": ([_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp], _i32),
    "rq_linear_group": ([_vp, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp], _i32),
    "rq_fp8_linear_noalloc": ([_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp], _i32),
    "rq_act_cache_invalidate": ([_vp], _i32),
    "rq_ctx_trace_begin": ([_vp, _i32], _i32),
    "rq_ctx_trace_end": ([_vp, _vp, _vp], _i32),
    "rq_ctx_trace_kinds": ([_vp, ctypes.c_uint], _i32),
    "rq_get_device_status": ([_vp], _i32),
    "rq_debug_wait_timeout": ([_i64, _vp], _i32),
    "rq_gemv_exact_outputs": ([_vp, ctypes.POINTER(_i64)], _i32),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


def lib():
    return _lib


def _check(status, where):
    if status != 0:
        raise RqError(status, where)


def _ptr(t):
    """Device (or host) address of a tensor, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def rq_abi_version():
    return _lib.rq_abi_version()


def rq_absmax(x, n, absmax_bits, stream=None):
    _check(_lib.rq_absmax(_ptr(x), n, _ptr(absmax_bits), _stream(stream)), "rq_absmax")


def rq_quant_e4m3(x, n, absmax_bits, out, dequant_out, stream=None):
    _check(_lib.rq_quant_e4m3(_ptr(x), n, _ptr(absmax_bits), _ptr(out),
                              _ptr(dequant_out), _stream(stream)), "rq_quant_e4m3")


def rq_q4k_gemv(w, x, y, M, N, K, stream=None):
    _check(_lib.rq_q4k_gemv(_ptr(w), _ptr(x), _ptr(y), M, N, K, _stream(stream)),
           "rq_q4k_gemv")


def rq_q6k_gemv(w, x, y, M, N, K, stream=None):
    _check(_lib.rq_q6k_gemv(_ptr(w), _ptr(x), _ptr(y), M, N, K, _stream(stream)),
           "rq_q6k_gemv")


def rq_fp8_gemm(x_fp8, x_dequant, w_fp8, w_dequant, y, M, N, K, stream=None):
    _check(_lib.rq_fp8_gemm(_ptr(x_fp8), _ptr(x_dequant), _ptr(w_fp8), _ptr(w_dequant),
                            _ptr(y), M, N, K, _stream(stream)), "rq_fp8_gemm")


NOALLOC_MAX_ACT_BYTES = 8 * 1024 * 1024


def rq_fp8_linear_noalloc(x, w_fp8, w_dequant, y, M, N, K, stream=None):
    """FP8 linear layer that allocates nothing (for callers that may not call
    cudaMalloc while serving): the activation's E4M3 copy lives in a fixed
    array inside the library, so (M rounded up to 16) * K must not exceed
    NOALLOC_MAX_ACT_BYTES.  w_fp8 / w_dequant are device tensors or the
    addresses Context.rq_fp8_weight_cache returns."""
    _check(_lib.rq_fp8_linear_noalloc(_ptr(x), _ptr(w_fp8), _ptr(w_dequant), _ptr(y), M, N,
                                      K, _stream(stream)), "rq_fp8_linear_noalloc")


def rq_get_device_status(stream=None):
    """Synchronise the stream; return the status code (0 = ok, 7 = timeout)."""
    return _lib.rq_get_device_status(_stream(stream))


def rq_debug_wait_timeout(limit_ns, stream=None):
    _check(_lib.rq_debug_wait_timeout(limit_ns, _stream(stream)), "rq_debug_wait_timeout")


def rq_gemv_exact_outputs(stream=None):
    """Synchronise the stream; return (and reset) how many GEMV outputs were
    recomputed on the exact fp64 path since the last call."""
    n = _i64()
    _check(_lib.rq_gemv_exact_outputs(_stream(stream), ctypes.byref(n)),
           "rq_gemv_exact_outputs")
    return n.value


class Context:
    """Owns an rq_ctx: FP8 weight cache, activation scratch, device scalars."""

    def __init__(self, gemm_threshold=None):
        h = _vp()
        _check(_lib.rq_ctx_create(ctypes.byref(h)), "rq_ctx_create")
        self._h = h
        if gemm_threshold is not None:
            self.set_gemm_threshold(gemm_threshold)

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            _lib.rq_ctx_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_gemm_threshold(self, m):
        _check(_lib.rq_ctx_set_gemm_threshold(self._h, m), "rq_ctx_set_gemm_threshold")

    @property
    def gemm_threshold(self):
        return _lib.rq_ctx_get_gemm_threshold(self._h)

    def stats(self):
        vals = [_i64() for _ in range(4)]
        _check(_lib.rq_ctx_get_stats(self._h, *[ctypes.byref(v) for v in vals]),
               "rq_ctx_get_stats")
        hits, misses, nw, nbytes = (v.value for v in vals)
        return {"act_hits": hits, "act_misses": misses, "weights": nw,
                "weight_bytes": nbytes}

    def rq_fp8_weight_cache(self, qtype, w, N, K, stream=None):
        """-> (device address of E4M3 [N x K], device address of the scale)."""
        wq = _vp()
        wd = _vp()
        _check(_lib.rq_fp8_weight_cache(self._h, qtype, _ptr(w), N, K, ctypes.byref(wq),
                                        ctypes.byref(wd), _stream(stream)),
               "rq_fp8_weight_cache")
        return wq.value, wd.value

    def rq_fp8_act_cache(self, x, M, K, stream=None):
        """-> (device address of E4M3 [M_pad x K], device address of the scale)."""
        xq = _vp()
        xd = _vp()
        _check(_lib.rq_fp8_act_cache(self._h, _ptr(x), M, K, ctypes.byref(xq),
                                     ctypes.byref(xd), _stream(stream)),
               "rq_fp8_act_cache")
        return xq.value, xd.value

    def rq_linear_group(self, qtypes, ws, x, ys, Ns, M, K, stream=None):
        """Linears sharing x: ys[i] = x . ws[i]^T, one call."""
        n = len(qtypes)
        qt = (_i32 * n)(*qtypes)
        wp = (_vp * n)(*[_ptr(w) for w in ws])
        yp = (_vp * n)(*[_ptr(y) for y in ys])
        nn = (_i32 * n)(*Ns)
        _check(_lib.rq_linear_group(self._h, n, qt, wp, _ptr(x), yp, nn, M, K,
                                    _stream(stream)), "rq_linear_group")

    def rq_linear(self, qtype, w, x, y, M, N, K, stream=None):
        _check(_lib.rq_linear(self._h, qtype, _ptr(w), _ptr(x), _ptr(y), M, N, K,
                              _stream(stream)), "rq_linear")

    TRACE_KINDS = ("gemv", "absmax", "quant", "gemm", "wcache")

    def rq_ctx_trace_begin(self, capacity):
        _check(_lib.rq_ctx_trace_begin(self._h, capacity), "rq_ctx_trace_begin")

    def rq_ctx_trace_kinds(self, kinds):
        """Trace only the named kinds (a subset of TRACE_KINDS)."""
        mask = 0
        for k in kinds:
            mask |= 1 << self.TRACE_KINDS.index(k)
        _check(_lib.rq_ctx_trace_kinds(self._h, mask), "rq_ctx_trace_kinds")

    def rq_ctx_trace_end(self):
        """-> {kind: (kernel count, summed device ms)}"""
        counts = (_i64 * 5)()
        ms = (ctypes.c_double * 5)()
        _check(_lib.rq_ctx_trace_end(self._h, counts, ms), "rq_ctx_trace_end")
        return {k: (counts[i], ms[i]) for i, k in enumerate(self.TRACE_KINDS)}

    def rq_act_cache_invalidate(self):
        _check(_lib.rq_act_cache_invalidate(self._h), "rq_act_cache_invalidate")
