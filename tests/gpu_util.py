"""Shared helpers for the GPU parity tests (device transfers, tolerances)."""
import numpy as np


def dev():
    import torch
    return torch.device("cuda:0")


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def empty(shape, dtype):
    import torch
    return torch.empty(shape, dtype=dtype, device=dev())


def u32(t):
    """First element of a device int32 tensor as an unsigned bit pattern."""
    return int(t.cpu().numpy().view(np.uint32).ravel()[0])


def gemv_ok(got, ref, absdot):
    """Decode GEMV bound: |gpu - ref| <= 1e-4 * sum_k |x_k w_k| per element."""
    err = np.abs(np.asarray(got, np.float64) - ref)
    bound = 1e-4 * absdot
    return bool(np.all(err <= bound)), float(np.max(err / np.maximum(bound, 1e-300)))


def gemm_ok(got, ref, row_rms):
    """FP8 GEMM bound: |gpu - ref| <= 2e-3*|ref| + 1e-3*rms(row of ref)."""
    got = np.asarray(got, np.float64)
    bound = 2e-3 * np.abs(ref) + 1e-3 * row_rms
    err = np.abs(got - ref)
    return bool(np.all(err <= bound)), float(np.max(err / np.maximum(bound, 1e-300)))


def random_e4m3(seed, shape):
    """Random E4M3 bytes without the NaN codes 0x7F / 0xFF."""
    import synthetic
    n = int(np.prod(shape))
    b = synthetic.random_bytes(seed, n)
    b[(b & 0x7F) == 0x7F] ^= 0x01
    return b.reshape(shape)


class _DevBuf:
    """Exposes a raw device allocation through __cuda_array_interface__."""

    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {
            "shape": (n,), "typestr": typestr, "data": (int(ptr), False),
            "version": 3, "strides": None}


def device_view(ptr, n, dtype):
    """torch tensor viewing n elements at a raw device address (no copy)."""
    import torch
    typestr = {torch.uint8: "|u1", torch.float32: "<f4"}[dtype]
    return torch.as_tensor(_DevBuf(ptr, n, typestr), device=dev())
