"""Q4_K / Q6_K super-block packers for the tests, written from the GGUF layout
description (the inverse of decoding), independently of the oracle's and the
kernels' decoders."""
import numpy as np


def pack_scale_min(sc, mn):
    """8 six-bit scales and mins -> the 12 packed bytes of a Q4_K block."""
    b = np.zeros(12, dtype=np.int64)
    for j in range(4):
        b[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        b[j + 4] = (mn[j] & 63) | ((mn[j + 4] >> 4) << 6)
        b[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return b.astype(np.uint8)


def pack_q4k(d, dmin, sc, mn, q):
    """Block from fp16 d/dmin, 8 scales, 8 mins, 256 quants (0..15)."""
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.array([d], np.float16).view(np.uint8)
    blk[2:4] = np.array([dmin], np.float16).view(np.uint8)
    blk[4:16] = pack_scale_min(sc, mn)
    qs = np.zeros(128, dtype=np.int64)
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    blk[16:144] = qs.astype(np.uint8)
    return blk


def pack_q6k(d, scales, q):
    """Block from fp16 d, 16 int8 scales, 256 quants (0..63)."""
    ql = np.zeros(128, np.int64)
    qh = np.zeros(64, np.int64)
    for h in range(2):
        for l in range(32):
            q0, q1, q2, q3 = (q[128 * h + l], q[128 * h + 32 + l],
                              q[128 * h + 64 + l], q[128 * h + 96 + l])
            ql[64 * h + l] = (q0 & 15) | ((q2 & 15) << 4)
            ql[64 * h + 32 + l] = (q1 & 15) | ((q3 & 15) << 4)
            qh[32 * h + l] = ((q0 >> 4) | ((q1 >> 4) << 2) | ((q2 >> 4) << 4)
                              | ((q3 >> 4) << 6))
    blk = np.zeros(210, np.uint8)
    blk[0:128] = ql.astype(np.uint8)
    blk[128:192] = qh.astype(np.uint8)
    blk[192:208] = np.asarray(scales, np.int8).view(np.uint8)
    blk[208:210] = np.array([d], np.float16).view(np.uint8)
    return blk


def q6_scale_slot(i):
    h, r = divmod(i, 128)
    quarter, l = divmod(r, 32)
    return 8 * h + l // 16 + 2 * quarter


def pack_q4k_matrix(d, dmin, sc, mn, q):
    """Vectorised pack_q4k over a matrix: d, dmin [N, nsb]; sc, mn [N, nsb, 8];
    q [N, nsb, 256] (0..15) -> uint8 [N, nsb * 144]."""
    d = np.asarray(d, np.float64)
    N, nsb = d.shape
    sc = np.asarray(sc, np.int64)
    mn = np.asarray(mn, np.int64)
    q = np.asarray(q, np.int64)
    blk = np.zeros((N, nsb, 144), np.uint8)
    blk[..., 0:2] = d.astype(np.float16)[..., None].view(np.uint8)
    blk[..., 2:4] = np.asarray(dmin, np.float64).astype(np.float16)[..., None].view(np.uint8)
    s = np.zeros((N, nsb, 12), np.int64)
    for j in range(4):
        s[..., j] = (sc[..., j] & 63) | ((sc[..., j + 4] >> 4) << 6)
        s[..., j + 4] = (mn[..., j] & 63) | ((mn[..., j + 4] >> 4) << 6)
        s[..., j + 8] = (sc[..., j + 4] & 15) | ((mn[..., j + 4] & 15) << 4)
    blk[..., 4:16] = s.astype(np.uint8)
    qc = q.reshape(N, nsb, 4, 2, 32)
    blk[..., 16:144] = (qc[:, :, :, 0, :] | (qc[:, :, :, 1, :] << 4)).reshape(N, nsb, 128)
    return blk.reshape(N, nsb * 144)


def pack_q6k_matrix(d, scales, q):
    """Vectorised pack_q6k: d [N, nsb]; scales [N, nsb, 16] (int8 range);
    q [N, nsb, 256] (0..63) -> uint8 [N, nsb * 210]."""
    d = np.asarray(d, np.float64)
    N, nsb = d.shape
    q = np.asarray(q, np.int64).reshape(N, nsb, 2, 4, 32)  # half, quarter, l
    ql = np.zeros((N, nsb, 2, 64), np.int64)
    ql[..., 0:32] = (q[:, :, :, 0] & 15) | ((q[:, :, :, 2] & 15) << 4)
    ql[..., 32:64] = (q[:, :, :, 1] & 15) | ((q[:, :, :, 3] & 15) << 4)
    qh = ((q[:, :, :, 0] >> 4) | ((q[:, :, :, 1] >> 4) << 2) | ((q[:, :, :, 2] >> 4) << 4)
          | ((q[:, :, :, 3] >> 4) << 6))
    blk = np.zeros((N, nsb, 210), np.uint8)
    blk[..., 0:128] = ql.reshape(N, nsb, 128).astype(np.uint8)
    blk[..., 128:192] = qh.reshape(N, nsb, 64).astype(np.uint8)
    blk[..., 192:208] = np.asarray(scales, np.int64).astype(np.int8).view(np.uint8)
    blk[..., 208:210] = d.astype(np.float16)[..., None].view(np.uint8)
    return blk.reshape(N, nsb * 210)
