"""Seeded synthetic inputs for the quantized linear layer.

This module is the one piece shared by the oracle side (tests, CPU baseline)
and the CUDA side (tests, benchmark): it only produces input bytes and floats
and holds none of the method's arithmetic (no decoding, scaling, encoding or
dot products).

Random numbers come from a counter-based SplitMix64 (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014; the constants
of Vigna's public-domain splitmix64): output i of stream `seed` is
mix(seed + (i + 1) * 0x9E3779B97F4A7C15).  Normal variates use the Box-Muller
transform.  Everything is vectorised numpy on uint64 with wrap-around, so the
same seed gives the same bytes on any machine.

Workload shapes (a 7B-class decoder: hidden 3584, intermediate 18944, 28 heads
with 4 KV heads of dim 128, so k/v have 512 rows) follow the decode and
prefill configurations of the benchmark; the pages themselves give only the
block sizes (144 bytes per 256 Q4_K weights).
"""
import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

HIDDEN = 3584
INTERMEDIATE = 18944
KV_DIM = 512
N_LAYERS = 28
Q4K = 12
Q6K = 14
Q4K_BLOCK = 144
Q6K_BLOCK = 210
QK = 256

# (name, qtype, N, K) of the seven linears of one decoder layer.
LAYER_LINEARS = (
    ("q", Q4K, HIDDEN, HIDDEN),
    ("k", Q4K, KV_DIM, HIDDEN),
    ("v", Q6K, KV_DIM, HIDDEN),
    ("o", Q4K, HIDDEN, HIDDEN),
    ("gate", Q4K, INTERMEDIATE, HIDDEN),
    ("up", Q4K, INTERMEDIATE, HIDDEN),
    ("down", Q4K, HIDDEN, INTERMEDIATE),
)


def _mix(z, tmp=None):
    """SplitMix64 finaliser, in place on a uint64 array (tmp: scratch of the
    same size; reusing buffers avoids first-touch page faults)."""
    if tmp is None:
        tmp = np.empty_like(z)
    with np.errstate(over="ignore"):
        np.right_shift(z, np.uint64(30), out=tmp)
        np.bitwise_xor(z, tmp, out=z)
        np.multiply(z, _M1, out=z)
        np.right_shift(z, np.uint64(27), out=tmp)
        np.bitwise_xor(z, tmp, out=z)
        np.multiply(z, _M2, out=z)
        np.right_shift(z, np.uint64(31), out=tmp)
        np.bitwise_xor(z, tmp, out=z)
    return z


def substream(seed, tag):
    """Seed of an independent stream derived from (seed, tag)."""
    z = np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF)], dtype=np.uint64)
    with np.errstate(over="ignore"):
        z += np.uint64(tag & 0xFFFFFFFFFFFFFFFF) * GOLDEN
        z += GOLDEN
    return int(_mix(z)[0])


def u64(seed, n, offset=0):
    """n consecutive SplitMix64 outputs of stream `seed`, starting at offset."""
    out = np.empty(n, dtype=np.uint64)
    base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    step = min(n, _CHUNK)
    ramp = np.arange(1, step + 1, dtype=np.uint64)
    tmp = np.empty(step, dtype=np.uint64)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        z = out[lo:hi]
        with np.errstate(over="ignore"):
            np.add(ramp[:hi - lo], np.uint64(offset + lo), out=z)
            np.multiply(z, GOLDEN, out=z)
            np.add(z, base, out=z)
        _mix(z, tmp[:hi - lo])
    return out


def random_bytes(seed, n):
    """n uniformly random bytes (little-endian bytes of the u64 stream)."""
    words = u64(seed, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def uniform(seed, n, lo=0.0, hi=1.0):
    """float64 uniform in [lo, hi) from the top 53 bits of each output."""
    u = (u64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return lo + (hi - lo) * u


def normal_f32(seed, n):
    """n standard normal float32 values (Box-Muller on pairs of uniforms)."""
    m = (n + 1) // 2
    w = u64(seed, 2 * m)
    u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return z[:n].astype(np.float32)


def activation(seed, M, K, outlier_frac=0.0, outlier_scale=50.0):
    """f32 [M, K] N(0,1) activations; a seeded `outlier_frac` of positions
    (without repeats) multiplied by `outlier_scale`."""
    x = normal_f32(substream(seed, 1), M * K)
    n_out = int(round(outlier_frac * M * K))
    if n_out:
        pos = outlier_positions(substream(seed, 2), M * K, n_out)
        x[pos] *= np.float32(outlier_scale)
    return x.reshape(M, K)


def outlier_positions(seed, n, count):
    """`count` distinct positions in [0, n), seeded."""
    chosen = np.empty(0, dtype=np.int64)
    offset = 0
    while chosen.size < count:
        cand = (u64(seed, 2 * count, offset) % np.uint64(n)).astype(np.int64)
        offset += 2 * count
        chosen = np.unique(np.concatenate([chosen, cand]))
    # unique() sorts; keep a seeded but order-free subset of exactly `count`
    keep = np.argsort(u64(substream(seed, 7), chosen.size))[:count]
    return np.sort(chosen[keep])


def _fp16_bits(values):
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def q4k_matrix(seed, N, K):
    """Packed GGUF Q4_K weights, uint8 [N, K/256*144].

    Per 144-byte super-block: bytes 0-1 fp16 d and 2-3 fp16 dmin, each
    uniform in [1e-3, 1e-2]; bytes 4-15 (packed 6-bit scales/mins) and
    16-143 (4-bit quants) uniformly random bytes."""
    assert K % QK == 0
    nsb = K // QK
    nblk = N * nsb
    blocks = random_bytes(substream(seed, 11), nblk * Q4K_BLOCK)
    blocks = blocks.reshape(nblk, Q4K_BLOCK)
    d = _fp16_bits(uniform(substream(seed, 12), nblk, 1e-3, 1e-2))
    dmin = _fp16_bits(uniform(substream(seed, 13), nblk, 1e-3, 1e-2))
    blocks[:, 0:2] = d.view(np.uint8).reshape(nblk, 2)
    blocks[:, 2:4] = dmin.view(np.uint8).reshape(nblk, 2)
    return blocks.reshape(N, nsb * Q4K_BLOCK)


def q6k_matrix(seed, N, K):
    """Packed GGUF Q6_K weights, uint8 [N, K/256*210].

    Per 210-byte super-block: ql[128] and qh[64] uniformly random bytes,
    16 int8 scales uniform on the integers -32..31, fp16 d uniform in
    [1e-3, 1e-2] (bytes 208-209)."""
    assert K % QK == 0
    nsb = K // QK
    nblk = N * nsb
    blocks = random_bytes(substream(seed, 21), nblk * Q6K_BLOCK)
    blocks = blocks.reshape(nblk, Q6K_BLOCK)
    sc = (u64(substream(seed, 22), nblk * 16) % np.uint64(64)).astype(np.int64) - 32
    blocks[:, 192:208] = sc.astype(np.int8).view(np.uint8).reshape(nblk, 16)
    d = _fp16_bits(uniform(substream(seed, 23), nblk, 1e-3, 1e-2))
    blocks[:, 208:210] = d.view(np.uint8).reshape(nblk, 2)
    return blocks.reshape(N, nsb * Q6K_BLOCK)


def weight_matrix(seed, qtype, N, K):
    if qtype == Q4K:
        return q4k_matrix(seed, N, K)
    if qtype == Q6K:
        return q6k_matrix(seed, N, K)
    raise ValueError("unknown qtype %r" % (qtype,))


def layer_seed(seed, layer, linear_index):
    return substream(substream(seed, 1000 + layer), 100 + linear_index)
