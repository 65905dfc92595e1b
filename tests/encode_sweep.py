"""Oracle side of the exhaustive E4M3 encoder sweep (tests/test_gpu_quant.py):
the oracle's bytes for a range of fp32 bit patterns, reduced to two 64-bit
checksums that the GPU side computes the same way.  A module of its own so
that spawned worker processes can import it."""
import numpy as np

SUB = 1 << 24  # patterns per oracle call


def patterns(start, count):
    """fp32 values whose bit patterns are start, start+1, ... (mod 2^32)."""
    return (np.arange(start, start + count, dtype=np.uint64) & np.uint64(0xFFFFFFFF)) \
        .astype(np.uint32).view(np.float32)


def checksums(codes, first_word):
    """(sum of w_i * (2 i + 1), sum of w_i) mod 2^64 over the 64-bit words w_i
    of the code bytes, i counted from first_word."""
    w = codes.view(np.uint64)
    v = np.arange(first_word, first_word + w.size, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    with np.errstate(over="ignore"):
        return int(np.sum(w * v, dtype=np.uint64)), int(np.sum(w, dtype=np.uint64))


def oracle_chunk(args):
    """(start, count, scale) -> the checksums of the oracle's codes for that
    range of patterns, each encoded as E4M3(fl(x * scale))."""
    import oracle
    start, count, scale = args
    c1 = c2 = 0
    for off in range(0, count, SUB):
        n = min(SUB, count - off)
        codes = oracle.encode_scaled(patterns(start + off, n), np.float32(scale))
        a, b = checksums(codes, off // 8)
        c1 = (c1 + a) & 0xFFFFFFFFFFFFFFFF
        c2 = (c2 + b) & 0xFFFFFFFFFFFFFFFF
    return c1, c2
