"""Pins for the oracle's GGUF Q4_K / Q6_K super-block decoders (CPU only).

The packers below build blocks from the layout description (the inverse of
decoding); a round trip through them, one-hot bytes and hand-built blocks
with known answers pin the decoder's indexing, nibble order and scale packing.
"""
import numpy as np
import pytest

import synthetic

Q4K, Q6K = 12, 14


def test_half_to_float_exhaustive_vs_numpy(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.half_to_float(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


from gguf_pack import pack_q4k, pack_q6k, pack_scale_min, q6_scale_slot  # noqa: E402


# ------------------------------------------------------------------ Q4_K --

def test_q4k_scale_min_round_trip(orc):
    rng = np.random.default_rng(0)
    for _ in range(200):
        sc = rng.integers(0, 64, 8)
        mn = rng.integers(0, 64, 8)
        packed = pack_scale_min(sc, mn)
        for j in range(8):
            assert orc.q4k_scale_min(packed, j) == (sc[j], mn[j])


def test_q4k_scale_min_one_hot_bytes(orc):
    # Which (scale j, min j) a set bit of byte b feeds, by the packing:
    #   bytes 0-3: low 6 bits -> scale b, top 2 bits -> scale b+4 (bits 4-5)
    #   bytes 4-7: low 6 bits -> min b-4, top 2 bits -> min b (bits 4-5)
    #   bytes 8-11: low nibble -> scale b-4 (bits 0-3), high nibble -> min b-4
    for b in range(12):
        for bit in range(8):
            packed = np.zeros(12, np.uint8)
            packed[b] = 1 << bit
            got = [orc.q4k_scale_min(packed, j) for j in range(8)]
            nz = [(j, s, m) for j, (s, m) in enumerate(got) if s or m]
            if b < 4:
                want = [(b, 1 << bit, 0)] if bit < 6 else [(b + 4, 1 << (bit - 2), 0)]
            elif b < 8:
                want = [(b - 4, 0, 1 << bit)] if bit < 6 else [(b, 0, 1 << (bit - 2))]
            else:
                want = [(b - 4, 1 << bit, 0)] if bit < 4 else [(b - 4, 0, 1 << (bit - 4))]
            assert nz == want, (b, bit, nz)


def test_q4k_unit_scales_give_raw_quants(orc):
    rng = np.random.default_rng(1)
    q = rng.integers(0, 16, 256)
    blk = pack_q4k(1.0, 0.0, [1] * 8, [0] * 8, q)
    assert np.array_equal(orc.decode_block(Q4K, blk), q.astype(np.float32))
    assert np.array_equal(orc.decode_block(Q4K, blk, exact=True), q.astype(np.float64))


def test_q4k_dmin_only_block(orc):
    mn = np.arange(8) * 7 + 1
    blk = pack_q4k(0.5, 0.25, [3] * 8, mn, np.zeros(256, np.int64))
    w = orc.decode_block(Q4K, blk)
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == -0.25 * mn[j])


def test_q4k_sub_block_of_each_weight(orc):
    # scale j = 1 << j (for j < 6) and all quants 1 reveal each weight's sub-block
    sc = [1, 2, 4, 8, 16, 32, 3, 5]
    blk = pack_q4k(1.0, 0.0, sc, [0] * 8, np.ones(256, np.int64))
    w = orc.decode_block(Q4K, blk)
    for i in range(256):
        assert w[i] == sc[i // 32]


def test_q4k_random_block_exact_definition(orc):
    rng = np.random.default_rng(4)
    for _ in range(50):
        d, dmin = rng.uniform(1e-3, 1e-2, 2)
        sc, mn, q = rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)
        blk = pack_q4k(d, dmin, sc, mn, q)
        dd = float(np.float16(d))
        dm = float(np.float16(dmin))
        exact = np.array([dd * sc[i // 32] * q[i] - dm * mn[i // 32] for i in range(256)])
        assert np.array_equal(orc.decode_block(Q4K, blk, exact=True), exact)
        # the fp32 form is the stated fp32 evaluation order
        d32, m32 = np.float32(dd), np.float32(dm)
        f32 = np.array([(d32 * np.float32(sc[i // 32])) * np.float32(q[i])
                        - m32 * np.float32(mn[i // 32]) for i in range(256)],
                       dtype=np.float32)
        assert np.array_equal(orc.decode_block(Q4K, blk), f32)


# ------------------------------------------------------------------ Q6_K --

def test_q6k_zero_quants(orc):
    sc = np.arange(-8, 8)
    blk = pack_q6k(0.5, sc, np.zeros(256, np.int64))
    w = orc.decode_block(Q6K, blk)
    for i in range(256):
        assert w[i] == -32 * 0.5 * sc[q6_scale_slot(i)]


def test_q6k_round_trip_of_quants(orc):
    rng = np.random.default_rng(6)
    for _ in range(30):
        q = rng.integers(0, 64, 256)
        blk = pack_q6k(1.0, np.ones(16, np.int64), q)
        assert np.array_equal(orc.decode_block(Q6K, blk), (q - 32).astype(np.float32))


def test_q6k_scale_slot_of_each_weight(orc):
    sc = np.arange(1, 17)
    blk = pack_q6k(1.0, sc, np.full(256, 33))
    w = orc.decode_block(Q6K, blk)
    for i in range(256):
        assert w[i] == sc[q6_scale_slot(i)]
    # every scale slot covers exactly 16 consecutive-in-l weights
    assert sorted(np.bincount([q6_scale_slot(i) for i in range(256)])) == [16] * 16


def test_q6k_random_block_exact_definition(orc):
    rng = np.random.default_rng(8)
    for _ in range(30):
        d = rng.uniform(1e-3, 1e-2)
        sc = rng.integers(-32, 32, 16)
        q = rng.integers(0, 64, 256)
        blk = pack_q6k(d, sc, q)
        dd = float(np.float16(d))
        exact = np.array([dd * sc[q6_scale_slot(i)] * (q[i] - 32) for i in range(256)])
        assert np.array_equal(orc.decode_block(Q6K, blk, exact=True), exact)


# --------------------------------------------------------------- matrices --

@pytest.mark.parametrize("qtype", [Q4K, Q6K])
def test_dequant_matrix_is_row_major_blocks(orc, qtype):
    N, K = 3, 768
    W = synthetic.weight_matrix(5, qtype, N, K)
    full = orc.dequant(qtype, W, N, K)
    bb = 144 if qtype == Q4K else 210
    for n in range(N):
        for s in range(K // 256):
            blk = W[n, s * bb:(s + 1) * bb]
            assert np.array_equal(full[n, s * 256:(s + 1) * 256],
                                  orc.decode_block(qtype, blk))


def test_synthetic_q4k_fields_in_range():
    W = synthetic.q4k_matrix(1, 64, 1024).reshape(-1, 144)
    d = W[:, 0:2].copy().view(np.float16).astype(np.float64).ravel()
    dm = W[:, 2:4].copy().view(np.float16).astype(np.float64).ravel()
    assert d.min() >= 0.00099 and d.max() <= 0.01001
    assert dm.min() >= 0.00099 and dm.max() <= 0.01001


def test_synthetic_q6k_fields_in_range():
    W = synthetic.q6k_matrix(1, 64, 1024).reshape(-1, 210)
    sc = W[:, 192:208].view(np.int8)
    assert sc.min() == -32 and sc.max() == 31


def test_matrix_packers_match_block_packers():
    """The vectorised packers the GPU tests use build the same bytes as the
    block packers pinned above."""
    from gguf_pack import pack_q4k_matrix, pack_q6k_matrix
    rng = np.random.default_rng(5)
    N, nsb = 3, 2
    d = rng.uniform(1e-3, 1e-2, (N, nsb))
    dmin = rng.uniform(1e-3, 1e-2, (N, nsb))
    sc = rng.integers(0, 64, (N, nsb, 8))
    mn = rng.integers(0, 64, (N, nsb, 8))
    q = rng.integers(0, 16, (N, nsb, 256))
    W = pack_q4k_matrix(d, dmin, sc, mn, q)
    for r in range(N):
        for b in range(nsb):
            assert np.array_equal(W[r, 144 * b:144 * (b + 1)],
                                  pack_q4k(d[r, b], dmin[r, b], sc[r, b], mn[r, b], q[r, b]))
    scales = rng.integers(-32, 32, (N, nsb, 16))
    q6 = rng.integers(0, 64, (N, nsb, 256))
    W6 = pack_q6k_matrix(d, scales, q6)
    for r in range(N):
        for b in range(nsb):
            assert np.array_equal(W6[r, 210 * b:210 * (b + 1)], pack_q6k(d[r, b], scales[r, b], q6[r, b]))


def q6k_one_hot_effect(byte, bit):
    """From the Q6_K layout alone: the weights that change when bit `bit` of
    byte `byte` is set in a block with d = 1, every scale 1 and every quant
    0 (every weight -32), and their new values.  Layout: ql[128] (low 4 bits
    of the quants), qh[64] (top 2 bits), int8 scales[16], fp16 d; half h
    holds weights 128h .. 128h+127; for l < 32 the low nibble of ql[64h+l]
    is quant 128h+l, of ql[64h+32+l] quant 128h+32+l, their high nibbles
    quants 128h+64+l and 128h+96+l; bits 2i..2i+1 of qh[32h+l] are the top
    bits of quant 128h+32i+l; weight 128h+32i+l uses scale 8h+l//16+2i."""
    if byte < 128:
        h, r = divmod(byte, 64)
        quarter = (0 if r < 32 else 1) + (2 if bit >= 4 else 0)
        q = 1 << (bit % 4)
        return {128 * h + 32 * quarter + r % 32: float(q - 32)}
    if byte < 192:
        h, l = divmod(byte - 128, 32)
        quarter, top = divmod(bit, 2)
        return {128 * h + 32 * quarter + l: float((16 << top) - 32)}
    if byte < 208:
        j = byte - 192
        h, r = divmod(j, 8)
        quarter, half = divmod(r, 2)
        scale = int(np.array([1 | (1 << bit)], np.uint8).view(np.int8)[0])
        if scale == 1:
            return {}
        return {128 * h + 32 * quarter + 16 * half + l: -32.0 * scale for l in range(16)}
    d = float(np.array([0x3C00 ^ (1 << (bit + 8 * (byte - 208)))], np.uint16).view(np.float16)[0])
    return {k: -32.0 * d for k in range(256)}


def test_q6k_one_hot_bytes(orc):
    """Every bit of every byte of a Q6_K block, set alone on a base block,
    changes exactly the weights the layout description predicts, to the
    predicted values (a table written independently of the packers)."""
    base = np.zeros(210, np.uint8)
    base[192:208] = 1
    base[208:210] = np.array([1.0], np.float16).view(np.uint8)
    w0 = orc.decode_block(Q6K, base)
    assert np.all(w0 == -32.0)
    for byte in range(210):
        for bit in range(8):
            blk = base.copy()
            blk[byte] |= np.uint8(1 << bit)
            if blk[byte] == base[byte]:
                continue
            w = orc.decode_block(Q6K, blk)
            want = q6k_one_hot_effect(byte, bit)
            changed = {int(k): float(w[k]) for k in np.flatnonzero(w != w0)}
            if byte >= 208 and not np.isfinite(list(want.values())[0]):
                continue  # d bits that make d Inf/NaN: checked by the half tests
            want = {k: v for k, v in want.items() if v != -32.0}
            assert changed == want, (byte, bit, changed, want)
