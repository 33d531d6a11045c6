"""Pins for the CPU oracle: closed forms, hand-built blocks, brute force on tiny
inputs, library special cases and structural cases of the decode block.  Each
test is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign, index or bit position, a transposed operand) fails it.  No GPU needed."""
import math

import numpy as np
import pytest

from quantised_gemv_norm_gb300 import synth

# ----------------------------------------------------------- fp16 / bf16 codecs


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0xBC00, -1.0), (0x7BFF, 65504.0), (0x0400, 2.0 ** -14),
    (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24), (0x3555, 0.333251953125),
    (0x0000, 0.0), (0x4248, 3.140625), (0xC580, -5.5),
])
def test_half_decode_textbook(orc, bits, value):
    assert orc.half_to_double(bits) == value


def test_half_encode_textbook(orc):
    assert orc.double_to_half(1.0) == 0x3C00
    assert orc.double_to_half(65504.0) == 0x7BFF
    assert orc.double_to_half(65519.99) == 0x7BFF
    assert orc.double_to_half(65520.0) == 0x7C00  # tie rounds to even -> inf
    assert orc.double_to_half(2.0 ** -24) == 0x0001
    assert orc.double_to_half(2.0 ** -25) == 0x0000  # tie to even (0)
    assert orc.double_to_half(3 * 2.0 ** -25) == 0x0002  # tie between 1 and 2 -> 2
    assert orc.double_to_half(1.0 + 2.0 ** -11) == 0x3C00  # tie -> even mantissa
    assert orc.double_to_half(1.0 + 3 * 2.0 ** -11) == 0x3C02
    assert orc.double_to_half(-0.1) == 0xAE66


def test_half_encode_matches_numpy(orc):
    # numpy's float64 -> float16 cast rounds to nearest even: a library special case.
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(3000) * s for s in (1e-6, 1e-3, 1.0, 100.0, 1e4)])
    want = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.double_to_half(v) for v in vals], np.uint16)
    assert np.array_equal(got, want)
    # and decode is the exact inverse on every finite half
    allh = np.arange(0, 0x7C00, 7, dtype=np.uint16)
    assert all(orc.half_to_double(int(h)) == float(np.uint16(h).view(np.float16)) for h in allh)


def test_bf16_decode(orc):
    assert orc.bf16_to_double(0x3F80) == 1.0
    assert orc.bf16_to_double(0xC040) == -3.0
    assert orc.bf16_to_double(0x3E80) == 0.25
    assert orc.bf16_to_double(0x0001) == 2.0 ** -133  # smallest subnormal


# ----------------------------------------------------------------- Q4_K blocks


def _q4k_bytes_by_hand(d_bits, dmin_bits, sc, m, q):
    """Independent encoder: the 96-bit scale string as one Python integer."""
    sc, m, q = [int(v) for v in sc], [int(v) for v in m], [int(v) for v in q]
    bits = 0
    for j in range(8):
        bits |= (sc[j] & 63) << (6 * j)
        bits |= (m[j] & 63) << (48 + 6 * j)
    out = bytearray(d_bits.to_bytes(2, "little") + dmin_bits.to_bytes(2, "little"))
    out += bits.to_bytes(12, "little")
    for j in range(8):
        for i in range(16):
            out.append((q[32 * j + i] & 15) | ((q[32 * j + 16 + i] & 15) << 4))
    return np.frombuffer(bytes(out), np.uint8)


def test_q4k_layout_matches_independent_encoder(orc):
    rng = np.random.default_rng(1)
    for _ in range(20):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        q = rng.integers(0, 16, 256)
        d_bits, dmin_bits = int(rng.integers(0, 0x7C00)), int(rng.integers(0, 0x7C00))
        ref = _q4k_bytes_by_hand(d_bits, dmin_bits, sc, m, q)
        blk = orc.pack_q4k(d_bits, dmin_bits, sc, m, q)
        assert np.array_equal(blk, ref)
        d, dmin, sc2, m2, q2 = orc.unpack_q4k(ref)
        assert d == orc.half_to_double(d_bits) and dmin == orc.half_to_double(dmin_bits)
        assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)


def test_q4k_scale_bits_by_hand(orc):
    # sc_0 = 1 -> bit 0 of byte 4; m_0 = 1 -> bit 48 = bit 0 of byte 10;
    # sc_5 = 63 straddles bytes 7 and 8 (bits 30..35).
    sc = [1, 0, 0, 0, 0, 63, 0, 0]
    m = [1, 0, 0, 0, 0, 0, 0, 0]
    blk = orc.pack_q4k(0, 0, sc, m, np.zeros(256, int))
    assert blk[4] == 1 and blk[10] == 1
    assert blk[7] == 0b11000000 and blk[8] == 0b00001111
    assert blk[5] == blk[6] == blk[9] == blk[11] == 0


def test_q4k_dequant_special_cases(orc):
    one, half = 0x3C00, 0x3800
    # all codes 15, scale 1, min 0, d = 1 -> every weight 15
    blk = orc.pack_q4k(one, 0, [1] * 8, [0] * 8, [15] * 256)
    assert np.all(orc.dequant_q4k(blk) == 15.0)
    # codes 0, min 63, dmin 0.5 -> -31.5
    blk = orc.pack_q4k(one, half, [5] * 8, [63] * 8, [0] * 256)
    assert np.all(orc.dequant_q4k(blk) == -31.5)
    # per-sub-block scale and min land on their own 32 weights, sign of the min term
    sc = [1, 2, 3, 4, 5, 6, 7, 8]
    m = [8, 7, 6, 5, 4, 3, 2, 1]
    q = [n % 16 for n in range(256)]
    w = orc.dequant_q4k(orc.pack_q4k(one, half, sc, m, q))
    want = [1.0 * sc[n // 32] * (n % 16) - 0.5 * m[n // 32] for n in range(256)]
    assert np.array_equal(w, np.array(want))


def test_q4k_single_code_moves_single_weight(orc):
    base = np.zeros(256, int)
    ref = orc.dequant_q4k(orc.pack_q4k(0x3C00, 0, [1] * 8, [0] * 8, base))
    for n in (0, 15, 16, 31, 32, 47, 200, 255):
        q = base.copy()
        q[n] = 9
        w = orc.dequant_q4k(orc.pack_q4k(0x3C00, 0, [1] * 8, [0] * 8, q))
        diff = np.nonzero(w != ref)[0]
        assert list(diff) == [n] and w[n] == 9.0


# ----------------------------------------------------------------- Q6_K blocks


def _q6k_bytes_by_hand(d_bits, sc, q):
    sc, q = [int(v) for v in sc], [int(v) for v in q]
    out = bytearray(210)
    for n in range(256):
        g, r = divmod(n, 32)
        h, rr = divmod(r, 16)
        t, e = divmod(rr, 4)
        out[16 * g + rr] |= (q[n] & 15) << (4 * h)
        out[128 + 8 * g + 4 * h + e] |= ((q[n] >> 4) & 3) << (2 * t)
    for s in range(16):
        out[192 + s] = sc[s] & 255
    out[208:210] = d_bits.to_bytes(2, "little")
    return np.frombuffer(bytes(out), np.uint8)


def test_q6k_layout_matches_independent_encoder(orc):
    rng = np.random.default_rng(2)
    for _ in range(20):
        sc = rng.integers(-128, 128, 16)
        q = rng.integers(0, 64, 256)
        d_bits = int(rng.integers(0, 0x7C00))
        ref = _q6k_bytes_by_hand(d_bits, sc, q)
        assert np.array_equal(orc.pack_q6k(d_bits, sc, q), ref)
        d, sc2, q2 = orc.unpack_q6k(ref)
        assert d == orc.half_to_double(d_bits)
        assert np.array_equal(sc2, sc) and np.array_equal(q2, q)


def test_q6k_dequant_special_cases(orc):
    # q = 32 is the zero code
    blk = orc.pack_q6k(0x3C00, [77] * 16, [32] * 256)
    assert np.all(orc.dequant_q6k(blk) == 0.0)
    # q = 63, sc = -128, d = 2^-14 -> (63 - 32) * -128 * 2^-14 = -0.2421875
    blk = orc.pack_q6k(0x0400, [-128] * 16, [63] * 256)
    assert np.all(orc.dequant_q6k(blk) == -0.2421875)
    # q = 0 -> -32 * sc * d ; each scale owns 16 weights
    sc = list(range(-8, 8))
    w = orc.dequant_q6k(orc.pack_q6k(0x3C00, sc, [0] * 256))
    assert np.array_equal(w, np.array([-32.0 * sc[n // 16] for n in range(256)]))


def test_q6k_single_code_moves_single_weight(orc):
    base = np.full(256, 32, int)
    for n in (0, 3, 4, 15, 16, 17, 31, 100, 255):
        q = base.copy()
        q[n] = 32 + 17 if n % 2 else 32 - 30  # exercises both the low and high bits
        w = orc.dequant_q6k(orc.pack_q6k(0x3C00, [1] * 16, q))
        assert list(np.nonzero(w)[0]) == [n] and w[n] == q[n] - 32


def test_generator_binades_make_dequant_exact_in_fp32(orc):
    # The synthetic blocks are drawn so every weight is an fp32 number; the
    # fp64 oracle result must then survive a round trip through float32.
    rng = np.random.default_rng(3)
    w4 = orc.dequant_q4k(synth.q4k_blocks(rng, 400))
    w6 = orc.dequant_q6k(synth.q6k_blocks(rng, 400))
    assert np.array_equal(w4.astype(np.float32).astype(np.float64), w4)
    assert np.array_equal(w6.astype(np.float32).astype(np.float64), w6)
    assert 0.01 < np.std(w4) < 0.2 and abs(np.mean(w4)) < 0.01
    assert 0.01 < np.std(w6) < 0.2


# ----------------------------------------------------------------- Q2_K blocks


def _q2k_bytes_by_hand(d_bits, dmin_bits, sc, m, q):
    # the layout as one little-endian integer: byte 4 + j = sc_j | m_j << 4; the code of
    # weight 16j + 4k + b sits at bit 2k of byte 20 + 4j + b
    v = d_bits | dmin_bits << 16
    for j in range(16):
        v |= (int(sc[j]) | int(m[j]) << 4) << (8 * (4 + j))
    for n in range(256):
        j, r = divmod(n, 16)
        k, b = divmod(r, 4)
        v |= int(q[n]) << (8 * (20 + 4 * j + b) + 2 * k)
    return np.frombuffer(v.to_bytes(84, "little"), np.uint8)


def test_q2k_layout_matches_independent_encoder(orc):
    rng = np.random.default_rng(11)
    for _ in range(20):
        sc, m, q = rng.integers(0, 16, 16), rng.integers(0, 16, 16), rng.integers(0, 4, 256)
        d_bits, dmin_bits = int(rng.integers(0, 0x7C00)), int(rng.integers(0, 0x7C00))
        ref = _q2k_bytes_by_hand(d_bits, dmin_bits, sc, m, q)
        assert np.array_equal(orc.pack_q2k(d_bits, dmin_bits, sc, m, q), ref)
        d, dmin, sc2, m2, q2 = orc.unpack_q2k(ref)
        assert d == orc.half_to_double(d_bits) and dmin == orc.half_to_double(dmin_bits)
        assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)


def test_q2k_bytes_by_hand(orc):
    # weight 0 is bits 0-1 of byte 20, weight 4 bits 2-3, weight 1 bits 0-1 of byte 21,
    # weight 16 (sub-block 1) bits 0-1 of byte 24; sc_3 = 5 and m_3 = 9 make byte 7 = 0x95
    q = np.zeros(256, int)
    q[0], q[4], q[1], q[16] = 3, 1, 2, 1
    sc, m = np.zeros(16, int), np.zeros(16, int)
    sc[3], m[3] = 5, 9
    blk = orc.pack_q2k(0x3C00, 0x3800, sc, m, q)
    assert blk[20] == 0b0111 and blk[21] == 0b10 and blk[24] == 1 and blk[7] == 0x95
    assert blk[0] == 0x00 and blk[1] == 0x3C and blk[2] == 0x00 and blk[3] == 0x38
    assert int(blk[22]) == int(blk[23]) == 0 and np.count_nonzero(blk[25:]) == 0


def test_q2k_dequant_special_cases(orc):
    one, half = 0x3C00, 0x3800
    # all codes 3, scale 1, min 0, d = 1 -> every weight 3
    assert np.all(orc.dequant_q2k(orc.pack_q2k(one, 0, [1] * 16, [0] * 16, [3] * 256)) == 3.0)
    # codes 0, min 15, dmin 0.5 -> -7.5
    assert np.all(orc.dequant_q2k(orc.pack_q2k(one, half, [7] * 16, [15] * 16, [0] * 256)) == -7.5)
    # per-sub-block scale and min on their own 16 weights, sign of the min term
    sc = [j % 16 for j in range(16)]
    m = [15 - j for j in range(16)]
    q = [n % 4 for n in range(256)]
    w = orc.dequant_q2k(orc.pack_q2k(one, half, sc, m, q))
    want = [1.0 * sc[n // 16] * (n % 4) - 0.5 * m[n // 16] for n in range(256)]
    assert np.array_equal(w, np.array(want))


def test_q2k_single_code_moves_single_weight(orc):
    base = np.zeros(256, int)
    ref = orc.dequant_q2k(orc.pack_q2k(0x3C00, 0, [1] * 16, [0] * 16, base))
    for n in (0, 1, 3, 4, 15, 16, 17, 100, 255):
        q = base.copy()
        q[n] = 2
        w = orc.dequant_q2k(orc.pack_q2k(0x3C00, 0, [1] * 16, [0] * 16, q))
        assert list(np.nonzero(w != ref)[0]) == [n] and w[n] == 2.0


def test_q2k_generator_exact_in_fp32_and_ledger(orc):
    w2 = orc.dequant_q2k(synth.q2k_blocks(np.random.default_rng(12), 400))
    assert np.array_equal(w2.astype(np.float32).astype(np.float64), w2)
    assert 0.001 < np.std(w2) < 0.2
    # 84 bytes per 256 weights: 2.625 bits per weight, 7/12 of Q4_K's bytes
    assert synth.Q2K_BLOCK_BYTES * 8 / 256 == 2.625 and synth.row_bytes(synth.FMT_Q2K, 4096) == 1344


def test_gemv_q2k_brute_force_integers(orc):
    rng = np.random.default_rng(13)
    rows, K = 4, 768
    blocks, Wint = [], np.zeros((rows, K), np.int64)
    for r in range(rows):
        for b in range(K // 256):
            sc, m, q = rng.integers(0, 16, 16), rng.integers(0, 16, 16), rng.integers(0, 4, 256)
            blocks.append(orc.pack_q2k(0x3C00, 0x3C00, sc, m, q))
            for n in range(256):
                Wint[r, 256 * b + n] = sc[n // 16] * q[n] - m[n // 16]
    x = rng.integers(-9, 10, K).astype(np.float32)
    want = [sum(int(Wint[r, k]) * int(x[k]) for k in range(K)) for r in range(rows)]
    assert np.array_equal(orc.gemv_q2k(np.concatenate(blocks), x, rows, K), np.array(want, np.float64))


# ----------------------------------------------------------------------- GEMV


def test_gemv_q4k_brute_force_integers(orc):
    # d = 1, dmin = 1 -> integer weights sc*q - m; integer x -> exact integer products
    rng = np.random.default_rng(4)
    rows, K = 5, 512
    blocks, Wint = [], np.zeros((rows, K), np.int64)
    for r in range(rows):
        for b in range(K // 256):
            sc, m, q = rng.integers(0, 64, 8), rng.integers(0, 64, 8), rng.integers(0, 16, 256)
            blocks.append(orc.pack_q4k(0x3C00, 0x3C00, sc, m, q))
            for n in range(256):
                Wint[r, 256 * b + n] = sc[n // 32] * q[n] - m[n // 32]
    W = np.concatenate(blocks)
    x = rng.integers(-9, 10, K).astype(np.float32)
    want = [sum(int(Wint[r, k]) * int(x[k]) for k in range(K)) for r in range(rows)]
    assert np.array_equal(orc.gemv_q4k(W, x, rows, K), np.array(want, np.float64))


def test_gemv_q6k_brute_force_integers(orc):
    rng = np.random.default_rng(5)
    rows, K = 3, 768
    blocks, Wint = [], np.zeros((rows, K), np.int64)
    for r in range(rows):
        for b in range(K // 256):
            sc, q = rng.integers(-128, 128, 16), rng.integers(0, 64, 256)
            blocks.append(orc.pack_q6k(0x3C00, sc, q))
            for n in range(256):
                Wint[r, 256 * b + n] = sc[n // 16] * (q[n] - 32)
    x = rng.integers(-9, 10, K).astype(np.float32)
    want = [sum(int(Wint[r, k]) * int(x[k]) for k in range(K)) for r in range(rows)]
    assert np.array_equal(orc.gemv_q6k(np.concatenate(blocks), x, rows, K), np.array(want, np.float64))


def test_gemv_quant_matches_numpy_matmul(orc):
    # GEMV = (dequantised matrix) @ x: numpy's float64 matmul as the library special case.
    rows, K = 37, 1024
    for fmt, deq, gemv in ((synth.FMT_Q4K, orc.dequant_q4k, orc.gemv_q4k),
                           (synth.FMT_Q6K, orc.dequant_q6k, orc.gemv_q6k),
                           (synth.FMT_Q2K, orc.dequant_q2k, orc.gemv_q2k)):
        W = synth.quant_matrix(7, fmt, rows, K)
        x = synth.activation(7, K)
        Wd = deq(W).reshape(rows, K)
        ref = Wd @ x.astype(np.float64)
        got = gemv(W, x, rows, K)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(Wd).sum())


def test_gemv_bf16_exact_products(orc):
    # bf16 x bf16 products are exact in fp64; small dyadic values make the sum exact too.
    vals = np.array([0x3F80, 0x4000, 0xBF80, 0x3F00, 0x4040, 0x0000], np.uint16)  # 1, 2, -1, .5, 3, 0
    dec = {0x3F80: 1.0, 0x4000: 2.0, 0xBF80: -1.0, 0x3F00: 0.5, 0x4040: 3.0, 0x0000: 0.0}
    rng = np.random.default_rng(6)
    W = vals[rng.integers(0, len(vals), (7, 64))]
    x = vals[rng.integers(0, len(vals), 64)]
    want = [sum(dec[int(W[r, k])] * dec[int(x[k])] for k in range(64)) for r in range(7)]
    assert np.array_equal(orc.gemv_bf16(W, x), np.array(want))


def test_gemv_bf16_matches_numpy(orc):
    W, x = synth.bf16_gemv_inputs(8, 33, 256)
    Wd = (W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xd = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(orc.gemv_bf16(W, x), Wd @ xd, rtol=1e-12, atol=1e-14)


def test_matmul_rows_are_gemvs_and_not_transposed(orc):
    rows, K, M = 9, 512, 3
    W = synth.quant_matrix(9, synth.FMT_Q4K, rows, K)
    X = np.stack([synth.activation(9, K, m) for m in range(M)])
    Y = orc.matmul_q4k(W, X, rows, K)
    assert Y.shape == (M, rows)
    for m in range(M):
        assert np.array_equal(Y[m], orc.gemv_q4k(W, X[m], rows, K))


# ---------------------------------------------------------------------- norms


def test_rmsnorm_closed_forms(orc):
    n = 4
    gamma = np.array([1.0, 2.0, -1.0, 0.5], np.float32)
    # constant row c: c / sqrt(c^2 + eps) * gamma  (negative c, large eps: catches mean vs
    # mean-of-squares, eps outside the root, and n-1 for n)
    for c, eps in ((-3.0, 0.0), (1.0, 0.5), (2.0, 1e-6)):
        x = np.full((1, n), c, np.float32)
        want = c / math.sqrt(c * c + eps) * gamma.astype(np.float64)
        assert np.allclose(orc.rmsnorm(x, gamma, eps)[0], want, rtol=1e-15, atol=0)
    # hand example: x = [1, 2, 3, 4]: mean square = 7.5
    x = np.array([[1, 2, 3, 4]], np.float32)
    want = np.array([1, 2, 3, 4]) / math.sqrt(7.5) * gamma
    assert np.allclose(orc.rmsnorm(x, gamma, 0.0)[0], want, rtol=1e-15)


def test_rmsnorm_scale_invariance_and_rows(orc):
    x, gamma, _ = synth.norm_inputs(0, 6, 2048)
    y = orc.rmsnorm(x, gamma, 0.0)
    y4 = orc.rmsnorm(x * 4, gamma, 0.0)  # x*4 is exact in fp32
    assert np.allclose(y, y4, rtol=1e-14, atol=0)
    # each row normalised on its own: mean of (y / gamma)^2 == 1
    r = y / gamma.astype(np.float64)
    assert np.allclose((r * r).mean(axis=1), 1.0, rtol=1e-12)


def test_layernorm_closed_forms(orc):
    gamma = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
    beta = np.array([0.5, -0.5, 0.25, 0.0], np.float32)
    # constant row -> beta exactly
    y = orc.layernorm(np.full((1, 4), 7.0, np.float32), gamma, beta, 1e-6)
    assert np.array_equal(y[0], beta.astype(np.float64))
    # hand example: x = [1,2,3,4]: mean 2.5, population variance 1.25
    x = np.array([[1, 2, 3, 4]], np.float32)
    want = (np.array([1, 2, 3, 4]) - 2.5) / math.sqrt(1.25 + 0.25) * gamma + beta
    assert np.allclose(orc.layernorm(x, gamma, beta, 0.25)[0], want, rtol=1e-15)


def test_layernorm_moments(orc):
    x, _, _ = synth.norm_inputs(1, 5, 2048)
    ones, zeros = np.ones(2048, np.float32), np.zeros(2048, np.float32)
    eps = 1e-6
    y = orc.layernorm(x, ones, zeros, eps)
    var = x.astype(np.float64).var(axis=1)
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-13)
    assert np.allclose(y.var(axis=1), var / (var + eps), rtol=1e-12)


def test_layernorm_matches_numpy(orc):
    x, gamma, beta = synth.norm_inputs(2, 4, 2048)
    xd = x.astype(np.float64)
    mu = xd.mean(axis=1, keepdims=True)
    ref = (xd - mu) / np.sqrt(xd.var(axis=1, keepdims=True) + 1e-6) * gamma + beta
    assert np.allclose(orc.layernorm(x, gamma, beta, 1e-6), ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ attention


def _halves(a):
    return np.asarray(a, np.float64).astype(np.float16).view(np.uint16)


def test_attention_single_key_returns_v(orc):
    rng = np.random.default_rng(10)
    n_q, n_kv, hd, ctx = 8, 2, 16, 4
    q = rng.standard_normal((n_q, hd))
    K = _halves(rng.standard_normal((n_kv, ctx, hd)))
    V = _halves(rng.standard_normal((n_kv, ctx, hd)))
    out = orc.attention(q, K, V, 1)
    Vd = V.view(np.float16).astype(np.float64)
    for h in range(n_q):
        assert np.array_equal(out[h], Vd[h // (n_q // n_kv), 0])  # GQA: group of 4 heads


def test_attention_identical_keys_average_v(orc):
    rng = np.random.default_rng(11)
    n_q, n_kv, hd, ctx = 4, 1, 8, 6
    q = rng.standard_normal((n_q, hd))
    K = _halves(np.tile(rng.standard_normal((1, 1, hd)), (n_kv, ctx, 1)))
    V = _halves(rng.standard_normal((n_kv, ctx, hd)))
    out = orc.attention(q, K, V, 5)
    Vd = V.view(np.float16).astype(np.float64)
    assert np.allclose(out, Vd[0, :5].mean(axis=0)[None, :], rtol=1e-13, atol=1e-15)


def test_attention_dominant_key_and_scale(orc):
    n_q, n_kv, hd, ctx = 2, 1, 16, 3
    q = np.zeros((n_q, hd))
    q[:, 0] = 100.0
    K = np.zeros((n_kv, ctx, hd))
    K[0, 1, 0] = 8.0       # score 800/4 = 200 against 0: weight e^-200 elsewhere
    V = np.zeros((n_kv, ctx, hd))
    V[0, :, 3] = [1.0, 2.0, 3.0]
    out = orc.attention(q, _halves(K), _halves(V), 3)
    assert np.allclose(out[:, 3], 2.0, rtol=0, atol=1e-80)
    # two keys with scores differing by exactly 1/sqrt(hd) * 4 -> softmax weights 1 : e^1
    q = np.zeros((1, hd)); q[0, 0] = 1.0
    K = np.zeros((1, 2, hd)); K[0, 1, 0] = 4.0      # scores 0 and 4 / sqrt(16) = 1
    V = np.zeros((1, 2, hd)); V[0, 0, 0], V[0, 1, 0] = 0.0, 1.0
    out = orc.attention(q, _halves(K), _halves(V), 2)
    assert math.isclose(out[0, 0], math.e / (1 + math.e), rel_tol=1e-15)


def test_attention_heads_of_a_group_use_their_own_query(orc):
    # two KV heads of two query heads each; key j of KV head g points along axis j, and
    # query head h points along axis h % 2 with a large norm: each head picks the value of
    # "its" key, so head h returns V[h // 2, h % 2]
    n_q, n_kv, hd, ctx = 4, 2, 16, 2
    q = np.zeros((n_q, hd))
    for h in range(n_q):
        q[h, h % 2] = 100.0
    K = np.zeros((n_kv, ctx, hd))
    K[:, 0, 0] = K[:, 1, 1] = 8.0          # scores 200 and 0: weight e^-200 on the other key
    V = np.arange(n_kv * ctx * hd, dtype=np.float64).reshape(n_kv, ctx, hd) / 64.0
    out = orc.attention(q, _halves(K), _halves(V), 2)
    for h in range(n_q):
        assert np.allclose(out[h], V[h // 2, h % 2], rtol=0, atol=1e-80)


def test_silu(orc):
    assert orc.silu(0.0) == 0.0
    assert math.isclose(orc.silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-16)
    assert math.isclose(orc.silu(-2.0), -2.0 / (1.0 + math.exp(2.0)), rel_tol=1e-16)
    assert orc.silu(40.0) == pytest.approx(40.0, rel=1e-15)


# ------------------------------------------------------- decode-block structure


def _tiny_model(seed=3, n_layers=1):
    return synth.make_model(seed, n_layers=n_layers, hidden=256, ffn=512, n_q_heads=4, n_kv_heads=2,
                            head_dim=64, vocab=300, max_ctx=8)


def _zero_q4k(a):
    z = np.zeros_like(a)  # d = dmin = 0 -> every weight 0
    return z


def _zero_q6k(a):
    return np.zeros_like(a)


def _rms(x, g, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt((x * x).mean() + eps) * np.asarray(g, np.float64)


def test_decode_zero_blocks_pass_residual_to_vocab(orc):
    m = _tiny_model(n_layers=2)
    for l in range(2):
        m.wo[l] = _zero_q4k(m.wo[l])
        m.wdown[l] = _zero_q4k(m.wdown[l]) if m.down_fmt[l] == synth.FMT_Q4K else _zero_q6k(m.wdown[l])
    x = synth.decode_input(0, m.hidden)
    kv = synth.make_kv_cache(0, m, 0)
    logits, hid = orc.decode_step(m, x, 0, kv, want_hidden=True)
    assert np.array_equal(hid, x.astype(np.float64))
    Wv = orc.dequant_q6k(m.wvocab).reshape(m.vocab, m.hidden)
    assert np.allclose(logits, Wv @ _rms(x, m.out_norm, m.eps), rtol=1e-12, atol=1e-12)


def test_decode_appends_k_and_v_rows_in_order(orc):
    m = _tiny_model(n_layers=1)
    x = synth.decode_input(1, m.hidden)
    kv = synth.make_kv_cache(1, m, 3)
    before = kv.copy()
    orc.decode_step(m, x, 3, kv)
    qdim, kvdim = m.n_q_heads * m.head_dim, m.n_kv_heads * m.head_dim
    Wqkv = orc.dequant_q4k(m.wqkv[0]).reshape(m.qkv_rows, m.hidden)
    qkv = Wqkv @ _rms(x, m.attn_norm[0], m.eps)
    k = qkv[qdim:qdim + kvdim].reshape(m.n_kv_heads, m.head_dim)
    v = qkv[qdim + kvdim:].reshape(m.n_kv_heads, m.head_dim)
    assert np.array_equal(kv[0, 0, :, 3, :], k.astype(np.float16).view(np.uint16))
    assert np.array_equal(kv[0, 1, :, 3, :], v.astype(np.float16).view(np.uint16))
    mask = np.ones(kv.shape, bool)
    mask[:, :, :, 3, :] = False
    assert np.array_equal(kv[mask], before[mask])  # nothing else touched


def test_decode_attention_path_empty_cache(orc):
    # FFN switched off: x1 = x + Wo . attn, and with one key attn(h) = v(h // group).
    m = _tiny_model(n_layers=1)
    m.wdown[0] = _zero_q4k(m.wdown[0])
    x = synth.decode_input(2, m.hidden)
    kv = synth.make_kv_cache(2, m, 0)
    _, hid = orc.decode_step(m, x, 0, kv, want_hidden=True)
    qdim, kvdim = m.n_q_heads * m.head_dim, m.n_kv_heads * m.head_dim
    Wqkv = orc.dequant_q4k(m.wqkv[0]).reshape(m.qkv_rows, m.hidden)
    v = (Wqkv @ _rms(x, m.attn_norm[0], m.eps))[qdim + kvdim:]
    v16 = v.astype(np.float16).astype(np.float64).reshape(m.n_kv_heads, m.head_dim)
    group = m.n_q_heads // m.n_kv_heads
    attn = np.concatenate([v16[h // group] for h in range(m.n_q_heads)])
    Wo = orc.dequant_q4k(m.wo[0]).reshape(m.hidden, qdim)
    assert np.allclose(hid, x + Wo @ attn, rtol=1e-12, atol=1e-10)


def test_decode_attention_path_qwen3_later_token(orc):
    # FFN switched off, Qwen3 attention inputs, pos 2 over a filled cache: x1 = x + Wo . attn,
    # with attn rebuilt from the pinned pieces in the layer's order: the q|k|v projection of
    # rms(x); per-head RMSNorm, then RoPE at pos, on every q head and on the new key; the new
    # k and v rounded to fp16 into row pos; attention over keys 0..pos (the new key included).
    m = synth.make_model(36, n_layers=1, hidden=256, ffn=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                         vocab=64, max_ctx=8, qwen3_attention=True)
    m.wdown[0] = _zero_q4k(m.wdown[0])
    pos, hd, nq, nkv = 2, m.head_dim, m.n_q_heads, m.n_kv_heads
    qdim, kvdim = nq * hd, nkv * hd
    kv = synth.make_kv_cache(36, m, pos)
    k_plane, v_plane = kv[0, 0].copy(), kv[0, 1].copy()
    x = synth.decode_input(36, m.hidden)
    _, hid = orc.decode_step(m, x, pos, kv, want_hidden=True)
    qkv = orc.dequant_q4k(m.wqkv[0]).reshape(m.qkv_rows, m.hidden) @ _rms(x, m.attn_norm[0], m.eps)

    def turn(v, w):
        return orc.rope(orc.head_rmsnorm(v, w, m.eps), pos, m.rope_theta)

    q = np.stack([turn(qkv[h * hd:(h + 1) * hd], m.q_norm[0]) for h in range(nq)])
    for g in range(nkv):
        k = turn(qkv[qdim + g * hd:qdim + (g + 1) * hd], m.k_norm[0])
        k_plane[g, pos] = k.astype(np.float16).view(np.uint16)
        v_plane[g, pos] = qkv[qdim + kvdim + g * hd:qdim + kvdim + (g + 1) * hd].astype(np.float16).view(np.uint16)
    attn = orc.attention(q, k_plane, v_plane, pos + 1).reshape(-1)
    Wo = orc.dequant_q4k(m.wo[0]).reshape(m.hidden, qdim)
    assert np.allclose(hid, x + Wo @ attn, rtol=1e-12, atol=1e-10)


def test_decode_ffn_path(orc):
    # attention output projection switched off: x1 = x + Wd . (silu(Wg h) * (Wu h)), h = rms(x)
    m = _tiny_model(n_layers=1)
    m.wo[0] = _zero_q4k(m.wo[0])
    x = synth.decode_input(3, m.hidden)
    kv = synth.make_kv_cache(3, m, 2)
    _, hid = orc.decode_step(m, x, 2, kv, want_hidden=True)
    h = _rms(x, m.ffn_norm[0], m.eps)
    g = orc.dequant_q4k(m.wgate[0]).reshape(m.ffn, m.hidden) @ h
    u = orc.dequant_q4k(m.wup[0]).reshape(m.ffn, m.hidden) @ h
    a = g / (1 + np.exp(-g)) * u
    Wd = orc.dequant_q4k(m.wdown[0]).reshape(m.hidden, m.ffn)
    assert np.allclose(hid, x + Wd @ a, rtol=1e-12, atol=1e-9)


# ------------------------------------------------- Qwen3 attention inputs


def test_rope_is_identity_at_position_zero(orc):
    v = synth.normal_f32(synth.rng_for(31, 1), (128,)).astype(np.float64)
    assert np.array_equal(orc.rope(v, 0, 1.0e6), v)


def test_rope_turns_the_first_pair_by_the_position(orc):
    # dimension 0 pairs with dimension 64 and turns by pos * theta^0 = pos radians
    for pos in (1, 7, 511, 4097):
        e0 = np.zeros(128)
        e0[0] = 1.0
        r = orc.rope(e0, pos, 1.0e6)
        assert abs(r[0] - np.cos(pos)) < 1e-12 and abs(r[64] - np.sin(pos)) < 1e-12
        assert np.count_nonzero(np.delete(r, [0, 64])) == 0


def test_rope_last_pair_angle(orc):
    # pair (63, 127) turns by pos * theta^(-126/128): with theta = 2^128 that is pos * 2^-126
    # (a tiny angle: its sine is checked relative to itself)
    pos = 3
    e = np.zeros(128)
    e[63] = 1.0
    r = orc.rope(e, pos, 2.0 ** 128)
    ang = pos * 2.0 ** -126
    assert abs(r[63] - np.cos(ang)) < 1e-15 and abs(r[127] - np.sin(ang)) <= 1e-12 * ang


def test_rope_middle_pair_angle(orc):
    # pair (32, 96) turns by pos * theta^(-64/128) = pos / sqrt(theta): one radian at
    # pos 1000 with theta 1e6; dimension 31 (pair (31, 95)) turns by 1000 * 1e6^(-62/128)
    e = np.zeros(128)
    e[32] = 1.0
    e[31] = 1.0
    r = orc.rope(e, 1000, 1.0e6)
    assert abs(r[32] - math.cos(1.0)) < 1e-12 and abs(r[96] - math.sin(1.0)) < 1e-12
    a31 = 1000 * 1.0e6 ** (-62 / 128)
    assert abs(r[31] - math.cos(a31)) < 1e-12 and abs(r[95] - math.sin(a31)) < 1e-12


def test_rope_keeps_pair_norms_and_relative_positions(orc):
    rng = synth.rng_for(32, 1)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    for pos in (5, 300):
        r = orc.rope(q, pos, 1.0e6)
        assert np.allclose(np.hypot(r[:64], r[64:]), np.hypot(q[:64], q[64:]), rtol=0, atol=1e-12)
    # a rotation by position: the score depends only on the distance between positions
    a = np.dot(orc.rope(q, 40, 1.0e6), orc.rope(k, 10, 1.0e6))
    b = np.dot(orc.rope(q, 130, 1.0e6), orc.rope(k, 100, 1.0e6))
    assert abs(a - b) < 1e-9 * max(1.0, abs(a))


def test_head_rmsnorm_closed_forms(orc):
    w = synth.normal_f32(synth.rng_for(33, 1), (128,), 1.0, 0.1)
    c = 3.0
    out = orc.head_rmsnorm(np.full(128, c), w, 1e-6)
    assert np.allclose(out, c / np.sqrt(c * c + 1e-6) * w.astype(np.float64), rtol=1e-14, atol=0)
    v = synth.normal_f32(synth.rng_for(33, 2), (128,)).astype(np.float64)
    ones = np.ones(128, np.float32)
    n1 = orc.head_rmsnorm(v, ones, 0.0)
    assert abs(np.sqrt(np.mean(n1 ** 2)) - 1.0) < 1e-14     # unit RMS with unit weights, eps 0
    assert np.allclose(orc.head_rmsnorm(v * 7.5, ones, 0.0), n1, rtol=1e-14, atol=0)  # scale invariant


def test_qwen3_attention_does_not_change_the_first_token(orc):
    # with one key the softmax is 1: the output is that key's value, whatever q and k are,
    # and v is not transformed: the logits at pos 0 equal those of plain attention
    plain = synth.make_model(34, n_layers=2, hidden=256, ffn=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                             vocab=300, max_ctx=8)
    qwen = synth.make_model(34, n_layers=2, hidden=256, ffn=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                            vocab=300, max_ctx=8, qwen3_attention=True)
    x = synth.decode_input(34, 256)
    a = orc.decode_step(plain, x, 0, synth.make_kv_cache(34, plain, 0))
    b = orc.decode_step(qwen, x, 0, synth.make_kv_cache(34, qwen, 0))
    assert np.array_equal(a, b)


def test_qwen3_attention_changes_later_tokens_and_caches_rotated_keys(orc):
    qwen = synth.make_model(35, n_layers=1, hidden=256, ffn=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                            vocab=64, max_ctx=8, qwen3_attention=True)
    plain = synth.make_model(35, n_layers=1, hidden=256, ffn=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                             vocab=64, max_ctx=8)
    kv_q = synth.make_kv_cache(35, qwen, 0)
    kv_p = synth.make_kv_cache(35, plain, 0)
    x = synth.decode_input(35, 256)
    orc.decode_step(qwen, x, 3, kv_q)
    orc.decode_step(plain, x, 3, kv_p)
    # the cached key at pos 3 is the normalised, rotated projection; the value is unchanged
    kq = kv_q.view(np.float16)[0, 0, :, 3, :].astype(np.float64)
    kp = kv_p.view(np.float16)[0, 0, :, 3, :].astype(np.float64)
    for h in range(2):
        want = orc.rope(orc.head_rmsnorm(kp[h], qwen.k_norm[0], qwen.eps), 3, qwen.rope_theta)
        assert np.max(np.abs(kq[h] - want)) <= 2e-3 * np.max(np.abs(want))  # fp16 rounding of both
    assert np.array_equal(kv_q.view(np.uint16)[0, 1], kv_p.view(np.uint16)[0, 1])
