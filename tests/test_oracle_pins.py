"""Pins for the CPU oracle, independent of the oracle's own code.

Each check ties the oracle to something other than itself: hand-derived
packed bytes (tests/golden), the INT8 dot product printed in BitLLM Fig. 2(c),
Python big-integer bit extraction (a different idiom from the oracle's per-bit
loop), exact rational brute force, a special case that reduces to a library
matmul, and closed forms.  They are chosen so that a dropped term, a wrong
sign, a wrong index or a transposed operand in the oracle fails at least one.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import SplitMix64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split("|")]


def _bigint_pack(codes_row, bits):
    """Independent packer: build one Python integer, write it little-endian."""
    v = 0
    for k, q in enumerate(codes_row):
        v |= int(q) << (k * bits)
    return np.frombuffer(v.to_bytes(len(codes_row) * bits // 8, "little"), dtype=np.uint8)


def _bigint_codes(row_bytes, K, bits):
    v = int.from_bytes(bytes(row_bytes), "little")
    return [(v >> (k * bits)) & ((1 << bits) - 1) for k in range(K)]


# ---- bitstream -----------------------------------------------------------------
@pytest.mark.parametrize("case", list(_golden_lines("bitstream_examples.txt")))
def test_hand_packed_examples(case):
    bits = int(case[0])
    codes = np.array([int(t) for t in case[1].split()], dtype=np.uint8)[None, :]
    expect = np.array([int(t, 16) for t in case[2].split()], dtype=np.uint8)[None, :]
    packed, bad = oracle.pack(codes, bits)
    assert bad == 0
    np.testing.assert_array_equal(packed, expect)
    np.testing.assert_array_equal(oracle.unpack(expect, codes.shape[1], bits), codes)
    for k in range(codes.shape[1]):
        assert oracle.code_at(expect[0], k, bits) == codes[0, k]


def test_golden_signed_int4_values():
    # the last golden line holds the weights -8 7 -1 0 3 -5 1 -2 as codes
    codes = [8, 7, 15, 0, 3, 11, 1, 14]
    assert [oracle.int4_value(c) for c in codes] == [-8, 7, -1, 0, 3, -5, 1, -2]


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("K", [8, 24, 40, 256, 1000])
def test_roundtrip_codes(bits, K):
    if (K * bits) % 8:
        pytest.skip("K*bits must be byte aligned")
    st = SplitMix64(bits * 1000 + K)
    codes = st.uniform_bits(3 * K, bits).reshape(3, K)
    packed, bad = oracle.pack(codes, bits)
    assert bad == 0
    assert packed.shape == (3, K * bits // 8)
    np.testing.assert_array_equal(oracle.unpack(packed, K, bits), codes)


@pytest.mark.parametrize("bits", range(1, 9))
def test_roundtrip_bytes_is_bijection(bits):
    K = 64
    st = SplitMix64(77 + bits)
    raw = st.uniform_bits(5 * K * bits // 8, 8).reshape(5, K * bits // 8)
    codes = oracle.unpack(raw, K, bits)
    assert codes.max() < (1 << bits)
    again, _ = oracle.pack(codes, bits)
    np.testing.assert_array_equal(again, raw)


@pytest.mark.parametrize("bits", range(1, 9))
def test_bigint_idiom_agrees(bits):
    K, N = 96, 4
    st = SplitMix64(500 + bits)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    packed, _ = oracle.pack(codes, bits)
    for n in range(N):
        np.testing.assert_array_equal(packed[n], _bigint_pack(codes[n], bits))
        assert _bigint_codes(packed[n], K, bits) == list(codes[n])


def test_view_bit_conservation():
    # eight b-bit codes fill exactly b bytes (u8[3] <-> i6[4] is the b=6 case:
    # four 6-bit codes in three bytes)
    for bits in range(1, 9):
        packed, _ = oracle.pack(np.zeros((1, 8), np.uint8), bits)
        assert packed.shape[1] == bits
    packed, _ = oracle.pack(np.array([[63, 0, 63, 0]], np.uint8), 6)
    assert packed.shape == (1, 3)
    np.testing.assert_array_equal(packed[0], [0x3F, 0xF0, 0x03])


def test_width8_identity_and_width4_nibbles():
    st = SplitMix64(9)
    c8 = st.uniform_bits(3 * 40, 8).reshape(3, 40)
    np.testing.assert_array_equal(oracle.pack(c8, 8)[0], c8)
    c4 = st.uniform_bits(3 * 40, 4).reshape(3, 40)
    p4 = oracle.pack(c4, 4)[0]
    np.testing.assert_array_equal(p4, c4[:, 0::2] | (c4[:, 1::2] << 4))


def test_pack_counts_and_truncates_out_of_range():
    codes = np.array([[0, 5, 8, 15, 16, 255, 3, 9]], np.uint8)
    packed, bad = oracle.pack(codes, 3)
    assert bad == 5  # 8, 15, 16, 255 and 9 do not fit in 3 bits
    np.testing.assert_array_equal(oracle.unpack(packed, 8, 3), codes & 7)


def test_columns_are_independent_streams():
    st = SplitMix64(11)
    for bits in (3, 5, 7):
        K = 40
        codes = st.uniform_bits(3 * K, bits).reshape(3, K)
        packed, _ = oracle.pack(codes, bits)
        for n in range(3):
            np.testing.assert_array_equal(packed[n], oracle.pack(codes[n:n + 1], bits)[0][0])


# ---- dequantize + matmul ---------------------------------------------------------
def _dyadic_fp16(st, n, den_bits, lo, hi):
    """Random dyadic values p / 2**den_bits, exactly representable in fp16."""
    span = hi - lo + 1
    raw = (st.next(n) % np.uint64(span)).astype(np.int64) + lo
    return (raw.astype(np.float64) / (1 << den_bits)).astype(np.float16)


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("zero_mode", ["const", "group"])
def test_qmm_brute_force_exact(bits, zero_mode):
    st = SplitMix64(1234 + bits)
    M, N, K, G = 3, 5, 64, 32
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    scales = _dyadic_fp16(st, N * (K // G), 6, 1, 63).reshape(N, K // G)
    x = _dyadic_fp16(st, M * K, 4, -64, 64).reshape(M, K)
    zc = (1 << bits) // 2 + 1 if bits > 1 else 1
    zeros = st.uniform_bits(N * (K // G), bits).reshape(N, K // G) if zero_mode == "group" else None
    packed = np.stack([_bigint_pack(codes[n], bits) for n in range(N)])
    y = oracle.qmm(x.astype(np.float64), packed, bits, G, scales.astype(np.float64),
                   zeros, zc, K, nthreads=2)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                z = int(zeros[n, k // G]) if zeros is not None else zc
                w = (int(codes[n, k]) - z) * Fraction(float(scales[n, k // G]))
                acc += Fraction(float(x[m, k])) * w
            assert y[m, n] == float(acc), (m, n)


def test_qmm_reduces_to_library_matmul():
    # s = 1, z = 0, b = 8: W is the code matrix itself, y = x . Q^T
    st = SplitMix64(42)
    M, N, K = 4, 7, 256
    codes = st.uniform_bits(N * K, 8).reshape(N, K)
    x = st.normal(M * K).reshape(M, K).astype(np.float16).astype(np.float64)
    packed, _ = oracle.pack(codes, 8)
    y = oracle.qmm(x, packed, 8, 128, np.ones((N, K // 128)), None, 0, K)
    ref = x @ codes.astype(np.float64).T
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-10)


@pytest.mark.parametrize("bits", [1, 4, 6])
def test_qmm_all_ones_closed_form(bits):
    st = SplitMix64(7 + bits)
    N, K, G = 6, 256, 64
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    zeros = st.uniform_bits(N * (K // G), bits).reshape(N, K // G)
    scales = (0.02 * np.abs(st.normal(N * (K // G))) + 1e-3).astype(np.float16).reshape(N, K // G)
    packed, _ = oracle.pack(codes, bits)
    y = oracle.qmm(np.ones((1, K)), packed, bits, G, scales.astype(np.float64), zeros, 0, K)
    for n in range(N):
        expect = sum(float(scales[n, g]) * sum(int(codes[n, k]) - int(zeros[n, g])
                                               for k in range(g * G, (g + 1) * G))
                     for g in range(K // G))
        assert abs(y[0, n] - expect) <= 1e-12 * max(1.0, abs(expect))


def test_qmm_thread_count_does_not_change_result():
    st = SplitMix64(3)
    M, N, K = 2, 33, 512
    codes = st.uniform_bits(N * K, 5).reshape(N, K)
    packed, _ = oracle.pack(codes, 5)
    x = st.normal(M * K).reshape(M, K)
    s = np.abs(st.normal(N * 4)).reshape(N, 4)
    a = oracle.qmm(x, packed, 5, 128, s, None, 16, K, nthreads=1)
    b = oracle.qmm(x, packed, 5, 128, s, None, 16, K, nthreads=5)
    np.testing.assert_array_equal(a, b)


# ---- W4A8 integer core -------------------------------------------------------------
@pytest.mark.parametrize("case", list(_golden_lines("int8_dot_example.txt")))
def test_int8_dot_printed_example(case):
    a = np.array([int(t) for t in case[0].split()], np.int8)
    b = np.array([int(t) for t in case[1].split()], np.int8)
    assert oracle.dot_i8(a, b, int(case[2])) == int(case[3])


def test_dp4a_identity_brute_force():
    st = SplitMix64(99)
    for _ in range(50):
        a = st.uniform_int8_sym(4)
        b = st.uniform_int8_sym(4)
        r = int(st.next(1)[0] >> np.uint64(40)) - (1 << 23)
        assert oracle.dot_i8(a, b, r) == r + sum(int(u) * int(v) for u, v in zip(a, b))


def test_w4a8_brute_force_exact():
    st = SplitMix64(5)
    M, N, K, G = 3, 4, 256, 128
    w4 = st.uniform_bits(N * K, 4).reshape(N, K)
    xq = st.uniform_int8_sym(M * K).reshape(M, K)
    ws = _dyadic_fp16(st, N * (K // G), 8, 1, 200).reshape(N, K // G)
    sa = _dyadic_fp16(st, M, 8, 1, 200)
    packed = np.stack([_bigint_pack(w4[n], 4) for n in range(N)])
    y, acc, ov = oracle.w4a8(xq, sa.astype(np.float64), packed, ws.astype(np.float64), G, K)
    assert not ov
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for g in range(K // G):
                a = 0
                for k in range(g * G, (g + 1) * G):
                    c = int(w4[n, k])
                    a += int(xq[m, k]) * (c - 16 if c >= 8 else c)
                assert acc[m, n, g] == a
                tot += Fraction(float(ws[n, g])) * a
            assert y[m, n] == float(Fraction(float(sa[m])) * tot)


def test_w4a8_extreme_accumulator_fits_int32():
    K, G = 256, 128
    xq = np.full((1, K), -127, np.int8)
    w4 = np.full((1, K), 8, np.uint8)  # -8
    packed, _ = oracle.pack(w4, 4)
    y, acc, ov = oracle.w4a8(xq, np.ones(1), packed, np.ones((1, 2)), G, K)
    assert not ov
    assert (acc == 127 * 8 * G).all()
    assert y[0, 0] == 2 * 127 * 8 * G


# ---- per-token int8 activation quantization (BitLLM sec. 2.2, Eq. (1)) -------------------
@pytest.mark.parametrize("case", list(_golden_lines("act_quant_examples.txt")))
def test_act_quant_worked_examples(case):
    xs, s, qs = (part.split() for part in case)
    x = np.array([float(v) for v in xs], dtype=np.float16).reshape(1, -1)
    q, sa = oracle.quantize_act(x.view(np.uint16))
    assert float(sa.view(np.float16)[0]) == float(s[0])
    assert q[0].tolist() == [int(v) for v in qs]


def _f16_round_exact(v):
    """Round a non-negative Fraction to the nearest fp16 value, ties to even,
    in exact rational arithmetic (normal and subnormal ranges; no overflow)."""
    from fractions import Fraction
    if v == 0:
        return Fraction(0)
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1                                   # now 2^e <= v < 2^(e+1)
    ulp = Fraction(2) ** (max(e, -14) - 10)      # 11 significant bits; subnormal ulp 2^-24
    return round(v / ulp) * ulp                  # Fraction.__round__ ties to even


@pytest.mark.parametrize("amax", [127.0, 12.7, 0.75, 1000.0, 3e-3, 60000.0, 1e-6])
def test_act_quant_equals_exact_rational_rounding_on_every_fp16(amax):
    # Eq. (1) read in exact arithmetic: s = fp16(max|x| / 127) and q = round(x / s),
    # both rounded once, ties to even, from the exact rational values.  The oracle
    # divides in IEEE single precision; this checks, for one token per amax that
    # holds EVERY finite fp16 value of magnitude <= amax, that no such division
    # ever decides a code (or the scale) differently from exact arithmetic.
    from fractions import Fraction
    a16 = np.float16(amax)
    bits = np.arange(0, 0x7C00, dtype=np.uint16)
    mags = bits.view(np.float16)
    mags = mags[mags <= a16]
    vals = np.concatenate([mags, -mags[1:], [a16]]).astype(np.float16)
    pad = (-vals.size) % 8
    vals = np.concatenate([vals, np.zeros(pad, dtype=np.float16)])
    q, sa = oracle.quantize_act(vals.reshape(1, -1).view(np.uint16))
    s = _f16_round_exact(Fraction(float(a16)) / 127)
    assert Fraction(float(sa.view(np.float16)[0])) == s
    # a scale that rounds to 0 (max|x| below about 127 x 2^-25) quantizes to 0
    want = [round(Fraction(float(v)) / s) if s else 0 for v in vals]
    assert q[0].tolist() == want


def test_act_quant_error_bound_and_range():
    # |x - s q| <= s / 2 (round to nearest, no clipping since |x| / s <= 127 up to
    # the scale's fp16 rounding), and |q| <= 127
    rng = np.random.default_rng(11)
    x = np.array(rng.standard_normal((8, 1024)) * rng.uniform(0.01, 100, (8, 1)), dtype=np.float16)
    q, sa = oracle.quantize_act(x.view(np.uint16))
    s = sa.view(np.float16).astype(np.float64)[:, None]
    err = np.abs(x.astype(np.float64) - s * q.astype(np.float64))
    assert np.all(err <= s / 2 * (1 + 1e-6))
    assert np.abs(q.astype(np.int32)).max() <= 127


# ---- W8A8: signed 8-bit weights (BitLLM, Experiment Setup) ------------------------------
def test_signed_value_table():
    assert [oracle.signed_value(c, 8) for c in (0, 1, 127, 128, 129, 255)] == [0, 1, 127, -128, -127, -1]
    assert [oracle.signed_value(c, 4) for c in (0, 7, 8, 9, 15)] == [0, 7, -8, -7, -1]
    assert [oracle.signed_value(c, 4) for c in range(16)] == [oracle.int4_value(c) for c in range(16)]


def test_w8a8_brute_force_exact():
    prob = synthetic.make_w8a8(3, 5, 96, 32, seed=3)
    y, acc, ov = oracle.solve_w8a8(prob)
    assert not ov
    ng = prob.K // prob.group
    for m in range(prob.M):
        for n in range(prob.N):
            yy = 0.0
            for g in range(ng):
                ks = range(g * prob.group, (g + 1) * prob.group)
                a = sum(int(prob.xq[m, k]) * int(prob.w8[n, k]) for k in ks)   # Python integers
                assert acc[m, n, g] == a
                yy += float(prob.ws[n, g]) * a
            assert y[m, n] == float(prob.sa[m]) * yy


def test_w8a8_extreme_accumulator():
    prob = synthetic.make_w8a8(2, 3, 256, 128, seed=4)
    prob.w8[:] = -128
    prob.xq[:] = -127
    _, acc, ov = oracle.solve_w8a8(prob)
    assert not ov and (acc == 128 * 127 * 128).all()


def test_wxa8_at_four_bits_is_w4a8():
    prob = synthetic.make_w4a8(3, 7, 256, 64, seed=9)
    packed, _ = oracle.pack(prob.w4, 4)
    y4, acc4, _ = oracle.w4a8(prob.xq, prob.sa.astype(np.float64), packed, prob.ws.astype(np.float64),
                              prob.group, prob.K)
    yx, accx, _ = oracle.wxa8(prob.xq, prob.sa.astype(np.float64), packed, 4, prob.ws.astype(np.float64),
                              prob.group, prob.K)
    np.testing.assert_array_equal(acc4, accx)
    np.testing.assert_array_equal(y4, yx)


# ---- signed b-bit weights: sign flip and the signed matmul ---------------------------------
@pytest.mark.parametrize("case", list(_golden_lines("sign_flip_masks.txt")))
def test_sign_flip_masks(case):
    bits = int(case[0])
    mask = [int(v, 16) for v in case[1].split()]
    K = 64
    flipped = oracle.flip_sign(np.zeros((1, K * bits // 8), dtype=np.uint8), K, bits)[0]
    assert flipped.tolist() == mask * (K // 8)


@pytest.mark.parametrize("bits", range(1, 9))
def test_sign_flip_is_an_involution_and_maps_codes(bits):
    st = SplitMix64(bits)
    N, K = 3, 96
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    packed, _ = oracle.pack(codes, bits)
    once = oracle.flip_sign(packed, K, bits)
    np.testing.assert_array_equal(oracle.flip_sign(once, K, bits), packed)
    np.testing.assert_array_equal(oracle.unpack(once, K, bits), codes ^ (1 << (bits - 1)))


@pytest.mark.parametrize("bits", [1, 3, 4, 6, 8])
def test_signed_matmul_is_offset_binary_with_half_range_zero(bits):
    st = SplitMix64(100 + bits)
    M, N, K, G = 2, 5, 128, 32
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    packed, _ = oracle.pack(codes, bits)
    s = (0.02 * np.abs(st.normal(N * K // G)) + 1e-3).astype(np.float16).reshape(N, K // G)
    x = st.normal(M * K).reshape(M, K).astype(np.float16).astype(np.float64)
    y_signed = oracle.qmm_signed(x, packed, bits, G, s.astype(np.float64), K)
    # explicit two's-complement weights from Python integers
    c = np.where(codes >= (1 << (bits - 1)), codes.astype(np.int64) - (1 << bits), codes)
    w = c * np.repeat(s.astype(np.float64), G, axis=1)
    np.testing.assert_allclose(y_signed, x @ w.T, rtol=1e-12, atol=1e-12)
    # the same through the unsigned definition: flipped stream, zero 2^(b-1)
    y_off = oracle.qmm(x, oracle.flip_sign(packed, K, bits), bits, G, s.astype(np.float64), None,
                       1 << (bits - 1), K)
    np.testing.assert_allclose(y_off, y_signed, rtol=1e-12, atol=1e-12)


# ---- float weight codes (Tilus review: float3-float8) --------------------------------------
@pytest.mark.parametrize("case", list(_golden_lines("float_code_values.txt")))
def test_float_code_worked_values(case):
    e, m = (int(v) for v in case[0].split())
    codes = [int(v) for v in case[1].split()]
    values = [float(v) for v in case[2].split()]
    assert [oracle.float_value(c, e, m) for c in codes] == values


def _float_fraction(code, e, m):
    """The definition with exact rationals (an independent implementation)."""
    b = 1 + e + m
    sign = -1 if (code >> (b - 1)) & 1 else 1
    E = (code >> m) & ((1 << e) - 1)
    M = code & ((1 << m) - 1)
    bias = (1 << (e - 1)) - 1
    if E > 0:
        v = Fraction(2) ** (E - bias) * (1 + Fraction(M, 1 << m))
    else:
        v = Fraction(2) ** (1 - bias) * Fraction(M, 1 << m)
    return sign * v


@pytest.mark.parametrize("bits", range(2, 9))
def test_float_values_all_splits_exact(bits):
    for e in range(1, bits):
        m = bits - 1 - e
        for c in range(1 << bits):
            assert Fraction(oracle.float_value(c, e, m)) == _float_fraction(c, e, m), (e, m, c)


@pytest.mark.parametrize("e,m", [(2, 1), (3, 2), (2, 3), (4, 3)])
def test_float_matmul_brute_force(e, m):
    bits = 1 + e + m
    st = SplitMix64(50 + bits + e)
    M, N, K, G = 2, 3, 64, 32
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    packed, _ = oracle.pack(codes, bits)
    s = (0.02 * np.abs(st.normal(N * K // G)) + 1e-3).astype(np.float16).reshape(N, K // G)
    x = st.normal(M * K).reshape(M, K).astype(np.float16)
    y = oracle.qmm_float(x.astype(np.float64), packed, e, m, G, s.astype(np.float64), K)
    for mm in range(M):
        for n in range(N):
            exact = sum(Fraction(float(x[mm, k])) * _float_fraction(int(codes[n, k]), e, m)
                        * Fraction(float(s[n, k // G])) for k in range(K))
            assert abs(y[mm, n] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


# ---- lane-interleaved int4 layout (BitLLM Fig. 6, sec. 4.3 Fig. 8(b)) ----------------
def _nibble_slots(packed_row):
    """The nibble slots of a byte row, slot 0 = low nibble of byte 0 upwards."""
    return [(int(b) >> (4 * h)) & 15 for b in packed_row for h in (0, 1)]


def test_interleave4_matches_the_printed_order():
    (line,) = list(_golden_lines("lane_interleave_order.txt"))
    pos_in = [int(v) for v in line[0].split()]
    pos_stored = [int(v) for v in line[1].split()]
    assert pos_in == list(range(32)) and sorted(pos_stored) == pos_in
    # codes 0..15 twice: each value names its position modulo 16
    codes = (np.arange(32) % 16).astype(np.uint8).reshape(1, 32)
    slots = _nibble_slots(oracle.interleave4(codes)[0])
    assert slots == [p % 16 for p in pos_stored]


def test_interleave4_one_shift_two_masks_give_byte_aligned_codes():
    st = synthetic.SplitMix64(2024)
    codes = st.uniform_bits(5 * 64, 4).reshape(5, 64)
    words = oracle.interleave4(codes).view("<u4")
    for n in range(5):
        for w, W in enumerate(words[n]):
            W = int(W)
            lo = [(W & 0x0F0F0F0F) >> (8 * i) & 0xFF for i in range(4)]
            hi = [((W & 0xF0F0F0F0) >> 4) >> (8 * i) & 0xFF for i in range(4)]
            assert lo == list(codes[n, 8 * w:8 * w + 4])
            assert hi == list(codes[n, 8 * w + 4:8 * w + 8])


def test_interleave4_is_the_canonical_pack_of_permuted_codes_and_inverts():
    st = synthetic.SplitMix64(77)
    codes = st.uniform_bits(3 * 136, 4).reshape(3, 136)
    order = np.array([0, 4, 1, 5, 2, 6, 3, 7])
    perm = (np.arange(136) // 8 * 8)[:, None].reshape(-1)
    perm = perm + np.tile(order, 136 // 8)
    canonical, _ = oracle.pack(codes[:, perm], 4)
    inter = oracle.interleave4(codes)
    np.testing.assert_array_equal(inter, canonical)
    np.testing.assert_array_equal(oracle.deinterleave4(inter, 136), codes)
    with pytest.raises(ValueError):
        oracle.interleave4(codes[:, :12])


# ---- fragment-ordered (tile16) layout ---------------------------------------------------
@pytest.mark.parametrize("case", list(_golden_lines("tile16_runs.txt")))
def test_tile16_worked_runs(case):
    run, hexbytes = (part.split() for part in case)
    n = np.arange(16)[:, None]
    k = np.arange(64)[None, :]
    codes = ((n + k) % 16).astype(np.uint8)
    out = oracle.tile16(codes, 4)
    r = int(run[0])
    assert out[8 * r:8 * r + 8].tolist() == [int(h, 16) for h in hexbytes]


def _tile16_by_chunks(codes, bits):
    """The tile16 stream built another way: the canonical stream cut into the
    2b-byte slices of 16 codes (byte-aligned: code 16t of a block starts at byte
    2bt), gathered run by run with numpy indexing."""
    N, K = codes.shape
    Np = -(-N // 16) * 16
    padded = np.zeros((Np, K), dtype=np.uint8)
    padded[:N] = codes
    canon, _ = oracle.pack(padded, bits)                          # [Np][K*b/8]
    runs = canon.reshape(Np // 16, 2, 8, K // 64, 4, 2 * bits)    # [T][h][g][kb][t][2b]
    return runs.transpose(0, 3, 1, 2, 4, 5).reshape(-1)           # [T][kb][h][g][t][2b]


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("N,K", [(16, 64), (37, 128), (5, 256), (48, 192)])
def test_tile16_is_a_permutation_of_canonical_runs(bits, N, K):
    st = SplitMix64(3 * bits + N + K)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    out = oracle.tile16(codes, bits)
    assert out.size == -(-N // 16) * 16 * K * bits // 8
    np.testing.assert_array_equal(out, _tile16_by_chunks(codes, bits))


@pytest.mark.parametrize("bits", range(1, 9))
def test_tile16_round_trip(bits):
    st = SplitMix64(bits + 700)
    N, K = 29, 320
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    np.testing.assert_array_equal(oracle.untile16(oracle.tile16(codes, bits), N, K, bits), codes)
