"""Host emulation of the decode kernel's bit-level steps (no GPU needed).

bit_weight_quantized_gb300/csrc/decode.cu turns each thread's packed words
into fp16 MMA operands with funnel shifts, byte permutes and LOP3s, and
permutes the MMA's k order so that the B fragment is one contiguous slice
of x.  These tests restate those integer operations in Python, exactly as
the kernel performs them, and check the invariants the kernel relies on:
- every extracted fp16 half is exactly 2^E + q for its code q;
- a thread's words for one row and 64-code block lie inside that block, and
  the 8- / 16-byte loads at b = 4 / 8 are aligned;
- the permuted k order, placed into the m16n8k16 fragment layout, gives the
  same product as the plain sum over the block's codes.
"""
import numpy as np
import pytest

from synthetic import SplitMix64

M32 = 0xFFFFFFFF


# ---- the kernel's integer operations, restated ------------------------------------
def funnelshift_r(lo, hi, s):
    return (((hi << 32) | lo) >> (s & 31)) & M32


def prmt(a, b, sel):
    by = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    return sum(by[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def lop3_and_or(a, mask, bits):
    return (a & mask) | bits


def dec_words(b):
    return (b + 1) // 2


def dec_exp(b):
    return 10 if b in (4, 8) else b


def dec_pair(b, win, c):
    """fp16 pair of codes c, c + 1 of a thread's 16 codes (code 0 at bit 0 of win[0])."""
    if b == 8:
        return prmt(win[c >> 2], 0x64646464, 0x4342 if c & 2 else 0x4140)
    if b == 4:
        w = win[c >> 3]
        byte = (c & 7) >> 1
        return lop3_and_or(prmt(w, w >> 4, byte | ((4 + byte) << 8)), 0x000F000F, 0x64006400)
    sh = c * b - (10 - b)
    u = (win[0] << (-sh)) & M32 if sh < 0 else funnelshift_r(win[sh >> 5], win[(sh >> 5) + 1], sh & 31)
    mask = ((1 << b) - 1) << (10 - b)
    magic = (b + 15) << 10
    lo = lop3_and_or(u, mask, magic | (magic << 16))
    return lop3_and_or((u << (16 - b)) & M32, (mask << 16) & M32, lo)


def thread_window(b, words, t):
    """The thread's shifted window: words read at its first word, shifted by its
    bit offset (odd widths only), plus one zero word."""
    nw = dec_words(b)
    o = 16 * (t & 1) if b & 1 else 0
    first = (16 * b * t) // 32
    raw = [int(words[first + k]) for k in range(nw)]
    win = [funnelshift_r(raw[k], raw[k + 1] if k + 1 < nw else 0, o) if b & 1 else raw[k]
           for k in range(nw)]
    return win + [0]


def pack_block(codes, b):
    """LSB-first bitstream of one 64-code block as 32-bit words (2b words)."""
    bits = ((codes[:, None].astype(np.int64) >> np.arange(b)) & 1).reshape(-1).astype(np.uint8)
    return np.packbits(bits, bitorder="little").view("<u4").astype(np.int64)


def half(bits16):
    return float(np.array([bits16 & 0xFFFF], dtype=np.uint16).view(np.float16)[0])


# ---- tests ------------------------------------------------------------------------
@pytest.mark.parametrize("b", range(1, 9))
def test_pairs_are_exactly_pow2_plus_code(b):
    st = SplitMix64(100 + b)
    for trial in range(24):
        codes = st.uniform_bits(64, b).astype(np.int64)
        if trial == 0:
            codes[:] = (1 << b) - 1          # all ones
        elif trial == 1:
            codes[:] = 0
        words = pack_block(codes, b)
        assert len(words) == 2 * b
        for t in range(4):
            win = thread_window(b, words, t)
            for c in range(0, 16, 2):
                pr = dec_pair(b, win, c)
                assert half(pr) == 2.0 ** dec_exp(b) + codes[16 * t + c], (b, t, c)
                assert half(pr >> 16) == 2.0 ** dec_exp(b) + codes[16 * t + c + 1], (b, t, c)


@pytest.mark.parametrize("b", range(1, 9))
@pytest.mark.parametrize("K", [512, 1024, 4096, 11008 // 512 * 512, 65536])
def test_thread_words_stay_in_block_and_vector_loads_align(b, K):
    row_words = K * b // 32
    kw = K // 8
    nw = dec_words(b)
    for row in (0, 1, 7):
        for warp in range(8):
            k0w = warp * kw
            for j in range(kw // 64):
                block_lo = (k0w * b + 64 * b * j) // 32
                block_hi = (k0w * b + 64 * b * (j + 1)) // 32
                for t in range(4):
                    first = (k0w * b + 16 * b * t) // 32 + 2 * b * j
                    assert block_lo <= first and first + nw <= block_hi
                    # the last code's bits lie inside the words read
                    o = (16 * b * t) % 32
                    assert o + 16 * b <= 32 * nw
                    if b in (4, 8):
                        # byte address relative to a 16-byte aligned base
                        assert ((row * row_words + first) * 4) % (4 * nw) == 0


@pytest.mark.parametrize("b", range(1, 9))
def test_permuted_k_order_gives_the_plain_dot_product(b):
    """One warp, one 64-code block, two 16-row tiles, 8 tokens: the fragments
    each thread supplies, placed by the m16n8k16 layout, multiply to
    sum_k (2^E + q[r][k]) x[m][k] for every row r and token m."""
    st = SplitMix64(7 * b)
    rows = 32
    codes = st.uniform_bits(rows * 64, b).reshape(rows, 64).astype(np.int64)
    x = (st.normal(8 * 64).reshape(8, 64)).astype(np.float16).astype(np.float64)
    words = [pack_block(codes[r], b) for r in range(rows)]
    D = np.zeros((rows, 8))
    for s in range(4):
        for i in range(2):
            A = np.zeros((16, 16))
            Bm = np.zeros((16, 8))
            for lane in range(32):
                g, t = lane >> 2, lane & 3
                wins = [thread_window(b, words[16 * i + 8 * h + g], t) for h in range(2)]
                regs = [dec_pair(b, wins[0], 4 * s), dec_pair(b, wins[1], 4 * s),
                        dec_pair(b, wins[0], 4 * s + 2), dec_pair(b, wins[1], 4 * s + 2)]
                places = [(g, 2 * t), (g + 8, 2 * t), (g, 2 * t + 8), (g + 8, 2 * t + 8)]
                for r, (row, k) in zip(regs, places):
                    A[row, k], A[row, k + 1] = half(r), half(r >> 16)
                base = 16 * t + 4 * s   # the B fragment: x[16t + 4s .. 16t + 4s + 3] of token g
                Bm[2 * t, g], Bm[2 * t + 1, g] = x[g, base], x[g, base + 1]
                Bm[2 * t + 8, g], Bm[2 * t + 9, g] = x[g, base + 2], x[g, base + 3]
            D[16 * i:16 * i + 16] += A @ Bm
    ref = (2.0 ** dec_exp(b) + codes.astype(np.float64)) @ x.T
    np.testing.assert_allclose(D, ref, rtol=0, atol=1e-9 * np.abs(ref).max())
