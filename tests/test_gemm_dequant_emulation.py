"""Host emulation of the tiled kernel's code extraction for widths other than 4
(bit_weight_quantized_gb300/csrc/gemm.cuh, run_pair): a funnel shift puts code
c of a 32-code run at the top of the low half's mantissa, two LOP3s (one after
a shift) set both halves' exponents to that of 2^b.  The integer operations are
restated here exactly; each half must read exactly 2^b + q in fp16 (10
mantissa bits) and in bf16 (7 mantissa bits), for every width, pair position
and code pattern, and the reads must stay inside the run's b words."""
import numpy as np
import pytest

from synthetic import SplitMix64

M32 = 0xFFFFFFFF


def funnelshift_r(lo, hi, s):
    return (((hi << 32) | lo) >> (s & 31)) & M32


def run_pair(b, mb, w, c):
    sh = c * b - (mb - b)
    if sh < 0:
        u = (w[0] << (-sh)) & M32
    else:
        i, s = sh >> 5, sh & 31
        assert i < b                           # the low word is inside the run
        hi = w[i + 1] if i + 1 < b else 0
        u = w[i] if s == 0 else funnelshift_r(w[i], hi, s)
    mask = ((1 << b) - 1) << (mb - b)
    magic = (b + 15) << 10 if mb == 10 else (b + 127) << 7
    lo = (u & mask) | (magic | (magic << 16))
    return (((u << (16 - b)) & M32) & (mask << 16)) | lo


def value(bits16, mb):
    if mb == 10:
        return float(np.array([bits16], dtype=np.uint16).view(np.float16)[0])
    return float(np.array([bits16 << 16], dtype=np.uint32).view(np.float32)[0])


def run_words(codes, b):
    v = 0
    for k, q in enumerate(codes):
        v |= int(q) << (k * b)
    return [(v >> (32 * i)) & M32 for i in range(b)]


@pytest.mark.parametrize("mb", [10, 7])
@pytest.mark.parametrize("b", [1, 2, 3, 5, 6, 7])
def test_run_pairs_are_exactly_pow2_plus_code(b, mb):
    st = SplitMix64(17 * b + mb)
    for trial in range(16):
        codes = st.uniform_bits(32, b).astype(np.int64)
        if trial == 0:
            codes[:] = (1 << b) - 1
        elif trial == 1:
            codes[:] = 0
        w = run_words(codes, b)
        for c in range(0, 32, 2):
            pr = run_pair(b, mb, w, c)
            assert value(pr & 0xFFFF, mb) == 2.0 ** b + codes[c], (b, mb, c)
            assert value(pr >> 16, mb) == 2.0 ** b + codes[c + 1], (b, mb, c)


@pytest.mark.parametrize("b", [1, 2, 3, 5, 6, 7, 8])
def test_stage_geometry(b):
    # widths 1, 2, 4, 8: 128-byte swizzled rows of 16 / b K steps; others: two K
    # steps of 16 b bytes; a thread's run (32 codes = b words at byte (2 j + qd) 4 b)
    # stays inside its row, and the TMA x coordinate of a stage is 16-byte aligned
    pow2 = b in (1, 2, 4, 8)
    ksteps = 16 // b if pow2 else 2
    box = ksteps * 8 * b
    assert box <= 128 and box % 16 == 0
    for j in range(ksteps):
        for qd in range(2):
            ob = (2 * j + qd) * 4 * b
            assert ob + 4 * b <= box
            if pow2 and b <= 2:
                assert ob // 16 == (ob + 4 * b - 1) // 16   # inside one 16-byte chunk
    for ks in range(0, 64, ksteps):
        assert (ks * 8 * b) % 16 == 0
