"""Host-side check of the generated register extraction plans.

Emulates, with numpy integers and numpy's float16, exactly what the kernel
does for each plan in bit_weight_quantized_gb300/csrc/unpack_plans.h: build
the windows of a run, AND with the mask, OR in the exponent bits, read the
halves as fp16 and subtract 2**E.  Every code of the run must come back once,
exactly, and the slot table must be the inverse of the pairing.  The run
words are built with Python big integers (LSB-first stream), independently
of the oracle's packer.
"""
import os
import re

import numpy as np
import pytest

from synthetic import SplitMix64

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "bit_weight_quantized_gb300", "csrc", "unpack_plans.h")


def parse_plans():
    text = open(HDR).read()
    plans = {}
    for m in re.finditer(r"struct UnpackPlan<(\d+), (\d+)> \{(.*?)\n\};", text, re.S):
        b, R, body = int(m.group(1)), int(m.group(2)), m.group(3)
        d = {}
        for f in re.finditer(r"static constexpr \w+ (\w+)\(int i\) \{\s*constexpr \w+ v\[\d+\] = \{([^}]*)\};", body):
            d[f.group(1)] = [int(v.rstrip("u"), 0) for v in f.group(2).split(",")]
        d["kWindows"] = int(re.search(r"kWindows = (\d+);", body).group(1))
        plans[(b, R)] = d
    return plans


PLANS = parse_plans()


def test_all_plans_present():
    assert set(PLANS) == {(b, R) for b in range(1, 8) for R in (8, 16, 32)}


def _window(words, P, v):
    nw = len(words)
    if P["kind"][v] == 1:
        a, b, sel = words[P["w0"][v]], words[P["w1"][v]], P["sel"][v]
        pool = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
        return sum(pool[(sel >> (4 * k)) & 7] << (8 * k) for k in range(4))
    o = P["off"][v]
    if o < 0:
        return (words[0] << (-o)) & 0xFFFFFFFF
    i, s = o >> 5, o & 31
    if s == 0:
        return words[i]
    hi = words[i + 1] if i + 1 < nw else 0
    return ((words[i] | (hi << 32)) >> s) & 0xFFFFFFFF


@pytest.mark.parametrize("key", sorted(PLANS))
def test_plan_recovers_every_code(key):
    b, R = key
    P = PLANS[key]
    st = SplitMix64(31 * b + R)
    for trial in range(20):
        codes = [int(c) for c in st.uniform_bits(R, b)]
        if trial == 0:
            codes = [(1 << b) - 1] * R      # all ones: catches mask overlap
        v = 0
        for k, q in enumerate(codes):
            v |= q << (k * b)
        nw = (R * b + 31) // 32
        # garbage above the run, as in the kernel (the next run's bits)
        v |= int(st.next(1)[0]) << (R * b)
        words = [(v >> (32 * i)) & 0xFFFFFFFF for i in range(nw)]
        wins = [_window(words, P, u) for u in range(P["kWindows"])]
        seen = {}
        for i in range(R // 2):
            x = (wins[P["win"][i]] & P["mask"][i]) | P["magic"][i]
            halves = np.array([x & 0xFFFF, x >> 16], dtype=np.uint16).view(np.float16).astype(np.float64)
            lo = halves[0] - 2.0 ** P["elo"][i]
            hi = halves[1] - 2.0 ** P["ehi"][i]
            assert lo == codes[P["lo"][i]], (i, "lo")
            assert hi == codes[P["hi"][i]], (i, "hi")
            seen[P["lo"][i]] = seen.get(P["lo"][i], 0) + 1
            seen[P["hi"][i]] = seen.get(P["hi"][i], 0) + 1
        assert sorted(seen) == list(range(R)) and set(seen.values()) == {1}


@pytest.mark.parametrize("key", sorted(PLANS))
def test_slot_table_inverts_pairing(key):
    b, R = key
    P = PLANS[key]
    for i in range(R // 2):
        j, half = divmod(i, 2)
        assert P["slot"][P["lo"][i]] == 4 * j + 2 * half
        assert P["slot"][P["hi"][i]] == 4 * j + 2 * half + 1
    assert sorted(P["slot"]) == list(range(R))


@pytest.mark.parametrize("key", sorted(PLANS))
def test_magic_exponents_keep_fields_in_mantissa(key):
    P = PLANS[key]
    b = key[0]
    for i in range(len(P["lo"])):
        for e, shift in ((P["elo"][i], 0), (P["ehi"][i], 16)):
            assert 1 <= e <= 10
            field = (P["mask"][i] >> shift) & 0xFFFF
            assert field & 0xFC00 == 0                  # mask never touches exponent/sign
            assert bin(field).count("1") == b
            assert (P["magic"][i] >> shift) & 0xFFFF == (e + 15) << 10
