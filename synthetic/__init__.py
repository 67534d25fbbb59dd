"""Seeded synthetic inputs for the quantized-matmul workloads.

This module holds random-number generation and storage-type casts only; it
contains none of the method's arithmetic (no packing, no dequantization, no
dot products).  Both the CPU oracle's tests and the CUDA path's tests and
benchmark draw their inputs from here, so that the two sides see identical
data without sharing any computational code.

Recipe (one stream per workload instance, seed 0 unless stated):

* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state advances by 0x9E3779B97F4A7C15 and each
  output is the state passed through the published 64-bit finaliser.
* Tensors are drawn in a fixed order from one stream: codes, zeros, scales,
  activations, activation scales.
* Uniform integers on a power-of-two range take the top bits of one output;
  other ranges use rejection sampling on the top byte.
* Normals use Box-Muller on two 53-bit uniforms in (0, 1].
* Values are rounded to fp16 with round-to-nearest-even (numpy), and to
  bf16 by fp64 -> fp32 (RNE) -> bf16 (RNE on the fp32 bit pattern).

Scales follow the workloads' law s = 0.02 * |N(0,1)| + 1e-3 rounded to fp16;
activations are N(0,1); int8 activations are uniform on [-127, 127]; signed
int4 weights are uniform on [-8, 7] and are returned as their 4-bit two's
complement codes.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


class SplitMix64:
    """Counter-based SplitMix64 stream; ``next(n)`` returns n uint64 draws."""

    def __init__(self, seed: int = 0):
        self.state = np.uint64(seed)
        self.count = 0  # number of outputs consumed so far

    def next(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint64)
        done = 0
        with np.errstate(over="ignore"):
            while done < n:
                m = min(_CHUNK, n - done)
                idx = np.arange(1, m + 1, dtype=np.uint64)
                z = self.state + idx * _GOLDEN
                z = (z ^ (z >> np.uint64(30))) * _M1
                z = (z ^ (z >> np.uint64(27))) * _M2
                z = z ^ (z >> np.uint64(31))
                out[done:done + m] = z
                self.state = self.state + np.uint64(m) * _GOLDEN
                done += m
        self.count += n
        return out

    # ---- derived draws ----------------------------------------------------
    def uniform_bits(self, n: int, bits: int) -> np.ndarray:
        """n integers uniform on [0, 2**bits), bits in 1..8, as uint8."""
        assert 1 <= bits <= 8
        return (self.next(n) >> np.uint64(64 - bits)).astype(np.uint8)

    def uniform_int8_sym(self, n: int) -> np.ndarray:
        """n integers uniform on [-127, 127] as int8 (rejects top byte 255)."""
        out = np.empty(n, dtype=np.int16)
        have = 0
        while have < n:
            want = n - have
            u = (self.next(want + want // 128 + 16) >> np.uint64(56)).astype(np.int16)
            u = u[u != 255][:want]
            out[have:have + u.size] = u - 127
            have += u.size
        return out.astype(np.int8)

    def normal(self, n: int) -> np.ndarray:
        """n standard normals in fp64 by Box-Muller (pairs of draws)."""
        pairs = (n + 1) // 2
        u = self.next(2 * pairs)
        f = ((u >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u1, u2 = f[0::2], f[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * pairs, dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * np.pi * u2)
        z[1::2] = r * np.sin(2.0 * np.pi * u2)
        return z[:n]


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (via fp32, both RNE); returns uint16 bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (f >> np.uint32(16)) & np.uint32(1)
    rounded = (f + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def scale_law(stream: SplitMix64, n: int) -> np.ndarray:
    """fp16(0.02 * |N(0,1)| + 1e-3)."""
    return (0.02 * np.abs(stream.normal(n)) + 1e-3).astype(np.float16)


@dataclass
class QmmProblem:
    """One FP16/BF16 x INT-b quantized matmul instance (unpacked codes)."""
    M: int
    N: int
    K: int
    bits: int
    group: int
    codes: np.ndarray            # uint8 [N][K], values < 2**bits
    scales: np.ndarray           # fp16 [N][K/group]
    zeros: Optional[np.ndarray]  # uint8 [N][K/group] or None
    zero_const: int              # used when zeros is None
    x: np.ndarray                # fp16 [M][K] or uint16 bf16 bits [M][K]
    x_dtype: str                 # "f16" or "bf16"
    y_dtype: str                 # "f16" or "bf16"
    label: str = ""

    def x_f64(self) -> np.ndarray:
        if self.x_dtype == "f16":
            return self.x.astype(np.float64)
        return bf16_bits_to_f64(self.x)

    def algorithmic_bytes(self) -> int:
        """Packed weights + scales + stored zeros + activations + outputs."""
        b = self.N * self.K * self.bits // 8
        b += self.scales.size * 2
        if self.zeros is not None:
            b += self.zeros.size
        b += self.M * self.K * 2 + self.M * self.N * 2
        return b

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


@dataclass
class W4A8Problem:
    """One integer-native W4A8 instance (signed int4 weights, int8 activations)."""
    M: int
    N: int
    K: int
    group: int
    w4: np.ndarray   # uint8 [N][K]: 4-bit two's-complement codes of weights in [-8, 7]
    ws: np.ndarray   # fp16 [N][K/group]
    xq: np.ndarray   # int8 [M][K]
    sa: np.ndarray   # fp16 [M]
    label: str = ""

    def algorithmic_bytes(self) -> int:
        return (self.N * self.K // 2 + self.ws.size * 2 + self.M * self.K
                + self.M * 2 + self.M * self.N * 2)

    def ops(self) -> int:
        return 2 * self.M * self.N * self.K


X_LAWS = ("normal", "shift2", "shift8", "abs4", "outlier")


def make_qmm(M: int, N: int, K: int, bits: int, group: int, *, zero_mode: str,
             x_dtype: str = "f16", y_dtype: str = "f16", seed: int = 0,
             label: str = "", x_law: str = "normal", code_fill: Optional[str] = None,
             scale_mult: float = 1.0) -> QmmProblem:
    """Draw one instance.

    zero_mode: "const8" (z = 8), "half" (z = 2**(bits-1)), "group" (uint8 per
    group, uniform on [0, 2**bits)), "none" (z = 0), "top" (z = 2**bits - 1)
    or "max" (z = 255, the largest stored zero).

    x_law (the activation law, N(0,1) unless stated):
      "normal"   N(0, 1)
      "shift2"   N(2, 1)        mean-shifted activations
      "shift8"   N(8, 1)
      "abs4"     4 |N(0, 1)|    non-negative, SiLU-like
      "outlier"  N(0, 1) with 8 channels (drawn after the activations, the
                 same channels for every token) multiplied by 100
    code_fill: None (codes drawn), "max" (every code 2**bits - 1) or "min"
    (every code 0); the codes are drawn either way, so the rest of the
    stream is unchanged.
    scale_mult multiplies the drawn fp16 scales (a power of two keeps them exact).
    """
    st = SplitMix64(seed)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    if code_fill == "max":
        codes[:] = (1 << bits) - 1
    elif code_fill == "min":
        codes[:] = 0
    elif code_fill is not None:
        raise ValueError(code_fill)
    ng = K // group
    zeros = None
    if zero_mode == "const8":
        zc = 8
    elif zero_mode == "half":
        zc = 1 << (bits - 1)
    elif zero_mode == "none":
        zc = 0
    elif zero_mode == "top":
        zc = (1 << bits) - 1
    elif zero_mode == "max":
        zc = 255
    elif zero_mode == "group":
        zc = 0
        zeros = st.uniform_bits(N * ng, bits).reshape(N, ng)
    else:
        raise ValueError(zero_mode)
    scales = scale_law(st, N * ng).reshape(N, ng)
    if scale_mult != 1.0:
        scales = (scales.astype(np.float64) * scale_mult).astype(np.float16)
    xn = st.normal(M * K).reshape(M, K)
    if x_law == "shift2":
        xn = xn + 2.0
    elif x_law == "shift8":
        xn = xn + 8.0
    elif x_law == "abs4":
        xn = 4.0 * np.abs(xn)
    elif x_law == "outlier":
        ch = (st.next(8) % np.uint64(K)).astype(np.int64)
        xn[:, ch] *= 100.0
    elif x_law != "normal":
        raise ValueError(x_law)
    if x_dtype == "f16":
        x = xn.astype(np.float16)
    elif x_dtype == "bf16":
        x = to_bf16_bits(xn).reshape(M, K)
    else:
        raise ValueError(x_dtype)
    return QmmProblem(M, N, K, bits, group, codes, scales, zeros, zc, x, x_dtype,
                      y_dtype, label)


def make_w4a8(M: int, N: int, K: int, group: int = 128, seed: int = 0,
              label: str = "") -> W4A8Problem:
    st = SplitMix64(seed)
    w4 = st.uniform_bits(N * K, 4).reshape(N, K)
    ws = scale_law(st, N * (K // group)).reshape(N, K // group)
    xq = st.uniform_int8_sym(M * K).reshape(M, K)
    sa = scale_law(st, M)
    return W4A8Problem(M, N, K, group, w4, ws, xq, sa, label)


# ---- the five workload families ------------------------------------------
def parity_ref() -> QmmProblem:
    """M=1, K=N=512, 4-bit, group 128, z=8, fp16 in/out."""
    return make_qmm(1, 512, 512, 4, 128, zero_mode="const8", label="parity_ref")


def decode_sweep(bits: int, seed: int = 0) -> QmmProblem:
    """M=1, K=N=4096 (7B-class q_proj), group 128, z = 2**(bits-1)."""
    return make_qmm(1, 4096, 4096, bits, 128, zero_mode="half", seed=seed,
                    label=f"decode_b{bits}")


def skinny(M: int, N: int, bits: int, seed: int = 0) -> QmmProblem:
    """M in {2,4,8,16}, K=4096, N in {11008, 14336}, group 64, uint8 zeros."""
    return make_qmm(M, N, 4096, bits, 64, zero_mode="group", seed=seed,
                    label=f"skinny_M{M}_N{N}_b{bits}")


def tiled(M: int, seed: int = 0) -> QmmProblem:
    """M in {128,512,2048}, K=8192, N=28672, int4 group 128, z=8, bf16."""
    return make_qmm(M, 28672, 8192, 4, 128, zero_mode="const8", x_dtype="bf16",
                    y_dtype="bf16", seed=seed, label=f"tiled_M{M}")


def w4a8(M: int, seed: int = 0) -> W4A8Problem:
    """M in {1,16,64}, K=N=4096, group 128."""
    return make_w4a8(M, 4096, 4096, 128, seed=seed, label=f"w4a8_M{M}")


def make_act(M: int, K: int, seed: int = 0) -> np.ndarray:
    """fp16 activations [M][K] for the per-token int8 quantizer: N(0,1) times a
    per-token magnitude 10**u, u uniform in [-2, 2) (from the same stream)."""
    st = SplitMix64(seed)
    mag = 10.0 ** (4.0 * (st.next(M) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53) - 2.0)
    return (st.normal(M * K).reshape(M, K) * mag[:, None]).astype(np.float16)


@dataclass
class W8A8Problem:
    """Integer-native W8A8: int8 weights and activations, per-group weight
    scales and per-token activation scales."""
    M: int
    N: int
    K: int
    group: int
    w8: np.ndarray   # int8 [N][K]
    ws: np.ndarray   # fp16 [N][K/group]
    xq: np.ndarray   # int8 [M][K]
    sa: np.ndarray   # fp16 [M]
    label: str = ""

    def algorithmic_bytes(self) -> int:
        return self.N * self.K + self.ws.size * 2 + self.M * self.K + self.M * 2 + self.M * self.N * 2


def make_w8a8(M: int, N: int, K: int, group: int = 32, seed: int = 0, label: str = "") -> W8A8Problem:
    """w ~ U[-128, 127] (all 256 byte values), xq ~ U[-127, 127], ws and sa by the scale law."""
    st = SplitMix64(seed)
    w8 = st.uniform_bits(N * K, 8).astype(np.uint8).view(np.int8).reshape(N, K)
    ws = scale_law(st, N * (K // group)).reshape(N, K // group)
    xq = st.uniform_int8_sym(M * K).reshape(M, K)
    sa = scale_law(st, M)
    return W8A8Problem(M, N, K, group, w8, ws, xq, sa, label)
