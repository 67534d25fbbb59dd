"""CPU oracle for the FP16/BF16 x INT-b quantized matmul and the W4A8 path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product library neither imports nor links it, and this package imports
nothing from the product.

The arithmetic lives in ``qmm_oracle.c`` (plain C, fp64/int64, per-bit
bitstream loops); this module only compiles it with gcc and marshals numpy
arrays.  Citations for each step are in the C file's header:

* bitstream unpack/pack  -- the workloads' little-endian bitstream along K
  (Tilus review, pith_extraction.core_discovery; BitLLM sec. 4.3 Fig. 8(a));
* dequantize ``w = s * (q - z)`` per group -- BitLLM Eq. (5), sec. 2.2;
* fp64 matmul ``y = x . W^T``;
* W4A8 integer core ``r + sum a_i b_i`` per group and fp64 epilogue --
  BitLLM sec. 4.3 (dp4a), sec. 4.4 (deferred dequantization, Fig. 9); the
  same core with signed 8-bit weights is W8A8 (BitLLM, Experiment Setup);
* per-token int8 quantization of fp16 activations -- BitLLM sec. 2.2 Eq. (1);
* signed b-bit weights: the sign-bit flip between two's complement and offset
  binary, and the signed dequantize-then-matmul;
* float b-bit weights (1 sign, e exponent, m mantissa bits) and their
  dequantize-then-matmul.

Every function here is pinned by a ``-m "not gpu"`` test (hand-packed
examples, round trips, brute force with Python integers/fractions, closed
forms); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc -O2 (no fast-math: fixed summation order)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, L, I = ctypes.c_void_p, ctypes.c_long, ctypes.c_int
            lib.oracle_code.argtypes = [P, L, I]
            lib.oracle_code.restype = I
            lib.oracle_unpack.argtypes = [P, P, L, L, I]
            lib.oracle_unpack.restype = None
            lib.oracle_pack.argtypes = [P, P, L, L, I]
            lib.oracle_pack.restype = L
            lib.oracle_qmm.argtypes = [P, P, I, I, P, P, I, P, L, L, L, I]
            lib.oracle_qmm.restype = None
            lib.oracle_int4_value.argtypes = [I]
            lib.oracle_int4_value.restype = I
            lib.oracle_dot_i8.argtypes = [P, P, L, ctypes.c_int64]
            lib.oracle_dot_i8.restype = ctypes.c_int64
            lib.oracle_w4a8.argtypes = [P, P, P, P, I, P, P, L, L, L, I]
            lib.oracle_w4a8.restype = I
            lib.oracle_wxa8.argtypes = [P, P, P, I, P, I, P, P, L, L, L, I]
            lib.oracle_wxa8.restype = I
            lib.oracle_signed_value.argtypes = [I, I]
            lib.oracle_signed_value.restype = I
            lib.oracle_flip_sign.argtypes = [P, L, L, I]
            lib.oracle_flip_sign.restype = None
            lib.oracle_float_value.argtypes = [I, I, I]
            lib.oracle_float_value.restype = ctypes.c_double
            lib.oracle_threads.argtypes = [I, L]
            lib.oracle_threads.restype = I
            lib.oracle_quantize_act.argtypes = [P, P, P, L, L]
            lib.oracle_quantize_act.restype = None
            lib.oracle_interleave4.argtypes = [P, P, L, L]
            lib.oracle_interleave4.restype = None
            lib.oracle_deinterleave4.argtypes = [P, P, L, L]
            lib.oracle_deinterleave4.restype = None
            lib.oracle_tile16_bytes.argtypes = [L, L, I]
            lib.oracle_tile16_bytes.restype = L
            lib.oracle_tile16.argtypes = [P, P, L, L, I]
            lib.oracle_tile16.restype = None
            lib.oracle_untile16.argtypes = [P, P, L, L, I]
            lib.oracle_untile16.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads_used(nthreads: int, N: int) -> int:
    return _load().oracle_threads(nthreads, N)


def pack(codes: np.ndarray, bits: int):
    """codes uint8 [N][K] -> (packed uint8 [N][K*bits/8], count of codes >= 2**bits)."""
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    if (K * bits) % 8:
        raise ValueError("K*bits must be a multiple of 8")
    out = np.empty((N, K * bits // 8), dtype=np.uint8)
    bad = _load().oracle_pack(_ptr(codes), _ptr(out), N, K, bits)
    return out, int(bad)


def unpack(packed: np.ndarray, K: int, bits: int) -> np.ndarray:
    """packed uint8 [N][K*bits/8] -> codes uint8 [N][K]."""
    packed = _c(packed, np.uint8)
    N = packed.shape[0]
    if packed.shape[1] * 8 != K * bits:
        raise ValueError("packed row length must be K*bits/8")
    out = np.empty((N, K), dtype=np.uint8)
    _load().oracle_unpack(_ptr(packed), _ptr(out), N, K, bits)
    return out


def code_at(row: np.ndarray, k: int, bits: int) -> int:
    row = _c(row, np.uint8)
    return int(_load().oracle_code(_ptr(row), k, bits))


def qmm(x_f64: np.ndarray, packed: np.ndarray, bits: int, group: int,
        scales: np.ndarray, zeros, zero_const: int, K: int, nthreads: int = 0) -> np.ndarray:
    """fp64 y[M][N] for the dequantize-then-matmul definition."""
    x = _c(x_f64, np.float64)
    packed = _c(packed, np.uint8)
    M = x.shape[0]
    N = packed.shape[0]
    if x.shape[1] != K or packed.shape[1] * 8 != K * bits or K % group:
        raise ValueError("shape mismatch")
    s = _c(scales, np.float64)
    if s.shape != (N, K // group):
        raise ValueError("scales must be [N][K/group]")
    z = None
    if zeros is not None:
        z = _c(zeros, np.uint8)
        if z.shape != (N, K // group):
            raise ValueError("zeros must be [N][K/group]")
    y = np.empty((M, N), dtype=np.float64)
    _load().oracle_qmm(_ptr(x), _ptr(packed), bits, group, _ptr(s),
                       None if z is None else _ptr(z), int(zero_const), _ptr(y),
                       M, N, K, nthreads)
    return y


def int4_value(code: int) -> int:
    return int(_load().oracle_int4_value(code))


def signed_value(code: int, bits: int) -> int:
    return _load().oracle_signed_value(int(code), bits)


def dot_i8(a: np.ndarray, b: np.ndarray, r: int = 0) -> int:
    a = _c(a, np.int8)
    b = _c(b, np.int8)
    if a.shape != b.shape:
        raise ValueError("shape mismatch")
    return int(_load().oracle_dot_i8(_ptr(a), _ptr(b), a.size, r))


def w4a8(xq: np.ndarray, sa_f64: np.ndarray, w4_packed: np.ndarray, ws_f64: np.ndarray,
         group: int, K: int, want_acc: bool = True, nthreads: int = 0):
    """Returns (y fp64 [M][N], acc int64 [M][N][K/group] or None, overflow flag)."""
    xq = _c(xq, np.int8)
    sa = _c(sa_f64, np.float64)
    w4 = _c(w4_packed, np.uint8)
    ws = _c(ws_f64, np.float64)
    M = xq.shape[0]
    N = w4.shape[0]
    if xq.shape[1] != K or w4.shape[1] * 2 != K or K % group or ws.shape != (N, K // group):
        raise ValueError("shape mismatch")
    y = np.empty((M, N), dtype=np.float64)
    acc = np.empty((M, N, K // group), dtype=np.int64) if want_acc else None
    ov = _load().oracle_w4a8(_ptr(xq), _ptr(sa), _ptr(w4), _ptr(ws), group,
                             None if acc is None else _ptr(acc), _ptr(y), M, N, K, nthreads)
    return y, acc, bool(ov)


# ---- convenience: a whole problem from the synthetic generator -----------------
def solve_qmm(prob, rows=None, cols=None, nthreads: int = 0):
    """Oracle y (fp64) for a synthetic.QmmProblem, optionally on a row/column
    subset (pure data selection; the arithmetic is unchanged)."""
    packed, bad = pack(prob.codes if cols is None else prob.codes[cols], prob.bits)
    assert bad == 0
    x = prob.x_f64() if rows is None else prob.x_f64()[rows]
    s = prob.scales.astype(np.float64)
    z = prob.zeros
    if cols is not None:
        s = s[cols]
        z = None if z is None else z[cols]
    return qmm(x, packed, prob.bits, prob.group, s, z, prob.zero_const, prob.K, nthreads)


def solve_w4a8(prob, rows=None, cols=None, want_acc=True, nthreads: int = 0):
    w4 = prob.w4 if cols is None else prob.w4[cols]
    packed, bad = pack(w4, 4)
    assert bad == 0
    xq = prob.xq if rows is None else prob.xq[rows]
    sa = prob.sa.astype(np.float64) if rows is None else prob.sa.astype(np.float64)[rows]
    ws = prob.ws.astype(np.float64) if cols is None else prob.ws.astype(np.float64)[cols]
    return w4a8(xq, sa, packed, ws, prob.group, prob.K, want_acc, nthreads)


def quantize_act(x_bits: np.ndarray):
    """Per-token int8 quantization of fp16 activations given as bit patterns
    (uint16 [M][K]); returns (xq int8 [M][K], sa fp16 bit patterns uint16 [M])."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    xq = np.zeros((M, K), dtype=np.int8)
    sa = np.zeros(M, dtype=np.uint16)
    _load().oracle_quantize_act(_ptr(x), _ptr(xq), _ptr(sa), M, K)
    return xq, sa


def wxa8(xq: np.ndarray, sa_f64: np.ndarray, w_packed: np.ndarray, bits: int, ws_f64: np.ndarray,
         group: int, K: int, want_acc: bool = True, nthreads: int = 0):
    """Signed b-bit weights x int8 activations (b = 4: W4A8, b = 8: W8A8).
    Returns (y fp64 [M][N], acc int64 [M][N][K/group] or None, overflow flag)."""
    xq = _c(xq, np.int8)
    sa = _c(sa_f64, np.float64)
    w = _c(w_packed, np.uint8)
    ws = _c(ws_f64, np.float64)
    M = xq.shape[0]
    N = w.shape[0]
    if xq.shape[1] != K or w.shape[1] * 8 != K * bits or K % group or ws.shape != (N, K // group):
        raise ValueError("shape mismatch")
    y = np.empty((M, N), dtype=np.float64)
    acc = np.empty((M, N, K // group), dtype=np.int64) if want_acc else None
    ov = _load().oracle_wxa8(_ptr(xq), _ptr(sa), _ptr(w), bits, _ptr(ws), group,
                             None if acc is None else _ptr(acc), _ptr(y), M, N, K, nthreads)
    return y, acc, bool(ov)


def solve_w8a8(prob, want_acc=True, nthreads: int = 0):
    """A synthetic.W8A8Problem: the weights are int8 values stored as bytes."""
    w = np.ascontiguousarray(prob.w8.view(np.uint8))
    return wxa8(prob.xq, prob.sa.astype(np.float64), w, 8, prob.ws.astype(np.float64),
                prob.group, prob.K, want_acc, nthreads)


def flip_sign(packed: np.ndarray, K: int, bits: int) -> np.ndarray:
    """A copy of the packed stream with the top bit of every b-bit code flipped
    (two's complement <-> offset binary)."""
    out = np.array(_c(packed, np.uint8), copy=True)
    if out.shape[1] * 8 != K * bits:
        raise ValueError("packed row length must be K*bits/8")
    _load().oracle_flip_sign(_ptr(out), out.shape[0], K, bits)
    return out


def qmm_signed(x_f64: np.ndarray, packed: np.ndarray, bits: int, group: int, scales: np.ndarray,
               K: int) -> np.ndarray:
    """fp64 y = x . W^T with W[n][k] = c[n][k] * s[n][k/G], c the two's-complement
    value of code k of column n (no zero point).  numpy's matmul is the last step."""
    codes = unpack(packed, K, bits)
    lib = _load()
    table = np.array([lib.oracle_signed_value(c, bits) for c in range(1 << bits)], dtype=np.float64)
    w = table[codes] * np.repeat(_c(scales, np.float64), group, axis=1)
    return _c(x_f64, np.float64) @ w.T


def interleave4(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [N][K] (4-bit, K % 8 == 0) -> the lane-interleaved layout
    uint8 [N][K/2]: per 32-bit word, nibble slots hold codes 0 4 1 5 2 6 3 7."""
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    if K % 8:
        raise ValueError("K must be a multiple of 8")
    out = np.empty((N, K // 2), dtype=np.uint8)
    _load().oracle_interleave4(_ptr(codes), _ptr(out), N, K)
    return out


def deinterleave4(packed: np.ndarray, K: int) -> np.ndarray:
    """Inverse of interleave4: uint8 [N][K/2] -> codes uint8 [N][K]."""
    packed = _c(packed, np.uint8)
    N = packed.shape[0]
    if K % 8 or packed.shape[1] * 2 != K:
        raise ValueError("packed row length must be K/2, K a multiple of 8")
    out = np.empty((N, K), dtype=np.uint8)
    _load().oracle_deinterleave4(_ptr(packed), _ptr(out), N, K)
    return out


def tile16_bytes(N: int, K: int, bits: int) -> int:
    return int(_load().oracle_tile16_bytes(N, K, bits))


def tile16(codes: np.ndarray, bits: int) -> np.ndarray:
    """uint8 codes [N][K] (K % 64 == 0) -> the fragment-ordered tile16 stream
    (uint8, ceil(N/16)*16*K*bits/8 bytes)."""
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    if K % 64:
        raise ValueError("K must be a multiple of 64")
    out = np.empty(tile16_bytes(N, K, bits), dtype=np.uint8)
    _load().oracle_tile16(_ptr(codes), _ptr(out), N, K, bits)
    return out


def untile16(stream: np.ndarray, N: int, K: int, bits: int) -> np.ndarray:
    """Inverse of tile16 -> codes uint8 [N][K]."""
    stream = _c(stream, np.uint8)
    if stream.size != tile16_bytes(N, K, bits):
        raise ValueError("stream length must be tile16_bytes(N, K, bits)")
    out = np.empty((N, K), dtype=np.uint8)
    _load().oracle_untile16(_ptr(stream), _ptr(out), N, K, bits)
    return out


def float_value(code: int, ebits: int, mbits: int) -> float:
    return _load().oracle_float_value(int(code), ebits, mbits)


def qmm_float(x_f64: np.ndarray, packed: np.ndarray, ebits: int, mbits: int, group: int,
              scales: np.ndarray, K: int) -> np.ndarray:
    """fp64 y = x . W^T with W[n][k] = value(code[n][k]) * s[n][k/G] for float codes of
    1 + ebits + mbits bits.  numpy's matmul is the last step."""
    bits = 1 + ebits + mbits
    codes = unpack(packed, K, bits)
    table = np.array([float_value(c, ebits, mbits) for c in range(1 << bits)], dtype=np.float64)
    w = table[codes] * np.repeat(_c(scales, np.float64), group, axis=1)
    return _c(x_f64, np.float64) @ w.T
