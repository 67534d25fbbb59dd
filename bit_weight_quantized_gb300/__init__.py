"""FP16/BF16 x INT1-8 quantized matmul on GB300 (sm_103a).

A thin ctypes binding over ``lib/libqmm.so`` (C ABI in ``include/qmm.h``).
The functions keep the C names and only marshal arguments: torch tensors are
used for device memory and the current CUDA stream, every step of the
computation runs in the library's kernels.  There is no CPU fallback: if the
library has not been built (``python -m bit_weight_quantized_gb300.build``) or
no sm_103a device is present, calls raise.

Storage: the b-bit weight matrix is a per-column LSB-first bitstream along K,
``packed[n]`` holding K*b/8 bytes (see qmm.h); scales are fp16 ``[N][K/G]``,
zeros are uint8 ``[N][K/G]`` or a constant.
"""
from __future__ import annotations

import ctypes
import importlib.util
import os
import sysconfig
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libqmm.so")

QMM_F16 = 0
QMM_BF16 = 1

STATUS_NAMES = {
    0: "QMM_OK", 1: "QMM_ERR_NULL", 2: "QMM_ERR_BITS", 3: "QMM_ERR_SHAPE",
    4: "QMM_ERR_ALIGN", 5: "QMM_ERR_UNSUPPORTED", 6: "QMM_ERR_CUDA",
    8: "QMM_ERR_TIMEOUT", 9: "QMM_ERR_DEVICE",
}

# C entry points and their ctypes signatures (must match include/qmm.h)
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "qmm_pack": ([_P, _P, _I, _I, _I, _P, _P], _I),
    "qmm_unpack": ([_P, _P, _I, _I, _I, _P], _I),
    "qmm_gemv": ([_P, _I, _P, _I, _I, _P, _P, _I, _P, _I, _I, _I, _I, _P], _I),
    "qmm_gemm": ([_P, _I, _P, _I, _I, _P, _P, _I, _P, _I, _I, _I, _I, _P], _I),
    "qmm_w4a8": ([_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P], _I),
    "qmm_w8a8": ([_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P], _I),
    "qmm_flip_sign": ([_P, _I, _I, _I, _P], _I),
    "qmm_gemv_float": ([_P, _P, _I, _I, _I, _P, _P, _I, _I, _I, _P], _I),
    "qmm_quantize_act": ([_P, _P, _P, _I, _I, _P], _I),
    "qmm_set_gemv_kernel": ([_I], _I),
    "qmm_gemv_route": ([_I, _I, _I, _I, _I, _I], _I),
    "qmm_repack_bytes": ([_I, _I, _I, _I], _SZ),
    "qmm_repack": ([_P, _P, _I, _I, _I, _I, _P], _I),
    "qmm_gemv_tile16": ([_P, _I, _P, _I, _I, _P, _P, _I, _P, _I, _I, _I, _I, _P], _I),
    "qmm_device_status": ([_P], _I),
    "qmm_watchdog_selftest": ([_P], _I),
    "qmm_status_string": ([_I], ctypes.c_char_p),
    "qmm_abi_version": ([], _I),
}

_lib = None
_FN = {}   # name -> the configured ctypes function, filled by load()

# The optional CPython fast-call extension (csrc/pyfast.c, built next to the
# library): it calls the 14-argument entry points through their addresses,
# without ctypes' per-argument conversion.  Without it the calls go through
# ctypes; either way the same library function runs.
FAST_PATH = os.path.join(_HERE, "lib", "_qmmfast" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))
_FAST_NAMES = ("qmm_gemv", "qmm_gemm", "qmm_gemv_tile16")
_call14 = None
_ADDR = {}   # name -> function address for _call14, filled by load()


def _load_fastcall(lib):
    global _call14
    if not os.path.exists(FAST_PATH):
        return
    try:
        spec = importlib.util.spec_from_file_location("_qmmfast", FAST_PATH)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    except (ImportError, OSError):
        return
    for name in _FAST_NAMES:
        _ADDR[name] = ctypes.cast(getattr(lib, name), ctypes.c_void_p).value
    _call14 = mod.call14


class QmmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libqmm.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"libqmm.so not built ({path}); run "
                              "`python -m bit_weight_quantized_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
            _FN[name] = fn
        _load_fastcall(lib)
        _lib = lib
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise QmmError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    # a plain int: ctypes converts it for a c_void_p argument without an object
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device=None):
    # the raw handle (an int) of the current stream, without building a Stream
    # object; `device` is a device index, a torch.device or None (the current one)
    if _raw_stream is not None:
        idx = device.index if isinstance(device, torch.device) else device
        if idx is None:
            idx = torch.cuda.current_device()
        return _raw_stream(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not (t.is_cuda and t.is_contiguous()) or (dtype is not None and t.dtype != dtype) or (
            shape is not None and t.shape != shape):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


_DT = {torch.float16: QMM_F16, torch.bfloat16: QMM_BF16}


def qmm_pack(codes: torch.Tensor, bits: int, bad_count: Optional[torch.Tensor] = None,
             out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """uint8 codes [N][K] -> packed bitstream [N][K*bits/8] (see qmm_pack)."""
    _dev(codes, "codes", torch.uint8)
    N, K = codes.shape
    if out is None:
        out = torch.empty((N, K * bits // 8), dtype=torch.uint8, device=codes.device)
    if bad_count is not None:
        _dev(bad_count, "bad_count", torch.int32)
    _check(load().qmm_pack(_ptr(codes), _ptr(out), N, K, bits, _ptr(bad_count),
                           _stream(codes.device)), "qmm_pack")
    return out


def qmm_unpack(packed: torch.Tensor, K: int, bits: int) -> torch.Tensor:
    _dev(packed, "packed", torch.uint8)
    N = packed.shape[0]
    out = torch.empty((N, K), dtype=torch.uint8, device=packed.device)
    _check(load().qmm_unpack(_ptr(packed), _ptr(out), N, K, bits, _stream(packed.device)),
           "qmm_unpack")
    return out


def _qmm_checks(x, packed, bits, group, scales, zeros, out, out_dtype):
    # the argument checks one by one, for a precise error message
    _dev(x, "x")
    M, K = x.shape
    _dev(packed, "packed", torch.uint8)
    N = packed.shape[0]
    if packed.shape[1] * 8 != K * bits:
        raise ValueError("packed must be [N][K*bits/8]")
    _dev(scales, "scales", torch.float16, (N, K // group))
    if zeros is not None:
        _dev(zeros, "zeros", torch.uint8, (N, K // group))
    if x.dtype not in _DT:
        raise ValueError("x must be float16 or bfloat16")
    _dev(out, "out", out_dtype, (M, N))


_U8, _F16 = torch.uint8, torch.float16


def _qmm(name, x, packed, bits, group, scales, zeros, zero_const, out, out_dtype):
    # the common path of the gemv/gemm calls, with the checks folded into one
    # expression (a call costs a few microseconds of host time; the checks were
    # a third of it); any failure re-runs them one by one for the message
    xdt = x.dtype
    M, K = x.shape
    N = packed.shape[0]
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else xdt
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    ng = K // group
    if not (x.is_cuda and x.is_contiguous() and xdt in _DT and packed.is_cuda and packed.is_contiguous()
            and packed.dtype is _U8 and packed.shape[1] * 8 == K * bits and scales.is_cuda
            and scales.is_contiguous() and scales.dtype is _F16 and scales.shape == (N, ng) and out.is_cuda
            and out.is_contiguous() and out.dtype is out_dtype and out.shape == (M, N)
            and (zeros is None or (zeros.is_cuda and zeros.is_contiguous() and zeros.dtype is _U8
                                   and zeros.shape == (N, ng)))):
        _qmm_checks(x, packed, bits, group, scales, zeros, out, out_dtype)
        raise ValueError(f"{name}: arguments do not match")
    if _lib is None:
        load()
    args = (x.data_ptr(), _DT[xdt], packed.data_ptr(), bits, group, scales.data_ptr(),
            None if zeros is None else zeros.data_ptr(), int(zero_const), out.data_ptr(),
            _DT[out_dtype], M, N, K, _stream(x.get_device()))
    st = _call14(_ADDR[name], *args) if _call14 is not None else _FN[name](*args)
    if st:
        raise QmmError(st, name)
    return out


def qmm_gemv(x, packed, bits, group, scales, zeros=None, zero_const=0, out=None,
             out_dtype=None) -> torch.Tensor:
    """y[M][N] = x . W^T for 1 <= M <= 16 (the decode or the skinny kernel)."""
    return _qmm("qmm_gemv", x, packed, bits, group, scales, zeros, zero_const, out, out_dtype)


LAYOUTS = {"tile16": 1, "interleave4": 2}


def qmm_repack_bytes(N: int, K: int, bits: int, layout: str) -> int:
    """Bytes of the `layout` form ("tile16" or "interleave4") of an N x K
    bits-bit weight matrix (0 if the layout does not take these sizes)."""
    return int(load().qmm_repack_bytes(N, K, bits, LAYOUTS[layout]))


def qmm_repack(packed: torch.Tensor, K: int, bits: int, layout: str, out: Optional[torch.Tensor] = None):
    """Canonical packed bitstream [N][K*bits/8] -> a flat uint8 tensor in `layout`."""
    _dev(packed, "packed", torch.uint8)
    N = packed.shape[0]
    if packed.shape[1] * 8 != K * bits:
        raise ValueError("packed must be [N][K*bits/8]")
    nbytes = qmm_repack_bytes(N, K, bits, layout)
    if nbytes == 0 and N * K:
        raise QmmError(3, "qmm_repack")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=packed.device)
    _dev(out, "out", torch.uint8, (nbytes,))
    _check(load().qmm_repack(packed.data_ptr(), out.data_ptr(), N, K, bits, LAYOUTS[layout],
                             _stream(packed.get_device())), "qmm_repack")
    return out


def qmm_gemv_tile16(x, tiled, N, bits, group, scales, zeros=None, zero_const=0, out=None,
                    out_dtype=None) -> torch.Tensor:
    """qmm_gemv on weights in the tile16 layout (`tiled`: the flat output of
    qmm_repack(..., "tile16") for N output columns)."""
    _dev(x, "x")
    M, K = x.shape
    _dev(tiled, "tiled", torch.uint8, (qmm_repack_bytes(N, K, bits, "tile16"),))
    _dev(scales, "scales", torch.float16, (N, K // group))
    if zeros is not None:
        _dev(zeros, "zeros", torch.uint8, (N, K // group))
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else x.dtype
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    _dev(out, "out", out_dtype, (M, N))
    if _lib is None:
        load()
    args = (x.data_ptr(), _DT[x.dtype], tiled.data_ptr(), bits, group, scales.data_ptr(),
            None if zeros is None else zeros.data_ptr(), int(zero_const), out.data_ptr(),
            _DT[out_dtype], M, N, K, _stream(x.get_device()))
    st = _call14(_ADDR["qmm_gemv_tile16"], *args) if _call14 is not None else _FN["qmm_gemv_tile16"](*args)
    if st:
        raise QmmError(st, "qmm_gemv_tile16")
    return out


GEMV_KERNELS = {"auto": 0, "skinny": 1}


def qmm_set_gemv_kernel(kernel: str):
    """Kernel choice of qmm_gemv for the calls that follow, process-wide:
    "auto" (the decode kernel where it applies, else the skinny kernel) or
    "skinny" (the skinny kernel for every shape; qmm_w4a8 / qmm_w8a8 then stay
    off the decode kernel too)."""
    if kernel not in GEMV_KERNELS:
        raise ValueError(f"kernel must be one of {sorted(GEMV_KERNELS)}")
    _check(load().qmm_set_gemv_kernel(GEMV_KERNELS[kernel]), "qmm_set_gemv_kernel")


def qmm_gemv_route(M: int, N: int, K: int, bits: int, group: int, stored_zeros: bool) -> str:
    """The kernel a qmm_gemv call of this shape runs on the current device:
    "decode" (the staged decode kernel) or "skinny"."""
    r = load().qmm_gemv_route(M, N, K, bits, group, 1 if stored_zeros else 0)
    if r < 0:
        raise QmmError(-r, "qmm_gemv_route")
    return "decode" if r == 0 else "skinny"


def qmm_gemm(x, packed, bits, group, scales, zeros=None, zero_const=0, out=None,
             out_dtype=None) -> torch.Tensor:
    """y[M][N] = x . W^T for M >= 17 (tiled tensor-core path)."""
    return _qmm("qmm_gemm", x, packed, bits, group, scales, zeros, zero_const, out, out_dtype)


def qmm_w4a8(xq, sa, w4, ws, group=128, want_acc=False, out=None, acc_out=None):
    """Integer-native W4A8: returns y (fp16 [M][N]) and, if requested, the int32
    accumulators [M][N][K/group]."""
    _dev(xq, "xq", torch.int8)
    M, K = xq.shape
    _dev(sa, "sa", torch.float16, (M,))
    _dev(w4, "w4", torch.uint8)
    N = w4.shape[0]
    if w4.shape[1] * 2 != K:
        raise ValueError("w4 must be [N][K/2]")
    _dev(ws, "ws", torch.float16, (N, K // group))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=xq.device)
    if want_acc and acc_out is None:
        acc_out = torch.empty((M, N, K // group), dtype=torch.int32, device=xq.device)
    _check(load().qmm_w4a8(_ptr(xq), _ptr(sa), _ptr(w4), _ptr(ws), group, _ptr(out),
                           _ptr(acc_out), M, N, K, _stream(xq.device)), "qmm_w4a8")
    return (out, acc_out) if want_acc else out


def qmm_gemv_float(x, packed, ebits, mbits, group, scales, out=None):
    """y[M][N] = x . W^T (fp16, 1 <= M <= 16) for float weight codes of
    1 + ebits + mbits bits (sign, exponent, mantissa; all encodings finite)."""
    _dev(x, "x", torch.float16)
    M, K = x.shape
    bits = 1 + ebits + mbits
    _dev(packed, "packed", torch.uint8)
    N = packed.shape[0]
    if packed.shape[1] * 8 != K * bits:
        raise ValueError("packed must be [N][K*bits/8]")
    _dev(scales, "scales", torch.float16, (N, K // group))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _dev(out, "out", torch.float16, (M, N))
    _check(load().qmm_gemv_float(_ptr(x), _ptr(packed), ebits, mbits, group, _ptr(scales), _ptr(out),
                                 M, N, K, _stream(x.device)), "qmm_gemv_float")
    return out


def qmm_flip_sign(packed, K, bits):
    """Flips the top bit of every b-bit code of `packed` ([N][K*bits/8]) in place:
    signed two's-complement codes become offset-binary codes for qmm_gemv /
    qmm_gemm with zero_const = 2**(bits-1).  Returns `packed`."""
    _dev(packed, "packed", torch.uint8)
    N = packed.shape[0]
    if packed.shape[1] * 8 != K * bits:
        raise ValueError("packed must be [N][K*bits/8]")
    _check(load().qmm_flip_sign(_ptr(packed), N, K, bits, _stream(packed.device)), "qmm_flip_sign")
    return packed


def qmm_w8a8(xq, sa, w8, ws, group=32, want_acc=False, out=None, acc_out=None):
    """Integer-native W8A8 (int8 weights [N][K]): returns y (fp16 [M][N]) and, if
    requested, the int32 accumulators [M][N][K/group]."""
    _dev(xq, "xq", torch.int8)
    M, K = xq.shape
    _dev(sa, "sa", torch.float16, (M,))
    _dev(w8, "w8", torch.int8)
    N = w8.shape[0]
    if w8.shape[1] != K:
        raise ValueError("w8 must be [N][K]")
    _dev(ws, "ws", torch.float16, (N, K // group))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=xq.device)
    if want_acc and acc_out is None:
        acc_out = torch.empty((M, N, K // group), dtype=torch.int32, device=xq.device)
    _check(load().qmm_w8a8(_ptr(xq), _ptr(sa), _ptr(w8), _ptr(ws), group, _ptr(out),
                           _ptr(acc_out), M, N, K, _stream(xq.device)), "qmm_w8a8")
    return (out, acc_out) if want_acc else out


def qmm_quantize_act(x, xq=None, sa=None):
    """Per-token int8 quantization of fp16 activations for qmm_w4a8: returns
    (xq int8 [M][K], sa fp16 [M]) with sa = fp16(max|x| / 127) and
    xq = round-half-even(x / sa) clipped to [-128, 127]."""
    _dev(x, "x", torch.float16)
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if sa is None:
        sa = torch.empty((M,), dtype=torch.float16, device=x.device)
    _dev(xq, "xq", torch.int8, (M, K))
    _dev(sa, "sa", torch.float16, (M,))
    _check(load().qmm_quantize_act(_ptr(x), _ptr(xq), _ptr(sa), M, K, _stream(x.device)),
           "qmm_quantize_act")
    return xq, sa


def qmm_device_status(stream=None) -> int:
    """Synchronizes the stream and returns (and clears) the device status word."""
    s = stream.cuda_stream if stream is not None else _stream()
    return load().qmm_device_status(s)


def qmm_status_string(status: int) -> str:
    return load().qmm_status_string(status).decode()


def native_library_path() -> str:
    return LIB_PATH


def qmm_watchdog_selftest(device=None):
    """Runs the library's bounded-wait watchdog once on a wait that never
    completes (about a second); qmm_device_status() then reports
    QMM_ERR_TIMEOUT."""
    _check(load().qmm_watchdog_selftest(_stream(device)), "qmm_watchdog_selftest")
