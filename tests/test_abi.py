"""The C ABI: the library builds for sm_103a, loads, exports every symbol that
include/qmm.h declares, and rejects bad arguments on the host before touching
a device.  Runs without a GPU (valid calls report QMM_ERR_DEVICE there)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")


@pytest.fixture(scope="module")
def lib():
    from bit_weight_quantized_gb300 import build
    import bit_weight_quantized_gb300 as q
    build.build()
    return q.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^QMM_API (?:qmm_status|const char \*|int|size_t)\s*(qmm_\w+)\s*\(", text, re.M)))


def test_header_declares_the_calls():
    syms = declared_symbols()
    for name in ("qmm_pack", "qmm_unpack", "qmm_gemv", "qmm_gemm", "qmm_w4a8", "qmm_w8a8",
                 "qmm_quantize_act", "qmm_flip_sign", "qmm_gemv_float", "qmm_set_gemv_kernel",
                 "qmm_gemv_route", "qmm_repack", "qmm_repack_bytes", "qmm_gemv_tile16",
                 "qmm_device_status", "qmm_status_string", "qmm_abi_version"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_header(lib):
    import bit_weight_quantized_gb300 as q
    assert set(declared_symbols()) <= set(q.SIGNATURES)


def test_abi_version_and_strings(lib):
    assert lib.qmm_abi_version() == 1
    for s in (0, 1, 2, 3, 4, 5, 6, 8, 9):
        assert lib.qmm_status_string(s)


def _fake(addr):
    return ctypes.c_void_p(addr)


A16 = _fake(0x10000)   # 16-byte aligned dummy addresses, never dereferenced
B16 = _fake(0x20000)


def gemv(lib, **kw):
    a = dict(x=A16, xdt=0, packed=B16, bits=4, group=128, scales=A16, zeros=None, zc=8,
             y=B16, ydt=0, M=1, N=64, K=128, stream=None)
    a.update(kw)
    return lib.qmm_gemv(a["x"], a["xdt"], a["packed"], a["bits"], a["group"], a["scales"],
                        a["zeros"], a["zc"], a["y"], a["ydt"], a["M"], a["N"], a["K"], a["stream"])


def test_gemv_argument_errors(lib):
    assert gemv(lib, bits=0) == 2
    assert gemv(lib, bits=9) == 2
    assert gemv(lib, group=48) == 3
    assert gemv(lib, K=96) == 3          # K % group
    assert gemv(lib, M=-1) == 3
    assert gemv(lib, M=17) == 3          # the skinny path takes M <= 16
    assert gemv(lib, zc=256) == 3
    assert gemv(lib, x=None) == 1
    assert gemv(lib, y=None) == 1
    assert gemv(lib, x=_fake(0x10008)) == 4   # activations must be 16-byte aligned
    assert gemv(lib, packed=_fake(0x20002)) == 4
    assert gemv(lib, xdt=7) == 5         # no such activation type
    assert gemv(lib, ydt=7) == 5
    # bf16 activations pass the host checks (the route is chosen on the device;
    # without a usable GPU the call stops there)
    assert gemv(lib, xdt=1) in (0, 9)


def test_empty_problems_are_noops(lib):
    assert gemv(lib, M=0) == 0
    assert gemv(lib, N=0, x=None, packed=None, scales=None) == 0


def test_gemm_and_w4a8_argument_errors(lib):
    assert lib.qmm_gemm(A16, 1, B16, 4, 128, A16, None, 8, B16, 1, 8, 64, 128, None) == 3
    assert lib.qmm_gemm(A16, 1, B16, 4, 128, A16, None, 8, B16, 0, 64, 64, 128, None) == 5
    # the tiled path needs 16-byte aligned x, y and packed, and a packed row
    # pitch (K * bits / 8 bytes) that is a multiple of 16
    assert lib.qmm_gemm(A16, 1, B16, 4, 128, A16, None, 8, _fake(0x20002), 1, 64, 64, 128, None) == 4
    assert lib.qmm_gemm(A16, 1, _fake(0x20004), 4, 128, A16, None, 8, B16, 1, 64, 64, 128, None) == 4
    assert lib.qmm_gemm(A16, 1, B16, 3, 32, A16, None, 4, B16, 1, 64, 64, 96, None) == 4
    assert lib.qmm_w4a8(A16, A16, B16, A16, 100, B16, None, 1, 64, 128, None) == 3
    assert lib.qmm_w4a8(A16, A16, B16, A16, 128, B16, None, 65, 64, 128, None) == 3
    assert lib.qmm_w4a8(None, A16, B16, A16, 128, B16, None, 1, 64, 128, None) == 1
    assert lib.qmm_w4a8(_fake(0x10004), A16, B16, A16, 128, B16, None, 1, 64, 128, None) == 4


def test_gemv_route_rejects_bad_shapes(lib):
    assert lib.qmm_gemv_route(17, 64, 512, 4, 128, 0) == -3     # M <= 16
    assert lib.qmm_gemv_route(1, 64, 512, 9, 128, 0) == -3      # bits
    assert lib.qmm_gemv_route(1, 64, 500, 4, 128, 0) == -3      # K % group
    assert lib.qmm_gemv_route(1, 64, 512, 4, 48, 0) == -3       # group


def test_repack_sizes_and_argument_errors(lib):
    lib.qmm_repack_bytes.restype = ctypes.c_size_t
    assert lib.qmm_repack_bytes(37, 128, 3, 1) == 48 * 128 * 3 // 8     # tile16 pads rows to 16
    assert lib.qmm_repack_bytes(37, 96, 3, 1) == 0                      # K % 64
    assert lib.qmm_repack_bytes(37, 96, 4, 2) == 37 * 48                # interleave4
    assert lib.qmm_repack_bytes(37, 96, 3, 2) == 0                      # interleave4 is 4-bit only
    assert lib.qmm_repack(A16, B16, 4, 96, 4, 1, None) == 3             # K % 64
    assert lib.qmm_repack(A16, B16, 4, 64, 9, 1, None) == 2             # bits
    assert lib.qmm_repack(None, B16, 4, 64, 4, 1, None) == 1
    assert lib.qmm_repack(A16, B16, 4, 64, 4, 7, None) == 3             # layout
    # the tile16 gemv needs a 16-byte aligned stream
    assert lib.qmm_gemv_tile16(A16, 0, _fake(0x20004), 4, 128, A16, None, 8, B16, 0, 1, 64, 128, None) == 4


def test_gemv_float_argument_errors(lib):
    assert lib.qmm_gemv_float(A16, B16, 0, 3, 32, A16, B16, 1, 64, 128, None) == 2    # ebits >= 1
    assert lib.qmm_gemv_float(A16, B16, 5, 3, 32, A16, B16, 1, 64, 128, None) == 2    # 9 bits
    assert lib.qmm_gemv_float(A16, B16, 3, 2, 32, A16, B16, 17, 64, 128, None) == 3   # M <= 16
    assert lib.qmm_gemv_float(A16, B16, 3, 2, 48, A16, B16, 1, 64, 128, None) == 3    # group
    assert lib.qmm_gemv_float(None, B16, 3, 2, 32, A16, B16, 1, 64, 128, None) == 1
    assert lib.qmm_gemv_float(_fake(0x10008), B16, 3, 2, 32, A16, B16, 1, 64, 128, None) == 4
    assert lib.qmm_gemv_float(A16, B16, 3, 2, 32, A16, B16, 0, 64, 128, None) == 0


def test_flip_sign_argument_errors(lib):
    assert lib.qmm_flip_sign(B16, 4, 8, 0, None) == 2
    assert lib.qmm_flip_sign(B16, 4, 8, 9, None) == 2
    assert lib.qmm_flip_sign(B16, 4, 3, 3, None) == 3     # K*bits not byte aligned
    assert lib.qmm_flip_sign(None, 4, 8, 3, None) == 1
    assert lib.qmm_flip_sign(None, 0, 8, 3, None) == 0


def test_w8a8_argument_errors(lib):
    assert lib.qmm_w8a8(A16, A16, B16, A16, 48, B16, None, 1, 64, 128, None) == 3   # group
    assert lib.qmm_w8a8(A16, A16, B16, A16, 32, B16, None, 65, 64, 128, None) == 3  # M <= 64
    assert lib.qmm_w8a8(A16, A16, B16, A16, 32, B16, None, 1, 64, 100, None) == 3   # K % group
    assert lib.qmm_w8a8(A16, A16, None, A16, 32, B16, None, 1, 64, 128, None) == 1
    assert lib.qmm_w8a8(A16, A16, _fake(0x20008), A16, 32, B16, None, 1, 64, 128, None) == 4
    assert lib.qmm_w8a8(A16, A16, B16, A16, 32, B16, None, 0, 64, 128, None) == 0


def test_quantize_act_argument_errors(lib):
    assert lib.qmm_quantize_act(A16, B16, A16, 2, 12, None) == 3            # K % 8
    assert lib.qmm_quantize_act(A16, B16, A16, -1, 64, None) == 3
    assert lib.qmm_quantize_act(None, B16, A16, 2, 64, None) == 1
    assert lib.qmm_quantize_act(A16, B16, None, 2, 64, None) == 1
    assert lib.qmm_quantize_act(_fake(0x10008), B16, A16, 2, 64, None) == 4  # x 16-byte aligned
    assert lib.qmm_quantize_act(A16, B16, _fake(0x10001), 2, 64, None) == 4
    assert lib.qmm_quantize_act(None, None, None, 0, 64, None) == 0          # no tokens


def test_pack_argument_errors(lib):
    assert lib.qmm_pack(A16, B16, 4, 3, 3, None, None) == 3   # K*bits not byte aligned
    assert lib.qmm_pack(A16, B16, 4, 8, 0, None, None) == 2
    assert lib.qmm_pack(None, B16, 4, 8, 3, None, None) == 1
    assert lib.qmm_unpack(A16, B16, 4, 8, 9, None) == 2


def test_gemv_kernel_choice(lib):
    import bit_weight_quantized_gb300 as q
    assert lib.qmm_set_gemv_kernel(2) == 3
    assert lib.qmm_set_gemv_kernel(-1) == 3
    assert lib.qmm_set_gemv_kernel(1) == 0
    assert lib.qmm_set_gemv_kernel(0) == 0
    with pytest.raises(ValueError):
        q.qmm_set_gemv_kernel("fastest")
    q.qmm_set_gemv_kernel("skinny")
    q.qmm_set_gemv_kernel("auto")


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="needs a machine without a GPU")
def test_valid_call_without_device_fails_loudly(lib):
    assert gemv(lib) == 9
    assert lib.qmm_pack(A16, B16, 4, 8, 3, None, None) == 9


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    import bit_weight_quantized_gb300 as q
    x = torch.zeros(1, 128, dtype=torch.float16)
    p = torch.zeros(64, 64, dtype=torch.uint8)
    s = torch.zeros(64, 1, dtype=torch.float16)
    with pytest.raises(ValueError):
        q.qmm_gemv(x, p, 4, 128, s)
