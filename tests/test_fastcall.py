"""The binding's CPython fast-call extension (csrc/pyfast.c): it must pass
every argument of the 14-argument entry points exactly as ctypes does.  Each
case below makes the library's host checks (which run before any device
work) reject one argument, so the returned status shows that the argument
reached its own parameter; the fast call and the ctypes call must agree on
all of them.  Runs without a GPU."""
import os

import pytest

import bit_weight_quantized_gb300 as q
from bit_weight_quantized_gb300 import build as qbuild

A = 1 << 20            # a 16-byte aligned stand-in address (never dereferenced by the checks)

# Host-only: with a GPU present a call that passed its checks would launch on
# the stand-in addresses, so the module runs only where no GPU is visible.
pytestmark = pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="host-only checks; a GPU is present")
OK_ARGS = dict(x=A, xdt=0, packed=A, bits=4, group=128, scales=A, zeros=None, zc=8, y=A, ydt=0,
               M=1, N=4096, K=4096, stream=None)


def _args(**kw):
    d = dict(OK_ARGS, **kw)
    return (d["x"], d["xdt"], d["packed"], d["bits"], d["group"], d["scales"], d["zeros"], d["zc"],
            d["y"], d["ydt"], d["M"], d["N"], d["K"], d["stream"])


CASES = [
    dict(M=-1), dict(N=-5), dict(K=-64),          # QMM_ERR_SHAPE from each size
    dict(bits=0), dict(bits=9),                   # QMM_ERR_BITS
    dict(group=48), dict(K=4000),                 # group rule, K % G
    dict(zc=300), dict(zc=-1), dict(zc=300, zeros=A),
    dict(M=0), dict(N=0),                         # nothing to do: QMM_OK
    dict(y=None), dict(K=0, y=None),              # y checked before K == 0 returns
    dict(x=None), dict(packed=None), dict(scales=None),
    dict(x=A + 8), dict(packed=A + 2), dict(scales=A + 1), dict(y=A + 1),
    dict(xdt=7), dict(ydt=7),
]
# Every case is rejected by the host checks (or has nothing to do) before any
# device work, so no case launches a kernel on the stand-in addresses.


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(q.LIB_PATH):
        pytest.skip("libqmm.so not built")
    return q.load()


def test_extension_is_built_and_loaded(lib):
    if qbuild.build_fastcall() is None:
        pytest.skip("no C compiler or Python headers here")
    assert os.path.exists(q.FAST_PATH)
    assert q._call14 is not None
    assert set(q._ADDR) == {"qmm_gemv", "qmm_gemm", "qmm_gemv_tile16"}


@pytest.mark.parametrize("name", ["qmm_gemv", "qmm_gemm", "qmm_gemv_tile16"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_fast_call_matches_ctypes(lib, name, case):
    if q._call14 is None:
        pytest.skip("fast-call extension not built")
    args = _args(**CASES[case])
    assert q._call14(q._ADDR[name], *args) == q._FN[name](*args)


def test_fast_call_statuses_are_the_checks(lib):
    # a few of the statuses spelled out, so that agreement above is not agreement on noise
    if q._call14 is None:
        pytest.skip("fast-call extension not built")
    f, a = q._call14, q._ADDR["qmm_gemv"]
    assert f(a, *_args(bits=9)) == 2
    assert f(a, *_args(group=48)) == 3
    assert f(a, *_args(x=None)) == 1
    assert f(a, *_args(x=A + 8)) == 4
    assert f(a, *_args(M=0)) == 0
    assert f(a, *_args(M=17)) == 3   # qmm_gemv takes M <= 16


def test_fast_call_rejects_bad_python_arguments(lib):
    if q._call14 is None:
        pytest.skip("fast-call extension not built")
    f, a = q._call14, q._ADDR["qmm_gemv"]
    with pytest.raises(OverflowError):
        f(a, *_args(M=1 << 40))
    with pytest.raises(TypeError):
        f(a, *_args()[:-1])
    with pytest.raises(ValueError):
        f(0, *_args())
