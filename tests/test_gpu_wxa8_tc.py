"""GPU parity of the tcgen05 W4A8 / W8A8 path (batches of 6 .. 64 tokens for
W4A8, 2 .. 64 for W8A8, K a multiple of 512): a cluster of four CTAs splits K,
each group accumulates exactly in its own tensor-memory accumulator, and the
partial totals meet in distributed shared memory.  The int32 per-group
accumulators must equal the oracle's bit for bit, the fp16 output must meet
the 2e-3 parity bound, at every group size, ragged N (row tiles of 128 cut by
N) and the extreme accumulators.  Up to eight tokens the decode kernel's
exact-integer mode takes the shapes it can (test_gpu_wxa8_decode.py), so this
module switches that route off (qmm_set_gemv_kernel("skinny")) to keep the
tcgen05 kernel on every case from 6 (W4A8) / 2 (W8A8) tokens."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests.helpers import REL_TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    q.qmm_set_gemv_kernel("skinny")   # the decode route off: small batches take tcgen05
    yield q
    q.qmm_set_gemv_kernel("auto")


def _f16(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.float16).cuda()


def run_w4(q, prob, want_acc=True):
    w4 = q.qmm_pack(torch.from_numpy(prob.w4).cuda(), 4)
    out = q.qmm_w4a8(torch.from_numpy(prob.xq).cuda(), _f16(prob.sa), w4, _f16(prob.ws), prob.group,
                     want_acc=want_acc)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    return out


def run_w8(q, prob, want_acc=True):
    out = q.qmm_w8a8(torch.from_numpy(prob.xq).cuda(), _f16(prob.sa), torch.from_numpy(prob.w8).cuda(),
                     _f16(prob.ws), prob.group, want_acc=want_acc)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    return out


def _check(out, ref):
    y, acc = out
    y_ref, acc_ref, ov = ref
    assert not ov
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    assert rel_err(y.float().cpu().numpy().astype(np.float64), y_ref) <= REL_TOL


@pytest.mark.parametrize("M", [6, 9, 24, 48, 64])
@pytest.mark.parametrize("G", [32, 64, 128])
@pytest.mark.parametrize("N,K", [(131, 512), (300, 2048)])
def test_w4a8_tc_parity(q, M, G, N, K):
    prob = synthetic.make_w4a8(M, N, K, G, seed=M * 7 + G + N)
    _check(run_w4(q, prob), oracle.solve_w4a8(prob))


@pytest.mark.parametrize("M", [2, 16, 33, 64])
@pytest.mark.parametrize("G", [32, 64, 128])
def test_w8a8_tc_parity(q, M, G):
    prob = synthetic.make_w8a8(M, 200, 1024, G, seed=M + G)
    _check(run_w8(q, prob), oracle.solve_w8a8(prob))


def test_w4a8_tc_extreme_accumulators(q):
    # every weight -8, every activation -128: each group accumulator is 8 * 128 * G
    M, N, K, G = 64, 140, 512, 128
    prob = synthetic.make_w4a8(M, N, K, G, seed=5)
    prob.w4[:] = 8
    prob.xq[:] = -128
    y, acc = run_w4(q, prob)
    assert (acc.cpu().numpy() == 8 * 128 * G).all()
    _check((y, acc), oracle.solve_w4a8(prob))


def test_w8a8_tc_extreme_accumulators(q):
    # every weight and activation -128: each group accumulator is 2^14 * G
    M, N, K, G = 64, 130, 512, 128
    prob = synthetic.make_w8a8(M, N, K, G, seed=6)
    prob.w8[:] = -128
    prob.xq[:] = -128
    y, acc = run_w8(q, prob)
    assert (acc.cpu().numpy() == 128 * 128 * G).all()
    _check((y, acc), oracle.solve_w8a8(prob))


def test_w4a8_tc_output_without_accumulators_and_twice(q):
    # no accumulator output; two calls in a row give the same bits
    prob = synthetic.make_w4a8(32, 256, 1024, 64, seed=9)
    y1 = run_w4(q, prob, want_acc=False)
    y2 = run_w4(q, prob, want_acc=False)
    assert torch.equal(y1, y2)
    y_ref, _, _ = oracle.solve_w4a8(prob, want_acc=False)
    assert rel_err(y1.float().cpu().numpy().astype(np.float64), y_ref) <= REL_TOL
