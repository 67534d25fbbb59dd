"""GPU parity of the integer-native W8A8 path (qmm_w8a8): the int32 per-group
accumulators equal the oracle's bit for bit; the fp16 output meets the
2e-3 parity bound."""
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
    return q


def run(q, prob):
    xq = torch.from_numpy(prob.xq).cuda()
    sa = torch.from_numpy(prob.sa.view(np.int16)).view(torch.float16).cuda()
    w8 = torch.from_numpy(prob.w8).cuda()
    ws = torch.from_numpy(prob.ws.view(np.int16)).view(torch.float16).cuda()
    y, acc = q.qmm_w8a8(xq, sa, w8, ws, prob.group, want_acc=True)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    return y.float().cpu().numpy().astype(np.float64), acc.cpu().numpy()


@pytest.mark.parametrize("M,N,K,G", [(1, 37, 256, 32), (5, 130, 512, 64), (16, 64, 384, 128),
                                     (17, 50, 1024, 32), (33, 29, 256, 64), (64, 40, 512, 32),
                                     (8, 300, 4096, 128)])
def test_w8a8_parity_small(q, M, N, K, G):
    prob = synthetic.make_w8a8(M, N, K, G, seed=M * 100 + N)
    y, acc = run(q, prob)
    y_ref, acc_ref, ov = oracle.solve_w8a8(prob)
    assert not ov
    np.testing.assert_array_equal(acc, acc_ref)
    assert rel_err(y, y_ref) <= REL_TOL


def test_w8a8_extreme_values(q):
    # all weights -128 and all activations -127: the largest |accumulator| at G = 128
    prob = synthetic.make_w8a8(3, 20, 256, 128, seed=2)
    prob.w8[:] = -128
    prob.xq[:] = -127
    y, acc = run(q, prob)
    assert (acc == 128 * 127 * 128).all()
    y_ref, acc_ref, _ = oracle.solve_w8a8(prob)
    np.testing.assert_array_equal(acc, acc_ref)
    assert rel_err(y, y_ref) <= REL_TOL


@pytest.mark.parametrize("M", [1, 16, 64])
def test_w8a8_decode_shapes(q, M):
    """K = N = 4096 with the pages' group of 32."""
    prob = synthetic.make_w8a8(M, 4096, 4096, 32, seed=M)
    y, acc = run(q, prob)
    y_ref, acc_ref, ov = oracle.solve_w8a8(prob)
    assert not ov
    np.testing.assert_array_equal(acc, acc_ref)
    assert rel_err(y, y_ref) <= REL_TOL


def test_w8a8_from_fp16_activations(q):
    """fp16 activations -> qmm_quantize_act -> qmm_w8a8 equals the oracle's chain."""
    prob = synthetic.make_w8a8(16, 256, 1024, 32, seed=8)
    x16 = synthetic.make_act(16, 1024, seed=9)
    prob.xq, sa_bits = oracle.quantize_act(x16.view(np.uint16))
    prob.sa = sa_bits.view(np.float16)
    x = torch.from_numpy(x16.view(np.int16)).view(torch.float16).cuda()
    xq, sa = q.qmm_quantize_act(x)
    w8 = torch.from_numpy(prob.w8).cuda()
    ws = torch.from_numpy(prob.ws.view(np.int16)).view(torch.float16).cuda()
    y, acc = q.qmm_w8a8(xq, sa, w8, ws, 32, want_acc=True)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    y_ref, acc_ref, ov = oracle.solve_w8a8(prob)
    assert not ov
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    assert rel_err(y.float().cpu().numpy().astype(np.float64), y_ref) <= REL_TOL
