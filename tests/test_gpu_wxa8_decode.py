"""GPU parity of the decode kernel's exact-integer mode, which serves qmm_w4a8
and qmm_w8a8 up to eight tokens when the group is 64 or 128 and K a multiple
of eight groups: int8 activations become exact fp16, the signed codes
offset-binary u = c xor 2^(b-1) with the plan's 2^E offset taken off before
the MMA, so every product and group sum is an integer below 2^24 and the
int32 accumulators must equal the oracle's bit for bit.  Each case also runs
with the decode route switched off (qmm_set_gemv_kernel("skinny"): the skinny
or the tcgen05 kernel), which must return the same accumulators."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import SplitMix64
from tests.helpers import REL_TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    return q


def run(q, prob, bits, kernel="auto"):
    xq = torch.from_numpy(prob.xq).cuda()
    sa = torch.from_numpy(prob.sa.view(np.int16)).view(torch.float16).cuda()
    ws = torch.from_numpy(prob.ws.view(np.int16)).view(torch.float16).cuda()
    q.qmm_set_gemv_kernel(kernel)
    try:
        if bits == 4:
            w = q.qmm_pack(torch.from_numpy(prob.w4).cuda(), 4)
            y, acc = q.qmm_w4a8(xq, sa, w, ws, prob.group, want_acc=True)
        else:
            w = torch.from_numpy(prob.w8).cuda()
            y, acc = q.qmm_w8a8(xq, sa, w, ws, prob.group, want_acc=True)
        torch.cuda.synchronize()
    finally:
        q.qmm_set_gemv_kernel("auto")
    assert q.qmm_device_status() == 0
    return y.float().cpu().numpy().astype(np.float64), acc.cpu().numpy()


def check(q, prob, bits):
    solve = oracle.solve_w4a8 if bits == 4 else oracle.solve_w8a8
    y_ref, acc_ref, ov = solve(prob)
    assert not ov
    y, acc = run(q, prob, bits)
    np.testing.assert_array_equal(acc, acc_ref)
    assert rel_err(y, y_ref) <= REL_TOL
    y2, acc2 = run(q, prob, bits, "skinny")
    np.testing.assert_array_equal(acc2, acc_ref)
    assert rel_err(y2, y_ref) <= REL_TOL


@pytest.mark.parametrize("M,N,K,G", [(1, 300, 1024, 128), (2, 130, 512, 64), (3, 4096, 4096, 128),
                                     (5, 257, 2048, 64), (4, 40, 8192, 128), (1, 152 * 27 + 5, 1024, 64),
                                     (6, 512, 4096, 128), (7, 99, 1024, 64), (8, 4096, 4096, 128)])
def test_w4a8_decode_mode(q, M, N, K, G):
    check(q, synthetic.make_w4a8(M, N, K, G, seed=M * 37 + N), 4)


@pytest.mark.parametrize("M,N,K,G", [(1, 300, 1024, 128), (1, 130, 512, 64), (1, 4096, 4096, 128),
                                     (1, 257, 2048, 64), (2, 600, 2048, 128), (5, 77, 1024, 64),
                                     (8, 4096, 4096, 128)])
def test_w8a8_decode_mode(q, M, N, K, G):
    check(q, synthetic.make_w8a8(M, N, K, G, seed=M + N + K), 8)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("w_fill,x_fill", [("min", -128), ("min", 127), ("max", -128), ("max", 127)])
def test_decode_mode_extreme_accumulators(q, bits, w_fill, x_fill):
    # every code at the width's extreme and every activation at an int8 extreme:
    # the largest |accumulator| the group allows (8 * 128 * 128 at b = 4,
    # 128 * 128 * 128 at b = 8)
    M, N, K, G = 1 if bits == 8 else 3, 64, 1024, 128
    prob = (synthetic.make_w4a8 if bits == 4 else synthetic.make_w8a8)(M, N, K, G, seed=bits)
    if bits == 4:
        prob.w4[:] = 8 if w_fill == "min" else 7      # codes of -8 and 7
    else:
        prob.w8[:] = -128 if w_fill == "min" else 127
    prob.xq[:] = x_fill
    check(q, prob, bits)


def test_w4a8_decode_mode_without_accumulators(q):
    prob = synthetic.make_w4a8(2, 512, 2048, 128, seed=9)
    xq = torch.from_numpy(prob.xq).cuda()
    sa = torch.from_numpy(prob.sa.view(np.int16)).view(torch.float16).cuda()
    ws = torch.from_numpy(prob.ws.view(np.int16)).view(torch.float16).cuda()
    w = q.qmm_pack(torch.from_numpy(prob.w4).cuda(), 4)
    y = q.qmm_w4a8(xq, sa, w, ws, 128)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    y_ref, _, _ = oracle.solve_w4a8(prob)
    assert rel_err(y.float().cpu().numpy().astype(np.float64), y_ref) <= REL_TOL
