"""GPU parity of the integer-native W4A8 path: the int32 per-group
accumulators must equal the oracle's bit for bit; the fp16 output must meet
the 2e-3 parity bound."""
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


def to_dev(prob):
    import bit_weight_quantized_gb300 as q
    w4 = q.qmm_pack(torch.from_numpy(prob.w4).cuda(), 4)
    ws = torch.from_numpy(prob.ws.view(np.int16)).view(torch.float16).cuda()
    xq = torch.from_numpy(prob.xq).cuda()
    sa = torch.from_numpy(prob.sa.view(np.int16)).view(torch.float16).cuda()
    return xq, sa, w4, ws


def run(q, prob, cols=None):
    xq, sa, w4, ws = to_dev(prob)
    y, acc = q.qmm_w4a8(xq, sa, w4, ws, prob.group, want_acc=True)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    return y.float().cpu().numpy().astype(np.float64), acc.cpu().numpy()


@pytest.mark.parametrize("M,N,K,G", [(1, 37, 256, 128), (5, 130, 512, 64), (16, 64, 384, 32),
                                     (17, 50, 1024, 128), (33, 29, 256, 64), (64, 40, 512, 128),
                                     (8, 300, 4096, 128)])
def test_w4a8_parity_small(q, M, N, K, G):
    prob = synthetic.make_w4a8(M, N, K, G, seed=M * 1000 + N)
    y, acc = run(q, prob)
    y_ref, acc_ref, ov = oracle.solve_w4a8(prob)
    assert not ov
    np.testing.assert_array_equal(acc, acc_ref)
    assert rel_err(y, y_ref) <= REL_TOL


def test_w4a8_extreme_values(q):
    # all weights -8 and all activations -127: the largest |accumulator|
    M, N, K, G = 3, 20, 256, 128
    prob = synthetic.make_w4a8(M, N, K, G, seed=1)
    prob.w4[:] = 8        # code of -8
    prob.xq[:] = -127
    y, acc = run(q, prob)
    assert (acc == 127 * 8 * G).all()
    y_ref, acc_ref, _ = oracle.solve_w4a8(prob)
    np.testing.assert_array_equal(acc, acc_ref)
    assert rel_err(y, y_ref) <= REL_TOL


@pytest.mark.parametrize("M", [1, 16, 64])
def test_w4a8_full_size(q, M):
    prob = synthetic.w4a8(M)
    y, acc = run(q, prob)
    st = SplitMix64(M)
    cols = np.unique((st.next(512) % np.uint64(prob.N)).astype(np.int64))
    cols = np.concatenate([cols, [0, prob.N - 1]])
    y_ref, acc_ref, ov = oracle.solve_w4a8(prob, cols=cols)
    assert not ov
    np.testing.assert_array_equal(acc[:, cols, :], acc_ref)
    assert rel_err(y[:, cols], y_ref) <= REL_TOL


def test_w4a8_without_accumulators(q):
    prob = synthetic.make_w4a8(4, 96, 512, 128, seed=3)
    xq, sa, w4, ws = to_dev(prob)
    y = q.qmm_w4a8(xq, sa, w4, ws, 128)
    y_ref, _, _ = oracle.solve_w4a8(prob, want_acc=False)
    assert rel_err(y.float().cpu().numpy().astype(np.float64), y_ref) <= REL_TOL


def test_w4a8_row_blocks_sampled(q):
    # more than 128 rows per CTA: two row blocks, accumulators still exact
    prob = synthetic.make_w4a8(64, 20000, 1024, 128, seed=11)
    y, acc = run(q, prob)
    st = SplitMix64(20000)
    cols = np.unique(np.concatenate([(st.next(256) % np.uint64(prob.N)).astype(np.int64),
                                     np.arange(0, 140), [prob.N - 1]]))
    y_ref, acc_ref, ov = oracle.solve_w4a8(prob, cols=cols)
    assert not ov
    np.testing.assert_array_equal(acc[:, cols, :], acc_ref)
    assert rel_err(y[:, cols], y_ref) <= REL_TOL
