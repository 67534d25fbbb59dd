"""GPU parity of the per-token int8 activation quantizer (qmm_quantize_act)
against the oracle: scales and int8 codes bit for bit, and the chain
quantize -> qmm_w4a8 against the oracle's chain."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    return q


def run(q, x16):
    x = torch.from_numpy(x16.view(np.int16)).view(torch.float16).cuda()
    xq = torch.full(x.shape, 99, dtype=torch.int8, device="cuda")
    sa = torch.full((x.shape[0],), float("nan"), dtype=torch.float16, device="cuda")
    q.qmm_quantize_act(x, xq, sa)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    return xq.cpu().numpy(), sa.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,K", [(1, 8), (1, 4096), (3, 96), (16, 4096), (64, 4096), (300, 1032),
                                 (2, 65536)])
def test_quantize_act_bit_exact(q, M, K):
    x16 = synthetic.make_act(M, K, seed=M * 31 + K)
    xq, sa = run(q, x16)
    xq_ref, sa_ref = oracle.quantize_act(x16.view(np.uint16))
    np.testing.assert_array_equal(sa, sa_ref)
    np.testing.assert_array_equal(xq, xq_ref)


def test_quantize_act_edge_tokens(q):
    K = 256
    rows = np.zeros((5, K), dtype=np.float64)
    rows[1] = ((np.arange(K) % 8) - 3.5) / 32.0   # s = 1/32: every x / s is a tie
    rows[1, 0] = 127.0 / 32.0
    rows[2, :] = 3e-6                       # the scale underflows fp16 to 0
    rows[3, :7] = [65504.0, -65504.0, 1.0, -1.0, 257.9, 0.0, -0.0]
    rows[4] = np.linspace(-1, 1, K) * 1e-3   # fp16 subnormal and normal values
    x16 = rows.astype(np.float16)
    xq, sa = run(q, x16)
    xq_ref, sa_ref = oracle.quantize_act(x16.view(np.uint16))
    np.testing.assert_array_equal(sa, sa_ref)
    np.testing.assert_array_equal(xq, xq_ref)
    assert sa[0] == 0 and sa[2] == 0 and not xq[0].any() and not xq[2].any()


def test_quantize_then_w4a8_chain(q):
    """fp16 activations -> qmm_quantize_act -> qmm_w4a8 equals the oracle's chain."""
    M, N, K, G = 16, 512, 1024, 128
    prob = synthetic.make_w4a8(M, N, K, G, seed=5)
    x16 = synthetic.make_act(M, K, seed=6)
    prob.xq, prob.sa = oracle.quantize_act(x16.view(np.uint16))
    prob.sa = prob.sa.view(np.float16)
    x = torch.from_numpy(x16.view(np.int16)).view(torch.float16).cuda()
    xq, sa = q.qmm_quantize_act(x)
    w4 = q.qmm_pack(torch.from_numpy(prob.w4).cuda(), 4)
    ws = torch.from_numpy(prob.ws.view(np.int16)).view(torch.float16).cuda()
    y, acc = q.qmm_w4a8(xq, sa, w4, ws, G, want_acc=True)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    y_ref, acc_ref, ov = oracle.solve_w4a8(prob)
    assert not ov
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    y64 = y.float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(y64 - y_ref)) / np.max(np.abs(y_ref)) <= 2e-3
