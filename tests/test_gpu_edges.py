"""Edge cases on the GPU: empty problems (K = 0 gives zero outputs; M = 0 or
N = 0 launches nothing), the smallest K (one group of 32), and a long K that
stages the activations in many K phases."""
import numpy as np
import pytest
import torch

import synthetic
from synthetic import SplitMix64
from tests.helpers import REL_TOL, oracle_y, rel_err, to_dev_problem, y_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    return q


def nan16(*shape, dtype=torch.float16):
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def test_k_zero_gives_zeros(q):
    M, N = 3, 40
    x = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    packed = torch.empty((N, 0), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, 0), dtype=torch.float16, device="cuda")
    y = q.qmm_gemv(x, packed, 4, 128, scales, None, 8, out=nan16(M, N))
    torch.cuda.synchronize()
    assert (y == 0).all()
    x17 = torch.empty((17, 0), dtype=torch.bfloat16, device="cuda")
    y = q.qmm_gemm(x17, packed, 4, 128, scales, None, 8, out=nan16(17, N, dtype=torch.bfloat16))
    torch.cuda.synchronize()
    assert (y == 0).all()
    xq = torch.empty((M, 0), dtype=torch.int8, device="cuda")
    sa = torch.ones(M, dtype=torch.float16, device="cuda")
    y = q.qmm_w4a8(xq, sa, packed, scales, 128, out=nan16(M, N))
    torch.cuda.synchronize()
    assert (y == 0).all()
    w8 = torch.empty((N, 0), dtype=torch.int8, device="cuda")
    y = q.qmm_w8a8(xq, sa, w8, scales, 32, out=nan16(M, N))
    torch.cuda.synchronize()
    assert (y == 0).all()
    y = q.qmm_gemv_float(x, packed, 3, 2, 32, scales, out=nan16(M, N))
    torch.cuda.synchronize()
    assert (y == 0).all()
    _, sa_out = q.qmm_quantize_act(x, torch.empty((M, 0), dtype=torch.int8, device="cuda"), nan16(M))
    torch.cuda.synchronize()
    assert (sa_out == 0).all()
    assert q.qmm_device_status() == 0


def test_empty_m_or_n_is_a_noop(q):
    prob = synthetic.make_qmm(1, 8, 128, 4, 128, zero_mode="const8", seed=1)
    x, packed, scales, _ = to_dev_problem(prob)
    y = q.qmm_gemv(x[:0], packed, 4, 128, scales, None, 8)
    assert y.shape == (0, 8)
    y = q.qmm_gemv(x, packed[:0], 4, 128, scales[:0], None, 8)
    assert y.shape == (1, 0)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0


@pytest.mark.parametrize("bits", [1, 3, 4, 8])
def test_single_group_k32(q, bits):
    prob = synthetic.make_qmm(5, 70, 32, bits, 32, zero_mode="group", seed=bits)
    x, packed, scales, zeros = to_dev_problem(prob)
    y = q.qmm_gemv(x, packed, bits, 32, scales, zeros, 0, out=nan16(5, 70))
    torch.cuda.synchronize()
    assert rel_err(y_to_f64(y), oracle_y(prob)) <= REL_TOL
    assert q.qmm_device_status() == 0


def test_long_k_many_phases_sampled(q):
    """M = 16, K = 65536: the activations (2 MB) are staged in about thirty K phases."""
    M, N, K = 16, 2000, 65536
    prob = synthetic.make_qmm(M, N, K, 3, 128, zero_mode="group", seed=77)
    x, packed, scales, zeros = to_dev_problem(prob)
    y = y_to_f64(q.qmm_gemv(x, packed, 3, 128, scales, zeros, 0, out=nan16(M, N)))
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    assert not np.isnan(y).any()
    st = SplitMix64(5)
    cols = np.unique(np.concatenate([(st.next(64) % np.uint64(N)).astype(np.int64), [0, N - 1]]))
    assert rel_err(y[:, cols], oracle_y(prob, cols=cols)) <= REL_TOL
