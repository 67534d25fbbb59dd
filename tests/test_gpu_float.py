"""GPU parity of the float-weight decode matmul (qmm_gemv_float) against the
oracle's definition, for float codes of 2 to 8 bits and several splits."""
import numpy as np
import pytest
import torch

import oracle
from synthetic import SplitMix64
from tests.helpers import REL_TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    return q


def run_case(q, e, m, M, N, K, G, seed):
    bits = 1 + e + m
    st = SplitMix64(seed)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    s16 = (0.02 * np.abs(st.normal(N * K // G)) + 1e-3).astype(np.float16).reshape(N, K // G)
    x16 = st.normal(M * K).reshape(M, K).astype(np.float16)
    packed_ref, _ = oracle.pack(codes, bits)
    ref = oracle.qmm_float(x16.astype(np.float64), packed_ref, e, m, G, s16.astype(np.float64), K)
    packed = q.qmm_pack(torch.from_numpy(codes).cuda(), bits)
    x = torch.from_numpy(x16.view(np.int16)).view(torch.float16).cuda()
    s = torch.from_numpy(s16.view(np.int16)).view(torch.float16).cuda()
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    q.qmm_gemv_float(x, packed, e, m, G, s, out=y)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    yv = y.float().cpu().numpy().astype(np.float64)
    assert not np.isnan(yv).any()
    return yv, ref


@pytest.mark.parametrize("e,m", [(1, 0), (1, 1), (2, 1), (1, 2), (2, 2), (3, 2), (2, 3), (3, 3),
                                 (4, 3), (5, 2), (1, 6)])
def test_float_weights_parity(q, e, m):
    y, ref = run_case(q, e, m, M=3, N=130, K=512, G=64, seed=e * 10 + m)
    assert rel_err(y, ref) <= REL_TOL


@pytest.mark.parametrize("M,N,K,G", [(1, 4096, 4096, 128), (16, 300, 1024, 32), (7, 33, 96, 32)])
def test_float6_e3m2_shapes(q, M, N, K, G):
    y, ref = run_case(q, 3, 2, M, N, K, G, seed=M + N)
    assert rel_err(y, ref) <= REL_TOL


@pytest.mark.parametrize("e,m", [(1, 0), (1, 1), (2, 0), (2, 1), (1, 2), (3, 0), (2, 2), (4, 0), (3, 2),
                                 (2, 3), (3, 3), (4, 2), (4, 3), (3, 4), (2, 5)])
@pytest.mark.parametrize("M", [1, 16])
def test_float_decode_shapes(q, e, m, M):
    # float codes of at most 4 exponent bits run on the decode kernel's
    # tensor-core path: the decode sweep shape, group 128
    y, ref = run_case(q, e, m, M, 4096, 4096, 128, seed=e * 100 + m * 10 + M)
    assert rel_err(y, ref) <= REL_TOL


@pytest.mark.parametrize("e,m", [(1, 1), (2, 1), (2, 2), (3, 2), (3, 3), (4, 3)])
def test_float_decode_group64_ragged(q, e, m):
    y, ref = run_case(q, e, m, 9, 333, 1024, 64, seed=e + m)
    assert rel_err(y, ref) <= REL_TOL
