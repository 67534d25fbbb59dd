"""Signed b-bit weights on the GPU: qmm_flip_sign equals the oracle's bit flip
byte for byte, and signed codes flipped to offset binary give the signed
matmul through qmm_gemv / qmm_gemm with zero point 2^(b-1)."""
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


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("N,K", [(1, 8), (37, 256), (300, 1000)])
def test_flip_sign_bit_exact(q, bits, N, K):
    if (K * bits) % 8:
        pytest.skip("K*bits not byte aligned")
    st = SplitMix64(bits * 1000 + N)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    ref_packed, _ = oracle.pack(codes, bits)
    dev = q.qmm_pack(torch.from_numpy(codes).cuda(), bits)
    q.qmm_flip_sign(dev, K, bits)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dev.cpu().numpy(), oracle.flip_sign(ref_packed, K, bits))


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("M", [1, 16, 40])
def test_signed_weights_matmul(q, bits, M):
    N, K, G = 300, 1024, 64
    st = SplitMix64(7 * bits + M)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)      # two's-complement signed codes
    s16 = (0.02 * np.abs(st.normal(N * K // G)) + 1e-3).astype(np.float16).reshape(N, K // G)
    x16 = st.normal(M * K).reshape(M, K).astype(np.float16)
    packed_ref, _ = oracle.pack(codes, bits)
    ref = oracle.qmm_signed(x16.astype(np.float64), packed_ref, bits, G, s16.astype(np.float64), K)
    packed = q.qmm_pack(torch.from_numpy(codes).cuda(), bits)
    q.qmm_flip_sign(packed, K, bits)
    x = torch.from_numpy(x16.view(np.int16)).view(torch.float16).cuda()
    s = torch.from_numpy(s16.view(np.int16)).view(torch.float16).cuda()
    if M <= 16:
        y = q.qmm_gemv(x, packed, bits, G, s, None, 1 << (bits - 1))
    elif bits == 4:
        y = q.qmm_gemm(x, packed, bits, G, s, None, 1 << (bits - 1))
    else:
        pytest.skip("the tiled path takes 4-bit weights")
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    assert rel_err(y.float().cpu().numpy().astype(np.float64), ref) <= REL_TOL
