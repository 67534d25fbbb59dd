"""GPU tests of the pre-permuted weight layouts (qmm_repack) and of the decode
kernel on the fragment-ordered layout (qmm_gemv_tile16), against the oracle.

* qmm_repack must reproduce the oracle's tile16 / interleave4 streams byte for
  byte (integer work: bit-exact).
* qmm_gemv_tile16 must meet the fp16 bound max|y - y_ref| / max|y_ref| <= 2e-3
  against the oracle on the same codes, like qmm_gemv on the canonical stream.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import SplitMix64
from tests.helpers import REL_TOL, oracle_y, rel_err, to_dev_problem, y_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    return q


@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("N,K", [(16, 64), (37, 128), (300, 1024), (5, 4096)])
def test_repack_tile16_bit_exact(q, bits, N, K):
    st = SplitMix64(bits * 13 + N)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    packed = q.qmm_pack(torch.from_numpy(codes).cuda(), bits)
    out = q.qmm_repack(packed, K, bits, "tile16")
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), oracle.tile16(codes, bits))


@pytest.mark.parametrize("N,K", [(1, 8), (33, 64), (300, 4096)])
def test_repack_interleave4_bit_exact(q, N, K):
    st = SplitMix64(N + K)
    codes = st.uniform_bits(N * K, 4).reshape(N, K)
    packed = q.qmm_pack(torch.from_numpy(codes).cuda(), 4)
    out = q.qmm_repack(packed, K, 4, "interleave4")
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().reshape(N, K // 2), oracle.interleave4(codes))


def test_repack_rejects_unsupported_sizes(q):
    packed = torch.zeros((4, 48), dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QmmError):
        q.qmm_repack(packed, 96, 4, "tile16")          # K % 64
    with pytest.raises(q.QmmError):
        q.qmm_repack(torch.zeros((4, 36), dtype=torch.uint8, device="cuda"), 96, 3, "interleave4")


def _gemv_tile16(q, prob, out_dtype=torch.float16):
    x, packed, scales, zeros = to_dev_problem(prob)
    tiled = q.qmm_repack(packed, prob.K, prob.bits, "tile16")
    y = torch.full((prob.M, prob.N), float("nan"), dtype=out_dtype, device="cuda")
    q.qmm_gemv_tile16(x, tiled, prob.N, prob.bits, prob.group, scales, zeros, prob.zero_const, out=y)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    yy = y_to_f64(y)
    assert not np.isnan(yy).any(), "unwritten outputs"
    return yy


CASES = []
for _b in range(1, 9):
    for (M, N, K, G, zm) in [(1, 4096, 4096, 128, "half"), (3, 37, 1024, 128, "group"),
                             (9, 300, 512, 64, "const8"), (16, 5000, 1024, 64, "group"),
                             (2, 4865, 2048, 128, "none"), (1, 8, 512, 64, "half")]:
        CASES.append((_b, M, N, K, G, zm))


@pytest.mark.parametrize("bits,M,N,K,G,zm", CASES)
def test_gemv_tile16_parity(q, bits, M, N, K, G, zm):
    prob = synthetic.make_qmm(M, N, K, bits, G, zero_mode=zm, seed=bits * 37 + M)
    assert rel_err(_gemv_tile16(q, prob), oracle_y(prob)) <= REL_TOL


@pytest.mark.parametrize("bits", [3, 6])
def test_gemv_tile16_skinny_config_sampled(q, bits):
    # M = 16, K = 4096, N = 14336, group 64, stored zeros: several row blocks per CTA
    prob = synthetic.skinny(16, 14336, bits)
    y = _gemv_tile16(q, prob)
    cols = np.unique(np.concatenate([np.arange(0, 14336, 53), np.arange(14320, 14336)]))
    assert rel_err(y[:, cols], oracle_y(prob, cols=cols)) <= REL_TOL


def test_gemv_tile16_bf16_output_and_adversarial_activations(q):
    prob = synthetic.make_qmm(4, 1000, 2048, 5, 128, zero_mode="group", x_law="shift8", seed=3)
    y = _gemv_tile16(q, prob, torch.bfloat16)
    ref = oracle_y(prob)
    assert np.all(np.abs(y - ref) <= REL_TOL * np.max(np.abs(ref)) + np.abs(ref) * 2.0 ** -8)


def test_gemv_tile16_rejects_shapes_outside_the_decode_kernel(q):
    prob = synthetic.make_qmm(1, 64, 256, 4, 32, zero_mode="half", seed=1)   # group 32
    x, packed, scales, _ = to_dev_problem(prob)
    tiled = q.qmm_repack(packed, 256, 4, "tile16")
    with pytest.raises(q.QmmError):
        q.qmm_gemv_tile16(x, tiled, 64, 4, 32, scales, None, 8)
