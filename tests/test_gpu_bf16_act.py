"""bf16 activations in qmm_gemv / qmm_gemv_tile16 (the decode kernel converts
them to fp16 while staging: exact for magnitudes in [2^-14, 65504]).  Parity
against the oracle on the same bf16 inputs, at the decode sweep's full size,
the skinny batched decode shape (sampled), bf16 outputs and a shifted
activation law; shapes the decode kernel does not take reject bf16."""
import numpy as np
import pytest
import torch

import synthetic
from tests.helpers import REL_TOL, oracle_y, rel_err, to_dev_problem, y_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    return q


def _run(q, prob, out_dtype=torch.float16, tile16=False):
    x, packed, scales, zeros = to_dev_problem(prob)
    assert x.dtype == torch.bfloat16
    if tile16:
        tiled = q.qmm_repack(packed, prob.K, prob.bits, "tile16")
        y = q.qmm_gemv_tile16(x, tiled, prob.N, prob.bits, prob.group, scales, zeros, prob.zero_const,
                              out_dtype=out_dtype)
    else:
        y = q.qmm_gemv(x, packed, prob.bits, prob.group, scales, zeros, prob.zero_const, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    return y_to_f64(y)


@pytest.mark.parametrize("bits", range(1, 9))
def test_bf16_activations_decode_sweep(q, bits):
    prob = synthetic.make_qmm(1, 4096, 4096, bits, 128, zero_mode="half", x_dtype="bf16", seed=bits)
    assert rel_err(_run(q, prob), oracle_y(prob)) <= REL_TOL


@pytest.mark.parametrize("tile16", [False, True])
def test_bf16_activations_skinny_shape_sampled(q, tile16):
    prob = synthetic.make_qmm(16, 14336, 4096, 6, 64, zero_mode="group", x_dtype="bf16", seed=16)
    y = _run(q, prob, tile16=tile16)
    cols = np.unique(np.concatenate([np.arange(0, 14336, 61), np.arange(14320, 14336)]))
    assert rel_err(y[:, cols], oracle_y(prob, cols=cols)) <= REL_TOL


@pytest.mark.parametrize("M", [3, 9])
def test_bf16_activations_shifted_law_bf16_out(q, M):
    prob = synthetic.make_qmm(M, 1000, 2048, 4, 128, zero_mode="group", x_dtype="bf16", x_law="shift8",
                              seed=M)
    y = _run(q, prob, out_dtype=torch.bfloat16)
    ref = oracle_y(prob)
    assert np.all(np.abs(y - ref) <= REL_TOL * np.max(np.abs(ref)) + np.abs(ref) * 2.0 ** -8)


def test_bf16_activations_outside_the_decode_kernel_are_rejected(q):
    prob = synthetic.make_qmm(2, 64, 256, 4, 32, zero_mode="half", x_dtype="bf16", seed=2)   # group 32
    x, packed, scales, zeros = to_dev_problem(prob)
    with pytest.raises(q.QmmError):
        q.qmm_gemv(x, packed, 4, 32, scales, zeros, prob.zero_const)
