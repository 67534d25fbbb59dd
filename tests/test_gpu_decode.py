"""GPU parity of qmm_gemv's two kernels on the shapes the staged decode kernel
takes (1 <= M <= 16, groups of 64 or 128, K a multiple of 512), against the
CPU oracle through the C ABI: the staged decode kernel (the default route for
these shapes, checked with qmm_gemv_route) and the skinny kernel (forced with
qmm_set_gemv_kernel)."""
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


@pytest.fixture(params=["auto", "skinny"])
def kernel(q, request):
    q.qmm_set_gemv_kernel(request.param)
    try:
        yield request.param
    finally:
        q.qmm_set_gemv_kernel("auto")


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _route(q, prob):
    return q.qmm_gemv_route(prob.M, prob.N, prob.K, prob.bits, prob.group, prob.zeros is not None)


def _run(q, prob, out_dtype=torch.float16):
    x, packed, scales, zeros = to_dev_problem(prob)
    y = torch.full((prob.M, prob.N), float("nan"), dtype=out_dtype, device="cuda")
    q.qmm_gemv(x, packed, prob.bits, prob.group, scales, zeros, prob.zero_const, out=y)
    torch.cuda.synchronize()
    yy = y_to_f64(y)
    assert not np.isnan(yy).any(), "unwritten outputs"
    return yy


CASES = []
for bits in range(1, 9):
    for (M, N, K, G, zm) in [(1, 37, 512, 64, "group"), (3, 300, 1024, 128, "half"),
                             (8, 4000, 512, 64, "const8"), (5, 1, 2048, 128, "none"),
                             (2, 153, 4096, 64, "group"), (7, 4096, 1024, 128, "group"),
                             (9, 500, 2048, 128, "group"), (16, 333, 1536, 64, "half"),
                             (12, 5000, 512, 64, "group")]:
        CASES.append((bits, M, N, K, G, zm))


@pytest.mark.parametrize("bits,M,N,K,G,zm", CASES)
def test_decode_shapes_parity(q, kernel, bits, M, N, K, G, zm):
    prob = synthetic.make_qmm(M, N, K, bits, G, zero_mode=zm, seed=bits * 31 + M)
    assert _route(q, prob) == ("decode" if kernel == "auto" else "skinny")
    assert rel_err(_run(q, prob), oracle_y(prob)) <= REL_TOL
    assert q.qmm_device_status() == 0


@pytest.mark.parametrize("bits", [1, 4, 7, 8])
@pytest.mark.parametrize("M", [2, 13])
def test_decode_several_row_blocks_per_cta(q, kernel, bits, M):
    # 32 x SMs + 1 columns: some CTAs own 33 rows, i.e. two row blocks
    N = 32 * _sms() + 1
    prob = synthetic.make_qmm(M, N, 512, bits, 64, zero_mode="group", seed=bits)
    assert rel_err(_run(q, prob), oracle_y(prob)) <= REL_TOL


@pytest.mark.parametrize("bits", [3, 4])
def test_group_32_takes_the_skinny_kernel(q, bits):
    # a 64-code block holds two groups of 32: the staged kernel does not take it
    prob = synthetic.make_qmm(1, 700, 1024, bits, 32, zero_mode="half", seed=bits)
    assert _route(q, prob) == "skinny"
    assert rel_err(_run(q, prob), oracle_y(prob)) <= REL_TOL


@pytest.mark.parametrize("bits", [2, 4, 5, 8])
def test_decode_bf16_output(q, kernel, bits):
    prob = synthetic.make_qmm(4, 200, 1024, bits, 128, zero_mode="group", seed=9)
    y = _run(q, prob, out_dtype=torch.bfloat16)
    ref = oracle_y(prob)
    # bf16 rounding of the output itself: half an ulp is 2^-8 of the element
    assert np.all(np.abs(y - ref) <= REL_TOL * np.max(np.abs(ref)) + np.abs(ref) * 2.0 ** -8)


def test_decode_deterministic(q):
    prob = synthetic.make_qmm(6, 3000, 4096, 5, 64, zero_mode="group", seed=4)
    x, packed, scales, zeros = to_dev_problem(prob)
    outs = [q.qmm_gemv(x, packed, 5, 64, scales, zeros).cpu().numpy().view(np.uint16).copy()
            for _ in range(3)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_decode_back_to_back_calls(q):
    # consecutive calls overlap under programmatic dependent launch: the second
    # call's activations are the first call's output
    p1 = synthetic.make_qmm(1, 1024, 1024, 4, 128, zero_mode="half", seed=11)
    x, packed, scales, _ = to_dev_problem(p1)
    p2 = synthetic.make_qmm(1, 2048, 1024, 3, 64, zero_mode="group", seed=12)
    _, packed2, scales2, zeros2 = to_dev_problem(p2)
    y1 = q.qmm_gemv(x, packed, 4, 128, scales, None, 8)
    y2 = q.qmm_gemv(y1, packed2, 3, 64, scales2, zeros2)
    torch.cuda.synchronize()
    p2.x = y1.cpu().numpy().astype(np.float16).reshape(1, 1024)
    assert rel_err(y_to_f64(y2), oracle_y(p2)) <= REL_TOL


@pytest.mark.parametrize("bits", [4, 8])
def test_decode_shape_with_unaligned_packed_base(q, bits):
    # a packed base that is 4- but not 16-byte aligned goes to the skinny kernel
    prob = synthetic.make_qmm(2, 300, 1024, bits, 128, zero_mode="half", seed=bits)
    x, packed, scales, _ = to_dev_problem(prob)
    buf = torch.zeros(packed.numel() + 16, dtype=torch.uint8, device="cuda")
    shifted = buf[4:4 + packed.numel()].view(packed.shape)
    shifted.copy_(packed)
    y = q.qmm_gemv(x, shifted, bits, 128, scales, None, prob.zero_const)
    assert rel_err(y_to_f64(y), oracle_y(prob)) <= REL_TOL
    assert q.qmm_device_status() == 0
