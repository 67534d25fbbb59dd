"""GPU parity: qmm_pack/qmm_unpack (bit exact) and qmm_gemv (within the
2e-3 parity bound) against the CPU oracle, through the C ABI."""
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


def _status_ok(q):
    assert q.qmm_device_status() == 0


# ---- pack / unpack ------------------------------------------------------------------
@pytest.mark.parametrize("bits", range(1, 9))
@pytest.mark.parametrize("N,K", [(1, 8), (37, 1000), (5, 4096), (300, 96)])
def test_pack_bit_exact(q, bits, N, K):
    if (K * bits) % 8:
        pytest.skip("K*bits not byte aligned")
    st = SplitMix64(bits * 7919 + N * K)
    codes = st.uniform_bits(N * K, bits).reshape(N, K)
    ref, _ = oracle.pack(codes, bits)
    packed = q.qmm_pack(torch.from_numpy(codes).cuda(), bits)
    np.testing.assert_array_equal(packed.cpu().numpy(), ref)
    back = q.qmm_unpack(packed, K, bits)
    np.testing.assert_array_equal(back.cpu().numpy(), codes)
    _status_ok(q)


def test_pack_counts_out_of_range(q):
    codes = np.array([[0, 5, 8, 15, 16, 255, 3, 9]] * 3, np.uint8)
    ref, bad = oracle.pack(codes, 3)
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    packed = q.qmm_pack(torch.from_numpy(codes).cuda(), 3, bad_count=cnt)
    np.testing.assert_array_equal(packed.cpu().numpy(), ref)
    assert int(cnt.item()) == bad == 15


# ---- skinny matmul --------------------------------------------------------------------
def run_gemv(q, prob, out_dtype=torch.float16):
    x, packed, scales, zeros = to_dev_problem(prob)
    y = torch.full((prob.M, prob.N), float("nan"), dtype=out_dtype, device="cuda")
    q.qmm_gemv(x, packed, prob.bits, prob.group, scales, zeros, prob.zero_const, out=y)
    torch.cuda.synchronize()
    return y


CASES = []
for bits in range(1, 9):
    for (M, N, K, G, zm) in [(1, 37, 640, 128, "half"), (3, 300, 256, 64, "group"),
                             (9, 130, 512, 32, "group"), (16, 64, 1024, 128, "group"),
                             (8, 1, 384, 128, "const8")]:
        CASES.append((bits, M, N, K, G, zm))


@pytest.mark.parametrize("bits,M,N,K,G,zm", CASES)
def test_gemv_parity_small(q, bits, M, N, K, G, zm):
    prob = synthetic.make_qmm(M, N, K, bits, G, zero_mode=zm, seed=bits * 100 + M)
    y = run_gemv(q, prob)
    yy = y_to_f64(y)
    assert not np.isnan(yy).any(), "unwritten outputs"
    ref = oracle_y(prob)
    assert rel_err(yy, ref) <= REL_TOL
    _status_ok(q)


@pytest.mark.parametrize("bits", [1, 3, 5, 6])
def test_gemv_unaligned_rows_use_plain_copies(q, bits):
    # K*bits/8 not a multiple of 16: the producer falls back to 4-byte copies
    prob = synthetic.make_qmm(2, 45, 96, bits, 32, zero_mode="group", seed=5)
    assert (96 * bits // 8) % 16 != 0
    y = run_gemv(q, prob)
    assert rel_err(y_to_f64(y), oracle_y(prob)) <= REL_TOL
    _status_ok(q)


def test_gemv_unaligned_base_uses_plain_copies(q):
    prob = synthetic.make_qmm(3, 50, 256, 4, 128, zero_mode="const8", seed=6)
    x, packed, scales, zeros = to_dev_problem(prob)
    buf = torch.zeros(packed.numel() + 16, dtype=torch.uint8, device="cuda")
    shifted = buf[4:4 + packed.numel()].view(packed.shape)
    shifted.copy_(packed)
    y = q.qmm_gemv(x, shifted, 4, 128, scales, None, 8)
    assert rel_err(y_to_f64(y), oracle_y(prob)) <= REL_TOL
    _status_ok(q)


def test_gemv_bf16_output(q):
    prob = synthetic.make_qmm(4, 200, 512, 5, 64, zero_mode="group", seed=9)
    y = run_gemv(q, prob, out_dtype=torch.bfloat16)
    ref = oracle_y(prob)
    # bf16 rounding of the output itself: half an ulp is 2^-8 of the element
    assert np.all(np.abs(y_to_f64(y) - ref) <= REL_TOL * np.max(np.abs(ref)) + np.abs(ref) * 2.0 ** -8)


def test_gemv_deterministic(q):
    prob = synthetic.make_qmm(5, 777, 2048, 3, 64, zero_mode="group", seed=2)
    x, packed, scales, zeros = to_dev_problem(prob)
    outs = []
    for _ in range(3):
        y = q.qmm_gemv(x, packed, 3, 64, scales, zeros)
        outs.append(y.cpu().numpy().view(np.uint16).copy())
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_parity_ref_workload(q):
    prob = synthetic.parity_ref()
    y = run_gemv(q, prob)
    assert rel_err(y_to_f64(y), oracle_y(prob)) <= REL_TOL


@pytest.mark.parametrize("bits", range(1, 9))
def test_decode_sweep_full_size(q, bits):
    prob = synthetic.decode_sweep(bits)
    y = run_gemv(q, prob)
    assert rel_err(y_to_f64(y), oracle_y(prob)) <= REL_TOL
    _status_ok(q)


@pytest.mark.parametrize("M", [2, 4, 8, 16])
@pytest.mark.parametrize("N", [11008, 14336])
@pytest.mark.parametrize("bits", [3, 4, 5, 6])
def test_skinny_full_size_sampled(q, M, N, bits):
    prob = synthetic.skinny(M, N, bits)
    y = y_to_f64(run_gemv(q, prob))
    assert not np.isnan(y).any()
    st = SplitMix64(N + bits)
    cols = np.unique((st.next(384) % np.uint64(N)).astype(np.int64))
    cols = np.concatenate([cols, [0, N - 1]])
    ref = oracle_y(prob, cols=cols)
    assert rel_err(y[:, cols], ref) <= REL_TOL
    _status_ok(q)


# ---- row blocks: a CTA with more than 128 rows (N > 152 * 128) takes them in
# blocks; with long K the activations are also staged in K phases, per block ----
@pytest.mark.parametrize("M,N,K,bits,G,zm", [
    (1, 20480, 512, 5, 64, "group"),
    (3, 20000, 1024, 4, 128, "const8"),
    (16, 19800, 8192, 3, 128, "half"),
])
def test_gemv_row_blocks_sampled(q, M, N, K, bits, G, zm):
    prob = synthetic.make_qmm(M, N, K, bits, G, zero_mode=zm, seed=N + K)
    y = y_to_f64(run_gemv(q, prob))
    assert not np.isnan(y).any()
    st = SplitMix64(N * 3 + K)
    cols = (st.next(384) % np.uint64(N)).astype(np.int64)
    # all rows of the first CTA (both of its blocks) and the last columns
    cols = np.unique(np.concatenate([cols, np.arange(0, 140), [N - 2, N - 1]]))
    ref = oracle_y(prob, cols=cols)
    assert rel_err(y[:, cols], ref) <= REL_TOL
    _status_ok(q)
