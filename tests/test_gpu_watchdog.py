"""Failure detection on the GPU without a fault: the bounded wait every kernel
uses gives up on a wait that never completes, reports QMM_ERR_TIMEOUT through
the device status word, and leaves the context usable."""
import pytest
import torch

import synthetic
from tests.helpers import REL_TOL, oracle_y, rel_err, to_dev_problem, y_to_f64

pytestmark = pytest.mark.gpu

QMM_ERR_TIMEOUT = 8


@pytest.fixture(scope="module")
def q():
    import bit_weight_quantized_gb300 as q
    q.load()
    return q


def test_watchdog_times_out_and_context_survives(q):
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    q.qmm_watchdog_selftest()
    assert q.qmm_device_status() == QMM_ERR_TIMEOUT
    assert q.qmm_device_status() == 0          # reading clears it
    prob = synthetic.parity_ref()
    x, packed, scales, zeros = to_dev_problem(prob)
    y = q.qmm_gemv(x, packed, prob.bits, prob.group, scales, zeros, prob.zero_const)
    torch.cuda.synchronize()
    assert q.qmm_device_status() == 0
    assert rel_err(y_to_f64(y), oracle_y(prob)) <= REL_TOL
