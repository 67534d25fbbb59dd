"""Shared helpers for the GPU parity tests (host-side marshalling only)."""
import numpy as np
import torch

import oracle

# The benchmark spec's tolerance for fp16 outputs: max|y - y_ref| / max|y_ref|.
REL_TOL = 2e-3


def rel_err(y: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(y.astype(np.float64) - ref))) / (den if den > 0 else 1.0)


def to_dev_problem(prob, device="cuda"):
    """Device tensors for a synthetic.QmmProblem (codes are packed by the
    library's own qmm_pack)."""
    import bit_weight_quantized_gb300 as q
    codes = torch.from_numpy(prob.codes).to(device)
    packed = q.qmm_pack(codes, prob.bits)
    scales = torch.from_numpy(prob.scales.view(np.int16)).view(torch.float16).to(device)
    zeros = None if prob.zeros is None else torch.from_numpy(prob.zeros).to(device)
    if prob.x_dtype == "f16":
        x = torch.from_numpy(prob.x.view(np.int16)).view(torch.float16).to(device)
    else:
        x = torch.from_numpy(prob.x.view(np.int16)).view(torch.bfloat16).to(device)
    return x, packed, scales, zeros


def y_to_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def oracle_y(prob, rows=None, cols=None):
    return oracle.solve_qmm(prob, rows=rows, cols=cols)
