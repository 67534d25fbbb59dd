"""Shared helpers for the GPU parity tests (host-side marshalling only)."""
import numpy as np
import torch

import oracle

# The parity bound for fp16 outputs: max|y - y_ref| / max|y_ref|.
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


def weight_rounding_sigma(prob, u, rows=None, cols=None):
    """Standard deviation of the error that rounding every dequantized weight
    w = (q - z) * s to the tensor-core operand type adds to y[m][n]: each
    rounding (RNE) moves w by at most u |w| (u = 2^-8 for bf16), taken as
    uniform and independent, so the sum's error has standard deviation at
    most u / sqrt(3) * sqrt(sum_k (x[m][k] w[n][k])^2).  Host-side tolerance
    arithmetic from the problem's own fields (the expected values come from
    the oracle)."""
    x = prob.x_f64()
    codes = prob.codes.astype(np.float64)
    s = prob.scales.astype(np.float64)
    z = (np.full(s.shape, float(prob.zero_const)) if prob.zeros is None
         else prob.zeros.astype(np.float64))
    if rows is not None:
        x = x[rows]
    if cols is not None:
        codes, s, z = codes[cols], s[cols], z[cols]
    w = (codes - np.repeat(z, prob.group, axis=1)) * np.repeat(s, prob.group, axis=1)
    return u / np.sqrt(3.0) * np.sqrt((x * x) @ (w * w).T)
