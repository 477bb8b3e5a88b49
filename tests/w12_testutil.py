"""Shared checks for the GPU parity tests: the GEMM error bound and the argmax near-tie rule.

Tolerances (the GEMM's stated accuracy bound for this path):
  fp32 y:  |y - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1e-6 per element (y_ref in fp64)
  bf16 y:  within one bf16 ulp of the fp64 reference, plus the fp32 bound above
  argmax:  top-1 must equal the fp64 oracle's wherever the oracle's top-1/top-2 gap exceeds
           1e-3 of the row's logit scale (max |y_ref|); closer rows are counted as near-ties.
"""
from __future__ import annotations

import numpy as np
import torch

REL = 2e-3
ABS = 1e-6


def gemm_violations(y_gpu: np.ndarray, y_ref: np.ndarray, absdot: np.ndarray, bf16: bool = False) -> int:
    y = y_gpu.astype(np.float64)
    tol = REL * absdot + ABS
    if bf16:
        a = np.abs(y_ref)
        with np.errstate(divide="ignore"):
            e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
        ulp = np.where(a > 0, np.exp2(e - 7), 0.0)
        tol = tol + ulp
    bad = ~(np.abs(y - y_ref) <= tol)
    return int(np.count_nonzero(bad))


def argmax_check(idx, val, gap, y_ref: np.ndarray, absdot: np.ndarray):
    """Returns (n_rows_checked, n_near_ties, n_wrong, details)."""
    import oracle

    ridx, rval, rgap, scale = oracle.argmax(y_ref)
    checked = near = wrong = 0
    details = []
    for m in range(y_ref.shape[0]):
        if rgap[m] > 1e-3 * scale[m]:
            checked += 1
            ok = int(idx[m]) == int(ridx[m])
            tol = REL * absdot[m, ridx[m]] + ABS
            ok = ok and abs(float(val[m]) - rval[m]) <= tol
            if not ok:
                wrong += 1
                details.append((m, int(idx[m]), int(ridx[m]), float(val[m]), rval[m], rgap[m]))
        else:
            near += 1
    return checked, near, wrong, details


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
