"""Shared parity helpers: the tolerance and how GPU results are compared with the oracle.

Tolerance (written here once, used by every GPU parity test):
  |O - O_ref|     <= 8e-3 + 1e-2 * |O_ref|   elementwise
  |LSE - LSE_ref| <= 1e-3                    where LSE_ref is finite
  LSE == -inf exactly where LSE_ref == -inf (no valid entry), and then O == 0.
"""

import numpy as np
import torch

O_ATOL, O_RTOL, LSE_ATOL = 8e-3, 1e-2, 1e-3


def to_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().double().numpy()


def parity_report(out, lse, ref_out, ref_lse):
    o = to_np(out)
    l = to_np(lse)
    err = np.abs(o - ref_out)
    excess = err - (O_ATOL + O_RTOL * np.abs(ref_out))
    fin = np.isfinite(ref_lse)
    lerr = np.abs(l[fin] - ref_lse[fin]) if fin.any() else np.zeros(1)
    return {
        "o_max_abs_err": float(err.max()) if err.size else 0.0,
        "o_worst_excess": float(excess.max()) if excess.size else -1.0,
        "lse_max_abs_err": float(lerr.max()) if lerr.size else 0.0,
        "neg_inf_match": bool(np.array_equal(np.isneginf(l), ~fin)),
        "empty_rows_zero": bool(np.all(o[~fin] == 0.0)) if (~fin).any() else True,
        "all_finite": bool(np.isfinite(o).all()),
    }


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    rep = parity_report(out, lse, ref_out, ref_lse)
    assert rep["all_finite"], f"{what}: non-finite outputs {rep}"
    assert rep["neg_inf_match"], f"{what}: -inf LSE pattern differs {rep}"
    assert rep["empty_rows_zero"], f"{what}: empty lists must give O = 0 {rep}"
    assert rep["o_worst_excess"] <= 0.0, f"{what}: O outside tolerance {rep}"
    assert rep["lse_max_abs_err"] <= LSE_ATOL, f"{what}: LSE outside tolerance {rep}"
    return rep
