"""Test helpers: exact torch -> float64 conversion for the oracle, and the
parity tolerances.

Tolerances (GPU result vs the fp64 oracle on the same inputs):
  bf16 K/V (fp32 accumulation): max |dO| <= 2e-2 and mean |dO| <= 2e-3
  fp32 inputs:                  max |dO| <= 1e-5
  LSE (either):                 |dLSE| <= 1e-3
  -inf LSE (empty history) and O = 0 must match exactly.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_BF16_MAX = 2e-2
TOL_BF16_MEAN = 2e-3
TOL_FP32_MAX = 1e-5
TOL_LSE = 1e-3


def to_f64(t: torch.Tensor) -> np.ndarray:
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(t.view(torch.uint16).numpy())
    if t.dtype in (torch.float32, torch.float64):
        return t.numpy().astype(np.float64)
    if t.dtype in (torch.int32, torch.int64):
        return t.numpy()
    raise TypeError(t.dtype)


def assert_parity(O, LSE, O_ref, LSE_ref, kv_dtype, label=""):
    O = np.asarray(O, np.float64)
    O_ref = np.asarray(O_ref, np.float64)
    assert O.shape == O_ref.shape, (O.shape, O_ref.shape)
    assert np.all(np.isfinite(O)), f"{label}: non-finite output"
    err = np.abs(O - O_ref)
    if kv_dtype == torch.bfloat16:
        assert err.max() <= TOL_BF16_MAX, f"{label}: max |dO| {err.max():.3e}"
        assert err.mean() <= TOL_BF16_MEAN, f"{label}: mean |dO| {err.mean():.3e}"
    else:
        assert err.max() <= TOL_FP32_MAX, f"{label}: max |dO| {err.max():.3e}"
    if LSE is not None:
        LSE = np.asarray(LSE, np.float64)
        LSE_ref = np.asarray(LSE_ref, np.float64)
        inf_ref = np.isneginf(LSE_ref)
        assert np.array_equal(np.isneginf(LSE), inf_ref), f"{label}: -inf pattern differs"
        if (~inf_ref).any():
            d = np.abs(LSE[~inf_ref] - LSE_ref[~inf_ref])
            assert d.max() <= TOL_LSE, f"{label}: max |dLSE| {d.max():.3e}"
        assert np.all(O[inf_ref] == 0), f"{label}: empty rows must be exactly 0"
