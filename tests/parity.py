"""Comparison metric shared by the GPU parity tests.

err = max_i |g_i - r_i| / max(|r_i|, rms(r)): a relative error with a floor at the RMS of
the reference, so that outputs near zero are judged against the tensor's own scale. Bounds:
2e-3 for bf16 inputs and 1e-5 for fp32 inputs (fp32 arithmetic in both cases). A bf16
output adds its own rounding, at most half a bf16 ulp, which is allowed on top of the bound.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3}


def as_f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rel_err(got, ref) -> float:
    g, r = as_f64(got), as_f64(ref)
    if r.size == 0:
        return 0.0
    assert np.all(np.isfinite(g)), "non-finite values in the GPU output"
    scale = max(float(np.sqrt(np.mean(r * r))), 1e-30)
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), scale)))


def half_ulp_bf16(x):
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 1e-38)))
    return np.exp2(e - 8)


def bf16_out_excess(got, ref, tol) -> float:
    """Largest excess of |g - r| over tol*max(|r|, rms) + half_ulp_bf16(max(|r|, |g|)), in
    units of the allowance; <= 1 passes."""
    g, r = as_f64(got), as_f64(ref)
    assert np.all(np.isfinite(g)), "non-finite values in the GPU output"
    scale = max(float(np.sqrt(np.mean(r * r))), 1e-30)
    allow = tol * np.maximum(np.abs(r), scale) + half_ulp_bf16(np.maximum(np.abs(r), np.abs(g)))
    return float(np.max(np.abs(g - r) / allow))


def _log(kind, value, tol, what):
    path = os.environ.get("SELSCAN_PARITY_LOG")
    if path:
        test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        with open(path, "a") as f:
            f.write(json.dumps({"test": test, "what": what, kind: value, "tol": tol}) + "\n")


def assert_close(got, ref, tol, what=""):
    if isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16:
        ex = bf16_out_excess(got, ref, tol)
        _log("bf16_excess", ex, tol, what)
        assert ex <= 1.0, f"{what}: bf16 output off by {ex:.3f}x the allowance (tol {tol:g} + 1/2 ulp)"
    else:
        e = rel_err(got, ref)
        _log("rel_err", e, tol, what)
        assert e <= tol, f"{what}: max relative error {e:.3e} > {tol:g}"
