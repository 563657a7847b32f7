"""Comparison rules for the CUDA path against the fp64 oracle.

* States and fp32 outputs: per block (one state, or one (sequence, head)
  output stream) rel = max|x - x_ref| / max|x_ref| <= 1e-4.
* bf16 outputs: one bf16 ulp is ~4e-3 relative, so a bf16 value passes when
  it is the round-to-nearest-even of the oracle's value, or the other
  neighbour when the oracle's value lies within 1e-4 * max|x_ref| of the
  rounding midpoint between the two.
* Indices: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = 1e-4


def to64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rel_err(x, ref) -> float:
    x, ref = to64(x), to64(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    m = np.max(np.abs(ref)) if ref.size else 0.0
    d = np.max(np.abs(x - ref)) if ref.size else 0.0
    if m == 0.0:
        return float(d)
    return float(d / m)


def assert_close(x, ref, what: str, tol: float = TOL) -> float:
    e = rel_err(x, ref)
    assert np.all(np.isfinite(to64(x))), f"{what}: non-finite values"
    assert e <= tol, f"{what}: rel err {e:.3e} > {tol:.0e}"
    return e


def _bf16_half_ulp(a: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |a| (8 significant bits)."""
    mag = np.abs(a)
    _, e = np.frexp(np.where(mag > 0, mag, 1.0))
    ulp = np.ldexp(1.0, e - 8)
    return np.where(mag > 0, 0.5 * ulp, np.ldexp(1.0, -133))


def assert_bf16_rounding(x_bf16: torch.Tensor, ref, what: str, tol: float = TOL) -> None:
    assert x_bf16.dtype == torch.bfloat16
    g = to64(x_bf16)
    r = to64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return
    M = np.max(np.abs(r))
    allowed = _bf16_half_ulp(np.maximum(np.abs(g), np.abs(r))) + tol * M
    bad = np.abs(g - r) > allowed
    assert not bad.any(), (f"{what}: {int(bad.sum())} bf16 values are neither the rounding of the oracle nor "
                           f"its neighbour within the midpoint tolerance; worst |diff|={np.max(np.abs(g - r)):.3e}")
    # and the bulk must be exactly the correctly rounded value
    exact = torch.from_numpy(r).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    frac = float(np.mean(g == exact))
    assert frac > 0.98, f"{what}: only {frac:.4f} of bf16 values equal RNE(oracle)"


def check_output(o_gpu: torch.Tensor, o_ref, what: str) -> None:
    if o_gpu.dtype == torch.bfloat16:
        assert_bf16_rounding(o_gpu, o_ref, what)
    else:
        assert_close(o_gpu, o_ref, what)
