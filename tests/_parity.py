"""Tolerances and comparison helpers for GPU-vs-oracle parity.

Output tolerance (fp32 accumulation of bf16 inputs): max |o_gpu - o_ref| <= 2e-2 * rms(o_ref).
That bound is applied to the fp32 output mode.  When the output is stored as
bf16 the final round-to-nearest-even adds at most half an ulp, 2^-8 |o|, per
element, so the bf16 mode is checked with |o_gpu - o_ref| <= 2e-2 rms(o_ref)
+ 2^-8 |o_ref| element by element.
State tolerance: relative Frobenius error <= 1e-3 for every (sequence, head)
final state and checkpoint.
"""
import numpy as np
import torch

O_TOL = 2e-2
S_TOL = 1e-3
BF16_HALF_ULP = 2.0 ** -8


def _np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def out_error(o_gpu, o_ref) -> float:
    """max |delta| / rms(ref)."""
    g, r = _np(o_gpu), _np(o_ref)
    return float(np.abs(g - r).max() / np.sqrt((r ** 2).mean()))


def check_out(o_gpu, o_ref, dtype, what="o"):
    g, r = _np(o_gpu), _np(o_ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    rms = np.sqrt((r ** 2).mean())
    err = np.abs(g - r)
    if dtype == torch.float32:
        worst = err.max() / rms
        assert worst <= O_TOL, f"{what}: max|d|/rms = {worst:.3e} > {O_TOL}"
        return worst
    bound = O_TOL * rms + BF16_HALF_ULP * np.abs(r)
    ratio = (err / bound).max()
    assert ratio <= 1.0, f"{what}: bf16 bound exceeded by x{ratio:.3f}"
    return err.max() / rms


def state_error(s_gpu, s_ref) -> float:
    """Largest relative Frobenius error over the leading (..., Dk, Dv) slices."""
    g, r = _np(s_gpu), _np(s_ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    g = g.reshape(-1, g.shape[-2] * g.shape[-1])
    r = r.reshape(-1, r.shape[-2] * r.shape[-1])
    num = np.linalg.norm(g - r, axis=1)
    den = np.linalg.norm(r, axis=1)
    rel = np.where(den > 0, num / np.where(den > 0, den, 1), num)
    return float(rel.max())


def check_state(s_gpu, s_ref, what="state"):
    assert np.isfinite(_np(s_gpu)).all(), f"{what}: non-finite"
    e = state_error(s_gpu, s_ref)
    assert e <= S_TOL, f"{what}: rel Frobenius {e:.3e} > {S_TOL}"
    return e
