"""Shared test helpers: tolerance check and small case runners."""
import numpy as np
import torch

# Acceptance: |out - ref| <= ATOL + RTOL*|ref| element-wise, |lse - ref| <= LSE_TOL
ATOL, RTOL, LSE_TOL = 8e-3, 1e-2, 1e-3


def assert_close_attn(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Element-wise acceptance check; returns (max |d out|, max |d lse|, rmse)."""
    o = out_gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(out_gpu, torch.Tensor) else out_gpu
    ls = lse_gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    ref_o = np.asarray(out_ref, np.float64)
    ref_l = np.asarray(lse_ref, np.float64)
    assert o.shape == ref_o.shape, (o.shape, ref_o.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - ref_o)
    bound = ATOL + RTOL * np.abs(ref_o)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of tolerance; first at {tuple(idx)}: "
                             f"gpu={o[tuple(idx)]:.6g} ref={ref_o[tuple(idx)]:.6g}")
    both_inf = np.isneginf(ls) & np.isneginf(ref_l)
    assert (np.isneginf(ls) == np.isneginf(ref_l)).all(), f"{what}: -inf lse mismatch"
    with np.errstate(invalid="ignore"):
        dl = np.abs(np.where(both_inf, 0.0, ls - ref_l))
    assert dl.max(initial=0.0) <= LSE_TOL, f"{what}: lse error {dl.max()}"
    rmse = float(np.sqrt(np.mean((o - ref_o) ** 2)))
    return float(err.max(initial=0.0)), float(dl.max(initial=0.0)), rmse
