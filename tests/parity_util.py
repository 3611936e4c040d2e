"""Shared helpers for the GPU parity tests: run the CUDA path, compare with the oracle.

Tolerances (per element, after widening the GPU output to fp64):
  bf16 O:  |ΔO| <= 1e-2 + 1e-2·|O_ref|
  f16  O:  |ΔO| <= 4e-3
  LSE:     |ΔLSE| <= 1e-3
"""

import numpy as np
import torch

BF16_ATOL, BF16_RTOL = 1e-2, 1e-2
F16_ATOL = 4e-3
LSE_ATOL = 1e-3


def o_within(o_gpu, o_ref, dtype: str):
    o = np.asarray(o_gpu, dtype=np.float64)
    err = np.abs(o - o_ref)
    if dtype == "bf16":
        bound = BF16_ATOL + BF16_RTOL * np.abs(o_ref)
    else:
        bound = np.full_like(o_ref, F16_ATOL)
    return err, bound


def assert_parity(o_gpu, lse_gpu, o_ref, lse_ref, dtype: str, what: str = ""):
    o = o_gpu.float().cpu().numpy() if isinstance(o_gpu, torch.Tensor) else o_gpu
    lse = lse_gpu.cpu().numpy() if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    assert np.isfinite(lse).all(), f"{what}: non-finite LSE"
    err, bound = o_within(o, o_ref, dtype)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} O elements out of tolerance; worst at {idx}: "
                             f"gpu={o[idx]:.6f} ref={o_ref[idx]:.6f} max|dO|={err.max():.3e}")
    dl = np.abs(lse.astype(np.float64) - lse_ref)
    if dl.max() > LSE_ATOL:
        idx = np.unravel_index(np.argmax(dl), dl.shape)
        raise AssertionError(f"{what}: max|dLSE|={dl.max():.3e} at {idx} "
                             f"(gpu={lse[idx]:.6f} ref={lse_ref[idx]:.6f})")
    return err.max(), dl.max()
