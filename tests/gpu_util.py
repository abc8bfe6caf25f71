"""Helpers for the GPU parity tests: move seeded inputs to the device and compare with the oracle."""
import numpy as np
import torch

TOL_F32 = 1e-4     # max|diff| <= 1e-4 max|ref| for the float32 path
TOL_BF16 = 5e-3    # max|diff| <= 5e-3 max|ref| for bf16 inputs on the tensor-core path


def dev(x, device="cuda"):
    return None if x is None else x.to(device).contiguous()


def rel_err(got, ref) -> float:
    got = got.detach().double().cpu().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), "non-finite values"
    denom = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (denom if denom > 0 else 1.0))


def assert_close(got, ref, tol, what=""):
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max|diff|/max|ref| = {e:.3e} > {tol:.1e}"
    return e
