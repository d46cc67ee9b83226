"""Tolerances of the GPU-vs-oracle comparisons (test infrastructure).

fp32 workloads: max |gpu - oracle| <= 1e-4.
bf16 workloads: max |gpu - oracle| <= 2e-2 AND max |gpu - oracle| / max |oracle| <= 1e-2.
"""
import numpy as np


def to64(x):
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def errors(got, ref):
    got, ref = to64(got), to64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    return err, scale


def assert_parity(got, ref, dtype: str, what: str):
    err, scale = errors(got, ref)
    if dtype == "f32":
        assert err <= 1e-4, f"{what}: max abs err {err:.3e} > 1e-4"
    else:
        assert err <= 2e-2, f"{what}: max abs err {err:.3e} > 2e-2"
        assert err <= 1e-2 * scale, f"{what}: relative err {err / max(scale, 1e-300):.3e} > 1e-2 (max |ref| {scale:.3e})"
    return err, scale
