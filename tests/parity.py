"""Tolerances of the parity tests (not a test module).

Floating point (the workload statement's bars):
  fp32 outputs and gradients: relative L2 error <= 1e-5;
  bf16 outputs and gradients: relative L2 error <= 1e-2 AND, for every row, the largest
  absolute error is <= 5e-2 of that row's largest |reference| value.
Integer (int8 accumulators): bit-exact.
"""
import numpy as np

F32_REL_L2 = 1e-5
BF16_REL_L2 = 1e-2
BF16_ROW_MAX = 5e-2


def to64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def row_max_rel(got, ref):
    got = np.atleast_2d(np.asarray(got, np.float64))
    ref = np.atleast_2d(np.asarray(ref, np.float64))
    err = np.abs(got - ref).max(axis=1)
    scale = np.abs(ref).max(axis=1)
    scale = np.where(scale > 0, scale, 1.0)
    return float((err / scale).max())


def assert_close(got, ref, dtype, what=""):
    got = to64(got) if hasattr(got, "detach") else np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    e = rel_l2(got, ref)
    if dtype == "f32":
        assert e <= F32_REL_L2, f"{what}: rel L2 {e:.3e} > {F32_REL_L2}"
    else:
        m = row_max_rel(got, ref)
        assert e <= BF16_REL_L2 and m <= BF16_ROW_MAX, f"{what}: rel L2 {e:.3e}, row max-abs {m:.3e}"
    return e
