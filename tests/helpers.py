"""Shared helpers of the GPU parity tests: moving seeded inputs to the
device and the comparison rules.

Tolerances (stated with the workloads): indices, block lists and cache
contents bit-exact; float32 outputs |delta| <= 1e-4; bf16 outputs
|delta| <= 2e-2 * max|reference|.
"""

import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16_REL = 2e-2


def to_dev(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(device="cuda", dtype=dtype).contiguous()


def assert_close_rel(got, want, rel=TOL_BF16_REL, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = float(np.max(np.abs(want))) or 1.0
    err = float(np.max(np.abs(got - want)))
    assert err <= rel * scale, f"{what}: max|delta| {err:.3e} > {rel} * {scale:.3e}"
    return err / scale


def assert_close_abs(got, want, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.max(np.abs(got - want)))
    assert err <= tol, f"{what}: max|delta| {err:.3e} > {tol}"
    return err
