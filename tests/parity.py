"""Helpers shared by the GPU parity tests: tolerance, sampling and device transfer.

The tolerance is the one the workloads are specified with:
|gpu - ref| <= 2e-4 + 2e-4 * |ref|, elementwise, ref from the float64 oracle.
"""
import numpy as np

ATOL = 2e-4
RTOL = 2e-4


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if np.any(bad):
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at flat "
                             f"{i}: got {got.reshape(-1)[i]!r} ref {ref.reshape(-1)[i]!r}")
    return float(err.max()) if err.size else 0.0


def sample_indices(shape, count, seed, include_corners=True):
    """Random multi-indices into `shape`, plus every corner (first/last of each dim)."""
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.integers(0, s, count) for s in shape], 1)
    if include_corners:
        corners = np.array(np.meshgrid(*[[0, s - 1] for s in shape], indexing="ij")).reshape(len(shape), -1).T
        idx = np.concatenate([idx, corners], 0)
    return idx


def to_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)
