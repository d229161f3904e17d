"""Shared helpers for the parity tests (GPU path vs the CPU oracle)."""
import numpy as np

# tolerance for every GEMV / MoE output element: |gpu - oracle| <= 1e-5 * B + 1e-6,
# with B the sum of |products| that form the element
REL = 1e-5
ABS = 1e-6


def assert_within_bound(got, ref, bound, rel=REL, abs_=ABS, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    lim = rel * bound + abs_
    bad = err > lim
    if bad.any():
        i = np.unravel_index(np.argmax(err / lim), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements exceed the bound; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} err {err[i]:.3e} lim {lim[i]:.3e}")


def to_dev(a, torch, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)
