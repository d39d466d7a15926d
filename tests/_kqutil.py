"""Helpers shared by the parity tests: device placement and the tolerance check."""
import numpy as np


def to_dev(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within_bound(y_gpu, y_ref, B, what=""):
    """|y_gpu - y_ref| <= 1e-3 * B + 1e-5 element by element (B = Sum_k |w_k x_k|)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    tol = 1e-3 * B + 1e-5
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside the bound; first at {idx.tolist()}: "
            f"gpu={y_gpu[tuple(idx[0])]!r} ref={y_ref[tuple(idx[0])]!r} bound={tol[tuple(idx[0])]!r}")
    return float(np.max(err / tol)) if err.size else 0.0
