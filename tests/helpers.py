"""Shared test helpers: move numpy inputs to the GPU, compare with the oracle."""
import numpy as np

import oracle


def to_dev(a, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def assert_within_bound(y_gpu, y_ref, absdot, what=""):
    """Element-wise |y - y_ref| <= 2^-9 |y_ref| + 1e-4 sum_k |x W^| ; returns max err/bound."""
    y = np.asarray(y_gpu).astype(np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    bound = oracle.tolerance(y_ref, absdot)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of bound; first at "
                             f"{tuple(i)}: gpu {y[tuple(i)]!r} ref {y_ref[tuple(i)]!r} bound {bound[tuple(i)]!r}")
    return float((err / np.maximum(bound, 1e-300)).max())
