"""Error measures for GPU-vs-oracle parity.

Normwise relative error of one slice: max|x - y| / max|y| (y = oracle).  A
tensor's error is the maximum over its per-head slices.  Bars (fixed in the
tests that use them): 2e-2 for bf16 / normalised outputs, 1e-2 for states.
"""
import numpy as np

OUT_TOL = 2e-2
STATE_TOL = 1e-2


def normwise_err(x, y, head_axis):
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    assert x.shape == y.shape, (x.shape, y.shape)
    if x.size == 0:
        return 0.0
    xs = np.moveaxis(x, head_axis, 0).reshape(x.shape[head_axis], -1)
    ys = np.moveaxis(y, head_axis, 0).reshape(y.shape[head_axis], -1)
    num = np.max(np.abs(xs - ys), axis=1)
    den = np.maximum(np.max(np.abs(ys), axis=1), 1e-30)
    assert np.all(np.isfinite(xs)), "non-finite GPU values"
    return float(np.max(num / den))


def to64(t):
    return t.detach().to("cpu").double().numpy()
