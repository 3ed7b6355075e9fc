"""Oracle of the split-product second moment and covariance.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this module; the library's product path
never imports it.  It shares no code with the CUDA path.

Source: page "Covariance" (neuro-kitchen dsp-kitchen, gpu/covariance): for a
window of n samples of a channel-major recording X (one row per channel),
the covariance C = (X - mu)(X - mu)^T / n, mu the channel means over the
window, and the uncentred second moment X X^T / n; a window is a column range
[t0, t0 + n) of the rows, which may start anywhere.  The page computes both in
splits of 4 096 samples for precision and parallelism; in exact arithmetic the
splits change nothing, so the oracle is the plain definition in float64 (the
products of the float32 inputs are exact in float64; the sums are float64
matrix products).
"""

from __future__ import annotations

import numpy as np

SPLIT = 4096


def window(X, t0: int, n: int) -> np.ndarray:
    """Columns [t0, t0 + n) of a channel-major [channels, samples] array, in float64."""
    X = np.asarray(X)
    if X.ndim != 2 or t0 < 0 or n < 1 or t0 + n > X.shape[1]:
        raise ValueError("window out of range")
    return X[:, t0:t0 + n].astype(np.float64)


def second_moment(X, t0: int, n: int, centred: bool) -> np.ndarray:
    """[channels, channels] float64: (V V^T) / n with V the window, centred
    on its channel means when ``centred``."""
    V = window(X, t0, n)
    if centred:
        V = V - V.mean(axis=1, keepdims=True)
    return (V @ V.T) / n


def abs_products(X, t0: int, n: int, centred: bool) -> np.ndarray:
    """sum_t |v_i[t] v_j[t]| / n: the scale of each entry's rounding error."""
    V = window(X, t0, n)
    if centred:
        V = V - V.mean(axis=1, keepdims=True)
    A = np.abs(V)
    return (A @ A.T) / n
