"""Pins of the second-moment / covariance oracle (oracle/moments.py), no GPU.

Page "Covariance": C = (X - mu)(X - mu)^T / n and X X^T / n over a window of
samples.  Checked against values worked out by hand, numpy's own covariance
(bias=True divides by n), and identities that a dropped term, a wrong sign,
a transposed operand or a wrong window would break.
"""

import numpy as np
import pytest

from oracle import moments as M


def test_hand_worked():
    """Two channels, three samples: x = (1, 2, 3), y = (2, 4, 7).
    Means 2 and 13/3.  Centred: x' = (-1, 0, 1), y' = (-7/3, -1/3, 8/3).
    C_xx = 2/3, C_xy = (7/3 + 8/3) / 3 = 5/3, C_yy = (49 + 1 + 64) / 27 = 114/27.
    Uncentred: X X^T / 3 = [[14, 31], [31, 69]] / 3."""
    X = np.array([[1, 2, 3], [2, 4, 7]], dtype=np.float32)
    C = M.second_moment(X, 0, 3, True)
    assert np.allclose(C, [[2 / 3, 5 / 3], [5 / 3, 114 / 27]], rtol=0, atol=1e-15)
    S = M.second_moment(X, 0, 3, False)
    assert np.allclose(S, np.array([[14, 31], [31, 69]]) / 3, rtol=0, atol=1e-15)


def test_window_offsets():
    """A window selects columns [t0, t0 + n): samples outside it change nothing."""
    X = np.array([[9, 1, 2, 3, -5], [9, 2, 4, 7, 8]], dtype=np.float32)
    assert np.array_equal(M.second_moment(X, 1, 3, True),
                          M.second_moment(X[:, 1:4], 0, 3, True))
    with pytest.raises(ValueError):
        M.window(X, 3, 3)


@pytest.mark.parametrize("n", [1, 2, 7, 4095, 4097, 9001])
def test_numpy_cov(n):
    rng = np.random.default_rng(n)
    X = (rng.standard_normal((5, n + 3)) * [[1], [10], [0.1], [3], [1e3]] + 7).astype(np.float32)
    C = M.second_moment(X, 3, n, True)
    ref = np.cov(X[:, 3:].astype(np.float64), bias=True)
    assert np.allclose(C, np.atleast_2d(ref), rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_identities():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((6, 1000)).astype(np.float32) + 2
    C = M.second_moment(X, 0, 1000, True)
    S = M.second_moment(X, 0, 1000, False)
    mu = X.astype(np.float64).mean(axis=1)
    # second moment = covariance + mu mu^T
    assert np.allclose(S, C + np.outer(mu, mu), rtol=1e-12, atol=1e-12)
    # symmetric, positive semi-definite, trace = mean squared deviation
    assert np.array_equal(C, C.T)
    assert np.linalg.eigvalsh(C).min() > -1e-12
    V = X.astype(np.float64) - mu[:, None]
    assert np.isclose(np.trace(C), (V ** 2).sum() / 1000, rtol=1e-12)
    # the covariance ignores a shift of each channel, and scales as a b
    shifted = X + np.arange(6, dtype=np.float32)[:, None] * 4
    assert np.allclose(M.second_moment(shifted, 0, 1000, True), C, rtol=1e-5, atol=1e-5)
    a = np.array([1, 2, 4, 0.5, 8, 1], dtype=np.float32)
    assert np.allclose(M.second_moment(X * a[:, None], 0, 1000, True), C * np.outer(a, a),
                       rtol=1e-12, atol=1e-12)
    # abs_products bounds every entry
    B = M.abs_products(X, 0, 1000, True)
    assert np.all(np.abs(C) <= B + 1e-12)
    assert np.allclose(np.diag(B), np.diag(C), rtol=1e-12)


# ---------------------------------------------------------------- planted mistakes

def _pins_pass():
    try:
        test_hand_worked()
        test_window_offsets()
        for n in (2, 7, 4097):
            test_numpy_cov(n)
        test_identities()
    except (AssertionError, ValueError):
        return False
    return True


_orig_window = M.window


def _divide_by_n_minus_1(X, t0, n, centred):
    V = _orig_window(X, t0, n)
    if centred:
        V = V - V.mean(axis=1, keepdims=True)
    return (V @ V.T) / max(n - 1, 1)


def _never_centred(X, t0, n, centred):
    V = _orig_window(X, t0, n)
    return (V @ V.T) / n


def _window_off_by_one(X, t0, n):
    X = np.asarray(X)
    return X[:, t0 + 1:t0 + n + 1].astype(np.float64) if t0 + n + 1 <= X.shape[1] else \
        X[:, t0:t0 + n].astype(np.float64)


def _mean_over_channels(X, t0, n, centred):
    V = _orig_window(X, t0, n)
    if centred:
        V = V - V.mean(axis=0, keepdims=True)
    return (V @ V.T) / n


@pytest.mark.parametrize("attr, bad", [
    ("second_moment", _divide_by_n_minus_1),
    ("second_moment", _never_centred),
    ("window", _window_off_by_one),
    ("second_moment", _mean_over_channels),
])
def test_planted_mistakes_fail_a_pin(monkeypatch, attr, bad):
    assert _pins_pass()
    monkeypatch.setattr(M, attr, bad)
    assert not _pins_pass()
