"""Split-product second moment and covariance on the GPU against the oracle
(oracle/moments.py; page "Covariance", sections "After: split products" and
"The bug a test with an odd length found": odd lengths and misaligned
windows are the cases that once went wrong).

Two kinds of check:

* exact: windows of integer channel levels plus sparse integer deviations,
  where the centring, every product and every partial sum is exact (values
  of at most 12 significant bits, sums below 2^24), so the result must equal
  the float64 oracle rounded to float32, bit for bit, wherever a "clean"
  channel (at most 11 significant bits, no low FP16 part) is involved;
  "dirty" channels (12 bits) then exercise the hi.lo' and lo.hi' products
  one at a time; both the covariance and the second moment (which the
  library forms from the centred products plus the means);
* bounded: random windows against the float64 oracle within the rounding
  bound of the arithmetic (below), at odd and even lengths across the
  4 096-sample split size and at misaligned starts.

The bound per entry (i, j), with B_ij = sum_t |v_i v_j| / n (oracle) and
h_c = channel c's flushing threshold of the two-part FP16 split in input
units (v the centred values the library splits):
  (3 * 4096 * 2^-24 + 4 * 2^-22) * 1.05 * B_ij        products and their sum
  + 2^-24 |C_ij|                                      final rounding
  + h_i mean|v_j| + mean|v_i| h_j + h_i h_j           flushed parts
(three products per sample into one float32 accumulator over a split, any
order; each product off by at most 3 * 2^-22 relative from the split, plus
2^-22 from centring).
"""

import numpy as np
import pytest

from oracle import moments as M
from gpu_common import H, dev, np_

pytestmark = pytest.mark.gpu


def f16_scale_h(X, t0, n):
    """Per channel, the flushing threshold of the split in input units:
    2^(-14 - e_c) with 2^e_c putting the channel's bound on its centred
    values, max |x| + |mean|, in [2^14, 2^15)."""
    W = X[:, t0:t0 + n].astype(np.float64)
    b = np.abs(W).max(axis=1) + np.abs(W.mean(axis=1))
    h = np.zeros(X.shape[0])
    for c, bc in enumerate(b):
        if bc > 0:
            e = max(-60, min(60, 14 - int(np.floor(np.log2(bc)))))
            h[c] = 2.0 ** (-14 - e)
    return h


def check_bounded(g, X, t0, n, centred, where=""):
    C = M.second_moment(X, t0, n, centred)
    B = M.abs_products(X, t0, n, centred)
    V = M.window(X, t0, n)
    V = V - V.mean(axis=1, keepdims=True)  # the library splits centred values
    ma = np.abs(V).mean(axis=1)
    h = f16_scale_h(X, t0, n)
    tol = ((3 * 4096 * 2.0 ** -24 + 4 * 2.0 ** -22) * 1.05 * B + 2.0 ** -24 * np.abs(C)
           + h[:, None] * ma[None, :] + ma[:, None] * h[None, :] + h[:, None] * h[None, :])
    err = np.abs(g.astype(np.float64) - C)
    bad = err > tol
    assert not bad.any(), (f"{where}: {int(bad.sum())} entries beyond the bound, e.g. "
                           f"{np.argwhere(bad)[:3].tolist()}: {g[bad][:3]} vs {C[bad][:3]}")
    assert np.array_equal(g, g.T), f"{where}: not symmetric"
    rel = err / np.maximum(B, np.finfo(np.float64).tiny)
    return float(np.median(rel)), float(rel.max())


def sparse_int_window(rng, C, T, t0, n):
    """Channels at a constant integer level plus two sparse integer
    deviations +a and -a (so every channel mean is an integer and the
    centred values are the deviations, exactly): even channels 'clean'
    (|a| <= 1000), odd channels 'dirty' (odd |a| in [2049, 2895], 12
    significant bits); every sum of products stays below 2^24."""
    X = np.zeros((C, T), dtype=np.float64)
    for c in range(C):
        X[c, :] = int(rng.integers(-7, 8)) * 16
        if n < 2:
            continue  # one sample: nothing deviates from the mean
        pos = rng.choice(n, 2, replace=False) + t0
        if c % 2 == 0:
            a = int(rng.integers(-1000, 1001))
        else:
            a = int(2 * rng.integers(1025, 1448) - 1) * int(rng.choice([-1, 1]))
        X[c, pos] += [a, -a]
    # samples outside the window: large values that must not leak in
    X[:, :t0] = 1e6
    X[:, t0 + n:] = -1e6
    return X.astype(np.float32)


@pytest.mark.parametrize("centred", [False, True])
@pytest.mark.parametrize("C, n, t0", [(5, 7, 1), (133, 5003, 3), (64, 4096, 0), (130, 8193, 5),
                                      (2, 1, 0), (257, 4097, 2)])
def test_exact_integer_windows(C, n, t0, centred):
    h = H()
    rng = np.random.default_rng(C * 7 + n)
    T = t0 + n + 3
    X = sparse_int_window(rng, C, T, t0, n)
    g = np_(h.second_moment(dev(X), t0, n, centred=centred))
    want = M.second_moment(X, t0, n, centred).astype(np.float32)
    dirty = (np.arange(C) % 2 == 1)
    exact = ~(dirty[:, None] & dirty[None, :])
    assert np.array_equal(g[exact], want[exact]), np.argwhere(g != want)[:5].tolist()
    check_bounded(g, X, t0, n, centred, "dirty pairs")


@pytest.mark.parametrize("centred", [False, True])
@pytest.mark.parametrize("C, n, t0", [
    (1, 1, 0), (1, 2, 0), (4, 7, 1), (61, 4095, 3), (64, 4096, 0), (61, 4097, 5),
    (127, 9001, 1), (128, 12288, 4), (129, 60000, 7), (384, 60000, 1001),
])
def test_random_windows(C, n, t0, centred):
    h = H()
    rng = np.random.default_rng(1000 + C + n)
    T = t0 + n + 11
    scale = rng.uniform(0.1, 10.0, (C, 1))
    level = rng.uniform(-50, 50, (C, 1))
    X = (rng.standard_normal((C, T)) * scale + level).astype(np.float32)
    g = np_(h.second_moment(dev(X), t0, n, centred=centred))
    med, mx = check_bounded(g, X, t0, n, centred, f"C={C} n={n} t0={t0}")
    print(f"C={C} n={n} t0={t0} centred={centred}: median rel err {med:.2e}, max {mx:.2e}")
    # in practice the error is far below the worst-case bound
    assert med < 1e-5


def test_channels_of_very_different_scale():
    """A channel a million times quieter than its neighbours keeps its
    precision: each channel has its own power-of-two scale."""
    h = H()
    rng = np.random.default_rng(21)
    X = rng.standard_normal((6, 9000)).astype(np.float32)
    X[2] *= 1e-6
    X[4] *= 1e4
    g = np_(h.second_moment(dev(X), 0, 9000, centred=True))
    check_bounded(g, X, 0, 9000, True, "scales")
    C = M.second_moment(X, 0, 9000, True)
    assert abs(g[2, 2] - C[2, 2]) <= 1e-5 * C[2, 2]


def test_accumulate_and_single_sample():
    h = H()
    rng = np.random.default_rng(9)
    X = rng.standard_normal((70, 5000)).astype(np.float32)
    Xd = dev(X)
    out = h.second_moment(Xd, 0, 2500, centred=False)
    h.second_moment(Xd, 2500, 2500, centred=False, out=out, accumulate=True)
    want = M.second_moment(X, 0, 2500, False) + M.second_moment(X, 2500, 2500, False)
    B = M.abs_products(X, 0, 2500, False) + M.abs_products(X, 2500, 2500, False)
    assert np.all(np.abs(np_(out) - want) <= 1e-3 * B + 1e-6 * np.abs(want))
    # one sample: its covariance is exactly zero
    assert not np.any(np_(h.second_moment(Xd, 17, 1, centred=True)))


def test_bad_inputs():
    h = H()
    X = np.ones((3, 10), dtype=np.float32)
    X[1, 4] = np.nan
    with pytest.raises(h.HdbmstError) as e:
        h.second_moment(dev(X), 0, 10)
    assert e.value.status == 4
    # the same NaN outside the window is not read
    assert np.all(np.isfinite(np_(h.second_moment(dev(X), 5, 5))))
    with pytest.raises(h.HdbmstError) as e:
        h.second_moment(dev(X), 6, 5)
    assert e.value.status == 1
