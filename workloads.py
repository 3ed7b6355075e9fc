"""Seeded synthetic point sets shaped like the spike-sorting workloads.

This module only draws random numbers: it holds none of the method's
arithmetic (no distances, no neighbour lists, no trees), so both the CUDA
path's tests and the oracle's tests may use it.

The workloads stand in for the recordings the pages measure on, which are
not available here:

* HDBSCAN on raw clips of 61 samples (page "HDBSCAN", neuro-kitchen dsp-kitchen
  gpu/hdbscan, section "Results": clip-like data, 61 dimensions, 20 000 to
  500 000 clips);
* the Kilosort4 k-NN graph over a section of 1 416 points of d = channels x 6
  features, every spike against a subset (page "Kilosort4 clustering and
  matching", sections "k-nearest neighbours are a matrix product" and "The
  measurement that changed the design").

Every set is a Gaussian mixture.  The draw order is fixed:

1. cluster means ``(K, d)``;
2. per-cluster standard deviations;
3. cluster labels, i.i.d. uniform over the K clusters;
4. noise;
5. outliers, uniform in the per-dimension min/max box of the inliers;
6. duplicate targets (uniform, without replacement) and their sources
   (uniform over the rows that are not targets, with replacement).

Values are drawn in float64 and stored as float32, feature-major ``[d, n]``
and C-contiguous.  Inliers occupy rows ``0 .. n_in-1`` and outliers the rows
after them; duplicates overwrite rows anywhere.
"""

from __future__ import annotations

import dataclasses
import hashlib

import numpy as np


@dataclasses.dataclass(frozen=True)
class Mixture:
    n: int
    d: int
    clusters: int
    mean_sd: float
    # isotropic per-cluster sigma: a fixed value, or a U(lo, hi) range
    sigma: float | None = 1.0
    sigma_range: tuple[float, float] | None = None
    # per-cluster, per-dimension sigma ~ U(lo, hi) (anisotropic noise)
    sigma_dim_range: tuple[float, float] | None = None
    outlier_frac: float = 0.0
    dup_frac: float = 0.0
    seed: int = 0


def draw(spec: Mixture) -> np.ndarray:
    """Draw the point set of ``spec`` as float32 ``[d, n]``."""
    rng = np.random.default_rng(spec.seed)
    n, d, K = spec.n, spec.d, spec.clusters
    n_out = int(round(spec.outlier_frac * n))
    n_in = n - n_out
    means = rng.normal(0.0, spec.mean_sd, size=(K, d))
    if spec.sigma_dim_range is not None:
        lo, hi = spec.sigma_dim_range
        sig = rng.uniform(lo, hi, size=(K, d))
    elif spec.sigma_range is not None:
        lo, hi = spec.sigma_range
        sig = rng.uniform(lo, hi, size=(K, 1))
    else:
        sig = np.full((K, 1), float(spec.sigma))
    labels = rng.integers(0, K, size=n_in)
    noise = rng.standard_normal(size=(n_in, d))
    pts = np.empty((n, d), dtype=np.float64)
    pts[:n_in] = means[labels] + sig[labels] * noise
    if n_out:
        box_lo = pts[:n_in].min(axis=0)
        box_hi = pts[:n_in].max(axis=0)
        pts[n_in:] = rng.uniform(box_lo, box_hi, size=(n_out, d))
    n_dup = int(round(spec.dup_frac * n))
    if n_dup:
        targets = rng.choice(n, size=n_dup, replace=False)
        keep = np.ones(n, dtype=bool)
        keep[targets] = False
        sources = rng.choice(np.flatnonzero(keep), size=n_dup, replace=True)
        pts[targets] = pts[sources]
    return np.ascontiguousarray(pts.astype(np.float32).T)


def digest(x: np.ndarray) -> str:
    """sha256 of the float32 bytes: lets stored expected values check that
    a machine drew the same set."""
    return hashlib.sha256(np.ascontiguousarray(x, dtype=np.float32).tobytes()).hexdigest()


# The five workloads.  Sizes, cluster counts and tasks follow the configurations
# the method is measured on; unstated generator details take the plainest reading
# (means and sigma as in the nearest stated config, seed 0 throughout).
WORKLOADS = {
    # HDBSCAN front half: 2 000 clips x 61, 8 clusters, unit isotropic noise, min_samples 5
    "hdbscan_2k_d61": dict(
        spec=Mixture(n=2000, d=61, clusters=8, mean_sd=4.0, sigma=1.0),
        task="mst", min_samples=5),
    # Kilosort4-style section: 1 416 x 102, 12 clusters, k = 10 against every 5th point
    "knn_1416_d102": dict(
        spec=Mixture(n=1416, d=102, clusters=12, mean_sd=3.0, sigma=1.0),
        task="knn", k=10, y_stride=5),
    # HDBSCAN: 50 000 clips x 61, 30 clusters, sigma ~ U(0.5, 2), 5% outliers, min_samples 10
    "hdbscan_50k_d61": dict(
        spec=Mixture(n=50000, d=61, clusters=30, mean_sd=4.0, sigma=None,
                     sigma_range=(0.5, 2.0), outlier_frac=0.05),
        task="mst", min_samples=10),
    # k-NN: 200 000 x 192 (32 channels x 6 PCs), 100 clusters, per-dim sigma ~ U(0.3, 1.5),
    # k = 10 against every 10th point (20 000)
    "knn_200k_d192": dict(
        spec=Mixture(n=200000, d=192, clusters=100, mean_sd=3.0, sigma=None,
                     sigma_dim_range=(0.3, 1.5)),
        task="knn", k=10, y_stride=10),
    # HDBSCAN at scale: 200 000 clips x 61, 50 clusters, sigma ~ U(0.5, 2), 10% outliers,
    # 1% exact duplicates, min_samples 10, full Boruvka
    "hdbscan_200k_d61": dict(
        spec=Mixture(n=200000, d=61, clusters=50, mean_sd=4.0, sigma=None,
                     sigma_range=(0.5, 2.0), outlier_frac=0.10, dup_frac=0.01),
        task="mst", min_samples=10),
}


def workload(name: str) -> tuple[np.ndarray, dict]:
    """Return ``(X [d, n] float32, task dict)`` for a named workload."""
    w = WORKLOADS[name]
    return draw(w["spec"]), w


def subset_columns(X: np.ndarray, stride: int) -> np.ndarray:
    """The subset every ``stride``-th point, as its own contiguous ``[d, m]`` array."""
    return np.ascontiguousarray(X[:, ::stride])


def small(n: int, d: int, seed: int, clusters: int = 3, dup_frac: float = 0.0,
          outlier_frac: float = 0.0, mean_sd: float = 4.0) -> np.ndarray:
    """A small mixture for edge-case and ragged-size tests."""
    return draw(Mixture(n=n, d=d, clusters=max(1, min(clusters, n)), mean_sd=mean_sd,
                        sigma=None, sigma_range=(0.5, 2.0), outlier_frac=outlier_frac,
                        dup_frac=dup_frac, seed=seed))
