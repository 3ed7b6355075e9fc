"""The tensor-memory load with a max reduction that the tensor-core tiles'
batch floor rests on (page "Kilosort4 clustering and matching", "k-nearest
neighbours are a matrix product": a batch whose least possible t reaches
every row's threshold holds no candidate).  If the reduction ever returned
less than the largest loaded value, the floor would drop batches that hold
candidates; the full-size parity tests would then fail, and this test names
the cause directly."""

import numpy as np
import pytest

from gpu_common import H, np_

pytestmark = pytest.mark.gpu


def expected_values():
    r = np.arange(128)[:, None]
    c = np.arange(64)[None, :]
    v = (((37 * r + 11 * c + 5 * (r ^ c)) % 97) - 48).astype(np.float32) * np.float32(0.75)
    v = np.broadcast_to(v, (128, 64)).copy()
    rows = np.arange(128)
    v[rows, rows % 64] = 100.0 + rows
    v[rows, (rows + 7) % 64] = -200.0 - rows
    return v


def test_max_reducing_loads_return_the_exact_maxima():
    out = np_(H().test_tmem_max())
    want = expected_values()
    # the values come back unchanged, so the maxima below are of these values
    assert np.array_equal(out[:, :64], want)
    m0, m1 = want[:, :32].max(axis=1), want[:, 32:].max(axis=1)
    assert np.array_equal(out[:, 64], m0), "one-batch load, columns 0..31"
    assert np.array_equal(out[:, 65], m1), "one-batch load, columns 32..63"
    assert np.array_equal(out[:, 66], m0), "two-batch load, columns 0..31"
    assert np.array_equal(out[:, 67], m1), "two-batch load, columns 32..63"
    # every row has its unique maximum in one of the two batches
    assert np.all(np.maximum(m0, m1) == 100.0 + np.arange(128))
