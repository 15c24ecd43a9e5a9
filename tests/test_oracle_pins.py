"""The CPU oracle against its pins (page values, closed forms, brute force,
PyTorch's float64 conv2d, IEEE single-precision arithmetic)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle(0)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_points_match_full(orc):
    """The point-wise entry computes the same accumulators as the full conv."""
    import numpy as np
    rng = np.random.default_rng(5)
    shape = (2, 32, 9, 7, 3, 3, 2, 1, 1, 2, 1, 1, 2)
    x = rng.integers(-128, 128, size=(2, 32, 9, 7)).astype(np.int8)
    f = rng.integers(-128, 128, size=(3, 32, 3, 2)).astype(np.int8)
    acc = orc.conv_acc(x, f, shape)
    N, K, P, Q = acc.shape
    pts = np.array([(n, k, p, q) for n in range(N) for k in range(K) for p in range(P) for q in range(Q)])
    assert np.array_equal(orc.conv_acc_points(x, f, shape, pts), acc.reshape(-1))


def test_f64_points_match_full(orc):
    """The point-wise fp32-path entry computes the same values (and magnitude
    sums) as the full convolution."""
    import numpy as np
    rng = np.random.default_rng(6)
    shape = (2, 3, 11, 9, 4, 3, 2, 1, 1, 2, 1, 1, 2)
    x = rng.random((2, 3, 11, 9)).astype(np.float32)
    w = (rng.random((4, 3, 3, 2)) - 0.5).astype(np.float32)
    b = (rng.random(4) - 0.5).astype(np.float32)
    y, mag = orc.conv_f64(x, w, shape, bias=b)
    N, K, P, Q = y.shape
    pts = np.array([(n, k, p, q) for n in range(N) for k in range(K) for p in range(P) for q in range(Q)])
    yp, mp = orc.conv_f64_points(x, w, shape, pts, bias=b)
    assert np.array_equal(yp, y.reshape(-1)) and np.array_equal(mp, mag.reshape(-1))
