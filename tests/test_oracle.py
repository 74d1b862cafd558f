"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle)


def test_oracle_empty_and_degenerate():
    q = np.zeros((2, 3, 0, 4), np.float32)
    v = np.zeros((2, 3, 0, 5), np.float32)
    assert oracle.fwd(q, q, v).shape == (2, 3, 0, 5)
    dq, dk, dv = oracle.bwd(q, q, v, v)
    assert dq.shape == (2, 3, 0, 4) and dv.shape == (2, 3, 0, 5)
    # N = 1: only the diagonal term.
    rng = np.random.default_rng(0)
    q1 = rng.standard_normal((1, 1, 1, 3)).astype(np.float32)
    k1 = rng.standard_normal((1, 1, 1, 3)).astype(np.float32)
    v1 = rng.standard_normal((1, 1, 1, 2)).astype(np.float32)
    ref = float(np.dot(q1[0, 0, 0].astype(np.float64), k1[0, 0, 0])) * v1[0, 0, 0].astype(np.float64)
    assert np.allclose(oracle.fwd(q1, k1, v1)[0, 0, 0], ref, rtol=1e-15)


def test_oracle_rejects_float64_inputs():
    x = np.zeros((1, 1, 2, 2))
    with pytest.raises(TypeError):
        oracle.fwd(x, x, x)


def test_oracle_threads_agree():
    """OpenMP over (b,h) slices only: the result is the same bitwise for any
    thread count."""
    rng = np.random.default_rng(3)
    q = rng.random((3, 4, 50, 8), dtype=np.float32)
    k = rng.random((3, 4, 50, 8), dtype=np.float32)
    v = rng.standard_normal((3, 4, 50, 6)).astype(np.float32)
    a = oracle.fwd(q, k, v, nthreads=1)
    b = oracle.fwd(q, k, v, nthreads=4)
    assert np.array_equal(a, b)
