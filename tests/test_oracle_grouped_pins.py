"""Pins for the oracle's grouped products: each product against pure-Python
integer arithmetic (so a mixed-up pairing of A_i with B_j, or a product
dropped from the group, fails), empty members, and the shape errors."""

import numpy as np
import pytest

import oracle
from test_oracle_pins import _brute, _narrowed, _store


@pytest.mark.parametrize("dtype", oracle.DTYPES)
def test_grouped_integer_exact_and_pairing(dtype):
    rng = np.random.default_rng(21)
    shapes = [(3, 5, 4), (1, 7, 2), (6, 1, 9), (4, 4, 4), (2, 3, 0), (0, 5, 3)]
    a_list = [rng.integers(-3, 4, size=(m, k)) for m, n, k in shapes]
    b_list = [rng.integers(-3, 4, size=(k, n)) for m, n, k in shapes]
    ys, ss = oracle.grouped([_store(a, dtype) for a in a_list], [_store(b, dtype) for b in b_list],
                            dtype)
    assert len(ys) == len(shapes)
    for (m, n, k), a, b, y, s in zip(shapes, a_list, b_list, ys, ss):
        want = np.array(_brute(a, b), dtype=np.float64).reshape(m, n)
        assert y.shape == (m, n)
        assert np.array_equal(oracle.to_float64(y, dtype), _narrowed(want, dtype))
        assert np.all(s >= np.abs(want))
    # planted: products paired with the wrong B (same shapes: 4x4x4 with itself swapped)
    sq_a = [rng.integers(-3, 4, size=(4, 4)) for _ in range(2)]
    sq_b = [rng.integers(-3, 4, size=(4, 4)) for _ in range(2)]
    right, _ = oracle.grouped(sq_a, [b.astype(np.float64) for b in sq_b], "float64")
    wrong, _ = oracle.grouped(sq_a, [b.astype(np.float64) for b in sq_b[::-1]], "float64")
    assert not np.array_equal(right[0], wrong[0])
    assert np.array_equal(right[0], np.array(_brute(sq_a[0], sq_b[0]), dtype=np.float64).reshape(4, 4))


def test_grouped_shape_errors():
    with pytest.raises(oracle.ShapeError):
        oracle.grouped([np.zeros((2, 3))], [], "float32")
    with pytest.raises(oracle.ShapeError):
        oracle.grouped([np.zeros((2, 3, 4))], [np.zeros((4, 5))], "float32")
    with pytest.raises(oracle.ShapeError):
        oracle.grouped([np.zeros((2, 3))], [np.zeros((4, 5))], "float32")
