"""Pins for the oracle's Gemm operator (rank-2, transA/transB, alpha, beta,
unidirectionally broadcast C): shapes against numpy's broadcasting, exact
integer results against pure-Python arithmetic, float results against numpy
in float64 within the accumulation bound, and MatMul as the alpha=1, no-C
special case.  Planted mistakes (swapped transposes, a dropped bias, alpha
applied to C) fail these checks."""

import math

import numpy as np
import pytest

import oracle
from test_oracle_pins import _narrowed, _store


def _brute_gemm(a, b, c, alpha, beta, ta, tb):
    ap = a.T if ta else a
    bp = b.T if tb else b
    m, k = ap.shape
    n = bp.shape[1]
    out = [[alpha * sum(int(ap[i][t]) * int(bp[t][j]) for t in range(k)) for j in range(n)]
           for i in range(m)]
    if c is not None:
        cb = np.broadcast_to(c.reshape([1] * (2 - c.ndim) + list(c.shape)), (m, n))
        out = [[out[i][j] + beta * int(cb[i][j]) for j in range(n)] for i in range(m)]
    return np.array(out, dtype=np.float64)


C_SHAPES = [None, (), (1,), (7,), (1, 7), (5, 1), (5, 7)]


@pytest.mark.parametrize("dtype", oracle.DTYPES)
@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
@pytest.mark.parametrize("c_shape", C_SHAPES, ids=str)
def test_gemm_integer_exact(dtype, ta, tb, c_shape):
    rng = np.random.default_rng(5 + 2 * ta + tb)
    m, n, k = 5, 7, 9
    a = rng.integers(-3, 4, size=(k, m) if ta else (m, k))
    b = rng.integers(-3, 4, size=(n, k) if tb else (k, n))
    c = None if c_shape is None else rng.integers(-3, 4, size=c_shape)
    alpha, beta = 2.0, -3.0
    y, s = oracle.gemm_op(_store(a, dtype), _store(b, dtype), dtype,
                          None if c is None else _store(c, dtype), alpha, beta, ta, tb)
    want = _brute_gemm(a, b, c, 2, -3, ta, tb)
    assert np.array_equal(oracle.to_float64(y, dtype), _narrowed(want, dtype))
    assert np.all(s >= np.abs(want) - 1e-9)


def test_gemm_alpha_one_no_c_is_matmul():
    rng = np.random.default_rng(1)
    for dtype in oracle.DTYPES:
        a = _store(rng.standard_normal((13, 21)), dtype)
        b = _store(rng.standard_normal((21, 9)), dtype)
        y1, s1 = oracle.gemm_op(a, b, dtype)
        y2, s2 = oracle.matmul(a, b, dtype)
        assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("c_shape", C_SHAPES[1:], ids=str)
def test_gemm_float_vs_numpy(c_shape):
    rng = np.random.default_rng(3)
    m, n, k = 5, 7, 300
    a = rng.uniform(-1, 1, (k, m)).astype(np.float32)
    b = rng.uniform(-1, 1, (n, k)).astype(np.float32)
    c = rng.uniform(-1, 1, c_shape).astype(np.float32)
    y, s = oracle.gemm_op(a, b, "float32", c, 0.5, 1.5, True, True)
    ref = 0.5 * (a.T.astype(np.float64) @ b.T.astype(np.float64)) + 1.5 * c.astype(np.float64)
    g = k * 2.0**-24 / (1 - k * 2.0**-24)
    assert np.all(np.abs(y - ref) <= (g + 4 * 2.0**-24) * s)


@pytest.mark.parametrize("shapes,ok", [
    (((3, 4), (4, 5), False, False, (3, 5)), True),
    (((4, 3), (4, 5), True, False, (5,)), True),
    (((3, 4), (5, 4), False, True, (1, 5)), True),
    (((3, 4), (4, 5), False, False, (3, 1)), True),
    (((3, 4), (4, 5), False, False, ()), True),
    (((3, 4), (4, 5), False, False, (4,)), False),      # C neither 1 nor N wide
    (((3, 4), (4, 5), False, False, (2, 5)), False),
    (((3, 4), (5, 4), False, False, None), False),      # inner dims differ without transB
    (((3, 4, 1), (4, 5), False, False, None), False),   # rank 3
])
def test_gemm_shapes(shapes, ok):
    a_shape, b_shape, ta, tb, c_shape = shapes
    if ok:
        m, n, k = oracle.gemm_output_shape(a_shape, b_shape, ta, tb, c_shape)
        ap = np.zeros(a_shape).T if ta else np.zeros(a_shape)
        bp = np.zeros(b_shape).T if tb else np.zeros(b_shape)
        out = ap @ bp
        assert out.shape == (m, n) and ap.shape[1] == k
        np.broadcast_to(np.zeros(c_shape), out.shape)    # numpy agrees C broadcasts
    else:
        with pytest.raises(oracle.ShapeError):
            oracle.gemm_output_shape(a_shape, b_shape, ta, tb, c_shape)


def test_gemm_planted_mistakes_are_caught():
    rng = np.random.default_rng(11)
    a = rng.integers(-3, 4, size=(9, 5))        # stored transposed: A' = a.T is 5 x 9
    b = rng.integers(-3, 4, size=(9, 7))
    c = rng.integers(-3, 4, size=(7,))
    want = _brute_gemm(a, b, c, 2, -3, True, False)
    f = lambda x: np.asarray(x, np.float32)
    good, _ = oracle.gemm_op(f(a), f(b), "float32", f(c), 2.0, -3.0, True, False)
    assert np.array_equal(good, want)
    # a dropped bias, alpha on the bias, beta on the product
    no_bias, _ = oracle.gemm_op(f(a), f(b), "float32", None, 2.0, -3.0, True, False)
    assert not np.array_equal(no_bias, want)
    swapped, _ = oracle.gemm_op(f(a), f(b), "float32", f(c), -3.0, 2.0, True, False)
    assert not np.array_equal(swapped, want)
    # a transposed operand read untransposed (square case so shapes still fit)
    sq_a = rng.integers(-3, 4, size=(6, 6))
    sq_b = rng.integers(-3, 4, size=(6, 6))
    right, _ = oracle.gemm_op(f(sq_a), f(sq_b), "float32", None, 1.0, 0.0, True, False)
    wrong, _ = oracle.gemm_op(f(sq_a), f(sq_b), "float32", None, 1.0, 0.0, False, False)
    assert np.array_equal(right, _brute_gemm(sq_a, sq_b, None, 1, 0, True, False))
    assert not np.array_equal(wrong, right)
