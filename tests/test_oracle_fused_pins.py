"""Pins for the oracle's fused epilogue (bias, residual, activation,
narrowing): the GELU against printed values of the standard normal
distribution function and the identity gelu(v) - gelu(-v) = v, its
Lipschitz constant against a numerical derivative, ReLU against its
definition, and whole fused products on integer inputs against pure-Python
arithmetic in the stated order (bias, then residual, then activation).
Planted mistakes (activation before the residual, a residual taken from the
wrong batch item, GELU with a wrong scale inside erf) fail these checks."""

import math

import numpy as np
import pytest

import oracle
from test_oracle_pins import _narrowed, _store

# Phi(x) of the standard normal distribution, as printed in statistical tables
PHI = {0.5: 0.6914624612740131, 1.0: 0.8413447460685429, 1.96: 0.9750021048517795,
       2.0: 0.9772498680518208, 3.0: 0.9986501019683699}


@pytest.mark.parametrize("x,phi", sorted(PHI.items()))
def test_gelu_is_x_times_normal_cdf(x, phi):
    got = oracle.activation(np.array([x, -x]), "gelu")
    assert got[0] == pytest.approx(x * phi, rel=1e-14, abs=1e-15)
    assert got[1] == pytest.approx(-x * (1.0 - phi), rel=1e-13, abs=1e-15)


def test_gelu_identity_and_limits():
    v = np.random.default_rng(0).uniform(-8, 8, 10_000)
    g, gm = oracle.activation(v, "gelu"), oracle.activation(-v, "gelu")
    assert np.allclose(g - gm, v, rtol=0, atol=1e-13)
    assert oracle.activation(np.array([0.0]), "gelu")[0] == 0.0
    assert oracle.activation(np.array([40.0]), "gelu")[0] == 40.0
    assert oracle.activation(np.array([-40.0]), "gelu")[0] == pytest.approx(0.0, abs=1e-300)


def test_gelu_lipschitz_constant():
    v = np.linspace(-6, 6, 120_001)
    h = 1e-6
    d = (oracle.activation(v + h, "gelu") - oracle.activation(v - h, "gelu")) / (2 * h)
    assert d.max() <= oracle.GELU_LIPSCHITZ
    assert d.max() >= oracle.GELU_LIPSCHITZ - 1e-3
    assert abs(v[np.argmax(d)] - math.sqrt(2.0)) < 1e-3     # the maximum sits at sqrt 2


def test_relu_definition():
    v = np.array([-3.0, -0.0, 0.0, 2.5, np.inf, -np.inf, np.nan])
    got = oracle.activation(v, "relu")
    assert np.array_equal(got[:6], [0.0, -0.0, 0.0, 2.5, np.inf, 0.0])
    assert np.isnan(got[6])
    assert np.array_equal(oracle.activation(v[:6], "none"), v[:6])


def _brute_fused(a, b, r, act):
    """Pure-Python batched product (a [Z, M, K] broadcast against b [K, N]),
    + residual r [Z, M, N], then the activation, one element at a time."""
    z, m, k = a.shape
    n = b.shape[1]
    out = np.zeros((z, m, n))
    for t in range(z):
        for i in range(m):
            for j in range(n):
                v = sum(int(a[t, i, p]) * int(b[p, j]) for p in range(k))
                if r is not None:
                    v += int(r[t, i, j])
                if act == "relu":
                    v = max(v, 0)
                out[t, i, j] = v
    return out


@pytest.mark.parametrize("dtype", oracle.DTYPES)
@pytest.mark.parametrize("act", ["none", "relu"])
@pytest.mark.parametrize("with_r", [False, True])
def test_fused_matmul_integer_exact(dtype, act, with_r):
    rng = np.random.default_rng(7)
    a = rng.integers(-3, 4, size=(3, 5, 6))
    b = rng.integers(-3, 4, size=(6, 4))
    r = rng.integers(-20, 21, size=(3, 5, 4)) if with_r else None
    y, s = oracle.matmul_fused(_store(a, dtype), _store(b, dtype), dtype,
                               None if r is None else _store(r, dtype), act)
    want = _brute_fused(a, b, r, act)
    assert np.array_equal(oracle.to_float64(y, dtype), _narrowed(want, dtype))
    assert np.all(s >= np.abs(want))


def test_fused_gemm_order_bias_residual_activation():
    rng = np.random.default_rng(9)
    a = rng.integers(-3, 4, size=(6, 8))
    b = rng.integers(-3, 4, size=(8, 5))
    c = rng.integers(-3, 4, size=(5,))
    r = rng.integers(-9, 10, size=(6, 5))
    f = lambda x: np.asarray(x, np.float32)
    y, _ = oracle.gemm_op(f(a), f(b), "float32", f(c), 2.0, -1.0, residual=f(r), act="relu")
    want = np.maximum(2 * (a @ b) - c[None, :] + r, 0)
    assert np.array_equal(y, want)
    # planted: the activation before the residual
    wrong = np.maximum(2 * (a @ b) - c[None, :], 0) + r
    assert not np.array_equal(wrong, want)


def test_fused_gelu_against_definition_and_planted_mistakes():
    rng = np.random.default_rng(4)
    a = rng.integers(-2, 3, size=(2, 4, 5))
    b = rng.integers(-2, 3, size=(5, 3))
    r = rng.integers(-3, 4, size=(2, 4, 3))
    y, _ = oracle.matmul_fused(a.astype(np.float64), b.astype(np.float64), "float64",
                               r.astype(np.float64), "gelu")
    v = _brute_fused(a, b, r, "none")
    phi = lambda x: 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))
    want = np.vectorize(lambda x: x * phi(x))(v)
    assert np.allclose(y, want, rtol=1e-15, atol=1e-15)
    assert y[1, 0, 0] == pytest.approx(v[1, 0, 0] * phi(v[1, 0, 0]), rel=1e-15, abs=1e-300)
    # planted: the residual of another batch item, a wrong scale inside erf
    swapped = np.vectorize(lambda x: x * phi(x))(_brute_fused(a, b, r[::-1], "none"))
    assert not np.allclose(swapped, want)
    bad = np.vectorize(lambda x: 0.5 * x * (1.0 + math.erf(x)))(v)
    assert not np.allclose(bad, want)


def test_fused_residual_shape_checked():
    with pytest.raises(oracle.ShapeError):
        oracle.matmul_fused(np.zeros((2, 3), np.float32), np.zeros((3, 4), np.float32),
                            "float32", np.zeros((2, 3), np.float32), "none")
