"""Pins for the oracle: checks against facts that do not come from the oracle
itself -- library conversions (numpy's float16, torch's bfloat16), exact
integer arithmetic, exactly rounded sums (math.fsum, fractions), closed-form
rounding cases, numpy's matmul shape rules, and the standard accumulation
error bound (Higham, Accuracy and Stability of Numerical Algorithms, 3.1).

Each mistake a restatement could plausibly make -- a dropped term, a wrong
sign, a transposed operand, a wrong batch index, the wrong accumulator
precision, narrowing per step instead of once -- fails at least one test here;
``test_planted_mistakes_are_caught`` plants each of them and checks that.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
U16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _same_bits_or_both_nan(x, y):
    with np.errstate(invalid="ignore"):         # NaN patterns widen quietly
        x = np.asarray(x, np.float64)
        y = np.asarray(y, np.float64)
    both_nan = np.isnan(x) & np.isnan(y)
    return np.all(both_nan | (x == y)) and np.all(np.signbit(x[~both_nan]) == np.signbit(y[~both_nan]))


# --------------------------------------------------------------------------
# 16-bit decode and encode


def test_decode_f16_all_patterns_match_numpy():
    got = oracle.decode(U16, "float16")
    want = U16.view(np.float16).astype(np.float32)
    assert _same_bits_or_both_nan(got, want)


def test_decode_bf16_all_patterns_match_torch():
    got = oracle.decode(U16, "bfloat16")
    want = torch.from_numpy(U16.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert _same_bits_or_both_nan(got, want)


def _probe_floats(n=400_000, seed=11):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 65504.0, 65519.996, 65520.0,
                        -65520.0, 65536.0, 2.0**-24, 2.0**-25, 3 * 2.0**-26, 2.0**-14,
                        2.0**-14 - 2.0**-25, 1.0, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11,
                        3.3895314e38, 3.4028235e38, 1e-40, -1e-45, 2.0**-126, 2.0**-133,
                        2.0**-134, 3 * 2.0**-135], np.float32)
    return np.concatenate([x, special, rng.standard_normal(50_000).astype(np.float32)])


def test_encode_f16_matches_numpy_rne():
    x = _probe_floats()
    got = oracle.encode(x, "float16")
    with np.errstate(over="ignore"):            # values past 65504 are meant to overflow
        want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    # NaN stays NaN
    assert np.all(np.isnan(got[nan].view(np.float16)))


def test_encode_bf16_matches_torch_rne():
    x = _probe_floats(seed=12)
    got = oracle.encode(x, "bfloat16")
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(oracle.decode(got[nan], "bfloat16")))


@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_encode_ties_go_to_even(dtype):
    # midpoints between consecutive finite positive values are exact in
    # float32; each must round to the neighbour whose last fraction bit is 0
    max_finite = 0x7BFF if dtype == "float16" else 0x7F7F
    lo = np.arange(1, max_finite, dtype=np.uint32).astype(np.uint16)
    lo_v = oracle.decode(lo, dtype).astype(np.float64)
    hi_v = oracle.decode(lo + 1, dtype).astype(np.float64)
    mid = ((lo_v + hi_v) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (lo_v + hi_v) / 2)  # exact midpoints
    got = oracle.encode(mid, dtype)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# the 2-D product


def _int_operands(m, k, n, seed, dtype):
    rng = np.random.default_rng(seed)
    a = rng.integers(-3, 4, size=(m, k))
    b = rng.integers(-3, 4, size=(k, n))
    return a, b, _store(a, dtype), _store(b, dtype)


def _store(x, dtype):
    if dtype in ("float16", "bfloat16"):
        return oracle.encode(np.asarray(x, np.float32), dtype)
    return np.asarray(x, {"float32": np.float32, "float64": np.float64}[dtype])


def _narrowed(exact, dtype):
    """Exact integer results narrowed by a library conversion (numpy float16,
    torch bfloat16); float32/float64 hold these integers exactly."""
    exact = np.asarray(exact, np.float64)
    if dtype == "float16":
        return exact.astype(np.float32).astype(np.float16).astype(np.float64)
    if dtype == "bfloat16":
        return torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).double().numpy()
    return exact


def _brute(a, b):
    """Pure-Python integer product, one term at a time."""
    m, k = a.shape
    n = b.shape[1]
    return [[sum(int(a[i][t]) * int(b[t][j]) for t in range(k)) for j in range(n)]
            for i in range(m)]


@pytest.mark.parametrize("dtype", oracle.DTYPES)
@pytest.mark.parametrize("mkn", [(1, 1, 1), (3, 5, 7), (7, 2, 3), (5, 17, 1), (17, 67, 19)])
def test_small_integer_products_are_exact(dtype, mkn):
    m, k, n = mkn
    a, b, sa, sb = _int_operands(m, k, n, seed=m * 100 + k * 10 + n, dtype=dtype)
    y, s = oracle.gemm2d(sa, sb, dtype)
    want = _narrowed(np.array(_brute(a, b), dtype=np.float64), dtype)
    assert np.array_equal(oracle.to_float64(y, dtype), want)
    want_s = np.array(_brute(np.abs(a), np.abs(b)), dtype=np.float64)
    assert np.array_equal(s, want_s)


@pytest.mark.parametrize("dtype", oracle.DTYPES)
def test_mid_size_integer_products_match_int64_matmul(dtype):
    a, b, sa, sb = _int_operands(130, 257, 70, seed=5, dtype=dtype)
    y, _ = oracle.gemm2d(sa, sb, dtype)
    assert np.array_equal(oracle.to_float64(y, dtype), _narrowed(a @ b, dtype))


@pytest.mark.parametrize("dtype", oracle.DTYPES)
def test_identity_and_permutation_are_exact(dtype):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 9)).astype(np.float32)
    sx = _store(x, dtype)
    eye = _store(np.eye(9), dtype)
    y, _ = oracle.gemm2d(sx, eye, dtype)
    assert np.array_equal(y, sx)
    y, _ = oracle.gemm2d(eye, sx, dtype)
    assert np.array_equal(y, sx)
    perm = rng.permutation(9)
    p = _store(np.eye(9)[perm], dtype)          # row i of P is e_{perm[i]}
    y, _ = oracle.gemm2d(p, sx, dtype)           # so (P X)[i] = X[perm[i]]
    assert np.array_equal(y, sx[perm])
    y, _ = oracle.gemm2d(sx, p.T.copy(), dtype)  # (X P^T)[:, i] = X[:, perm[i]]
    assert np.array_equal(y, sx[:, perm])


def test_fp32_accumulator_and_k_order():
    # 2^24 + 1 + 1 in float32, k ascending: each +1 is lost (ties to even)
    a = np.array([[2.0**24, 1.0, 1.0]], np.float32)
    ones = np.ones((3, 1), np.float32)
    y, s = oracle.gemm2d(a, ones, "float32")
    assert y[0, 0] == np.float32(2.0**24) and s[0, 0] == 2.0**24 + 2
    # reversed order: 1 + 1 = 2 first, then 2^24 + 2 is representable
    y, _ = oracle.gemm2d(a[:, ::-1].copy(), ones, "float32")
    assert y[0, 0] == np.float32(2.0**24 + 2)
    # float64 keeps every term
    y, _ = oracle.gemm2d(a.astype(np.float64), ones.astype(np.float64), "float64")
    assert y[0, 0] == 2.0**24 + 2


@pytest.mark.parametrize("dtype,big", [("float16", 2048.0), ("bfloat16", 256.0)])
def test_half_types_accumulate_in_fp32_and_narrow_once(dtype, big):
    # big + 1 + 1: a 16-bit accumulator would lose both ones (spacing 2 at
    # `big`, ties to even); float32 accumulation gives big + 2, which the
    # final narrowing represents exactly
    a = _store(np.array([[big, 1.0, 1.0]]), dtype)
    ones = _store(np.ones((3, 1)), dtype)
    y, _ = oracle.gemm2d(a, ones, dtype)
    assert oracle.to_float64(y, dtype)[0, 0] == big + 2
    # and the narrowing of a non-representable float32 sum rounds to nearest:
    # big + 1 + 0.5 + 0.25 = big + 1.75 -> big + 2
    a = _store(np.array([[big, 1.0, 0.5, 0.25]]), dtype)
    y, _ = oracle.gemm2d(a, _store(np.ones((4, 1)), dtype), dtype)
    assert oracle.to_float64(y, dtype)[0, 0] == big + 2


def _gamma(k, u):
    return k * u / (1 - k * u)


@pytest.mark.parametrize("mkn", [(13, 300, 11), (4, 2000, 3)])
def test_fp32_within_accumulation_bound_of_exact(mkn):
    m, k, n = mkn
    rng = np.random.default_rng(k)
    a = rng.uniform(-1, 1, (m, k)).astype(np.float32)
    b = rng.uniform(-1, 1, (k, n)).astype(np.float32)
    y, s = oracle.gemm2d(a, b, "float32")
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    for i in range(m):
        for j in range(n):
            exact = math.fsum(a64[i] * b64[:, j])   # products exact in float64
            assert abs(float(y[i, j]) - exact) <= _gamma(k, 2.0**-24) * s[i, j]
            assert s[i, j] == pytest.approx(math.fsum(np.abs(a64[i] * b64[:, j])), rel=1e-15)


def test_fp64_within_accumulation_bound_of_exact_rational():
    m, k, n = 4, 60, 5
    rng = np.random.default_rng(9)
    a = rng.uniform(-1, 1, (m, k))
    b = rng.uniform(-1, 1, (k, n))
    y, s = oracle.gemm2d(a, b, "float64")
    for i in range(m):
        for j in range(n):
            exact = sum(Fraction(a[i, t]) * Fraction(b[t, j]) for t in range(k))
            err = abs(Fraction(float(y[i, j])) - exact)
            assert err <= Fraction(_gamma(k, 2.0**-53)) * Fraction(float(s[i, j]))


@pytest.mark.parametrize("dtype,u_out", [("float16", 2.0**-11), ("bfloat16", 2.0**-8)])
def test_half_within_bound_of_exact(dtype, u_out):
    m, k, n = 9, 500, 7
    rng = np.random.default_rng(21)
    a = _store(rng.standard_normal((m, k)), dtype)
    b = _store(rng.standard_normal((k, n)) * 0.02, dtype)
    y, s = oracle.gemm2d(a, b, dtype)
    a64 = oracle.to_float64(a, dtype)
    b64 = oracle.to_float64(b, dtype)
    yv = oracle.to_float64(y, dtype)
    g = _gamma(k, 2.0**-24)
    for i in range(m):
        for j in range(n):
            exact = math.fsum(a64[i] * b64[:, j])
            bound = u_out * (abs(exact) + g * s[i, j]) + g * s[i, j]
            assert abs(yv[i, j] - exact) <= bound


def test_k_zero_gives_zeros():
    for dtype in oracle.DTYPES:
        a = _store(np.zeros((3, 0)), dtype)
        b = _store(np.zeros((0, 4)), dtype)
        y, s = oracle.gemm2d(a, b, dtype)
        assert y.shape == (3, 4) and np.all(oracle.to_float64(y, dtype) == 0) and np.all(s == 0)


def test_row_sample_equals_full_rows():
    rng = np.random.default_rng(2)
    for dtype in oracle.DTYPES:
        a = _store(rng.standard_normal((40, 33)), dtype)
        b = _store(rng.standard_normal((33, 21)), dtype)
        full, sfull = oracle.gemm2d(a, b, dtype)
        rows = [0, 39, 7, 7, 20]
        part, spart = oracle.gemm2d(a, b, dtype, rows=rows)
        assert np.array_equal(part, full[rows]) and np.array_equal(spart, sfull[rows])


# --------------------------------------------------------------------------
# shapes and batch broadcasting


def _parse_shape(s):
    s = s.strip()
    if s == "()":
        return ()
    return tuple(int(t) for t in s.split(","))


def _golden_shapes():
    cases = []
    with open(os.path.join(HERE, "golden", "shapes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b, out = [t.strip() for t in line.split("|")]
            cases.append((_parse_shape(a), _parse_shape(b), None if out == "error" else _parse_shape(out)))
    return cases


@pytest.mark.parametrize("a_shape,b_shape,want", _golden_shapes())
def test_output_shape_golden_table(a_shape, b_shape, want):
    if want is None:
        with pytest.raises(oracle.ShapeError):
            oracle.output_shape(a_shape, b_shape)
    else:
        assert oracle.output_shape(a_shape, b_shape) == want


@pytest.mark.parametrize("a_shape,b_shape,want", _golden_shapes())
def test_output_shape_agrees_with_numpy_matmul(a_shape, b_shape, want):
    a, b = np.zeros(a_shape), np.zeros(b_shape)
    try:
        np_shape = np.matmul(a, b).shape
    except ValueError:
        np_shape = None
    assert np_shape == want


BROADCAST_CASES = [
    ((8, 1, 12, 16), (1, 4, 16, 6)),
    ((2, 1, 3, 1, 4, 5), (7, 1, 6, 5, 2)),
    ((5,), (3, 5, 4)),
    ((3, 4, 5), (5,)),
    ((2, 3, 4), (4, 5)),
    ((3, 4), (2, 4, 5)),
    ((1, 1, 4, 5), (3, 5, 6)),
    ((6,), (6,)),
]


@pytest.mark.parametrize("dtype", oracle.DTYPES)
@pytest.mark.parametrize("a_shape,b_shape", BROADCAST_CASES)
def test_broadcast_equals_explicit_repeat_and_numpy(dtype, a_shape, b_shape):
    a, b = synth.operands(a_shape, b_shape, dtype, synth.UNIFORM, synth.UNIFORM, seed=1)
    na, nb = synth.to_numpy_storage(a), synth.to_numpy_storage(b)
    y, s = oracle.matmul(na, nb, dtype)
    assert y.shape == np.matmul(np.zeros(a_shape), np.zeros(b_shape)).shape
    # explicit repeat: materialise both operands at the broadcast batch shape
    a2 = na.reshape((1,) + na.shape) if na.ndim == 1 else na
    b2 = nb.reshape(nb.shape + (1,)) if nb.ndim == 1 else nb
    batch = np.broadcast_shapes(a2.shape[:-2], b2.shape[:-2])
    ar = np.ascontiguousarray(np.broadcast_to(a2, batch + a2.shape[-2:]))
    br = np.ascontiguousarray(np.broadcast_to(b2, batch + b2.shape[-2:]))
    yr, sr = oracle.matmul(ar, br, dtype)
    assert np.array_equal(y.reshape(-1), yr.reshape(-1))
    assert np.array_equal(s.reshape(-1), sr.reshape(-1))
    # numpy's own batched matmul on the exact (float64) values: the batch
    # index mapping must agree with it
    av = oracle.to_float64(na, dtype)
    bv = oracle.to_float64(nb, dtype)
    ref = np.matmul(av, bv)
    tol = {"float32": 1e-5, "float64": 1e-12, "float16": 2e-3, "bfloat16": 1e-2}[dtype]
    assert np.all(np.abs(oracle.to_float64(y, dtype) - ref) <= tol * s + 1e-300)


def test_empty_outputs_do_not_read_inputs():
    for a_shape, b_shape in [((0, 16, 32), (32, 8)), ((0, 5), (5, 3)), ((4, 5), (5, 0)),
                             ((0, 1, 2, 3), (1, 5, 3, 4))]:
        out = oracle.output_shape(a_shape, b_shape)
        assert 0 in out
        # operands hold NaN: an empty product must not care
        y, s = oracle.matmul(np.full(a_shape, np.nan, np.float32),
                             np.full(b_shape, np.nan, np.float32), "float32")
        assert y.shape == out and y.size == 0


# --------------------------------------------------------------------------
# planted mistakes: each broken restatement below must fail a pin above


def _check_small_int(gemm):
    a, b, sa, sb = _int_operands(5, 9, 4, seed=77, dtype="float32")
    y = gemm(sa, sb)
    return np.array_equal(y.astype(np.float64), (a @ b).astype(np.float64))


def test_planted_mistakes_are_caught():
    good = lambda a, b: oracle.gemm2d(a, b, "float32")[0]
    assert _check_small_int(good)
    mutants = {
        "dropped last term": lambda a, b: oracle.gemm2d(a[:, :-1].copy(), b[:-1].copy(), "float32")[0],
        "dropped first term": lambda a, b: oracle.gemm2d(a[:, 1:].copy(), b[1:].copy(), "float32")[0],
        "wrong sign": lambda a, b: -oracle.gemm2d(a, b, "float32")[0],
        "B read transposed": lambda a, b: oracle.gemm2d(
            a, b.reshape(b.shape[1], b.shape[0]).T.copy(), "float32")[0],
        "A row offset": lambda a, b: np.roll(oracle.gemm2d(a, b, "float32")[0], 1, axis=0),
        "B column offset": lambda a, b: np.roll(oracle.gemm2d(a, b, "float32")[0], 1, axis=1),
    }
    for name, fn in mutants.items():
        assert not _check_small_int(fn), name

    # a 16-bit accumulator (narrowing per step) fails the accumulation pin
    def narrow_each_step(a, b):
        acc = np.float16(0)
        for t in range(a.shape[1]):
            acc = np.float16(acc + np.float16(a[0, t]) * np.float16(b[t, 0]))
        return acc
    a = np.array([[2048.0, 1.0, 1.0]])
    assert float(narrow_each_step(a, np.ones((3, 1)))) != 2050.0

    # a wrong batch index (B indexed by A's batch position) fails the
    # broadcast pin against numpy
    a = np.arange(2 * 3 * 4, dtype=np.float32).reshape(2, 3, 4)
    b = np.arange(1 * 4 * 2, dtype=np.float32).reshape(1, 4, 2) - 3
    b2 = np.concatenate([b, b + 1])     # a B with two different batch items
    right = oracle.matmul(a, b2, "float32")[0]
    wrong = np.stack([oracle.gemm2d(a[i], b2[0], "float32")[0] for i in range(2)])
    assert np.array_equal(right, np.matmul(a, b2))
    assert not np.array_equal(wrong, np.matmul(a, b2))
