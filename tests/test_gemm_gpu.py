"""The Gemm operator on the GPU against the oracle: every transpose
combination, every C shape, alpha/beta, each feasible algorithm, all four
types; integer-valued inputs bit for bit; K == 0 gives beta * C."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import GemmPlan, OlcError, synth
from parity import TOL

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "float64", "float16", "bfloat16"]


def _run(a, b, c, dtype, ta, tb, alpha, beta, algorithm=None, variant=None):
    A, B = a.cuda(), b.cuda()
    C = None if c is None else c.cuda()
    with GemmPlan(a.shape, b.shape, dtype, ta, tb, alpha, beta,
                  None if c is None else c.shape) as p:
        if algorithm:
            p.force(algorithm)
        if variant is not None:
            p.set_tc_variant(variant)
        m, n = p.output_shape
        buf = torch.full((m * n + 16,), float("nan"), dtype=A.dtype, device="cuda")
        Y = buf[:m * n].view(m, n)
        p.execute(A, B, Y, C=C)
        torch.cuda.synchronize()
        assert torch.isnan(buf[m * n:].float()).all()
        return Y.cpu(), p.algorithm


def _check(a, b, c, dtype, ta, tb, alpha, beta, exact=False, **kw):
    y, algo = _run(a, b, c, dtype, ta, tb, alpha, beta, **kw)
    nc = None if c is None else synth.to_numpy_storage(c)
    ref, s = oracle.gemm_op(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype, nc,
                            alpha, beta, ta, tb)
    yg = oracle.to_float64(synth.to_numpy_storage(y), dtype)
    yr = oracle.to_float64(ref, dtype)
    if exact:
        assert np.array_equal(yg, yr), (algo, np.argwhere(yg != yr)[:3])
    else:
        err = np.abs(yg - yr)
        assert np.all(err <= TOL[dtype] * s + 1e-30), (algo, float((err / (TOL[dtype] * s + 1e-30)).max()))
    return algo


def _operands(m, n, k, ta, tb, c_shape, dtype, dist, seed):
    a_shape = (k, m) if ta else (m, k)
    b_shape = (n, k) if tb else (k, n)
    a, b = synth.operands(a_shape, b_shape, dtype, dist, dist, seed)
    c = None
    if c_shape is not None:
        c, _ = synth.operands(c_shape, (1,), dtype, dist, dist, seed + 100)
    return a, b, c


C_CASES = [None, (), (96,), (1, 96), (72, 1), (72, 96)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("c_shape", C_CASES, ids=str)
def test_gemm_small_all_algorithms(dtype, ta, tb, c_shape):
    m, n, k = 72, 96, 136
    for dist, exact in ((synth.UNIFORM, False), (synth.SMALL_INT, True)):
        a, b, c = _operands(m, n, k, ta, tb, c_shape, dtype, dist, seed=3)
        for algo in (None, "direct", "general_simt", "general_tc"):
            try:
                _check(a, b, c, dtype, ta, tb, 2.0, -1.5 if not exact else -3.0, exact=exact,
                       algorithm=algo)
            except OlcError:
                assert algo in ("general_tc",)   # not every type / layout has it


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("variant", [1, 2])
# N = 832 = 13 x 64: the CTA pairs load MN-major B as 4-D boxes of two 64-column
# blocks, the last one past N
@pytest.mark.parametrize("n", [776, 832])
def test_gemm_tensor_cores_large(dtype, ta, tb, variant, n):
    m, k = 520, 264
    a, b, c = _operands(m, n, k, ta, tb, (n,), dtype, synth.normal(1.0), seed=4)
    algo = _check(a, b, c, dtype, ta, tb, 0.5, 2.0, variant=variant)
    assert algo == "general_tc"
    ai, bi, ci = _operands(m, n, k, ta, tb, (m, 1), dtype, synth.SMALL_INT, seed=5)
    _check(ai, bi, ci, dtype, ta, tb, 1.0, 1.0, exact=True, variant=variant)


@pytest.mark.parametrize("dtype", DTYPES)
def test_gemm_non_transposed_special_paths(dtype):
    # skinny-M, skinny-N, split-K with the epilogue
    for (m, n, k) in [(4, 1024, 512), (512, 8, 1024), (32, 32, 16384)]:
        a, b, c = _operands(m, n, k, False, False, (n,), dtype, synth.SMALL_INT, seed=6)
        _check(a, b, c, dtype, False, False, 2.0, -1.0, exact=True)


@pytest.mark.parametrize("dtype", DTYPES)
def test_gemm_k_zero_is_beta_c(dtype):
    a = torch.empty((5, 0), dtype=synth.TORCH_DTYPES[dtype])
    b = torch.empty((0, 7), dtype=synth.TORCH_DTYPES[dtype])
    c, _ = synth.operands((5, 7), (1,), dtype, synth.SMALL_INT, synth.SMALL_INT, 1)
    y, algo = _run(a, b, c, dtype, False, False, 2.0, 3.0)
    assert algo == "zero_fill"
    assert torch.equal(y.double(), 3.0 * c.double())
