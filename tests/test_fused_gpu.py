"""The fused epilogue on the GPU against the oracle: residual add and
ReLU / GELU in every kernel's store (SIMT direct, general, skinny-M,
skinny-N, split-K; tensor-core single-CTA, CTA-pair, swapped skinny-M,
skinny-N, split and the small mma.sync split-K), for MatMul (batched,
broadcast) and Gemm (bias, transposes) plans; integer-valued inputs with
ReLU bit for bit; an in-place residual (R == Y); unaligned R; K == 0; the
constant-B fused execute; and the errors."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import GemmPlan, OlcError, Plan, synth
from parity import compare

pytestmark = pytest.mark.gpu


def _draw(shape, dtype, dist, seed):
    x, _ = synth.operands(shape, (1,), dtype, dist, dist, seed)
    return x


def _fused(a, b, r, dtype, act, algorithm=None, variant=None, inplace=False, r_offset=0):
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        if algorithm is not None:
            p.force(algorithm)
        if variant is not None:
            p.set_tc_variant(variant)
        p.set_epilogue(act, r is not None)
        shape = p.output_shape
        n = int(np.prod(shape, dtype=np.int64))
        buf = torch.full((n + 64,), float("nan"), dtype=A.dtype, device="cuda")
        Y = buf[:n].view(shape)
        R = None
        if r is not None:
            if inplace:
                Y.copy_(r.cuda())
                R = Y
            else:
                rbuf = torch.empty(n + r_offset, dtype=A.dtype, device="cuda")
                R = rbuf[r_offset:].view(shape)
                R.copy_(r.cuda())
        p.execute_fused(A, B, Y, R=R)
        torch.cuda.synchronize()
        assert torch.isnan(buf[n:].float()).all(), "kernel wrote past the end of Y"
        algo = p.algorithm
    nr = None if r is None else synth.to_numpy_storage(r)
    ref, s = oracle.matmul_fused(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                                 nr, act)
    return Y.cpu(), ref, s, algo


# (a shape, b shape, dtypes, algorithm, tensor-core variant)
KERNEL_CASES = [
    ((2, 3, 40, 24), (24, 40), ["float32", "float64", "float16", "bfloat16"], "direct", None),
    ((2, 130, 72), (72, 136), ["float32", "float64"], "general_simt", None),
    ((300, 256), (256, 264), ["float32"], "general_simt", None),
    ((4, 8192), (8192, 520), ["float32", "bfloat16"], "skinny_m", None),
    ((3, 2, 5, 64), (2, 64, 384), ["float16"], "skinny_m", None),
    ((4096, 1024), (1024, 8), ["float32", "bfloat16"], "skinny_n", None),
    ((2, 130, 72), (2, 72, 16), ["float16"], "skinny_n", None),
    ((64, 16384), (16384, 96), ["float32", "bfloat16"], "split_k", None),
    ((24, 16384), (16384, 32), ["bfloat16", "float16"], "split_k", None),     # mma.sync tiles
    ((300, 520), (520, 264), ["bfloat16", "float16"], "general_tc", 1),
    ((3, 1, 260, 64), (1, 2, 64, 264), ["bfloat16"], "general_tc", 1),
    ((300, 520), (520, 264), ["bfloat16", "float16"], "general_tc", 2),       # CTA pairs
    ((1024, 2048), (2048, 1024), ["bfloat16"], "general_tc", 2),
    ((300, 200), (200, 320), ["bfloat16", "float16"], "general_tc", 2),   # 4-D B loads, blocks past N
    ((100, 2048), (2048, 520), ["bfloat16", "float16"], "general_tc", None),  # cluster split-K
]
CASES = [(a, b, dt, al, v) for a, b, dts, al, v in KERNEL_CASES for dt in dts]


@pytest.mark.parametrize("act", ["relu", "gelu"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%s-%s" % (
    c[3] + ("" if c[4] is None else str(c[4])), c[2], "x".join(map(str, c[0] + c[1]))))
def test_fused_every_kernel(case, act):
    a_shape, b_shape, dtype, algo, variant = case
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.05), seed=21)
    with Plan(a_shape, b_shape, dtype) as p:
        out_shape = p.output_shape
    r = _draw(out_shape, dtype, synth.UNIFORM, 22)
    y, ref, s, ran = _fused(a, b, r, dtype, act, algo, variant)
    assert ran == algo
    compare(y, ref, s, dtype)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%s-%s" % (
    c[3] + ("" if c[4] is None else str(c[4])), c[2], "x".join(map(str, c[0] + c[1]))))
def test_fused_relu_integers_bit_exact(case):
    a_shape, b_shape, dtype, algo, variant = case
    a, b = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=23)
    with Plan(a_shape, b_shape, dtype) as p:
        out_shape = p.output_shape
    r = _draw(out_shape, dtype, synth.Dist("int", -40, 40), 24)
    y, ref, s, _ = _fused(a, b, r, dtype, "relu", algo, variant)
    # integer sums are exact in the accumulator, so both sides narrow the
    # same value (bfloat16 and float16 round large sums the same way)
    compare(y, ref, s, dtype, exact=True)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_activation_only_and_inplace_residual(dtype, act):
    a, b = synth.operands((2, 300, 512), (512, 264), dtype, synth.normal(1.0), synth.normal(0.05), 25)
    y, ref, s, _ = _fused(a, b, None, dtype, act)
    compare(y, ref, s, dtype)
    r = _draw((2, 300, 264), dtype, synth.UNIFORM, 26)
    y, ref, s, _ = _fused(a, b, r, dtype, act, inplace=True)
    compare(y, ref, s, dtype)


@pytest.mark.parametrize("dtype", ["float32", "float16"])
def test_unaligned_residual_takes_the_direct_kernel(dtype):
    a, b = synth.operands((256, 512), (512, 256), dtype, synth.normal(1.0), synth.normal(0.05), 27)
    r = _draw((256, 256), dtype, synth.UNIFORM, 28)
    y, ref, s, _ = _fused(a, b, r, dtype, "gelu", r_offset=1)
    compare(y, ref, s, dtype)


@pytest.mark.parametrize("dtype", ["float64", "bfloat16"])
def test_k_zero_is_activation_of_residual(dtype):
    a = torch.zeros(2, 5, 0, dtype=synth.TORCH_DTYPES[dtype])
    b = torch.zeros(0, 24, dtype=synth.TORCH_DTYPES[dtype])
    r = _draw((2, 5, 24), dtype, synth.UNIFORM, 29)
    y, ref, s, algo = _fused(a, b, r, dtype, "relu")
    assert algo == "zero_fill"
    compare(y, ref, s, dtype, exact=True)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True), (True, True)])
def test_gemm_bias_residual_gelu(dtype, ta, tb):
    m, n, k = 264, 136, 520
    a, b = synth.operands((k, m) if ta else (m, k), (n, k) if tb else (k, n), dtype,
                          synth.normal(1.0), synth.normal(0.05), 30)
    c = _draw((n,), dtype, synth.UNIFORM, 31)
    r = _draw((m, n), dtype, synth.UNIFORM, 32)
    with GemmPlan(a.shape, b.shape, dtype, ta, tb, 0.75, 1.5, c.shape) as p:
        p.set_epilogue("gelu", True)
        Y = torch.empty(m, n, dtype=a.dtype, device="cuda")
        p.execute_fused(a.cuda(), b.cuda(), Y, R=r.cuda(), C=c.cuda())
        torch.cuda.synchronize()
    ref, s = oracle.gemm_op(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                            synth.to_numpy_storage(c), 0.75, 1.5, ta, tb,
                            residual=synth.to_numpy_storage(r), act="gelu")
    compare(Y.cpu(), ref, s, dtype)


def test_fused_with_constant_b_and_errors():
    dtype = "bfloat16"
    a, b = synth.operands((512, 1024), (1024, 512), dtype, synth.normal(1.0), synth.normal(0.05), 33)
    r = _draw((512, 512), dtype, synth.UNIFORM, 34)
    A, R = a.cuda(), r.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        p.set_epilogue("relu", True)
        Y1 = torch.empty(512, 512, dtype=a.dtype, device="cuda")
        Y2 = torch.empty_like(Y1)
        with pytest.raises(OlcError) as ei:
            p.execute(A, b.cuda(), Y1)                 # the residual has no slot here
        assert ei.value.name == "OLC_ERR_NEEDS_RESIDUAL"
        with pytest.raises(OlcError) as ei:
            p.execute_fused(A, b.cuda(), Y1)           # R missing
        assert ei.value.name == "OLC_ERR_NULL"
        with pytest.raises(OlcError) as ei:
            p.execute_fused(A, None, Y1, R=R)          # no B and none owned
        assert ei.value.name == "OLC_ERR_NO_CONSTANT_B"
        p.execute_fused(A, b.cuda(), Y1, R=R)
        p.set_constant_b(b)
        p.execute_fused(A, None, Y2, R=R)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2)
    ref, s = oracle.matmul_fused(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                                 synth.to_numpy_storage(r), "relu")
    compare(Y1.cpu(), ref, s, dtype)


@pytest.mark.parametrize("dtype", ["float32", "float64"])
def test_device_gelu_within_its_error_bound(dtype):
    """GELU alone (K = 1, B = [[1]], so the accumulator is x exactly) against
    the exact x Phi(x).  FLOAT uses erfc from Abramowitz and Stegun 7.1.26,
    absolute error at most 1.5e-7, so |gelu - exact| <= |x| / 2 (1.5e-7 +
    float32 evaluation rounding); the test allows |x| / 2 * 1e-6.  DOUBLE
    uses the library erfc (x / 2 * erfc(-x / sqrt 2)): a few units in the last
    place, times erfc's condition number for the argument's rounding."""
    xs = np.concatenate([np.linspace(-12, 12, 20001), [0.0, -0.0, 1e-30, -1e-30, 40.0, -40.0,
                                                       1e6, -1e6]])
    np_t = np.float32 if dtype == "float32" else np.float64
    x = xs.astype(np_t)
    a = torch.from_numpy(x.reshape(-1, 1).copy())
    b = torch.ones(1, 1, dtype=a.dtype)
    y, _, _, _ = _fused(a, b, None, dtype, "gelu")
    y = y.numpy().reshape(-1).astype(np.float64)
    exact = oracle.activation(x.astype(np.float64), "gelu")
    err = np.abs(y - exact)
    if dtype == "float32":
        bound = 0.5 * np.abs(x.astype(np.float64)) * 1e-6 + 1e-38
    else:
        # erfc(u) has condition number about 2 u^2: the argument's own rounding
        # (x / sqrt 2 here, multiplied by 1 / sqrt 2 there) moves it by that
        xd = x.astype(np.float64)
        bound = np.abs(exact) * 2 * (xd * xd + 16) * 2.3e-16 + 1e-300   # both sides
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), "x=%r gpu %r exact %r" % (x[worst], y[worst], exact[worst])
    nan = _fused(torch.tensor([[float("nan")]], dtype=a.dtype), b, None, dtype, "gelu")[0]
    assert torch.isnan(nan).all()
