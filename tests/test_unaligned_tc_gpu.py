"""FLOAT16 / BFLOAT16 products the TMA cannot read in place stay on the
tensor cores ("Gemm and MatMul Performance Roadmap", Phase 4: the required
test classes include tails and non-contiguous shapes; "MatMul Kernel Design",
section "Types and algorithm selection": one algorithm choice per shape, any
layout).  Odd N or K (rows that are not 16-byte multiples) and operands or
outputs that start off a 16-byte boundary: the operand is staged into padded
rows by a copy kernel, the general tiles read it through a row pitch and
store Y at any alignment.  Every case is compared with the oracle element by
element (integer inputs bit for bit), with canaries around Y."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import GemmPlan, Plan, synth
from parity import compare, sample_rows

pytestmark = pytest.mark.gpu

HALF = ["float16", "bfloat16"]

ODD_SHAPES = [
    ((300, 520), (520, 263)),          # odd N, tails in M and N
    ((257, 515), (515, 300)),          # odd K
    ((600, 1001), (1001, 777)),        # both odd, several tiles
    ((513, 2051), (2051, 1023)),       # CTA pairs with odd K and N
    ((3, 1, 130, 67), (1, 2, 67, 133)),   # broadcast batch, odd K and N
    ((67,), (67, 301)),                # rank-one A
    ((40, 9), (9, 3)),                 # tiny, odd everything
]


def _offset_tensor(t_cpu: torch.Tensor, off: int, canary: float):
    """A device copy of t starting `off` elements into a buffer filled with
    `canary` (off = 1: a 2-byte offset from the 256-byte aligned base)."""
    buf = torch.full((t_cpu.numel() + off + 8,), canary, dtype=t_cpu.dtype, device="cuda")
    view = buf[off:off + t_cpu.numel()].view(t_cpu.shape)
    view.copy_(t_cpu.cuda())
    return buf, view


def _run(a, b, dtype, a_off=0, b_off=0, y_off=0, variant=None, algo=None, expect=None):
    A_buf, A = _offset_tensor(a, a_off, 0.0)
    B_buf, B = _offset_tensor(b, b_off, 0.0)
    with Plan(a.shape, b.shape, dtype) as p:
        if algo:
            p.force(algo)
        if variant is not None:
            p.set_tc_variant(variant)
        shape = p.output_shape
        n = int(np.prod(shape, dtype=np.int64))
        ybuf = torch.full((n + y_off + 16,), 0.5, dtype=synth.TORCH_DTYPES[dtype], device="cuda")
        Y = ybuf[y_off:y_off + n].view(shape)
        if expect is not None:
            assert p.algorithm_for(A, B, Y) == expect
        p.execute_checked(A, B, Y)
        torch.cuda.synchronize()
        rest = torch.cat([ybuf[:y_off], ybuf[y_off + n:]]).float().cpu()
        assert bool((rest == 0.5).all()), "write outside Y"
        return Y.cpu(), p


@pytest.mark.parametrize("dtype", HALF)
@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("shapes", ODD_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_odd_rows_on_tensor_cores(dtype, variant, shapes):
    a_shape, b_shape = shapes
    with Plan(a_shape, b_shape, dtype) as p:
        # small products take DIRECT by the size rule: force the tiles there
        force = None if p.algorithm == "general_tc" else "general_tc"
    for dist, exact in [(synth.normal(1.0), False), (synth.SMALL_INT, True)]:
        a, b = synth.operands(a_shape, b_shape, dtype, dist, synth.normal(0.02) if not exact else dist,
                              seed=31)
        y, _ = _run(a, b, dtype, variant=variant, algo=force, expect="general_tc")
        y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        compare(y, y_ref, s, dtype, exact=exact)


@pytest.mark.parametrize("dtype", HALF)
@pytest.mark.parametrize("algo,shapes,variant", [
    ("general_tc", ((300, 520), (520, 264)), 1),
    ("general_tc", ((512, 256), (256, 512)), 2),
    ("skinny_m", ((4, 8192), (8192, 512)), 2),
    ("skinny_m", ((4, 8192), (8192, 512)), 1),
    ("skinny_n", ((600, 4096), (4096, 8)), 2),
    ("skinny_n", ((600, 4096), (4096, 8)), 1),
    ("split_k", ((32, 16384), (16384, 32)), 0),
    ("split_k", ((300, 5000), (5000, 264)), 0),
], ids=lambda x: x if isinstance(x, str) else None)
@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 5, 7)],
                         ids=lambda o: "A%d_B%d_Y%d" % o)
def test_misaligned_pointers_stay_on_tensor_cores(dtype, algo, shapes, variant, offs):
    a_off, b_off, y_off = offs
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=32)
    # a misaligned Y moves skinny and split-K products to the general tiles;
    # misaligned operands alone keep the planned kernel (with a dense copy)
    expect = algo if y_off == 0 else "general_tc"
    y, p = _run(a, b, dtype, a_off, b_off, y_off, variant=variant, algo=algo, expect=expect)
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(y, y_ref, s, dtype, exact=True)


@pytest.mark.parametrize("dtype", HALF)
def test_staging_copy_counts(dtype):
    a, b = synth.operands((300, 515), (515, 263), dtype, synth.UNIFORM, synth.UNIFORM, seed=33)
    with Plan(a.shape, b.shape, dtype) as p:
        assert p.algorithm == "general_tc"
        assert p.launches == 3            # A and B padded, then the product
        A, B = a.cuda(), b.cuda()
        Y = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
        assert p.staging_copies(A, B, Y) == 2
        p.set_constant_b(b)
        assert p.launches == 2            # the constant B is kept padded
    a, b = synth.operands((300, 520), (520, 264), dtype, synth.UNIFORM, synth.UNIFORM, seed=33)
    with Plan(a.shape, b.shape, dtype) as p:
        A, B = a.cuda(), b.cuda()
        Y = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
        assert p.launches == 1 and p.staging_copies(A, B, Y) == 0


@pytest.mark.parametrize("dtype", HALF)
def test_constant_b_with_odd_n(dtype):
    a, b = synth.operands((8, 300, 1024), (1024, 1001), dtype, synth.normal(1.0), synth.normal(0.02),
                          seed=34)
    A = a.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        Y1 = torch.full(p.output_shape, 0.5, dtype=A.dtype, device="cuda")
        Y2 = torch.full(p.output_shape, 0.5, dtype=A.dtype, device="cuda")
        p.execute(A, b.cuda(), Y1)
        p.set_constant_b(b)
        p.execute_constant(A, Y2)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2)
    a2 = synth.to_numpy_storage(a).reshape(-1, 1024)
    rows = sample_rows(a2.shape[0], extra=64)
    y_ref, s = oracle.gemm2d(a2, synth.to_numpy_storage(b), dtype, rows=rows)
    compare(Y2.cpu().reshape(-1, 1001)[rows], y_ref, s, dtype)


@pytest.mark.parametrize("dtype", HALF)
@pytest.mark.parametrize("act", ["none", "gelu"])
def test_fused_residual_with_odd_n_and_offsets(dtype, act):
    a, b = synth.operands((520, 264), (264, 777), dtype, synth.UNIFORM, synth.UNIFORM, seed=35)
    r, _ = synth.operands((520, 777), (1,), dtype, synth.UNIFORM, synth.UNIFORM, seed=36)
    _, A = _offset_tensor(a, 1, 0.0)
    _, B = _offset_tensor(b, 0, 0.0)
    _, R = _offset_tensor(r, 3, 0.0)
    with Plan(a.shape, b.shape, dtype) as p:
        p.set_epilogue(act, True)
        ybuf = torch.full((520 * 777 + 9,), 0.5, dtype=A.dtype, device="cuda")
        Y = ybuf[5:5 + 520 * 777].view(520, 777)
        assert p.algorithm_for(A, B, Y, R) == "general_tc"
        p.execute_fused(A, B, Y, R=R)
        torch.cuda.synchronize()
        assert bool((ybuf[:5].float() == 0.5).all()) and bool((ybuf[5 + 520 * 777:].float() == 0.5).all())
    y_ref, s = oracle.matmul_fused(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                                   synth.to_numpy_storage(r), act)
    compare(Y.cpu(), y_ref, s, dtype)


@pytest.mark.parametrize("dtype", HALF)
@pytest.mark.parametrize("trans", [(True, False), (False, True), (True, True)])
def test_gemm_transposed_with_offsets(dtype, trans):
    ta, tb = trans
    m, k, n = 264, 520, 777 if not tb else 776
    a_shape = (k, m) if ta else (m, k)
    b_shape = (n, k) if tb else (k, n)
    a, b = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=37)
    c, _ = synth.operands((n,), (1,), dtype, synth.SMALL_INT, synth.SMALL_INT, seed=38)
    _, A = _offset_tensor(a, 1, 0.0)
    _, B = _offset_tensor(b, 1, 0.0)
    with GemmPlan(a_shape, b_shape, dtype, ta, tb, 1.0, 2.0, c.shape) as p:
        assert p.algorithm == "general_tc"
        ybuf = torch.full((m * n + 3,), 0.5, dtype=A.dtype, device="cuda")
        Y = ybuf[1:1 + m * n].view(m, n)
        p.execute(A, B, Y, C=c.cuda())
        torch.cuda.synchronize()
        assert float(ybuf[0]) == 0.5 and bool((ybuf[1 + m * n:].float() == 0.5).all())
    y_ref, s = oracle.gemm_op(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                              c=synth.to_numpy_storage(c), alpha=1.0, beta=2.0, trans_a=ta, trans_b=tb)
    compare(Y.cpu(), y_ref, s, dtype, exact=True)


def test_misaligned_pointer_to_its_element_is_rejected():
    with Plan((64, 64), (64, 64), "float32") as p:
        buf = torch.zeros(64 * 64 + 1, device="cuda")
        A = buf[1:].view(64, 64)
        lib = p.lib
        base = buf.data_ptr()
        # a float operand two bytes into a float: not a float address
        assert lib.olc_matmul_execute(p.handle, base + 2, A.data_ptr(), A.data_ptr(), None) == 13


def test_vocab_projection_odd_n_sampled_rows():
    """[16384, 4096] x [4096, 50257] BF16 (an output projection onto a
    50257-entry vocabulary: N odd) on the tensor cores, checked on sampled
    rows including the first and last of every 128-row band."""
    a, b = synth.operands((16384, 4096), (4096, 50257), "bfloat16", synth.normal(1.0),
                          synth.normal(0.02), seed=39)
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, "bfloat16") as p:
        assert p.algorithm == "general_tc"
        ybuf = torch.full((16384 * 50257 + 16,), 0.5, dtype=torch.bfloat16, device="cuda")
        Y = ybuf[:16384 * 50257].view(16384, 50257)
        p.execute_checked(A, B, Y)
        torch.cuda.synchronize()
        assert bool((ybuf[16384 * 50257:].float() == 0.5).all())
    rows = sample_rows(16384, extra=32)
    y_ref, s = oracle.gemm2d(synth.to_numpy_storage(a), synth.to_numpy_storage(b), "bfloat16",
                             rows=rows)
    compare(Y[rows].cpu(), y_ref, s, "bfloat16")


def test_up_projection_with_a_offset_by_one_element_sampled_rows():
    """The transformer up projection [8, 2048, 4096] x [4096, 14336] BF16 with
    A starting one element into its buffer: A is staged, the pair tiles run."""
    a, b = synth.operands((8, 2048, 4096), (4096, 14336), "bfloat16", synth.normal(1.0),
                          synth.normal(0.02), seed=2)
    _, A = _offset_tensor(a, 1, 0.0)
    B = b.cuda()
    with Plan(a.shape, b.shape, "bfloat16") as p:
        Y = torch.empty(p.output_shape, dtype=torch.bfloat16, device="cuda")
        assert p.algorithm_for(A, B, Y) == "general_tc" and p.staging_copies(A, B, Y) == 1
        p.execute_checked(A, B, Y)
        torch.cuda.synchronize()
    a2 = synth.to_numpy_storage(a).reshape(-1, 4096)
    rows = sample_rows(a2.shape[0], extra=32)
    y_ref, s = oracle.gemm2d(a2, synth.to_numpy_storage(b), "bfloat16", rows=rows)
    compare(Y.reshape(-1, 14336)[rows].cpu(), y_ref, s, "bfloat16")
