"""Plan-owned constant B: executes without B compute the planned product
(checked against the oracle) and equal executes with it bit for bit (the
same kernels read the owned copy), the copy outlives the source buffer, the
size must be the planned one, and the B-less execute is rejected when the
plan owns no B."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import GemmPlan, OlcError, Plan, binding, synth
from parity import compare, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["float32", "float64", "float16", "bfloat16"])
@pytest.mark.parametrize("shapes", [((8, 2048, 512), (512, 1024)), ((4, 4096), (4096, 2048)),
                                    ((2, 64, 96), (2, 96, 40)), ((300, 8192), (8192, 8))],
                         ids=lambda s: "x".join(map(str, s[0] + s[1])))
@pytest.mark.parametrize("source", ["device", "host"])
def test_constant_b_matches_per_call_b(dtype, shapes, source):
    a, b = synth.operands(shapes[0], shapes[1], dtype, synth.UNIFORM, synth.UNIFORM, seed=2)
    A = a.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        Y1 = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
        Y2 = torch.empty_like(Y1)
        p.execute(A, b.cuda(), Y1)
        src = b.cuda() if source == "device" else b.clone().pin_memory()
        p.set_constant_b(src)
        assert p.has_constant_b
        src.fill_(7)          # the plan's copy must not depend on the source
        del src
        p.execute_constant(A, Y2)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2)
    _check_against_oracle(a, b, Y2.cpu(), dtype)


def _check_against_oracle(a, b, y, dtype):
    """The constant-B result against the oracle: on sampled rows of the
    folded product when B is one matrix, in full otherwise."""
    an, bn = synth.to_numpy_storage(a), synth.to_numpy_storage(b)
    if b.dim() == 2 and an.size // an.shape[-1] > 512:
        k = an.shape[-1]
        a2 = an.reshape(-1, k)
        rows = sample_rows(a2.shape[0], extra=64)
        y_ref, s = oracle.gemm2d(a2, bn, dtype, rows=rows)
        compare(y.reshape(-1, bn.shape[-1])[rows], y_ref, s, dtype)
    else:
        y_ref, s = oracle.matmul(an, bn, dtype)
        compare(y, y_ref, s, dtype)


def test_constant_b_rejections():
    with Plan((16, 32), (32, 24), "float32") as p:
        A = torch.zeros(16, 32, device="cuda")
        Y = torch.zeros(16, 24, device="cuda")
        assert not p.has_constant_b
        with pytest.raises(OlcError) as ei:
            p.execute_constant(A, Y)
        assert ei.value.name == "OLC_ERR_NO_CONSTANT_B"
        with pytest.raises(OlcError) as ei:
            p.set_constant_b(torch.zeros(32, 23, device="cuda"))   # not the planned B
        assert ei.value.name == "OLC_ERR_BUFFER_TOO_SMALL"
        assert not p.has_constant_b


def test_gemm_constant_b_with_bias():
    a, b = synth.operands((96, 512), (256, 512), "bfloat16", synth.UNIFORM, synth.UNIFORM, 4)
    c, _ = synth.operands((256,), (1,), "bfloat16", synth.UNIFORM, synth.UNIFORM, 5)
    A, C = a.cuda(), c.cuda()
    with GemmPlan(a.shape, b.shape, "bfloat16", False, True, 0.5, 2.0, c.shape) as p:
        Y1 = torch.empty(96, 256, dtype=torch.bfloat16, device="cuda")
        Y2 = torch.empty_like(Y1)
        p.execute(A, b.cuda(), Y1, C=C)
        p.set_constant_b(b)
        p.execute_constant(A, Y2, C=C)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2)
    y_ref, s = oracle.gemm_op(synth.to_numpy_storage(a), synth.to_numpy_storage(b), "bfloat16",
                              c=synth.to_numpy_storage(c), alpha=0.5, beta=2.0, trans_a=False,
                              trans_b=True)
    compare(Y2.cpu(), y_ref, s, "bfloat16")
