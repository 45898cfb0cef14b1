"""Brute force on tiny products: every M, N, K in {0, 1, 2, 3, 5, 8, 17},
each with one of four batch patterns (none, equal batches, broadcast both
ways, rank 3 with 1s sprinkled), in every type, through every algorithm the
plan accepts for the shape (forced), on integer inputs compared bit for bit
with the oracle.  Outputs are written into canary-guarded buffers."""

import itertools

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import OlcError, Plan, synth
from parity import compare

pytestmark = pytest.mark.gpu

SIZES = [0, 1, 2, 3, 5, 8, 17]
BATCHES = [((), ()), ((2,), (2,)), ((1, 3), (2, 1)), ((2, 1, 2), (1, 3, 1))]
ALGOS = ["direct", "general_simt", "skinny_m", "skinny_n", "split_k", "general_tc"]


@pytest.mark.parametrize("dtype", ["float32", "float64", "float16", "bfloat16", "float8_e4m3fn"])
def test_every_tiny_shape_every_algorithm(dtype):
    ran = 0
    for i, (m, n, k) in enumerate(itertools.product(SIZES, SIZES, SIZES)):
        ab, bb = BATCHES[i % len(BATCHES)]
        a_shape, b_shape = ab + (m, k), bb + (k, n)
        a, b = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=i)
        y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        A, B = a.cuda(), b.cuda()
        ydt = synth.TORCH_DTYPES[synth.output_dtype(dtype)]
        for algo in ALGOS + [None]:
            with Plan(a_shape, b_shape, dtype) as p:
                if algo is not None:
                    try:
                        p.force(algo)
                    except OlcError:
                        continue
                count = int(np.prod(p.output_shape, dtype=np.int64))
                buf = torch.full((count + 16,), float("nan"), dtype=ydt, device="cuda")
                Y = buf[:count].view(p.output_shape)
                p.execute_checked(A, B, Y)
                torch.cuda.synchronize()
                assert torch.isnan(buf[count:].float()).all(), "write past Y: %s %s %s" % (
                    a_shape, b_shape, p.algorithm)
                if count:
                    compare(Y.cpu(), y_ref, s, dtype, exact=True)
                ran += 1
    assert ran >= len(SIZES) ** 3
