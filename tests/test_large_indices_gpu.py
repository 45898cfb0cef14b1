"""Products whose element offsets pass 2^31 (64-bit index arithmetic in the
kernels): a 4 GB FP16 A through the skinny-N streaming kernel, an 8 GB BF16
output from the CTA-pair kernel, a 16 GB FLOAT output from the SIMT kernel.
Parity on sampled rows (the first and last row of every 128-row band, rows 0
and M - 1, and seeded random rows), each computed by the oracle."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import Plan, synth
from parity import TOL, sample_rows

pytestmark = pytest.mark.gpu


def _sampled(a_shape, b_shape, dtype, expect_algo):
    a, b = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.normal(1.0), seed=77)
    with Plan(a_shape, b_shape, dtype) as p:
        assert p.algorithm == expect_algo
        Y = torch.empty(p.output_shape, dtype=a.dtype, device="cuda")
        p.execute(a.cuda(), b.cuda(), Y)
        torch.cuda.synchronize()
    m = a_shape[0]
    rows = sample_rows(m, extra=64, seed=5)
    an, bn = synth.to_numpy_storage(a), synth.to_numpy_storage(b)
    ref, s = oracle.gemm2d(an, bn, dtype, rows=rows)
    got = oracle.to_float64(synth.to_numpy_storage(Y[torch.tensor(rows, device="cuda")].cpu()), dtype)
    err = np.abs(got - oracle.to_float64(ref, dtype))
    assert np.all(err <= TOL[dtype] * s), "max err %g" % float(err.max())
    del Y
    torch.cuda.empty_cache()


def test_skinny_n_a_of_2_pow_31_elements():
    _sampled((262144, 8192), (8192, 8), "float16", "skinny_n")


def test_pair_kernel_output_of_2_pow_32_elements():
    _sampled((131072, 64), (64, 32768), "bfloat16", "general_tc")


def test_simt_output_of_2_pow_32_elements():
    _sampled((65536, 64), (64, 65536), "float32", "general_simt")
