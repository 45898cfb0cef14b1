"""Shared helpers for the GPU parity tests: run a product through the C ABI,
compute the oracle on the same seeded inputs, compare element by element.

Tolerances: |y_gpu - y_oracle| <= tol * sum_k |a||b| per element, with tol =
1e-5 (FLOAT), 1e-12 (DOUBLE), 2e-3 (FLOAT16), 1e-2 (BFLOAT16).  Integer-valued
inputs whose sums are exact in the accumulator must match bit for bit.

Special values follow the oracle exactly: an output is NaN where, and only
where, the oracle's is NaN, and an infinite output must be the oracle's
infinity with its sign ("MatMul Kernel Design", section "Types and algorithm
selection": float32 accumulation, then one narrowing; NaN stays NaN and a sum
beyond the output type's range becomes an infinity)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import Plan
from gemm_matmulplan_broadcast_gb300 import synth

TOL = {"float32": 1e-5, "float64": 1e-12, "float16": 2e-3, "bfloat16": 1e-2,
       # 8-bit float operands: exact products, float32 sums, float32 output
       "float8_e4m3fn": 1e-5, "float8_e5m2": 1e-5, "float8_e4m3fnuz": 1e-5,
       "float8_e5m2fnuz": 1e-5}


def gpu_matmul(a_cpu: torch.Tensor, b_cpu: torch.Tensor, dtype: str, algorithm=None,
               checked=True, guard=64, variant=None, fill=float("nan")):
    """Y = MatMul(A, B) through the library (kernel-family override `variant`
    if given); Y is allocated filled with `fill`, with `guard` trailing canary
    elements of that value that must stay untouched.  Products whose correct
    output holds NaNs pass a finite `fill` that no correct output takes, so
    that an unwritten element still shows.  Returns (Y on CPU, plan
    algorithm)."""
    A = a_cpu.cuda()
    B = b_cpu.cuda()
    with Plan(a_cpu.shape, b_cpu.shape, dtype) as p:
        if algorithm is not None:
            p.force(algorithm)
        if variant is not None:
            p.set_tc_variant(variant)
        shape = p.output_shape
        n = int(np.prod(shape, dtype=np.int64))
        buf = torch.full((n + guard,), fill, dtype=synth.TORCH_DTYPES[synth.output_dtype(dtype)], device="cuda")
        Y = buf[:n].view(shape)
        if checked:
            p.execute_checked(A, B, Y)
        else:
            p.execute(A, B, Y)
        torch.cuda.synchronize()
        tail = buf[n:].double().cpu()
        if np.isnan(fill):
            assert torch.isnan(tail).all(), "kernel wrote past the end of Y"
        else:
            want = torch.tensor(fill, dtype=buf.dtype).double()
            assert bool((tail == want).all()), "kernel wrote past the end of Y"
        return Y.cpu(), p.algorithm


def compare(y_gpu: torch.Tensor, y_ref: np.ndarray, s: np.ndarray, dtype: str, exact=False):
    """Element-by-element comparison; returns the largest error / (tol * S).
    NaN must appear exactly where the oracle has NaN (with the usual NaN
    fill of gpu_matmul an unwritten element therefore fails), an infinity
    must equal the oracle's, and finite outputs must be within tol * S (equal
    with `exact`)."""
    yg = oracle.to_float64(synth.to_numpy_storage(y_gpu), dtype).reshape(y_ref.shape)
    yr = oracle.to_float64(y_ref, dtype)
    assert yg.shape == yr.shape
    nan_g, nan_r = np.isnan(yg), np.isnan(yr)
    if (nan_g != nan_r).any():
        i = tuple(np.argwhere(nan_g != nan_r)[0])
        raise AssertionError("NaN pattern differs (unwritten or wrong) at %s: gpu %r oracle %r" % (
            i, yg[i], yr[i]))
    inf = ~nan_r & (np.isinf(yg) | np.isinf(yr))
    if inf.any() and (yg[inf] != yr[inf]).any():
        i = tuple(np.argwhere(inf & (yg != yr))[0])
        raise AssertionError("infinity differs at %s: gpu %r oracle %r" % (i, yg[i], yr[i]))
    fin = ~nan_r & ~inf
    if exact:
        bad = np.argwhere(fin & (yg != yr))
        assert bad.size == 0, "first mismatch at %s: gpu %r oracle %r" % (
            tuple(bad[0]), yg[tuple(bad[0])], yr[tuple(bad[0])])
        return 0.0
    yg, yr = np.where(fin, yg, 0.0), np.where(fin, yr, 0.0)
    s = np.where(fin, s, 0.0)
    err = np.abs(yg - yr)
    bound = TOL[dtype] * s
    ok = err <= bound
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError("parity: at %s gpu %r oracle %r |err| %g > tol*S %g" % (
            i, yg[i], yr[i], err[i], bound[i]))
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / np.where(bound > 0, bound, 1), 0)
    return float(r.max()) if r.size else 0.0


def check_product(a_cpu, b_cpu, dtype, algorithm=None, exact=False, variant=None):
    y, algo = gpu_matmul(a_cpu, b_cpu, dtype, algorithm, variant=variant)
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a_cpu), synth.to_numpy_storage(b_cpu), dtype)
    compare(y, y_ref, s, dtype, exact=exact)
    return y, algo


def sample_rows(m: int, band: int = 128, extra: int = 256, seed: int = 0):
    """Rows 0 and m-1, the first and last row of every `band`-row band (at most
    256 of them, spread evenly), plus `extra` seeded random rows."""
    rows = {0, m - 1}
    bands = list(range(0, m, band))
    if len(bands) > 128:
        idx = np.linspace(0, len(bands) - 1, 128).round().astype(int)
        bands = [bands[i] for i in idx]
    for b in bands:
        rows.add(b)
        rows.add(min(m - 1, b + band - 1))
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, m, size=min(extra, m)).tolist())
    return sorted(rows)
