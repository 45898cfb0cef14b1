"""Grouped products on the GPU against the oracle: hundreds of members of
irregular shapes in one launch, every type, integer inputs bit for bit,
empty and K == 0 members, and repeated execution."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import GroupedPlan, synth
from parity import compare

pytestmark = pytest.mark.gpu


def _members(count, seed, lo=1, hi=200):
    rng = np.random.default_rng(seed)
    return [tuple(int(x) for x in rng.integers(lo, hi + 1, size=3)) for _ in range(count)]


def _run(shapes, dtype, dist, seed):
    As, Bs = [], []
    for i, (m, n, k) in enumerate(shapes):
        a, b = synth.operands((m, k), (k, n), dtype, dist, dist if dist is synth.SMALL_INT else synth.normal(0.1), seed + i)
        As.append(a)
        Bs.append(b)
    tdt = synth.TORCH_DTYPES[dtype]
    with GroupedPlan(shapes, dtype) as g:
        Ys = [torch.full((m, n), float("nan"), dtype=tdt, device="cuda") for m, n, k in shapes]
        g.execute([a.cuda() for a in As], [b.cuda() for b in Bs], Ys)
        torch.cuda.synchronize()
    refs, ss = oracle.grouped([synth.to_numpy_storage(a) for a in As],
                              [synth.to_numpy_storage(b) for b in Bs], dtype)
    return Ys, refs, ss


@pytest.mark.parametrize("dtype", ["float32", "float64", "float16", "bfloat16"])
def test_grouped_irregular_members(dtype):
    shapes = _members(300, 5)
    Ys, refs, ss = _run(shapes, dtype, synth.UNIFORM, 100)
    for y, r, s in zip(Ys, refs, ss):
        compare(y.cpu(), r, s, dtype)


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_grouped_integers_bit_exact_with_empty_members(dtype):
    shapes = _members(64, 7, 1, 130) + [(0, 5, 7), (6, 0, 3), (9, 4, 0), (1, 1, 1), (65, 129, 257)]
    Ys, refs, ss = _run(shapes, dtype, synth.SMALL_INT, 200)
    for y, r, s in zip(Ys, refs, ss):
        compare(y.cpu(), r, s, dtype, exact=True)


def test_grouped_repeated_and_tile_count():
    shapes = [(64, 64, 64), (65, 1, 8), (1, 200, 3)]
    with GroupedPlan(shapes, "float32") as g:
        assert g.tiles == 1 + 2 + 4
        a = [torch.randn(m, k, device="cuda") for m, n, k in shapes]
        b = [torch.randn(k, n, device="cuda") for m, n, k in shapes]
        y1 = [torch.empty(m, n, device="cuda") for m, n, k in shapes]
        y2 = [torch.empty(m, n, device="cuda") for m, n, k in shapes]
        g.execute(a, b, y1)
        g.execute(a, b, y2)
        torch.cuda.synchronize()
        for p, q in zip(y1, y2):
            assert torch.equal(p, q)
