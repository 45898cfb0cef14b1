"""The narrowing contract on the device: NaN stays NaN, infinities keep their
sign, and a float32 sum beyond FLOAT16's range becomes an infinity, through
every kernel family ("MatMul Kernel Design", section "Types and algorithm
selection": FLOAT16 / BFLOAT16 accumulate in float32 and narrow once; "Gemm
and MatMul Performance Roadmap", the PR10.3 tuning record: the scalar
contract for NaNs and tails holds on every path).

Inputs are small integers (exact float32 sums, so every finite output is
bit-exact) with planted special values:
  - one NaN in A (row NAN_ROW): that whole output row is NaN;
  - one +Inf in A (row 1) and one -Inf in B (last row, last column): +-Inf
    where the infinity meets a non-zero factor, NaN where it meets a zero or
    where +Inf and -Inf terms meet;
  - row 2 of A all ones, and B's columns 0..4 built so that row 2's exact
    sums are 65520, 65519, -65520, 65504 and 67583: FLOAT16 must give +inf,
    65504, -inf, 65504 and +inf (65520 is the tie between 65504 and 2^16, and
    round-to-nearest-even goes to 2^16, i.e. inf); BFLOAT16 stays finite.
    B's other rows hold 2047s in these columns, so most other rows overflow
    FLOAT16 too.
FLOAT and DOUBLE run the same inputs (no narrowing; NaN and Inf propagate).
Each output is compared with the oracle element by element: NaN exactly where
the oracle has NaN, equal infinities, equal finite values."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import OlcError, Plan, synth
from parity import compare, gpu_matmul

pytestmark = pytest.mark.gpu

# (A shape, B shape, forced algorithm, kernel-family variant or None).  The
# variants pick the kernels behind one algorithm: skinny-M 1 = SIMT
# streaming, 2 = swapped-operand tcgen05; skinny-N 1 = tcgen05 16-column
# tiles, 2 = register-streaming mma.sync; general_tc 1 = one CTA per
# 128 x 256 tile, 2 = CTA pairs (cta_group::2, 256 x 256 tiles).
CASES = [
    ((40, 72), (72, 24), "direct", None),
    ((130, 200), (200, 72), "general_simt", None),
    ((4, 8192), (8192, 512), "skinny_m", 1),
    ((4, 8192), (8192, 512), "skinny_m", 2),
    ((600, 4096), (4096, 8), "skinny_n", 1),
    ((600, 4096), (4096, 8), "skinny_n", 2),
    ((32, 16384), (16384, 32), "split_k", None),      # small-output cluster kernel
    ((300, 5000), (5000, 264), "split_k", None),      # tcgen05 split tiles
    ((300, 520), (520, 264), "general_tc", 1),
    ((512, 256), (256, 512), "general_tc", 2),
    ((3, 1, 130, 64), (1, 2, 64, 136), "general_tc", None),   # broadcast batch
]

NAN_ROW_FROM_END = 1          # the NaN sits in the last row (a tail tile)
# row 2's target sums (A row of ones) and what FLOAT16 narrowing gives
TARGETS = [65520.0, 65519.0, -65520.0, 65504.0, 67583.0]
F16_EXPECT = [np.inf, 65504.0, -np.inf, 65504.0, np.inf]


def _plant(a_cpu: torch.Tensor, b_cpu: torch.Tensor, dtype: str):
    """Special values in every batch item of A [..., M, K] and B [..., K, N]
    (small-integer draws, modified in float64 and cast back to the storage
    type with round-to-nearest-even)."""
    a = a_cpu.double().clone()
    b = b_cpu.double().clone()
    m, k = a.shape[-2], a.shape[-1]
    n = b.shape[-1]
    a[..., m - NAN_ROW_FROM_END, k // 2] = float("nan")
    a[..., 1, 3] = float("inf")
    a[..., 2, :] = 1.0
    for j, t in enumerate(TARGETS[:n]):
        col = torch.zeros(k, dtype=torch.float64)
        big = 2047.0 if t > 0 else -2047.0
        col[:32] = big
        col[32] = t - 32 * big
        b[..., :, j] = col
    b[..., k - 1, n - 1] = float("-inf")
    tdt = synth.TORCH_DTYPES[dtype]
    return a.to(tdt), b.to(tdt)


def _feasible(a_shape, b_shape, dtype, algo):
    try:
        with Plan(a_shape, b_shape, dtype) as p:
            p.force(algo)
        return True
    except OlcError:
        return False


@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32", "float64"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-v%s-%s" % (
    c[2], c[3], "x".join(map(str, c[0] + c[1]))))
def test_special_values_follow_the_oracle(dtype, case):
    a_shape, b_shape, algo, variant = case
    if not _feasible(a_shape, b_shape, dtype, algo):
        pytest.skip("%s does not take %s" % (algo, dtype))
    if variant is not None and dtype not in ("float16", "bfloat16"):
        if variant == 2:
            pytest.skip("kernel-family variants select among 16-bit kernels")
        variant = None
    a0, b0 = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=21)
    a, b = _plant(a0, b0, dtype)
    # 0.5 is no correct output here (all finite outputs are integers), so an
    # element the kernel never wrote cannot pass
    y, got = gpu_matmul(a, b, dtype, algo, variant=variant, fill=0.5)
    assert got == algo
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(y, y_ref, s, dtype, exact=True)

    yg = oracle.to_float64(synth.to_numpy_storage(y), dtype).reshape(y_ref.shape)
    m = a_shape[-2]
    # the NaN in A turns its whole output row to NaN
    assert np.isnan(yg[..., m - NAN_ROW_FROM_END, :]).all()
    row2 = yg[..., 2, :len(TARGETS)]
    if dtype == "float16":
        want = np.broadcast_to(np.array(F16_EXPECT[:row2.shape[-1]]), row2.shape)
        assert np.array_equal(row2, want), row2
    elif dtype == "bfloat16":
        assert np.isfinite(row2).all()
    else:
        # the targets are exact for FLOAT and DOUBLE (2047 and the remainders
        # are exact there); the last column may meet B's -Inf in row 2
        want = np.broadcast_to(np.array(TARGETS[:row2.shape[-1]]), row2.shape)
        cols = row2.shape[-1] if b_shape[-1] - 1 >= len(TARGETS) else row2.shape[-1] - 1
        assert np.array_equal(row2[..., :cols], want[..., :cols]), row2


@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_overflow_to_inf_in_the_pair_kernel_at_size(dtype):
    """A product large enough for many CTA-pair tiles per cluster, with
    integer operands whose exact sums pass FLOAT16's range in a seeded set
    of rows and columns: bit-exact with the oracle on sampled rows."""
    m, k, n = 2048, 1024, 2048
    a0, b0 = synth.operands((m, k), (k, n), dtype, synth.SMALL_INT, synth.SMALL_INT, seed=22)
    a, b = a0.double(), b0.double()
    rng = np.random.default_rng(22)
    rows = rng.choice(m, size=64, replace=False)
    a[rows, :64] = 64.0                       # 64 * 64 * 3 * ... : beyond 65504
    b[:64, :] = torch.where(b[:64, :] == 0, torch.ones_like(b[:64, :]), b[:64, :]) * 64.0
    tdt = synth.TORCH_DTYPES[dtype]
    a, b = a.to(tdt), b.to(tdt)
    y, got = gpu_matmul(a, b, dtype, "general_tc", variant=2, fill=0.5, guard=16)
    assert got == "general_tc"
    yg_rows = np.sort(np.concatenate([rows, rng.choice(m, size=64, replace=False), [0, m - 1]]))
    yg_rows = np.unique(yg_rows)
    y_ref, s = oracle.gemm2d(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                             rows=yg_rows)
    compare(y[yg_rows], y_ref, s, dtype, exact=True)
    ygv = oracle.to_float64(synth.to_numpy_storage(y[yg_rows]), dtype)
    if dtype == "float16":
        assert np.isinf(ygv).sum() > 1000       # the planted rows overflow
    else:
        assert np.isfinite(ygv).all()
