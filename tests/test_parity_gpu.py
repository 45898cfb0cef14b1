"""GPU parity: the CUDA path (through the C ABI) against the oracle on the same
seeded inputs, for every named workload, every algorithm on small ragged
shapes, and the edge cases (empty outputs, K == 0, rank-one operands,
broadcast batches, unaligned pointers, buffer checks)."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import OlcError, Plan, synth
from parity import TOL, check_product, compare, gpu_matmul, sample_rows

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "float64", "float16", "bfloat16"]


# --------------------------------------------------------------------------
# the named workloads at their own sizes


def test_fp32_64x128x96_uniform_and_exact_integers():
    w = synth.workload("fp32_64x128x96")
    for prod in w.products:
        a, b = prod.draw()
        check_product(a, b, prod.dtype, exact=(prod.name == "small_int"))


def test_fp32_broadcast_batch_and_rank_one_and_empty():
    w = synth.workload("fp32_broadcast_batch")
    for prod in w.products:
        a, b = prod.draw()
        y, algo = check_product(a, b, prod.dtype)
        assert y.shape == oracle.output_shape(prod.a_shape, prod.b_shape)
        if prod.name == "empty_batch":
            assert algo == "empty" and y.numel() == 0


@pytest.mark.parametrize("algorithm", [None, "direct", "general_simt"])
def test_broadcast_equals_explicit_repeat_bit_exact(algorithm):
    a, b = synth.operands((8, 1, 128, 256), (1, 4, 256, 64), "float32", synth.UNIFORM,
                          synth.UNIFORM, seed=1)
    y_bc, _ = gpu_matmul(a, b, "float32", algorithm)
    ar = a.expand(8, 4, 128, 256).contiguous()
    br = b.expand(8, 4, 256, 64).contiguous()
    y_rep, _ = gpu_matmul(ar, br, "float32", algorithm)
    assert torch.equal(y_bc, y_rep)


def test_bf16_transformer_projection_sampled_rows():
    w = synth.workload("bf16_transformer_projection")
    for prod in w.products:
        a, b = prod.draw()
        y, algo = gpu_matmul(a, b, prod.dtype, checked=True, guard=16)
        k = prod.a_shape[-1]
        a2 = synth.to_numpy_storage(a).reshape(-1, k)
        rows = sample_rows(a2.shape[0], seed=len(prod.name))
        y_ref, s = oracle.gemm2d(a2, synth.to_numpy_storage(b), prod.dtype, rows=rows)
        y2 = y.reshape(-1, prod.b_shape[-1])[rows]
        compare(y2, y_ref, s, prod.dtype)


def test_fp16_skinny_and_split_k_full():
    w = synth.workload("fp16_skinny_splitk")
    want = {"skinny_m": "skinny_m", "skinny_n": "skinny_n", "split_k": "split_k"}
    for prod in w.products:
        a, b = prod.draw()
        y, algo = check_product(a, b, prod.dtype)
        assert algo == want[prod.name]


@pytest.mark.parametrize("dtype", ["float32", "float64"])
def test_square_sweep_and_chain(dtype):
    w = synth.workload("%s_square_chain" % dtype)
    for prod in w.products:
        a, b = prod.draw()
        y, _ = gpu_matmul(a, b, dtype, guard=16)
        rows = None if prod.a_shape[0] <= 1024 else sample_rows(prod.a_shape[0], extra=64)
        y_ref, s = oracle.gemm2d(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                                 rows=rows)
        compare(y if rows is None else y[rows], y_ref, s, dtype)
    # the chain: every stage on the GPU feeds the next; the oracle runs its
    # own chain on the sampled rows (row i of each stage depends only on row i
    # of the previous one).  The bound adds the previous stage's propagated
    # tolerance: tol * (S_prev @ |W|).
    (chain,) = w.chains
    xs = chain.draw()
    cur = xs[0].cuda()
    rows = sample_rows(chain.shapes[0][0], extra=64)
    ref = synth.to_numpy_storage(xs[0])[rows]
    prev_bound = np.zeros(ref.shape)
    for wt in xs[1:]:
        with Plan(tuple(cur.shape), tuple(wt.shape), dtype) as p:
            out = torch.empty(p.output_shape, dtype=cur.dtype, device="cuda")
            p.execute(cur, wt.cuda(), out)
        cur = out
        wn = synth.to_numpy_storage(wt)
        ref, s = oracle.gemm2d(ref, wn, dtype)
        bound = TOL[dtype] * s + prev_bound @ np.abs(wn)
        yg = cur.cpu().numpy()[rows].astype(np.float64)
        err = np.abs(yg - ref)
        assert np.all(err <= bound), float((err / bound).max())
        prev_bound = bound


# --------------------------------------------------------------------------
# every algorithm on small ragged shapes

ALGOS = ["direct", "general_simt", "skinny_m", "skinny_n", "split_k", "general_tc"]

SMALL_SHAPES = [
    ((1, 8), (8, 16)),
    ((3, 40), (40, 24)),
    ((16, 72), (72, 64)),
    ((17, 65), (65, 255)),
    ((127, 129), (129, 33)),
    ((129, 64), (64, 257)),
    ((200, 3000), (3000, 8)),
    ((33, 9000), (9000, 40)),
    ((2, 3, 5, 16), (3, 16, 24)),
    ((5, 1, 7, 40), (1, 3, 40, 16)),
    ((64,), (64, 48)),
    ((3, 80, 64), (64,)),
    ((2, 1, 2, 1, 2, 1, 5, 24), (1, 2, 1, 2, 1, 2, 24, 16)),   # rank 8: 64 broadcast items
]


def _feasible(a_shape, b_shape, dtype, algo):
    try:
        with Plan(a_shape, b_shape, dtype) as p:
            p.force(algo)
        return True
    except OlcError:
        return False


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shapes", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_every_algorithm_uniform(dtype, shapes):
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.UNIFORM, synth.UNIFORM, seed=7)
    ran = 0
    for algo in ALGOS:
        if _feasible(a_shape, b_shape, dtype, algo):
            check_product(a, b, dtype, algorithm=algo)
            ran += 1
    assert ran >= 2


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shapes", SMALL_SHAPES[:9], ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_every_algorithm_integers_bit_exact(dtype, shapes):
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=8)
    for algo in ALGOS:
        if _feasible(a_shape, b_shape, dtype, algo):
            check_product(a, b, dtype, algorithm=algo, exact=True)


@pytest.mark.parametrize("algo,shapes", [
    ("split_k", ((32, 131072), (131072, 32))),
    ("skinny_m", ((4, 8192), (8192, 28672))),
])
def test_split_reductions_are_reproducible(algo, shapes):
    a, b = synth.operands(shapes[0], shapes[1], "float16", synth.normal(1.0), synth.normal(0.02),
                          seed=3)
    y1, _ = gpu_matmul(a, b, "float16", algo)
    y2, _ = gpu_matmul(a, b, "float16", algo)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


# --------------------------------------------------------------------------
# the tensor-core path: one tile first, then tails, batches, many tiles


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_tc_single_tile(dtype):
    a, b = synth.operands((128, 64), (64, 256), dtype, synth.SMALL_INT, synth.SMALL_INT, seed=1)
    y, algo = check_product(a, b, dtype, algorithm="general_tc", exact=True)
    assert algo == "general_tc"


TC_SHAPES = [
    ((128, 128), (128, 256)),
    ((300, 520), (520, 264)),        # M, N and K tails
    ((1, 8), (8, 8)),
    ((129, 4104), (4104, 520)),
    ((3, 1, 130, 64), (1, 2, 64, 136)),   # broadcast batch through 3-D tensor maps
    ((2, 3, 40, 32), (3, 32, 24)),
    ((64,), (64, 48)),
]


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("shapes", TC_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_tc_shapes(dtype, shapes):
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.02), seed=9)
    check_product(a, b, dtype, algorithm="general_tc")
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=9)
    check_product(ai, bi, dtype, algorithm="general_tc", exact=True)


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("variant", [1, 2])
def test_tc_many_tiles_per_cta_sampled(dtype, variant):
    # 32 x 8 = 256 tiles of 128 x 256 (128 pair tiles): more than one tile per
    # CTA or CTA pair, both TMEM accumulators in use
    a, b = synth.operands((4096, 1024), (1024, 2048), dtype, synth.normal(1.0),
                          synth.normal(0.02), seed=10)
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        p.force("general_tc")
        p.set_tc_variant(variant)
        Y = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
        p.execute_checked(A, B, Y)
    y = Y.cpu()
    rows = sample_rows(4096, extra=128)
    y_ref, s = oracle.gemm2d(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                             rows=rows)
    compare(y[rows], y_ref, s, dtype)


TC_SPLIT_SHAPES = [
    ((32, 131072), (131072, 32)),      # the FP16 corner's split-K product
    ((17, 8008), (8008, 24)),          # row and K tails of the streaming kernel
    ((1, 65536), (65536, 8)),          # one row, one 8-column plane
    ((32, 4096), (4096, 32)),          # 32-column tiles
    ((40, 20000), (20000, 24)),        # 32-column tiles, N tail
    ((16, 9000), (9000, 16)),          # 16-column tiles
    ((8, 3000), (3000, 8)),
    ((32, 1536), (1536, 32)),          # clusters of 4 CTAs
    ((24, 640), (640, 16)),            # clusters of 2 CTAs
    ((300, 5000), (5000, 264)),        # 256-column tiles, several tiles
    ((2, 24, 2048), (2048, 40)),       # folded batch
    ((3, 24, 1024), (3, 1024, 32)),    # batched B
]


def _split_product(a, b, dtype, variant, exact):
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        p.force("split_k")
        p.set_tc_variant(variant)
        n = int(np.prod(p.output_shape))
        buf = torch.full((n + 64,), float("nan"), dtype=A.dtype, device="cuda")
        Y = buf[:n].view(p.output_shape)
        p.execute_checked(A, B, Y)
        Y2 = torch.empty_like(Y)
        p.execute_checked(A, B, Y2)          # reproducible: the reduction order is fixed
        torch.cuda.synchronize()
        assert torch.isnan(buf[n:].float()).all()
        assert torch.equal(Y, Y2)
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(Y.cpu(), y_ref, s, dtype, exact=exact)


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("shapes", TC_SPLIT_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_tc_split_k(dtype, shapes):
    """FLOAT16 / BFLOAT16 split-K (the small mma.sync ring for one item of at
    most 32 x 32 outputs, tcgen05 split tiles otherwise): parity, integer
    inputs bit for bit, and two runs identical."""
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.02), seed=12)
    _split_product(a, b, dtype, 0, exact=False)
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=12)
    _split_product(ai, bi, dtype, 0, exact=True)


@pytest.mark.parametrize("splits", [2, 5, 13, 24, 64, 200])
def test_tiny_split_k_slice_counts(splits):
    """The small-output split-K kernel with requested slice counts (clusters
    of 2, 4 and 8 CTAs, more clusters than run at once): integer inputs bit
    for bit, normal inputs within the bound, two runs identical."""
    shapes = ((32, 16384), (16384, 32))
    for dist_a, dist_b, exact in [(synth.SMALL_INT, synth.SMALL_INT, True),
                                  (synth.normal(1.0), synth.normal(0.02), False)]:
        a, b = synth.operands(shapes[0], shapes[1], "float16", dist_a, dist_b, seed=13)
        A, B = a.cuda(), b.cuda()
        with Plan(a.shape, b.shape, "float16") as p:
            p.force("split_k")
            p.set_splits(splits)
            assert p.splits >= 2
            Y = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
            Y2 = torch.empty_like(Y)
            p.execute_checked(A, B, Y)
            p.execute_checked(A, B, Y2)
            torch.cuda.synchronize()
            assert torch.equal(Y, Y2)
        y_ref, sabs = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), "float16")
        compare(Y.cpu(), y_ref, sabs, "float16", exact=exact)


@pytest.mark.parametrize("splits", [0, 1, 2, 3, 7, 16])
def test_fp32_simt_k_slices(splits):
    """FLOAT products with fewer 128 x 128 tiles than SMs run K slices whose
    partial tiles the last slice sums in slice order: integer inputs bit for
    bit, normal inputs within the bound, two runs identical; 0 is the
    automatic choice, 1 no slicing."""
    shapes = ((2, 200, 2048), (2048, 392))
    for dist, exact in [(synth.SMALL_INT, True), (synth.UNIFORM, False)]:
        a, b = synth.operands(shapes[0], shapes[1], "float32", dist, dist, seed=14)
        A, B = a.cuda(), b.cuda()
        with Plan(a.shape, b.shape, "float32") as p:
            p.force("general_simt")
            p.set_splits(splits)
            if splits == 1:
                assert p.splits == 1
            elif splits > 1:
                assert p.splits > 1
            Y = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
            Y2 = torch.empty_like(Y)
            p.execute_checked(A, B, Y)
            p.execute_checked(A, B, Y2)
            torch.cuda.synchronize()
            assert torch.equal(Y, Y2)
        y_ref, sabs = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), "float32")
        compare(Y.cpu(), y_ref, sabs, "float32", exact=exact)


FP32_SIMT_SHAPES = [
    ((128, 16), (16, 128)),            # one tile, one slice
    ((300, 1000), (1000, 260)),        # M, N, K tails (K, N multiples of 4)
    ((3, 1, 130, 68), (1, 2, 68, 132)),   # broadcast batch through 3-D tensor maps
    ((8, 2048, 256), (256, 512)),      # folded batch, many tiles
    ((64,), (64, 48)),                 # rank-one A
]


@pytest.mark.parametrize("shapes", FP32_SIMT_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_fp32_simt_register_tiles(shapes):
    """The FLOAT register-tile kernel on tails, batches and a rank-one A:
    integer inputs bit for bit, uniform inputs within the bound."""
    a_shape, b_shape = shapes
    for dist, exact in [(synth.SMALL_INT, True), (synth.UNIFORM, False)]:
        a, b = synth.operands(a_shape, b_shape, "float32", dist, dist, seed=16)
        check_product(a, b, "float32", algorithm="general_simt", exact=exact)


def test_fp32_square_1024_sampled():
    """The 1024-cube FLOAT product (64 tiles: sliced over K automatically)
    on sampled rows."""
    a, b = synth.operands((1024, 1024), (1024, 1024), "float32", synth.UNIFORM, synth.UNIFORM, seed=4)
    with Plan(a.shape, b.shape, "float32") as p:
        assert p.algorithm == "general_simt"
        assert p.splits > 1
        A, B = a.cuda(), b.cuda()
        Y = torch.empty(1024, 1024, device="cuda")
        p.execute_checked(A, B, Y)
    rows = sample_rows(1024, extra=64)
    y_ref, sabs = oracle.gemm2d(synth.to_numpy_storage(a), synth.to_numpy_storage(b), "float32",
                                rows=rows)
    compare(Y.cpu()[rows], y_ref, sabs, "float32")


TC_SKINNY_N_SHAPES = [
    ((4096, 1024), (1024, 8)),         # 32 row tiles: stream-K shares over the SMs
    ((16384, 4096), (4096, 8)),        # the FP16 corner's skinny-N product
    ((1000, 6144), (6144, 5)),         # widest K whose transposed B fits; row tail; N < 8
    ((777, 8200), (8200, 12)),         # K too long for the staged B: tcgen05 kernel
    ((3, 50, 40), (40, 3)),            # K not a multiple of 32, tiny rows per item
    ((2, 2048, 512), (512, 16)),       # folded batch, stream-K
    ((256, 1024), (1024, 8)),
    ((1000, 520), (520, 16)),
    ((3, 200, 64), (64, 8)),
    ((2, 130, 72), (2, 72, 16)),
]


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("shapes", TC_SKINNY_N_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
@pytest.mark.parametrize("variant", [0, 1, 2], ids=["auto", "tcgen05", "mma_sync_stream"])
def test_tc_skinny_n(dtype, shapes, variant):
    """Both FLOAT16 / BFLOAT16 skinny-N kernels: the register-streaming
    mma.sync kernel (the automatic choice up to 8 columns; forced with
    variant 2 up to 16) and the tcgen05 16-column kernel (variant 1)."""
    a_shape, b_shape = shapes
    for dist, seed, exact in ((synth.normal(1.0), 13, False), (synth.SMALL_INT, 13, True)):
        a, b = synth.operands(a_shape, b_shape, dtype, dist,
                              synth.normal(0.02) if not exact else synth.SMALL_INT, seed=seed)
        A, B = a.cuda(), b.cuda()
        with Plan(a.shape, b.shape, dtype) as p:
            p.force("skinny_n")
            p.set_tc_variant(variant)
            n = int(np.prod(p.output_shape))
            buf = torch.full((n + 64,), float("nan"), dtype=A.dtype, device="cuda")
            Y = buf[:n].view(p.output_shape)
            p.execute_checked(A, B, Y)
            torch.cuda.synchronize()
            assert torch.isnan(buf[n:].float()).all()
        y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        compare(Y.cpu(), y_ref, s, dtype, exact=exact)


TC_SKINNY_M_SHAPES = [
    ((1, 64), (64, 256)),
    ((16, 520), (520, 136)),           # N tail inside the second 128-column tile
    ((4, 8192), (8192, 2048)),         # long K: split over K
    ((3, 2, 5, 64), (2, 64, 384)),     # broadcast batch
    ((64,), (64, 48)),                 # rank-one A
    ((2, 16, 1024), (2, 1024, 264)),   # batched B: 2 items of 16 rows
]


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("shapes", TC_SKINNY_M_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
@pytest.mark.parametrize("variant", [0, 1, 2], ids=["auto", "simt", "tcgen05"])
def test_tc_skinny_m(dtype, shapes, variant):
    """FLOAT16 / BFLOAT16 skinny-M: automatic choice, the SIMT streaming
    kernel (variant 1) and the swapped-operand tcgen05 kernel (variant 2)."""
    a_shape, b_shape = shapes
    for dist_a, dist_b, exact in ((synth.normal(1.0), synth.normal(0.02), False),
                                  (synth.SMALL_INT, synth.SMALL_INT, True)):
        a, b = synth.operands(a_shape, b_shape, dtype, dist_a, dist_b, seed=14)
        A, B = a.cuda(), b.cuda()
        with Plan(a.shape, b.shape, dtype) as p:
            p.force("skinny_m")
            p.set_tc_variant(variant)
            n = int(np.prod(p.output_shape))
            buf = torch.full((n + 64,), float("nan"), dtype=A.dtype, device="cuda")
            Y = buf[:n].view(p.output_shape)
            p.execute_checked(A, B, Y)
            torch.cuda.synchronize()
            assert torch.isnan(buf[n:].float()).all()
        y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        compare(Y.cpu(), y_ref, s, dtype, exact=exact)


def _pair_product(a, b, dtype, exact=False):
    """The product through the CTA-pair (cta_group::2) tensor-core kernel."""
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        p.force("general_tc")
        p.set_tc_variant(2)
        n = int(np.prod(p.output_shape))
        buf = torch.full((n + 64,), float("nan"), dtype=A.dtype, device="cuda")
        Y = buf[:n].view(p.output_shape)
        p.execute_checked(A, B, Y)
        torch.cuda.synchronize()
        assert torch.isnan(buf[n:].float()).all()
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(Y.cpu(), y_ref, s, dtype, exact=exact)


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_tc_pair_single_tile(dtype):
    a, b = synth.operands((256, 64), (64, 256), dtype, synth.SMALL_INT, synth.SMALL_INT, seed=2)
    _pair_product(a, b, dtype, exact=True)


TC_PAIR_SHAPES = [
    ((256, 128), (128, 512)),
    ((300, 520), (520, 264)),          # M, N, K tails inside a pair tile
    ((130, 64), (64, 136)),            # the peer CTA's rows and columns out of range
    ((3, 1, 260, 64), (1, 2, 64, 264)),
    ((1024, 2048), (2048, 1024)),      # several pair tiles per cluster
    # a last partial wave of at most half the clusters runs as 256 x 128
    # half tiles (on 76 clusters): 77 tiles -> 76 whole and one split; 256
    # tiles -> 228 whole and 28 split; 10 tiles -> all split
    ((1792, 512), (512, 2816)),
    ((4096, 256), (256, 4096)),
    ((3, 1, 500, 128), (1, 2, 128, 600)),
    # N a multiple of 64: B's two 64-column blocks come in one 4-D load, and
    # blocks past N (the peer CTA's, or the second of a pair) read as zeros
    ((300, 200), (200, 320)),
    ((512, 64), (64, 448)),
    ((3, 1, 260, 96), (1, 2, 96, 384)),   # broadcast batch through the 4-D map
    ((1792, 128), (128, 2880)),           # 84 tiles: 8 run as halves, the last column tile partial
]


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("shapes", TC_PAIR_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_tc_pair_shapes(dtype, shapes):
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.02), seed=15)
    _pair_product(a, b, dtype)
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=15)
    _pair_product(ai, bi, dtype, exact=True)


# --------------------------------------------------------------------------
# edge cases


@pytest.mark.parametrize("dtype", DTYPES)
def test_k_zero_fills_zeros(dtype):
    a = torch.empty((5, 0), dtype=synth.TORCH_DTYPES[dtype])
    b = torch.empty((0, 7), dtype=synth.TORCH_DTYPES[dtype])
    y, algo = gpu_matmul(a, b, dtype)
    assert algo == "zero_fill" and y.shape == (5, 7) and bool((y == 0).all())


def test_empty_outputs_launch_nothing_and_accept_null():
    for a_shape, b_shape in [((0, 16, 32), (32, 8)), ((4, 5), (5, 0)), ((0, 1, 2, 3), (1, 5, 3, 4))]:
        with Plan(a_shape, b_shape, "float32") as p:
            assert p.algorithm == "empty" and p.launches == 0
            st = p.lib.olc_matmul_execute(p.handle, None, None, None, None)
            assert st == 0


@pytest.mark.parametrize("dtype", DTYPES)
def test_unaligned_pointers_still_correct(dtype):
    # operands that start one element into their buffers
    a, b = synth.operands((16, 64), (64, 256), dtype, synth.UNIFORM, synth.UNIFORM, seed=5)
    tdt = synth.TORCH_DTYPES[dtype]
    abuf = torch.zeros(a.numel() + 1, dtype=tdt, device="cuda")
    bbuf = torch.zeros(b.numel() + 1, dtype=tdt, device="cuda")
    ybuf = torch.zeros(16 * 256 + 1, dtype=tdt, device="cuda")
    A = abuf[1:].view(16, 64)
    B = bbuf[1:].view(64, 256)
    Y = ybuf[1:].view(16, 256)
    A.copy_(a.cuda())
    B.copy_(b.cuda())
    with Plan((16, 64), (64, 256), dtype) as p:
        p.execute_checked(A, B, Y)
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(Y.cpu(), y_ref, s, dtype)


def test_checked_execute_rejects_small_buffers():
    with Plan((8, 16), (16, 4), "float32") as p:
        A = torch.zeros(8, 16, device="cuda")
        B = torch.zeros(16, 4, device="cuda")
        Y = torch.zeros(8, 4, device="cuda")
        lib = p.lib
        assert lib.olc_matmul_execute_checked(p.handle, A.data_ptr(), 127, B.data_ptr(), 64,
                                              Y.data_ptr(), 32, None) == 8
        assert lib.olc_matmul_execute_checked(p.handle, A.data_ptr(), 128, B.data_ptr(), 64,
                                              Y.data_ptr(), 31, None) == 8
        assert lib.olc_matmul_execute_checked(p.handle, A.data_ptr(), 128, B.data_ptr(), 64,
                                              Y.data_ptr(), 32, None) == 0


@pytest.mark.parametrize("dtype", DTYPES)
def test_execute_host_round_trip(dtype):
    a, b = synth.operands((3, 40, 64), (64, 48), dtype, synth.UNIFORM, synth.UNIFORM, seed=6)
    tdt = synth.TORCH_DTYPES[dtype]
    with Plan(a.shape, b.shape, dtype) as p:
        ah, bh = a.pin_memory(), b.pin_memory()
        yh = torch.empty(p.output_shape, dtype=tdt).pin_memory()
        ad = torch.empty_like(a, device="cuda")
        bd = torch.empty_like(b, device="cuda")
        yd = torch.empty(p.output_shape, dtype=tdt, device="cuda")
        p.execute_host(ah, bh, yh, ad, bd, yd)
        torch.cuda.synchronize()
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(yh, y_ref, s, dtype)


@pytest.mark.parametrize("dtype,shapes", [
    ("bfloat16", ((8, 1024, 512), (512, 768))),      # folded to 8192 rows, tensor cores
    ("float32", ((5000, 256), (256, 136))),          # 5000 rows, SIMT, ragged last chunk
])
def test_execute_host_pipelined_matches_device_execute(dtype, shapes):
    """Large 2-D products from host buffers run as a copy-in / compute /
    copy-out pipeline over row chunks on internal streams; the result equals
    the device-buffer execute bit for bit, and a second call on the same plan
    (events and streams reused) does too."""
    a, b = synth.operands(shapes[0], shapes[1], dtype, synth.normal(1.0), synth.normal(0.05), 31)
    tdt = synth.TORCH_DTYPES[dtype]
    with Plan(a.shape, b.shape, dtype) as p:
        ref = torch.empty(p.output_shape, dtype=tdt, device="cuda")
        p.execute(a.cuda(), b.cuda(), ref)
        ah, bh = a.pin_memory(), b.pin_memory()
        ad = torch.empty_like(a, device="cuda")
        bd = torch.empty_like(b, device="cuda")
        yd = torch.empty(p.output_shape, dtype=tdt, device="cuda")
        s = torch.cuda.Stream()
        for _ in range(2):
            yh = torch.full(p.output_shape, float("nan"), dtype=tdt).pin_memory()
            p.execute_host(ah, bh, yh, ad, bd, yd, stream=s)
            s.synchronize()
            assert torch.equal(yh, ref.cpu())


def test_plan_reuse_across_streams_and_inputs():
    with Plan((64, 96), (96, 80), "float32") as p:
        s = torch.cuda.Stream()
        for seed in range(3):
            a, b = synth.operands((64, 96), (96, 80), "float32", synth.UNIFORM, synth.UNIFORM, seed)
            A, B = a.cuda(), b.cuda()
            Y = torch.empty(64, 80, device="cuda")
            with torch.cuda.stream(s):
                p.execute(A, B, Y, stream=s)
            s.synchronize()
            y_ref, sm = oracle.matmul(a.numpy(), b.numpy(), "float32")
            compare(Y.cpu(), y_ref, sm, "float32")


# --------------------------------------------------------------------------
# cluster split-K: general FP16/BF16 products whose 128 x 256 tiles fill at
# most half the SMs run each tile's K slices on the CTAs of a cluster and sum
# them through distributed shared memory

CSPLIT_SHAPES = [
    ((17, 4096), (4096, 1024)),          # few rows, B in 4-D loads, 8 slices
    ((100, 2056), (2056, 264)),          # N not a multiple of 64: 3-D loads, a partial last run
    ((129, 4104), (4104, 520)),          # two row tiles, K tail
    ((300, 1024), (1024, 320)),          # three row tiles, blocks past N
    ((2, 3, 40, 512), (3, 512, 256)),    # broadcast batch through the 3-D / 4-D maps
]


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("shapes", CSPLIT_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_cluster_split_k_shapes(dtype, shapes):
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.02), seed=61)
    check_product(a, b, dtype, algorithm="general_tc")
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, seed=61)
    check_product(ai, bi, dtype, algorithm="general_tc", exact=True)


def test_cluster_split_k_is_reproducible():
    """The slices are summed in slice order, whatever order the CTAs finish
    in: repeated executes give the same bits."""
    a, b = synth.operands((64, 8192), (8192, 512), "bfloat16", synth.normal(1.0), synth.normal(0.02), 62)
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, "bfloat16") as p:
        p.force("general_tc")
        ys = []
        for _ in range(3):
            Y = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
            p.execute(A, B, Y)
            ys.append(Y)
        torch.cuda.synchronize()
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
