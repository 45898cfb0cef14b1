"""8-bit float operands (E4M3FN, E5M2) on the GPU against the oracle:
the tcgen05 kind::f8f6f4 kernel (B transposed into the workspace) and the
SIMT decode kernel, float32 output; ragged tiles, batches, integer inputs
bit for bit, the fused epilogue, K == 0 and the rejections."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import GemmPlan, OlcError, Plan, synth
from parity import check_product, compare

pytestmark = pytest.mark.gpu

FP8 = ["float8_e4m3fn", "float8_e5m2"]

TC_SHAPES = [
    ((128, 128), (128, 256)),          # one tile, one K block
    ((256, 128), (128, 256)),          # one pair tile
    ((260, 2064), (2064, 516)),        # pair tiles with the peer CTA's rows and columns ragged
    ((300, 1040), (1040, 264)),        # M, N, K tails (K a multiple of 16, N of 4)
    ((200, 1040), (1040, 400)),        # 16-byte B transpose with ragged K and N tiles
    ((2, 512, 2048), (2048, 1024)),    # folded batch, several tiles and K blocks
    ((64, 4096), (4096, 4096)),
]


def _tc(a, b, dtype, variant, exact):
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        p.force("general_tc")
        p.set_tc_variant(variant)
        n = int(np.prod(p.output_shape))
        buf = torch.full((n + 64,), float("nan"), device="cuda")
        Y = buf[:n].view(p.output_shape)
        p.execute_checked(A, B, Y)
        torch.cuda.synchronize()
        assert torch.isnan(buf[n:]).all()
    ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(Y.cpu(), ref, s, dtype, exact=exact)


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("shapes", TC_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
@pytest.mark.parametrize("variant", [0, 1], ids=["auto_pairs", "one_cta"])
def test_fp8_tensor_core(dtype, shapes, variant):
    """Automatic choice (CTA pairs with 256 x 256 tiles once M and N reach
    256) and variant 1 (one CTA per 128 x 256 tile)."""
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.5), 41)
    _tc(a, b, dtype, variant, exact=False)
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, 42)
    _tc(ai, bi, dtype, variant, exact=True)


SIMT_SHAPES = [
    ((1, 8), (8, 16)),
    ((37, 55), (55, 29)),              # no 16-byte rows at all
    ((3, 2, 40, 24), (2, 24, 48)),     # broadcast batch with batched B
    ((64,), (64, 48)),                 # rank-one A
    ((300, 1040), (1040, 264)),
]


FNUZ = ["float8_e4m3fnuz", "float8_e5m2fnuz"]


@pytest.mark.parametrize("dtype", FP8 + FNUZ)
@pytest.mark.parametrize("shapes", SIMT_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_fp8_simt(dtype, shapes):
    a_shape, b_shape = shapes
    a, b = synth.operands(a_shape, b_shape, dtype, synth.UNIFORM, synth.UNIFORM, 43)
    check_product(a, b, dtype, algorithm="general_simt")
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, 44)
    check_product(ai, bi, dtype, algorithm="direct", exact=True)


@pytest.mark.parametrize("dtype", FP8)
def test_fp8_fused_relu_residual_and_k_zero(dtype):
    a, b = synth.operands((256, 512), (512, 256), dtype, synth.normal(1.0), synth.normal(0.5), 45)
    r = torch.randn(256, 256)
    with Plan(a.shape, b.shape, dtype) as p:
        assert p.algorithm == "general_tc"
        p.set_epilogue("relu", True)
        Y = torch.empty(256, 256, device="cuda")
        p.execute_fused(a.cuda(), b.cuda(), Y, R=r.cuda())
        torch.cuda.synchronize()
    ref, s = oracle.matmul_fused(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                                 r.numpy(), "relu")
    compare(Y.cpu(), ref, s, dtype)
    with Plan((5, 0), (0, 7), dtype) as p:
        assert p.algorithm == "zero_fill"
        Y = torch.full((5, 7), float("nan"), device="cuda")
        p.execute(torch.empty(5, 0, dtype=a.dtype, device="cuda"),
                  torch.empty(0, 7, dtype=a.dtype, device="cuda"), Y)
        torch.cuda.synchronize()
        assert torch.equal(Y.cpu(), torch.zeros(5, 7))


def test_fp8_rejections():
    with pytest.raises(OlcError) as ei:
        GemmPlan((4, 8), (8, 4), "float8_e4m3fn")
    assert ei.value.name == "OLC_ERR_DTYPE"
    with Plan((64, 40), (40, 30), "float8_e5m2") as p:    # N not a multiple of 4
        with pytest.raises(OlcError):
            p.force("general_tc")
        with pytest.raises(OlcError):
            p.force("split_k")


def test_fp8_convenience_call_returns_float32():
    from gemm_matmulplan_broadcast_gb300 import matmul
    a, b = synth.operands((64, 96), (96, 40), "float8_e5m2", synth.SMALL_INT, synth.SMALL_INT, 46)
    y = matmul(a.cuda(), b.cuda())
    torch.cuda.synchronize()
    assert y.dtype == torch.float32 and tuple(y.shape) == (64, 40)
    ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), "float8_e5m2")
    compare(y.cpu(), ref, s, "float8_e5m2", exact=True)


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("shapes", [((260, 2064), (2064, 516)), ((512, 1024), (1024, 2048)),
                                    ((96, 272), (272, 48)), ((37, 55), (55, 29))],
                         ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_fp8_constant_b_prepacked(dtype, shapes):
    """A constant B is kept transposed by the plan (tensor-core plans); the
    executes without B give the per-call result bit for bit, also after the
    source is overwritten."""
    a, b = synth.operands(shapes[0], shapes[1], dtype, synth.normal(1.0), synth.normal(0.5), 43)
    A = a.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        Y1 = torch.empty(p.output_shape, device="cuda")
        Y2 = torch.empty_like(Y1)
        p.execute(A, b.cuda(), Y1)
        src = b.cuda()
        p.set_constant_b(src)
        src.view(torch.uint8).fill_(0x38)
        p.execute_constant(A, Y2)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2)
    ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    compare(Y2.cpu(), ref, s, dtype)


@pytest.mark.parametrize("dtype", FNUZ)
def test_fnuz_runs_on_the_decode_kernel(dtype):
    """The FNUZ encodings are not tensor-core formats: the plan takes the SIMT
    decode kernel, forcing the tensor cores is rejected; a large product and
    the special patterns (0x80 is NaN, 0x7F and 0xFF the largest finite
    values) against the oracle."""
    a, b = synth.operands((512, 1024), (1024, 768), dtype, synth.normal(1.0), synth.normal(0.5), 47)
    with Plan(a.shape, b.shape, dtype) as p:
        assert p.algorithm == "general_simt"
        with pytest.raises(OlcError):
            p.force("general_tc")
    check_product(a, b, dtype)
    a8 = np.full((4, 16), 0x00, np.uint8)
    b8 = np.full((16, 8), 0x00, np.uint8)
    a8[0, 0] = 0x80            # NaN: row 0 of Y is NaN
    a8[1, :2] = [0x7F, 0xFF]   # +max, -max
    b8[:2, :] = 0x40           # 1.0
    a8[2, 5] = 0x01            # the smallest subnormal
    b8[5, :] = 0x01
    ta, tb = synth.from_numpy_storage(a8, dtype), synth.from_numpy_storage(b8, dtype)
    ref, s = oracle.matmul(a8, b8, dtype)
    with Plan(ta.shape, tb.shape, dtype) as p:
        Y = torch.empty(4, 8, device="cuda")
        p.execute_checked(ta.cuda(), tb.cuda(), Y)
        torch.cuda.synchronize()
    y = Y.cpu().numpy()
    assert np.isnan(y[0]).all() and np.isnan(ref[0]).all()
    assert np.array_equal(y[1:], ref[1:])
    assert y[1, 0] == 0.0 and y[2, 0] == ref[2, 0] and ref[2, 0] > 0


SKINNY_SHAPES = [
    ((4, 8192), (8192, 2048)),         # K sliced across blocks
    ((1, 4096), (4096, 4096)),
    ((16, 1024), (1024, 512)),
    ((3, 2, 64), (64, 256)),           # batch folded into 6 rows
    ((5, 1000), (1000, 272)),          # K tail, partial column group
    ((64,), (64, 512)),                # rank-one A
    ((4, 2048), (2048, 4096)),         # 4 rows: 8 columns per lane
    ((16, 4096), (4096, 1024)),        # 16 rows: 4 columns per lane
    ((6, 1001), (1001, 256)),          # A rows not 8-byte aligned: element loads
    ((12, 999), (999, 512)),           # the same with 16 rows
    ((2, 5, 256), (2, 256, 512)),      # batched B: 2 items of 5 rows
    ((3, 1, 12, 64), (1, 2, 64, 256)), # broadcast on both sides: 6 items of 12 rows
]


SKINNY_VARIANTS = {"auto": 0, "simt": 1, "mma": 2, "tcgen05": 3}


@pytest.mark.parametrize("dtype", FP8 + FNUZ)
@pytest.mark.parametrize("shapes", SKINNY_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
@pytest.mark.parametrize("variant", list(SKINNY_VARIANTS), ids=list(SKINNY_VARIANTS))
def test_fp8_skinny_m(dtype, shapes, variant):
    """Up to 16 rows, chosen automatically from N >= 256: the SIMT streaming
    kernel (16, 8 or 4 one-byte B elements per lane load, decoded to float32;
    A rows that are not 8-byte aligned take element loads) and, for E4M3FN
    and E5M2, the warp-level MMA kernel (m16n8k32, B fragments transposed in
    registers; automatic from 4 rows) and the tcgen05 kernel with swapped
    operands and B transposed in shared memory (variant 3; one item, N and K
    multiples of 16, else the warp-level MMA kernel).  The FNUZ formats take
    the SIMT kernel whatever the variant."""
    a_shape, b_shape = shapes
    with Plan(a_shape, b_shape, dtype) as p:
        if b_shape[-1] >= 256:
            assert p.algorithm == "skinny_m"
    v = SKINNY_VARIANTS[variant]
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.5), 48)
    check_product(a, b, dtype, algorithm="skinny_m", variant=v)
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, 49)
    check_product(ai, bi, dtype, algorithm="skinny_m", exact=True, variant=v)


ONE = {"float8_e4m3fn": 0x38, "float8_e5m2": 0x3C, "float8_e4m3fnuz": 0x40, "float8_e5m2fnuz": 0x40}


@pytest.mark.parametrize("dtype", FP8 + FNUZ)
@pytest.mark.parametrize("m", [2, 4, 16])
@pytest.mark.parametrize("variant", [1, 2, 3], ids=["simt", "mma", "tcgen05"])
def test_fp8_skinny_m_decodes_every_pattern(dtype, m, variant):
    """Every one of the 256 patterns through the skinny kernel's B decode
    (16, 8 or 4 one-byte columns per lane for 2, 4 or 16 rows; element i of a
    vector in byte i): Y row 0 = 1.0 x B row 0 (patterns 0..255), Y row 1 =
    1.0 x B row 8 (255..0), all other terms 0."""
    a8 = np.zeros((m, 16), np.uint8)
    a8[0, 0] = ONE[dtype]
    a8[1, 8] = ONE[dtype]
    b8 = np.zeros((16, 256), np.uint8)
    b8[0] = np.arange(256)
    b8[8] = np.arange(255, -1, -1)
    assert oracle.decode_fp8(np.array([ONE[dtype]], np.uint8), dtype)[0] == 1.0
    ref, _ = oracle.matmul(a8, b8, dtype)
    ta, tb = synth.from_numpy_storage(a8, dtype), synth.from_numpy_storage(b8, dtype)
    with Plan(ta.shape, tb.shape, dtype) as p:
        p.force("skinny_m")
        p.set_tc_variant(variant)
        Y = torch.empty(m, 256, device="cuda")
        p.execute_checked(ta.cuda(), tb.cuda(), Y)
        torch.cuda.synchronize()
    y = Y.cpu().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan)
    assert np.array_equal(y[~nan], ref[~nan])


@pytest.mark.parametrize("dtype", FP8 + FNUZ)
@pytest.mark.parametrize("variant", [1, 2, 3], ids=["simt", "mma", "tcgen05"])
def test_fp8_skinny_m_decodes_every_a_pattern(dtype, variant):
    """Every pattern through the skinny kernel's A decode (A rows kept as
    packed bytes, decoded two k positions at a time): A[i, k] = 16 i + k for
    16 rows and K = 16, B[k, j] = 1.0 where j == k < 16, else 0.  Y[i, j] =
    A[i, j] exactly, except in rows holding a NaN or an infinity, where every
    other term is NaN x 0 or inf x 0 and the oracle's row is NaN too."""
    a8 = np.arange(256, dtype=np.uint8).reshape(16, 16)
    b8 = np.zeros((16, 256), np.uint8)
    b8[np.arange(16), np.arange(16)] = ONE[dtype]
    ref, _ = oracle.matmul(a8, b8, dtype)
    dec = oracle.decode_fp8(a8.reshape(-1), dtype).reshape(16, 16)
    clean = ~np.isnan(ref).any(axis=1)
    assert clean.sum() >= 14
    assert np.array_equal(ref[clean][:, :16], dec[clean])
    ta, tb = synth.from_numpy_storage(a8, dtype), synth.from_numpy_storage(b8, dtype)
    with Plan(ta.shape, tb.shape, dtype) as p:
        p.force("skinny_m")
        p.set_tc_variant(variant)
        Y = torch.empty(16, 256, device="cuda")
        p.execute_checked(ta.cuda(), tb.cuda(), Y)
        torch.cuda.synchronize()
    y = Y.cpu().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan)
    assert np.array_equal(y[~nan], ref[~nan])


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("shapes,splits", [
    (((4, 8192), (8192, 28672)), 0),     # the named few-row workload's product, automatic slices
    (((16, 8192), (8192, 2048)), 5),     # several K slices summed in slice order
    (((1, 300), (300, 4112)), 1),        # one row, K and N tails of the boxes
    (((7, 4096), (4096, 512)), 32),      # many slices
])
def test_fp8_skinny_m_tcgen05(dtype, shapes, splits):
    """The tcgen05 few-row kernel (variant 3): normal inputs within the
    bound, integer inputs bit for bit, two runs identical (fixed-order
    reduction of the K slices)."""
    a_shape, b_shape = shapes
    for dist, exact in [(synth.normal(1.0), False), (synth.SMALL_INT, True)]:
        a, b = synth.operands(a_shape, b_shape, dtype, dist, dist if exact else synth.normal(0.5), 50)
        A, B = a.cuda(), b.cuda()
        with Plan(a_shape, b_shape, dtype) as p:
            p.force("skinny_m")
            p.set_tc_variant(3)
            if splits:
                p.set_splits(splits)
            Y = torch.full(p.output_shape, float("nan"), device="cuda")
            Y2 = torch.empty_like(Y)
            p.execute_checked(A, B, Y)
            p.execute_checked(A, B, Y2)
            torch.cuda.synchronize()
            assert torch.equal(Y, Y2)
        y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        compare(Y.cpu(), y_ref, s, dtype, exact=exact)


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("shapes", [((4, 8192), (8192, 2048)), ((16, 1024), (1024, 512)),
                                    ((2, 300), (300, 4112)), ((1, 512), (512, 1024))],
                         ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_fp8_skinny_m_constant_b(dtype, shapes):
    """An 8-bit few-row plan of 2 or more rows given a constant B keeps it
    transposed and runs the tcgen05 kernel on that copy (no shared-memory
    transposition; one row stays on the SIMT kernel): against
    the oracle (integer inputs bit for bit), two executes identical; an
    execute with a caller's B on the same plan (the same kernel, transposing
    in shared memory) too."""
    a_shape, b_shape = shapes
    for dist, exact in [(synth.normal(1.0), False), (synth.SMALL_INT, True)]:
        a, b = synth.operands(a_shape, b_shape, dtype, dist, dist if exact else synth.normal(0.5), 51)
        A = a.cuda()
        with Plan(a_shape, b_shape, dtype) as p:
            assert p.algorithm == "skinny_m"
            p.set_constant_b(b)
            Y = torch.full(p.output_shape, float("nan"), device="cuda")
            Y2 = torch.empty_like(Y)
            Y3 = torch.full(p.output_shape, float("nan"), device="cuda")
            p.execute_constant(A, Y)
            p.execute_constant(A, Y2)
            p.execute(A, b.cuda(), Y3)
            torch.cuda.synchronize()
            assert torch.equal(Y, Y2)
        y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        compare(Y.cpu(), y_ref, s, dtype, exact=exact)
        compare(Y3.cpu(), y_ref, s, dtype, exact=exact)


def test_fp8_skinny_decode_workload_full():
    """The named FP8 few-row workload at full size ([1|4|16, 8192] x [8192,
    28672]): SKINNY_M chosen, every element against the oracle."""
    w = synth.workload("fp8_skinny_decode")
    for prod in w.products:
        a, b = prod.draw()
        y, algo = check_product(a, b, prod.dtype)
        assert algo == "skinny_m"


F8_SPLIT_SHAPES = [
    ((32, 131072), (131072, 32)),          # the tiny-output long-K corner: two 16-row tiles
    ((16, 40000), (40000, 48)),            # one tile, K tail inside a chunk
    ((20, 9000), (9000, 128)),             # two column groups
    ((3, 2, 8, 3000), (2, 3000, 16)),      # six batch items, batched B
    ((17, 10001), (10001, 32)),            # A rows not 4-byte aligned: byte loads
]


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("shapes", F8_SPLIT_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_fp8_split_k(dtype, shapes):
    """Small outputs over long K: the warp-MMA split-K (about one K slice
    per SM, partials summed in slice order within groups of 16, then in
    group order); normal inputs within the float32 bar, integers exact."""
    a_shape, b_shape = shapes
    with Plan(a_shape, b_shape, dtype) as p:
        if a_shape == (32, 131072):
            assert p.algorithm == "split_k" and p.splits > 16
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.5), 50)
    check_product(a, b, dtype, algorithm="split_k")
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, 51)
    check_product(ai, bi, dtype, algorithm="split_k", exact=True)


@pytest.mark.parametrize("splits", [1, 3, 16, 17, 40])
def test_fp8_split_k_slice_counts_and_reproducibility(splits):
    """Requested slice counts: one level (1..16 slices) and two levels (17:
    groups of 16 and 1; 40: 16, 16, 8); the same inputs give bit-identical
    results on every run."""
    dtype = "float8_e4m3fn"
    a, b = synth.operands((24, 20000), (20000, 64), dtype, synth.normal(1.0), synth.normal(0.5), 52)
    ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    A, B = a.cuda(), b.cuda()
    with Plan(a.shape, b.shape, dtype) as p:
        p.force("split_k")
        p.set_splits(splits)
        assert p.splits == splits
        outs = []
        for _ in range(3):
            Y = torch.full((24, 64), float("nan"), device="cuda")
            p.execute_checked(A, B, Y)
            torch.cuda.synchronize()
            outs.append(Y.cpu())
    for y in outs[1:]:
        assert torch.equal(y, outs[0])
    compare(outs[0], ref, s, dtype)


F8_SKINNY_N_SHAPES = [
    ((16384, 4096), (4096, 8)),            # the skinny-N corner shape
    ((1000, 4096), (4096, 16)),            # two 8-column blocks, rows not a multiple of 16
    ((300, 1040), (1040, 5)),              # N padded to 8 columns, K tail of a warp's range
    ((2, 3, 100, 2048), (2048, 12)),       # batch folded into 600 rows
    ((513, 64), (64, 3)),                  # K shorter than the sixteen warps' ranges
]


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("shapes", F8_SKINNY_N_SHAPES, ids=lambda s: "x".join(map(str, s[0] + s[1])))
def test_fp8_skinny_n(dtype, shapes):
    """Few columns: the register-streaming kernel of FLOAT16 skinny-N on
    mma.sync.m16n8k32 (A rows streamed in 16-byte pieces, B transposed in
    shared memory), chosen up to 8 columns and forced up to 16; normal
    inputs within the float32 bar, integers exact."""
    a_shape, b_shape = shapes
    with Plan(a_shape, b_shape, dtype) as p:
        assert (p.algorithm == "skinny_n") == (b_shape[-1] <= 8)
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.5), 53)
    check_product(a, b, dtype, algorithm="skinny_n")
    ai, bi = synth.operands(a_shape, b_shape, dtype, synth.SMALL_INT, synth.SMALL_INT, 54)
    check_product(ai, bi, dtype, algorithm="skinny_n", exact=True)


FP8_FUSED_CASES = [
    ("skinny_m", 1, (4, 2048), (2048, 512)),       # SIMT skinny-M
    ("skinny_m", 2, (12, 2048), (2048, 512)),      # warp-MMA skinny-M
    ("skinny_m", 3, (12, 8192), (8192, 512)),      # tcgen05 skinny-M, K slices
    ("split_k", None, (24, 20000), (20000, 64)),   # warp-MMA split-K, two reduction levels
    ("skinny_n", None, (1000, 1024), (1024, 8)),   # warp-MMA skinny-N
    ("general_simt", None, (100, 300), (300, 200)),
    ("direct", None, (7, 33), (33, 9)),
]


@pytest.mark.parametrize("dtype", FP8)
@pytest.mark.parametrize("act", ["relu", "gelu"])
@pytest.mark.parametrize("case", FP8_FUSED_CASES, ids=lambda c: "%s-%s" % (c[0], c[1]))
def test_fp8_fused_epilogue_every_kernel(dtype, act, case):
    """Residual and activation fused into the store of every FP8 kernel,
    against the oracle's float64 activation of the float32 sum plus the
    residual."""
    algo, variant, a_shape, b_shape = case
    a, b = synth.operands(a_shape, b_shape, dtype, synth.normal(1.0), synth.normal(0.5), 55)
    M, N = a_shape[0], b_shape[1]
    r = torch.randn(M, N, generator=torch.Generator().manual_seed(56))
    with Plan(a.shape, b.shape, dtype) as p:
        p.force(algo)
        if variant is not None:
            p.set_tc_variant(variant)
        p.set_epilogue(act, True)
        Y = torch.full((M, N), float("nan"), device="cuda")
        p.execute_fused(a.cuda(), b.cuda(), Y, R=r.cuda())
        torch.cuda.synchronize()
    ref, s = oracle.matmul_fused(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype,
                                 r.numpy(), act)
    compare(Y.cpu(), ref, s, dtype)
