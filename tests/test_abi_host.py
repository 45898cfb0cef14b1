"""Host-side checks of the C ABI (no GPU needed, no kernel launched): the
library loads and exports every function the header declares; plans resolve
shapes, batch strides and errors as the shape rules say; the algorithm choice
and its feasibility rules; workspace sizing."""

import ctypes
import itertools

import numpy as np
import pytest

import oracle
from gemm_matmulplan_broadcast_gb300 import Plan, binding
from gemm_matmulplan_broadcast_gb300.binding import OlcError
from gemm_matmulplan_broadcast_gb300 import GemmPlan

from test_oracle_pins import _golden_shapes


def test_library_exports_every_declared_function():
    lib = binding.load()
    names = binding.header_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name
    assert lib.olc_version() >= 100


def test_status_and_algorithm_strings():
    lib = binding.load()
    for code in binding.STATUS:
        assert lib.olc_status_string(code)
    assert lib.olc_status_string(999) == b"unknown status"
    for name, code in binding.ALGORITHMS.items():
        assert lib.olc_algorithm_name(code).decode() == name


@pytest.mark.parametrize("a_shape,b_shape,want", _golden_shapes())
def test_plan_output_shape_matches_golden_table(a_shape, b_shape, want):
    if want is None:
        with pytest.raises(OlcError):
            Plan(a_shape, b_shape, "float32")
    else:
        with Plan(a_shape, b_shape, "float32") as p:
            assert p.output_shape == want
            assert p.output_shape == oracle.output_shape(a_shape, b_shape)


def _numpy_batch_strides(a_shape, b_shape):
    """Reference batch strides: numpy's broadcast_to view of each operand's
    matrix index array (stride 0 along broadcast dimensions)."""
    a2 = (1,) + tuple(a_shape) if len(a_shape) == 1 else tuple(a_shape)
    b2 = tuple(b_shape) + (1,) if len(b_shape) == 1 else tuple(b_shape)
    batch = np.broadcast_shapes(a2[:-2], b2[:-2])
    out = []
    for op in (a2, b2):
        mat = op[-2] * op[-1]
        idx = np.arange(int(np.prod(op[:-2], dtype=np.int64)) if len(op) > 2 else 1,
                        dtype=np.int64).reshape(op[:-2])
        view = np.broadcast_to(idx, batch)
        out.append(tuple(s // 8 * mat for s in view.strides))
    return batch, out[0], out[1]


STRIDE_CASES = [
    ((8, 1, 128, 256), (1, 4, 256, 64)),
    ((2, 1, 3, 1, 4, 5), (7, 1, 6, 5, 2)),
    ((1, 1, 4, 5), (3, 5, 6)),
    ((256,), (4, 256, 64)),
    ((4, 32, 256), (256,)),
    ((3, 2, 4, 5), (2, 5, 6)),
    ((5, 6), (2, 3, 6, 7)),
]


@pytest.mark.parametrize("a_shape,b_shape", STRIDE_CASES)
def test_batch_strides_match_numpy_broadcast_views(a_shape, b_shape):
    batch, sa_ref, sb_ref = _numpy_batch_strides(a_shape, b_shape)
    with Plan(a_shape, b_shape, "float32") as p:
        shape, sa, sb = p.batch()
        assert shape == tuple(batch)
        for d, e in enumerate(batch):
            if e > 1:   # strides of extent-1 dimensions are never used
                assert sa[d] == sa_ref[d] and sb[d] == sb_ref[d]
            else:
                assert sa[d] == 0 and sb[d] == 0
        m, n, k, nb = p.dims()
        assert nb == int(np.prod(batch, dtype=np.int64))


def _random_shape_pair(rng):
    """Shapes of rank 1-5 with small extents (0 included), K matched most of
    the time and batch extents drawn so that broadcasts, matches and
    mismatches all occur."""
    ra, rb = int(rng.integers(1, 6)), int(rng.integers(1, 6))
    k = int(rng.integers(0, 4))
    a = [int(x) for x in rng.integers(0, 4, size=ra)]
    b = [int(x) for x in rng.integers(0, 4, size=rb)]
    if rng.random() < 0.85:
        a[-1] = k
        b[0 if rb == 1 else -2] = k
    ba, bb = a[:-2], b[:-2]
    for i in range(1, min(len(ba), len(bb)) + 1):
        r = rng.random()
        if r < 0.4:
            bb[-i] = ba[-i]
        elif r < 0.6:
            bb[-i] = 1
        elif r < 0.8:
            ba[-i] = 1
    return tuple(ba + a[len(ba):]), tuple(bb + b[len(bb):])


def test_random_shapes_agree_with_numpy_matmul():
    """A seeded sweep of 3,000 shape pairs: the plan (and the oracle's shape
    rule) accept exactly the pairs numpy.matmul accepts, with numpy's output
    shape; its batch strides
    are numpy's broadcast-view strides (where the batch is not empty), and
    collapse / fold keep every row (launch rows x items = M x batch)."""
    rng = np.random.default_rng(20261202)
    accepted = rejected = 0
    for _ in range(3000):
        a_shape, b_shape = _random_shape_pair(rng)
        try:
            want = np.matmul(np.zeros(a_shape, np.float32), np.zeros(b_shape, np.float32)).shape
        except ValueError:
            want = None
        if want is None:
            with pytest.raises(OlcError):
                Plan(a_shape, b_shape, "float32")
            with pytest.raises(oracle.ShapeError):
                oracle.output_shape(a_shape, b_shape)
            rejected += 1
            continue
        accepted += 1
        assert oracle.output_shape(a_shape, b_shape) == tuple(want), (a_shape, b_shape)
        with Plan(a_shape, b_shape, "float32") as p:
            assert p.output_shape == tuple(want), (a_shape, b_shape)
            batch, sa_ref, sb_ref = _numpy_batch_strides(a_shape, b_shape)
            shape, sa, sb = p.batch()
            assert shape == tuple(batch)
            m, n, k, nb = p.dims()
            for d, e in enumerate(batch):
                if e > 1 and nb > 0:    # an empty batch addresses no item
                    assert sa[d] == sa_ref[d] and sb[d] == sb_ref[d], (a_shape, b_shape)
            if m * n * nb > 0:
                rows, items, _ = p.launch_shape()
                assert rows * items == m * nb, (a_shape, b_shape)
    assert accepted > 1000 and rejected > 300


def test_random_gemm_shapes_agree_with_numpy():
    """A seeded sweep of 2,000 Gemm shape sets (transA / transB, C of rank
    0-3): the plan and the oracle's shape rule accept exactly the sets whose
    A' B' numpy can multiply and whose C numpy.broadcast_to takes to [M, N]
    (ONNX's unidirectional broadcast), and the plan's output is [M, N]."""
    rng = np.random.default_rng(20261203)
    accepted = rejected = 0
    for _ in range(2000):
        m, n, k = (int(x) for x in rng.integers(0, 4, size=3))
        ta, tb = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
        kb = k if rng.random() < 0.85 else int(rng.integers(0, 4))
        a_shape = (k, m) if ta else (m, k)
        b_shape = (n, kb) if tb else (kb, n)
        c_shape = None
        if rng.random() < 0.8:
            rank = int(rng.integers(0, 4))
            c_shape = tuple(int(rng.choice([1, m, n, int(rng.integers(0, 4))])) for _ in range(rank))
        try:
            a = np.zeros(a_shape, np.float32)
            b = np.zeros(b_shape, np.float32)
            want = ((a.T if ta else a) @ (b.T if tb else b)).shape
            if c_shape is not None:
                np.broadcast_to(np.zeros(c_shape, np.float32), want)
        except ValueError:
            want = None
        if want is None:
            with pytest.raises(OlcError):
                GemmPlan(a_shape, b_shape, "float32", ta, tb, 1.0, 1.0, c_shape)
            with pytest.raises(oracle.ShapeError):
                oracle.gemm_output_shape(a_shape, b_shape, ta, tb, c_shape)
            rejected += 1
            continue
        accepted += 1
        assert oracle.gemm_output_shape(a_shape, b_shape, ta, tb, c_shape)[:2] == want
        with GemmPlan(a_shape, b_shape, "float32", ta, tb, 1.0, 1.0, c_shape) as p:
            assert p.output_shape == want, (a_shape, b_shape, ta, tb, c_shape)
    assert accepted > 1000 and rejected > 200


def test_random_plans_choose_a_feasible_algorithm():
    """A seeded sweep over shapes from tiny to projection-sized and every
    element type: EMPTY exactly for empty outputs, ZERO_FILL exactly for
    K = 0 with a non-empty output, the chosen algorithm can be forced again
    (it is feasible) and stays chosen, plans that launch no product own no
    workspace, and the description names the choice."""
    rng = np.random.default_rng(20261204)
    dtypes = ["float32", "float64", "float16", "bfloat16", "float8_e4m3fn", "float8_e5m2",
              "float8_e4m3fnuz"]
    ms = [0, 1, 2, 4, 16, 17, 64, 128, 300, 4096, 16384]
    ks = [0, 8, 64, 520, 4096, 131072]
    ns = [1, 8, 16, 24, 32, 64, 256, 4096, 14336]
    seen = set()
    for _ in range(600):
        m, k, n = (int(rng.choice(v)) for v in (ms, ks, ns))
        batch = [int(x) for x in rng.choice([1, 2, 3, 8], size=int(rng.integers(0, 3)))]
        a_shape = tuple(batch + [m, k])
        b_shape = (k, n) if rng.random() < 0.5 else tuple(batch + [k, n])
        dt = str(rng.choice(dtypes))
        with Plan(a_shape, b_shape, dt) as p:
            algo = p.algorithm
            seen.add(algo)
            empty = int(np.prod(p.output_shape, dtype=np.int64)) == 0
            assert (algo == "empty") == empty, (a_shape, b_shape, dt, algo)
            assert (algo == "zero_fill") == (not empty and k == 0), (a_shape, b_shape, dt, algo)
            assert p.describe().startswith("algo=%s " % algo)
            if algo in ("empty", "zero_fill", "direct"):
                assert p.workspace_bytes == 0
            p.force(algo)
            assert p.algorithm == algo
    assert {"empty", "zero_fill", "direct", "skinny_m", "skinny_n", "split_k", "general_tc",
            "general_simt"} <= seen


def test_batch_collapse_and_fold():
    # B shared by every item and A's items consecutive: folded into rows
    with Plan((8, 2048, 64), (64, 32), "float32") as p:
        assert p.launch_shape() == (8 * 2048, 1, 0)
    with Plan((2, 3, 16, 8), (8, 4), "float32") as p:
        assert p.launch_shape() == (2 * 3 * 16, 1, 0)
    # rank-2 A with rank-one B: folds too (B shared)
    with Plan((4, 32, 256), (256,), "float32") as p:
        assert p.launch_shape() == (128, 1, 0)
    # both sides broadcast along different dims: two collapsed dims, 32 items
    with Plan((8, 1, 128, 256), (1, 4, 256, 64), "float32") as p:
        assert p.launch_shape() == (128, 32, 2)
    # contiguous batch dims on both sides collapse into one
    with Plan((2, 3, 4, 5), (2, 3, 5, 6), "float32") as p:
        assert p.launch_shape() == (4, 6, 1)
    # extent-1 dims drop out
    with Plan((1, 3, 1, 4, 5), (1, 1, 5, 6), "float32") as p:
        assert p.launch_shape() == (12, 1, 0)
    # B broadcast but A too: cannot fold
    with Plan((1, 4, 5), (3, 5, 6), "float32") as p:
        assert p.launch_shape() == (4, 3, 1)


@pytest.mark.parametrize("bad,status", [
    (((2, 3), (4, 5)), "OLC_ERR_K_MISMATCH"),
    (((2, 3, 4), (3, 4, 5)), "OLC_ERR_BATCH_MISMATCH"),
    (((-1, 3), (3, 4)), "OLC_ERR_NEGATIVE_DIM"),
    (((1,) * 9, (1, 1)), "OLC_ERR_RANK"),
])
def test_create_errors(bad, status):
    with pytest.raises(OlcError) as ei:
        Plan(bad[0], bad[1], "float32")
    assert ei.value.name == status


def test_create_rejects_sizes_whose_offsets_overflow():
    """Operands or outputs of more than 2^62 bytes are refused before any
    allocation (their element offsets could overflow int64); a zero extent
    makes a tensor empty whatever its other extents."""
    big = 1 << 31
    for a, b in [((big, big), (big, 4)),                 # A: 2^62 elements x 4 bytes
                 ((4, 8), (8, big, big)),               # B batch dims
                 ((big, 2), (2, big))]:                 # Y only
        with pytest.raises(OlcError) as ei:
            Plan(a, b, "float32")
        assert ei.value.name == "OLC_ERR_INVALID"
    with pytest.raises(OlcError) as ei:
        GemmPlan((big, big), (big, 2), "float16")
    assert ei.value.name == "OLC_ERR_INVALID"
    # 2^61 bytes of FP16 output: accepted (nothing is allocated for Y)
    with Plan((1 << 30, 2), (2, 1 << 30), "float16") as p:
        assert p.output_shape == (1 << 30, 1 << 30)
    # empty: a zero extent next to huge ones
    with Plan((0, big, big), (big, 4), "float32") as p:
        assert p.algorithm == "empty"


def test_fp8_split_k_choice_and_workspace():
    """FP8 products with small outputs and long K plan the warp-MMA split-K
    (about one slice per SM, a workspace for both reduction levels); the
    FNUZ formats, columns not a multiple of 16 and more than 32 rows do not
    take it."""
    with Plan((32, 131072), (131072, 32), "float8_e4m3fn") as p:
        assert p.algorithm == "split_k"
        s = p.splits
        assert 16 < s <= 152
        groups = -(-s // 16)
        assert p.workspace_bytes >= (s + groups) * 32 * 64 * 4 + (groups + 1) * 4
    for a, b, dt in [((32, 131072), (131072, 32), "float8_e4m3fnuz"),
                     ((32, 131072), (131072, 24), "float8_e4m3fn"),
                     ((40, 131072), (131072, 32), "float8_e5m2")]:
        with Plan(a, b, dt) as p:
            assert p.algorithm != "split_k"
            with pytest.raises(OlcError):
                p.force("split_k")


def test_fp8_skinny_n_choice():
    """FP8 products with at most 8 columns and one B stream A through the
    warp-MMA skinny-N kernel (up to 16 when forced); the FNUZ formats and K
    not a multiple of 16 do not take it."""
    for a, b in [((16384, 4096), (4096, 8)), ((2, 3, 100, 2048), (2048, 5))]:
        with Plan(a, b, "float8_e5m2") as p:
            assert p.algorithm == "skinny_n"
    # 9-16 columns: the tensor-core tile kernel by default, this one on request
    with Plan((1000, 4096), (4096, 16), "float8_e4m3fn") as p:
        assert p.algorithm == "general_tc"
        p.force("skinny_n")
    for a, b, dt in [((16384, 4096), (4096, 8), "float8_e4m3fnuz"),
                     ((16384, 4104), (4104, 8), "float8_e4m3fn")]:
        with Plan(a, b, dt) as p:
            assert p.algorithm != "skinny_n"
            with pytest.raises(OlcError):
                p.force("skinny_n")


def test_create_rejects_rank0_null_and_bad_dtype():
    lib = binding.load()
    h = ctypes.c_void_p()
    a = (ctypes.c_int64 * 2)(3, 4)
    assert lib.olc_matmul_plan_create(a, 0, a, 2, 1, ctypes.byref(h)) == 2    # rank 0
    assert lib.olc_matmul_plan_create(a, 2, a, 2, 7, ctypes.byref(h)) == 6    # dtype 7
    assert lib.olc_matmul_plan_create(None, 2, a, 2, 1, ctypes.byref(h)) == 1
    assert lib.olc_matmul_plan_create(a, 2, a, 2, 1, None) == 1
    assert h.value is None
    lib.olc_matmul_plan_destroy(None)   # NULL is accepted
    assert lib.olc_matmul_plan_algorithm(None) == -1


def test_algorithm_choice_for_named_shapes():
    cases = [
        ((64, 128), (128, 96), "float32", "direct"),
        # 32 items of one 128 x 128 tile each (fewer than half the SMs), K =
        # 256: latency-bound, DIRECT's whole-K tiles
        ((8, 1, 128, 256), (1, 4, 256, 64), "float32", "direct"),
        ((8, 1, 128, 512), (1, 4, 512, 64), "float32", "general_simt"),   # K past the whole-K bound
        ((0, 16, 32), (32, 8), "float32", "empty"),
        ((5, 0), (0, 7), "float32", "zero_fill"),
        ((4, 8192), (8192, 28672), "float16", "skinny_m"),
        ((16384, 4096), (4096, 8), "float16", "skinny_n"),
        ((32, 131072), (131072, 32), "float16", "split_k"),
        ((4096, 4096), (4096, 4096), "float32", "general_simt"),
        ((4096, 4096), (4096, 4096), "float64", "general_simt"),
    ]
    for a, b, dt, want in cases:
        with Plan(a, b, dt) as p:
            assert p.algorithm == want, (a, b, dt, p.describe())


def test_force_algorithm_feasibility():
    with Plan((40, 24), (24, 20), "float16") as p:
        p.force("direct")
        assert p.algorithm == "direct"
        p.force("general_simt")
        with pytest.raises(OlcError):
            p.force("skinny_m")          # 40 rows > 16
        with pytest.raises(OlcError):
            p.force("empty")
        p.force("auto")
    with Plan((3, 24), (24, 20), "float16") as p:
        with pytest.raises(OlcError):
            p.force("skinny_m")          # N * 2 bytes not a multiple of 16
    with Plan((3, 24), (24, 24), "float16") as p:
        p.force("skinny_m")
    with Plan((0, 4), (4, 4), "float32") as p:
        assert p.algorithm == "empty"
        with pytest.raises(OlcError):
            p.force("direct")
        p.force("empty")
    with Plan((2, 0), (0, 4), "float32") as p:
        assert p.algorithm == "zero_fill"
        p.force("zero_fill")


def test_workspace_and_launch_counts():
    with Plan((32, 131072), (131072, 32), "float16") as p:
        assert p.algorithm == "split_k"
        assert p.workspace_bytes > 0 and p.launches == 1
    with Plan((0, 16, 32), (32, 8), "float32") as p:
        assert p.launches == 0 and p.workspace_bytes == 0
    with Plan((64, 128), (128, 96), "float32") as p:
        assert p.workspace_bytes == 0 and p.launches == 1
        assert "direct" in p.describe()


def _field(v, lo, hi):
    return (v >> lo) & ((1 << (hi - lo + 1)) - 1)


def test_tcgen05_descriptor_bit_layout():
    """Field-by-field check of the descriptors the tensor-core kernel builds,
    against the PTX ISA tables (tcgen05 shared memory descriptor; instruction
    descriptor for kind::f16)."""
    lib = binding.load()
    lib.olc_debug_tc_smem_desc.argtypes = [ctypes.c_uint32] * 4
    lib.olc_debug_tc_smem_desc.restype = ctypes.c_uint64
    lib.olc_debug_tc_instr_desc.argtypes = [ctypes.c_int] * 5
    lib.olc_debug_tc_instr_desc.restype = ctypes.c_uint32
    d = lib.olc_debug_tc_smem_desc(0x1A400, 8192, 1024, 2)
    assert _field(d, 0, 13) == 0x1A400 >> 4      # start address >> 4
    assert _field(d, 14, 15) == 0
    assert _field(d, 16, 29) == 8192 >> 4        # leading byte offset >> 4
    assert _field(d, 32, 45) == 1024 >> 4        # stride byte offset >> 4
    assert _field(d, 46, 47) == 1                # fixed 0b01 for tcgen05
    assert _field(d, 49, 51) == 0                # base offset
    assert _field(d, 52, 52) == 0                # relative LBO mode
    assert _field(d, 61, 63) == 2                # 128-byte swizzle
    # the address field keeps 18 bits of byte address (256 KiB window)
    assert _field(lib.olc_debug_tc_smem_desc(0x3FFF0, 16, 1024, 2), 0, 13) == 0x3FFF
    for layout in (4, 6):   # 64-byte and 32-byte swizzle codes
        d = lib.olc_debug_tc_smem_desc(0x2000, 4096, 512, layout)
        assert _field(d, 61, 63) == layout and _field(d, 32, 45) == 512 >> 4
    for bf16 in (0, 1):
        i = lib.olc_debug_tc_instr_desc(bf16, 128, 256, 0, 1)
        assert _field(i, 0, 3) == 0                  # dense, no saturate
        assert _field(i, 4, 5) == 1                  # D = F32
        assert _field(i, 7, 9) == bf16               # A: 0 F16, 1 BF16
        assert _field(i, 10, 12) == bf16             # B
        assert _field(i, 13, 14) == 0                # no negation
        assert _field(i, 15, 15) == 0                # A K-major
        assert _field(i, 16, 16) == 1                # B MN-major
        assert _field(i, 17, 22) == 256 >> 3         # N
        assert _field(i, 23, 23) == 0
        assert _field(i, 24, 28) == 128 >> 4         # M
        assert _field(i, 29, 31) == 0
    # swapped operands: A MN-major, B K-major, N = 16
    i = lib.olc_debug_tc_instr_desc(0, 128, 16, 1, 0)
    assert _field(i, 15, 15) == 1 and _field(i, 16, 16) == 0
    assert _field(i, 17, 22) == 16 >> 3 and _field(i, 24, 28) == 128 >> 4


def test_constant_b_host_rejections():
    """No kernel runs: a plan without an owned B rejects the B-less execute,
    NULL plans are rejected, and a wrong-size B is refused before any copy."""
    lib = binding.load()
    assert lib.olc_matmul_plan_has_constant_b(None) == 0
    assert binding.STATUS[lib.olc_matmul_plan_set_constant_b(None, None, 0, None)] == "OLC_ERR_NULL"
    assert binding.STATUS[lib.olc_matmul_execute_constant(None, None, None, None)] == "OLC_ERR_NULL"
    with Plan((16, 32), (32, 24), "float32") as p:
        assert not p.has_constant_b
        st = lib.olc_matmul_execute_constant(p._h, None, None, None)
        assert binding.STATUS[st] == "OLC_ERR_NO_CONSTANT_B"
        st = lib.olc_gemm_execute_constant(p._h, None, None, None, None)
        assert binding.STATUS[st] == "OLC_ERR_NO_CONSTANT_B"
        st = lib.olc_matmul_plan_set_constant_b(p._h, None, 32 * 23, None)
        assert binding.STATUS[st] in ("OLC_ERR_BUFFER_TOO_SMALL", "OLC_ERR_NULL")
        assert not p.has_constant_b


def test_grouped_plan_host_checks():
    """No kernel runs: creation errors and the tile count of a group."""
    lib = binding.load()
    arr = ctypes.c_int64 * 3
    h = ctypes.c_void_p()
    m, n, k = arr(64, 65, 0), arr(64, 1, 5), arr(64, 8, 3)
    assert binding.STATUS[lib.olc_grouped_plan_create(0, m, n, k, 1, ctypes.byref(h))] == "OLC_ERR_INVALID"
    assert binding.STATUS[lib.olc_grouped_plan_create(3, None, n, k, 1, ctypes.byref(h))] == "OLC_ERR_NULL"
    assert binding.STATUS[lib.olc_grouped_plan_create(3, m, n, k, 7, ctypes.byref(h))] == "OLC_ERR_DTYPE"
    bad = arr(64, -1, 3)
    assert binding.STATUS[lib.olc_grouped_plan_create(3, m, bad, k, 1, ctypes.byref(h))] == "OLC_ERR_NEGATIVE_DIM"
    # a member above 2^62 bytes, or more than 2^31 - 1 tiles in all
    big = arr(1 << 31, 1, 1)
    assert binding.STATUS[lib.olc_grouped_plan_create(3, big, arr(1 << 31, 1, 1), k, 1,
                                                      ctypes.byref(h))] == "OLC_ERR_INVALID"
    assert binding.STATUS[lib.olc_grouped_plan_create(3, arr(1 << 22, 1, 1), arr(1 << 22, 1, 1), k, 10,
                                                      ctypes.byref(h))] == "OLC_ERR_INVALID"
    assert h.value is None
    assert lib.olc_grouped_plan_create(3, m, n, k, 1, ctypes.byref(h)) == 0
    assert lib.olc_grouped_plan_tiles(h) == 1 + 2 + 0      # a 0-row member owns no tiles
    assert lib.olc_grouped_plan_count(h) == 3
    lib.olc_grouped_plan_destroy(h)
    lib.olc_grouped_plan_destroy(None)
    assert lib.olc_grouped_plan_tiles(None) == -1


def test_f8_instruction_descriptor_layout():
    """kind::f8f6f4 instruction descriptor fields, as the FP8 kernel builds
    them: float32 accumulator (bits 4-5 = 1), A / B format (bits 7-9 /
    10-12: 0 = E4M3, 1 = E5M2), K-major operands (bits 15, 16 clear),
    N / 8 in bits 17-22, M / 16 in bits 24-28."""
    lib = binding.load()
    lib.olc_debug_f8_instr_desc.restype = ctypes.c_uint32
    for fmt in (0, 1):
        for m, n in ((128, 256), (128, 16), (64, 8)):
            d = lib.olc_debug_f8_instr_desc(fmt, m, n)
            assert (d >> 4) & 3 == 1
            assert (d >> 7) & 7 == fmt and (d >> 10) & 7 == fmt
            assert (d >> 15) & 3 == 0
            assert (d >> 17) & 0x3F == n // 8
            assert (d >> 24) & 0x1F == m // 16
            assert d & 0b1111 == 0 and (d >> 13) & 3 == 0 and (d >> 23) & 1 == 0 and d >> 29 == 0


def test_route_for_misaligned_pointers_and_odd_rows():
    """The host-side route an execute takes (no device needed): FP16 / BF16
    stay on their tensor-core kernels with staging copies for operands the
    TMA cannot read in place; a misaligned Y moves skinny and split-K
    products to the general tiles; other types fall back to DIRECT."""
    lib = binding.load()
    al, off = 1 << 20, (1 << 20) + 2          # 16-byte aligned, and two bytes off
    with Plan((300, 520), (520, 264), "bfloat16") as p:
        assert p.algorithm == "general_tc"
        h = p.handle
        assert lib.olc_matmul_plan_algorithm_for(h, al, al, al, None) == 6
        assert lib.olc_matmul_plan_staging_copies(h, al, al, al, None) == 0
        assert lib.olc_matmul_plan_staging_copies(h, off, al, al, None) == 1
        assert lib.olc_matmul_plan_staging_copies(h, off, off, off, None) == 2
        assert lib.olc_matmul_plan_algorithm_for(h, off, off, off, None) == 6
    with Plan((300, 515), (515, 263), "float16") as p:       # odd K and N: both staged
        assert p.algorithm == "general_tc" and p.launches == 3
        assert lib.olc_matmul_plan_staging_copies(p.handle, al, al, al, None) == 2
    with Plan((4, 8192), (8192, 512), "float16") as p:       # skinny-M
        h = p.handle
        assert p.algorithm == "skinny_m"
        assert lib.olc_matmul_plan_algorithm_for(h, off, al, al, None) == 3   # A copied densely
        assert lib.olc_matmul_plan_staging_copies(h, off, al, al, None) == 1
        assert lib.olc_matmul_plan_algorithm_for(h, al, al, off, None) == 6   # Y off: general tiles
    with Plan((64, 128), (128, 96), "float32") as p:
        h = p.handle
        assert lib.olc_matmul_plan_algorithm_for(h, al, al, al, None) == 2
    with Plan((1024, 1024), (1024, 1024), "float32") as p:
        h = p.handle
        assert p.algorithm == "general_simt"
        # the FFMA register tiles load element by element: any alignment
        assert lib.olc_matmul_plan_algorithm_for(h, al + 4, al, al, None) == 7
        assert lib.olc_matmul_plan_staging_copies(h, al + 4, al, al, None) == 0
    with Plan((4, 8192), (8192, 512), "float32") as p:
        h = p.handle
        assert p.algorithm == "skinny_m"
        assert lib.olc_matmul_plan_algorithm_for(h, al, al, al, None) == 3
        assert lib.olc_matmul_plan_algorithm_for(h, al + 4, al, al, None) == 2   # vector loads: DIRECT
    assert lib.olc_matmul_plan_algorithm_for(None, al, al, al, None) == -1


def test_few_tile_half_products_take_the_cluster_split_k():
    """FLOAT16 / BFLOAT16 products whose 128 x 256 tiles fill at most half the
    SMs stay on the general tiles, which then own a workspace of whole
    128 x 256 float32 partial tiles (tiles x K slices); the tiny-output
    corner (at most 32 x 32) and other types keep SPLIT_K, and products with
    many tiles own no workspace."""
    tile_bytes = 128 * 256 * 4
    for dt in ("bfloat16", "float16"):
        with Plan((64, 8192), (8192, 512), dt) as p:
            assert p.algorithm == "general_tc"
            ws = p.workspace_bytes
            assert ws > 0 and ws % (2 * tile_bytes) == 0 and 2 * 2 <= ws // tile_bytes <= 2 * 8
            # two tiles, each cut into the slices the description names
            assert " cluster_slices=%d " % (ws // (2 * tile_bytes)) in p.describe()
        with Plan((32, 131072), (131072, 32), dt) as p:
            assert p.algorithm == "split_k"
        with Plan((8, 2048, 4096), (4096, 14336), dt) as p:
            assert p.algorithm == "general_tc" and p.workspace_bytes == 0
            assert "cluster_slices" not in p.describe()
    with Plan((64, 8192), (8192, 512), "float32") as p:
        assert p.algorithm == "split_k"
    with Plan((64, 8192), (8192, 512), "bfloat16") as p:
        p.set_tc_variant(2)                  # forced pairs: no split, no workspace
        assert p.workspace_bytes == 0
