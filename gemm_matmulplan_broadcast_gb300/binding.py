"""ctypes binding over libolc_matmul.so (argument marshalling only).

Every computation happens in the library's CUDA kernels; this module turns
torch tensors into pointers, sizes and a stream handle, and status codes into
exceptions.  It never computes a result itself, and it raises if the library
has not been built -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libolc_matmul.so")
HEADER = os.path.join(ROOT, "include", "olc_matmul.h")

DTYPE_CODES = {"float32": 1, "float16": 10, "float64": 11, "bfloat16": 16,
               "float8_e4m3fn": 17, "float8_e4m3fnuz": 18, "float8_e5m2": 19,
               "float8_e5m2fnuz": 20}
ALGORITHMS = {
    "auto": -1, "empty": 0, "zero_fill": 1, "direct": 2, "skinny_m": 3, "skinny_n": 4,
    "split_k": 5, "general_tc": 6, "general_simt": 7,
}
ALGORITHM_NAMES = {v: k for k, v in ALGORITHMS.items()}
STATUS = {
    0: "OLC_OK", 1: "OLC_ERR_NULL", 2: "OLC_ERR_RANK", 3: "OLC_ERR_NEGATIVE_DIM",
    4: "OLC_ERR_K_MISMATCH", 5: "OLC_ERR_BATCH_MISMATCH", 6: "OLC_ERR_DTYPE",
    7: "OLC_ERR_ALIGNMENT", 8: "OLC_ERR_BUFFER_TOO_SMALL", 9: "OLC_ERR_NO_CONSTANT_B",
    10: "OLC_ERR_CUDA", 11: "OLC_ERR_DEVICE_TIMEOUT", 12: "OLC_ERR_OOM",
    13: "OLC_ERR_INVALID", 14: "OLC_ERR_WRONG_DEVICE", 15: "OLC_ERR_SCRATCH_LIMIT",
    16: "OLC_ERR_NEEDS_RESIDUAL",
}
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}
MAX_RANK = 8

_lock = threading.Lock()
_lib = None


class OlcError(RuntimeError):
    """A non-OK status from the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.name = STATUS.get(self.status, "status %d" % status)
        msg = load().olc_status_string(self.status).decode()
        super().__init__("%s: %s (%s)" % (where, self.name, msg))


def header_functions() -> list:
    """Names of the functions include/olc_matmul.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(olc_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def load():
    """Load libolc_matmul.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libolc_matmul.so is not built; run `python -m gemm_matmulplan_broadcast_gb300.build` "
                "(the CUDA library is required: there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        i64p = ctypes.POINTER(ctypes.c_int64)
        vp = ctypes.c_void_p
        sig = {
            "olc_matmul_plan_create": ([i64p, ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(vp)], ctypes.c_int),
            "olc_matmul_plan_destroy": ([vp], None),
            "olc_gemm_plan_create": ([i64p, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                      ctypes.c_double, i64p, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(vp)], ctypes.c_int),
            "olc_gemm_execute": ([vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_matmul_plan_set_constant_b": ([vp, vp, ctypes.c_int64, vp], ctypes.c_int),
            "olc_matmul_plan_has_constant_b": ([vp], ctypes.c_int),
            "olc_matmul_execute_constant": ([vp, vp, vp, vp], ctypes.c_int),
            "olc_matmul_plan_set_epilogue": ([vp, ctypes.c_int, ctypes.c_int], ctypes.c_int),
            "olc_grouped_plan_create": ([ctypes.c_int, i64p, i64p, i64p, ctypes.c_int,
                                         ctypes.POINTER(vp)], ctypes.c_int),
            "olc_grouped_plan_destroy": ([vp], None),
            "olc_grouped_plan_tiles": ([vp], ctypes.c_int64),
            "olc_grouped_plan_count": ([vp], ctypes.c_int),
            "olc_grouped_execute": ([vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_matmul_execute_fused": ([vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_gemm_execute_constant": ([vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_matmul_execute": ([vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_matmul_execute_checked": ([vp, vp, ctypes.c_int64, vp, ctypes.c_int64, vp,
                                            ctypes.c_int64, vp], ctypes.c_int),
            "olc_matmul_execute_host": ([vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_matmul_plan_output_shape": ([vp, i64p, ctypes.c_int, ctypes.POINTER(ctypes.c_int)],
                                             ctypes.c_int),
            "olc_matmul_plan_dims": ([vp, i64p, i64p, i64p, i64p], ctypes.c_int),
            "olc_matmul_plan_batch": ([vp, ctypes.POINTER(ctypes.c_int), i64p, i64p, i64p],
                                      ctypes.c_int),
            "olc_matmul_plan_launch_shape": ([vp, i64p, i64p, ctypes.POINTER(ctypes.c_int)],
                                             ctypes.c_int),
            "olc_matmul_plan_algorithm": ([vp], ctypes.c_int),
            "olc_matmul_plan_force_algorithm": ([vp, ctypes.c_int], ctypes.c_int),
            "olc_matmul_plan_launches": ([vp], ctypes.c_int),
            "olc_matmul_plan_set_splits": ([vp, ctypes.c_int], ctypes.c_int),
            "olc_matmul_plan_splits": ([vp], ctypes.c_int),
            "olc_matmul_plan_set_tc_variant": ([vp, ctypes.c_int], ctypes.c_int),
            "olc_matmul_plan_workspace_bytes": ([vp], ctypes.c_size_t),
            "olc_matmul_plan_describe": ([vp, ctypes.c_char_p, ctypes.c_size_t], ctypes.c_int),
            "olc_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "olc_algorithm_name": ([ctypes.c_int], ctypes.c_char_p),
            "olc_version": ([], ctypes.c_int),
            "olc_matmul_plan_algorithm_for": ([vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_matmul_plan_staging_copies": ([vp, vp, vp, vp, vp], ctypes.c_int),
            "olc_debug_alu_rate": ([ctypes.c_int, ctypes.c_int64, vp, ctypes.POINTER(ctypes.c_double)],
                                   ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _shape_arr(shape: Sequence[int]):
    arr = (ctypes.c_int64 * max(1, len(shape)))(*[int(d) for d in shape])
    return arr


def _check(status: int, where: str):
    if status != 0:
        raise OlcError(status, where)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr() if t.numel() > 0 else None


class Plan:
    """A MatMul plan: Y = MatMul(A, B) for fixed shapes and element type.

    MatMul Kernel Design, section "Shape and plan model": the plan resolves
    promotion, broadcasting, batch strides and the GEMM algorithm once;
    ``execute`` then enqueues the kernels.
    """

    def __init__(self, a_shape, b_shape, dtype: str):
        self.lib = load()
        self.a_shape = tuple(int(d) for d in a_shape)
        self.b_shape = tuple(int(d) for d in b_shape)
        if dtype not in DTYPE_CODES:
            raise ValueError("unsupported dtype %r" % (dtype,))
        self.dtype = dtype
        h = ctypes.c_void_p()
        st = self.lib.olc_matmul_plan_create(_shape_arr(self.a_shape), len(self.a_shape),
                                             _shape_arr(self.b_shape), len(self.b_shape),
                                             DTYPE_CODES[dtype], ctypes.byref(h))
        _check(st, "olc_matmul_plan_create")
        self._h = h

    # -- lifetime --------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self.lib.olc_matmul_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def handle(self):
        return self._h

    # -- queries ---------------------------------------------------------
    @property
    def output_shape(self):
        buf = (ctypes.c_int64 * MAX_RANK)()
        r = ctypes.c_int()
        _check(self.lib.olc_matmul_plan_output_shape(self._h, buf, MAX_RANK, ctypes.byref(r)),
               "olc_matmul_plan_output_shape")
        return tuple(buf[i] for i in range(r.value))

    def dims(self):
        m, n, k, b = (ctypes.c_int64() for _ in range(4))
        _check(self.lib.olc_matmul_plan_dims(self._h, ctypes.byref(m), ctypes.byref(n),
                                             ctypes.byref(k), ctypes.byref(b)), "dims")
        return m.value, n.value, k.value, b.value

    def batch(self):
        r = ctypes.c_int()
        shape, sa, sb = ((ctypes.c_int64 * MAX_RANK)() for _ in range(3))
        _check(self.lib.olc_matmul_plan_batch(self._h, ctypes.byref(r), shape, sa, sb), "batch")
        n = r.value
        return tuple(shape[:n]), tuple(sa[:n]), tuple(sb[:n])

    def launch_shape(self):
        rows, items, rank = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int()
        _check(self.lib.olc_matmul_plan_launch_shape(self._h, ctypes.byref(rows), ctypes.byref(items),
                                                     ctypes.byref(rank)), "launch_shape")
        return rows.value, items.value, rank.value

    @property
    def algorithm(self) -> str:
        return ALGORITHM_NAMES[self.lib.olc_matmul_plan_algorithm(self._h)]

    def algorithm_for(self, A, B, Y, R=None) -> str:
        """The algorithm an execute with these tensors runs (host query)."""
        a = self.lib.olc_matmul_plan_algorithm_for(self._h, _ptr(A), _ptr(B), _ptr(Y), _ptr(R))
        return ALGORITHM_NAMES.get(a, str(a))

    def staging_copies(self, A, B, Y, R=None) -> int:
        """Staging copies an execute with these tensors makes (host query)."""
        return int(self.lib.olc_matmul_plan_staging_copies(self._h, _ptr(A), _ptr(B), _ptr(Y), _ptr(R)))

    def force(self, algorithm: str):
        _check(self.lib.olc_matmul_plan_force_algorithm(self._h, ALGORITHMS[algorithm]),
               "olc_matmul_plan_force_algorithm(%s)" % algorithm)
        return self

    def set_splits(self, splits: int):
        """Tuning override of the K-slice count (0 = automatic)."""
        _check(self.lib.olc_matmul_plan_set_splits(self._h, int(splits)), "set_splits")
        return self

    def set_tc_variant(self, variant: int):
        """Tuning override of the tensor-core tiling: 0 automatic, 1 one CTA
        per 128 x 256 tile, 2 CTA pairs with 256 x 256 tiles."""
        _check(self.lib.olc_matmul_plan_set_tc_variant(self._h, int(variant)), "set_tc_variant")
        return self

    @property
    def splits(self) -> int:
        return int(self.lib.olc_matmul_plan_splits(self._h))

    @property
    def launches(self) -> int:
        return int(self.lib.olc_matmul_plan_launches(self._h))

    @property
    def workspace_bytes(self) -> int:
        return int(self.lib.olc_matmul_plan_workspace_bytes(self._h))

    def describe(self) -> str:
        buf = ctypes.create_string_buffer(512)
        self.lib.olc_matmul_plan_describe(self._h, buf, 512)
        return buf.value.decode()

    # -- execution -------------------------------------------------------
    def _check_tensors(self, A, B, Y):
        import torch
        from .synth import TORCH_DTYPES, output_dtype
        for name, t, shape in (("A", A, self.a_shape), ("B", B, self.b_shape),
                               ("Y", Y, self.output_shape)):
            if t is None:
                continue
            want = TORCH_DTYPES[output_dtype(self.dtype) if name == "Y" else self.dtype]
            if t.dtype != want:
                raise TypeError("%s has dtype %s, plan is %s" % (name, t.dtype, self.dtype))
            if tuple(t.shape) != tuple(shape):
                raise ValueError("%s has shape %s, plan wants %s" % (name, tuple(t.shape), shape))
            if t.numel() > 0 and not t.is_contiguous():
                raise ValueError("%s must be contiguous" % name)
            if t.numel() > 0 and t.device.type != "cuda":
                raise ValueError("%s must be a CUDA tensor" % name)
        return torch

    def execute(self, A, B, Y, stream=None):
        """Enqueue Y = MatMul(A, B) (device tensors) on ``stream``."""
        self._check_tensors(A, B, Y)
        st = self.lib.olc_matmul_execute(self._h, _ptr(A), _ptr(B), _ptr(Y),
                                         _stream_handle(stream))
        _check(st, "olc_matmul_execute")
        return Y

    def execute_checked(self, A, B, Y, stream=None):
        """Execute with buffer-size validation, then synchronise and read the
        device error word."""
        st = self.lib.olc_matmul_execute_checked(
            self._h, _ptr(A), A.numel() if A is not None else 0, _ptr(B),
            B.numel() if B is not None else 0, _ptr(Y), Y.numel() if Y is not None else 0,
            _stream_handle(stream))
        _check(st, "olc_matmul_execute_checked")
        return Y

    def execute_host(self, A_host, B_host, Y_host, A_dev, B_dev, Y_dev, stream=None):
        """Host buffers in and out, staged through the caller's device
        buffers; everything is enqueued on ``stream``."""
        st = self.lib.olc_matmul_execute_host(self._h, _ptr(A_host), _ptr(B_host), _ptr(Y_host),
                                              _ptr(A_dev), _ptr(B_dev), _ptr(Y_dev),
                                              _stream_handle(stream))
        _check(st, "olc_matmul_execute_host")
        return Y_host

    def set_constant_b(self, B, stream=None):
        """Copy B (host or device tensor of the planned shape) into storage
        the plan owns; later executes may omit B."""
        st = self.lib.olc_matmul_plan_set_constant_b(self._h, _ptr(B), B.numel(),
                                                     _stream_handle(stream))
        _check(st, "olc_matmul_plan_set_constant_b")
        return self

    @property
    def has_constant_b(self) -> bool:
        return bool(self.lib.olc_matmul_plan_has_constant_b(self._h))

    def execute_constant(self, A, Y, stream=None):
        """Y = MatMul(A, plan-owned B)."""
        self._check_tensors(A, None, Y)
        st = self.lib.olc_matmul_execute_constant(self._h, _ptr(A), _ptr(Y), _stream_handle(stream))
        _check(st, "olc_matmul_execute_constant")
        return Y

    def set_epilogue(self, act: str = "none", residual: bool = False):
        """Fuse a residual add and an activation into the product's store."""
        if act not in ACTIVATIONS:
            raise ValueError("activation must be one of %s" % sorted(ACTIVATIONS))
        st = self.lib.olc_matmul_plan_set_epilogue(self._h, ACTIVATIONS[act], int(bool(residual)))
        _check(st, "olc_matmul_plan_set_epilogue")
        self.epilogue = (act, bool(residual))
        return self

    def execute_fused(self, A, B, Y, R=None, C=None, stream=None):
        """Y = act(product (+ bias) + R); B None = the plan-owned B."""
        self._check_tensors(A, B, Y)
        if R is not None:
            self._check_tensors(None, None, R)
        st = self.lib.olc_matmul_execute_fused(self._h, _ptr(A), _ptr(B), _ptr(C), _ptr(R),
                                               _ptr(Y), _stream_handle(stream))
        _check(st, "olc_matmul_execute_fused")
        return Y

    def __call__(self, A, B, out=None, stream=None):
        import torch
        from .synth import TORCH_DTYPES, output_dtype
        if out is None:
            out = torch.empty(self.output_shape, dtype=TORCH_DTYPES[output_dtype(self.dtype)],
                              device=A.device)
        return self.execute(A, B, out, stream)


class GemmPlan(Plan):
    """A Gemm plan: Y = alpha * A' B' + beta * C (rank-2, transA / transB,
    C broadcast to [M, N]; c_shape None = no C)."""

    def __init__(self, a_shape, b_shape, dtype: str, trans_a=False, trans_b=False, alpha=1.0,
                 beta=1.0, c_shape=None):
        self.lib = load()
        self.a_shape = tuple(int(d) for d in a_shape)
        self.b_shape = tuple(int(d) for d in b_shape)
        if dtype not in DTYPE_CODES:
            raise ValueError("unsupported dtype %r" % (dtype,))
        if len(self.a_shape) != 2 or len(self.b_shape) != 2:
            raise ValueError("Gemm takes rank-2 A and B")
        self.dtype = dtype
        self.trans_a, self.trans_b = bool(trans_a), bool(trans_b)
        self.c_shape = None if c_shape is None else tuple(int(d) for d in c_shape)
        h = ctypes.c_void_p()
        c_rank = -1 if self.c_shape is None else len(self.c_shape)
        st = self.lib.olc_gemm_plan_create(
            _shape_arr(self.a_shape), _shape_arr(self.b_shape), int(self.trans_a),
            int(self.trans_b), float(alpha), float(beta),
            _shape_arr(self.c_shape or ()), c_rank, DTYPE_CODES[dtype], ctypes.byref(h))
        _check(st, "olc_gemm_plan_create")
        self._h = h

    def execute(self, A, B, Y, stream=None, C=None):
        """Enqueue the Gemm (device tensors) on ``stream``."""
        self._check_tensors(A, B, Y)
        st = self.lib.olc_gemm_execute(self._h, _ptr(A), _ptr(B), _ptr(C), _ptr(Y),
                                       _stream_handle(stream))
        _check(st, "olc_gemm_execute")
        return Y

    def execute_constant(self, A, Y, stream=None, C=None):
        """The Gemm with the plan-owned B."""
        self._check_tensors(A, None, Y)
        st = self.lib.olc_gemm_execute_constant(self._h, _ptr(A), _ptr(C), _ptr(Y),
                                                _stream_handle(stream))
        _check(st, "olc_gemm_execute_constant")
        return Y


class GroupedPlan:
    """A group of independent rank-2 products Y_i = A_i @ B_i with their own
    shapes, run in one launch.  `shapes`: list of (m, n, k)."""

    def __init__(self, shapes, dtype: str):
        from .synth import ONNX_CODES
        self.lib = load()
        self.shapes = [tuple(int(x) for x in sh) for sh in shapes]
        self.dtype = dtype
        cnt = len(self.shapes)
        arr = ctypes.c_int64 * max(cnt, 1)
        m = arr(*[sh[0] for sh in self.shapes])
        n = arr(*[sh[1] for sh in self.shapes])
        k = arr(*[sh[2] for sh in self.shapes])
        h = ctypes.c_void_p()
        _check(self.lib.olc_grouped_plan_create(cnt, m, n, k, ONNX_CODES[dtype], ctypes.byref(h)),
               "olc_grouped_plan_create")
        self._h = h
        self._keep = None

    @property
    def tiles(self) -> int:
        return int(self.lib.olc_grouped_plan_tiles(self._h))

    def execute(self, As, Bs, Ys, stream=None):
        """As, Bs, Ys: lists of CUDA tensors (member i: [m, k], [k, n], [m, n])."""
        import torch
        from .synth import TORCH_DTYPES
        if not (len(As) == len(Bs) == len(Ys) == len(self.shapes)):
            raise ValueError("need one A, B and Y per member")
        want = TORCH_DTYPES[self.dtype]
        for (m, n, k), a, b, y in zip(self.shapes, As, Bs, Ys):
            for name, t, shp in (("A", a, (m, k)), ("B", b, (k, n)), ("Y", y, (m, n))):
                if tuple(t.shape) != shp or t.dtype != want:
                    raise ValueError("%s of a member is %s %s, want %s %s" % (name, tuple(t.shape), t.dtype, shp, want))
                if t.numel() > 0 and (not t.is_contiguous() or t.device.type != "cuda"):
                    raise ValueError("%s must be a contiguous CUDA tensor" % name)
        ptrs = self.pointer_arrays(As, Bs, Ys)
        self.execute_ptrs(*ptrs, stream=stream)
        self._keep = ptrs        # the kernel reads the pointer arrays asynchronously
        return Ys

    @staticmethod
    def pointer_arrays(As, Bs, Ys):
        """Device int64 arrays of the members' A, B and Y addresses (built
        once, reusable while the tensors live; synchronous upload)."""
        import torch
        dev = next((t.device for t in list(As) + list(Ys) if t.numel() > 0), torch.device("cuda"))
        return tuple(torch.tensor([_ptr(t) or 0 for t in ts], dtype=torch.int64, device=dev)
                     for ts in (As, Bs, Ys))

    def execute_ptrs(self, a_ptrs, b_ptrs, y_ptrs, stream=None):
        """Run the group from prebuilt device pointer arrays (no host work
        beyond the launch; capturable in a CUDA graph)."""
        st = self.lib.olc_grouped_execute(self._h, a_ptrs.data_ptr(), b_ptrs.data_ptr(),
                                          y_ptrs.data_ptr(), _stream_handle(stream))
        _check(st, "olc_grouped_execute")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self.lib.olc_grouped_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def alu_rate(kind: int, iters: int, stream=None) -> float:
    """flop/s of the library's FMA-pipe probe (olc_debug_alu_rate): kind 0
    paired FP32 FMA, 1 FP32 FMA, 2 FP64 FMA, 3 FP64 tensor-core MMA."""
    out = ctypes.c_double(0.0)
    st = load().olc_debug_alu_rate(int(kind), int(iters), _stream_handle(stream), ctypes.byref(out))
    _check(st, "olc_debug_alu_rate")
    return float(out.value)


def gemm(A, B, C=None, alpha=1.0, beta=1.0, trans_a=False, trans_b=False, out=None, stream=None):
    """ONNX Gemm of CUDA tensors through a fresh plan."""
    import torch
    from .synth import TORCH_DTYPES
    inv = {v: k for k, v in TORCH_DTYPES.items()}
    with GemmPlan(A.shape, B.shape, inv[A.dtype], trans_a, trans_b, alpha, beta,
                  None if C is None else C.shape) as plan:
        if out is None:
            out = torch.empty(plan.output_shape, dtype=A.dtype, device=A.device)
        return plan.execute(A, B, out, stream=stream, C=C)


def matmul(A, B, out=None, stream=None, algorithm: Optional[str] = None):
    """ONNX MatMul of two CUDA tensors through a fresh plan."""
    from .synth import TORCH_DTYPES
    inv = {v: k for k, v in TORCH_DTYPES.items()}
    if A.dtype != B.dtype:
        raise TypeError("MatMul needs equal-typed operands, got %s and %s" % (A.dtype, B.dtype))
    if A.dtype not in inv:
        raise TypeError("unsupported dtype %s" % A.dtype)
    with Plan(A.shape, B.shape, inv[A.dtype]) as plan:
        if algorithm is not None:
            plan.force(algorithm)
        return plan(A, B, out=out, stream=stream)
