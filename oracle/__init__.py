"""ORACLE -- test infrastructure only.

A plain CPU restatement of the ONNX ``MatMul`` operator used to check the CUDA
library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it; the product package never does, and this
package imports nothing from the product.

Two halves:

* ``oracle.c`` (compiled on first use with gcc into ``oracle/_build``): the
  2-D product with the pages' accumulation rules and the binary16 / bfloat16
  encode and decode.
* this module: the shape rules and the batch loop.

Shape rules (MatMul Kernel Design, section "Shape and plan model"; Gemm and
MatMul Performance Roadmap, section "Phase 4: complete MatMul"):

1. a rank-one A ``[K]`` is read as ``[1, K]`` and a rank-one B ``[K]`` as
   ``[K, 1]``; the promoted dimension is dropped from the output;
2. the leading (batch) dimensions of the two operands are aligned on the
   right and broadcast: equal extents stay, an extent of 1 stretches to the
   other operand's extent, anything else is an error;
3. every output batch item ``b`` multiplies the A matrix and the B matrix that
   ``b`` selects, where an operand's index along a dimension it broadcasts
   (extent 1) is 0;
4. an output with no elements is returned without reading the inputs.

Readings where the pages are silent: rank-0
operands are rejected; broadcasting an extent 0 against 1 gives 0 and against
n > 1 is an error; K == 0 with a non-empty output gives zeros; two rank-one
operands give a rank-0 (one element) output.

Values are passed as numpy arrays: float32 / float64 for FLOAT / DOUBLE, and
uint16 bit patterns for FLOAT16 / BFLOAT16 (numpy has no bfloat16).
"""

from __future__ import annotations

import ctypes
import itertools
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_lock = threading.Lock()
_lib = None

DTYPES = ("float32", "float64", "float16", "bfloat16")
FP8_DTYPES = ("float8_e4m3fn", "float8_e5m2", "float8_e4m3fnuz", "float8_e5m2fnuz")


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        for name in ("oracle_gemm_f32", "oracle_gemm_f64", "oracle_gemm_f16", "oracle_gemm_bf16",
                     "oracle_gemm_f16_acc", "oracle_gemm_bf16_acc"):
            fn = getattr(lib, name)
            fn.argtypes = [i64, i64, i64, p, p, p, i64, p, p]
            fn.restype = None
        for name in ("oracle_decode_f16", "oracle_decode_bf16", "oracle_encode_f16",
                     "oracle_encode_bf16"):
            fn = getattr(lib, name)
            fn.argtypes = [p, p, i64]
            fn.restype = None
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_threads.restype = None
        _lib = lib
        return lib


def threads() -> int:
    """Host threads the oracle's parallel loops use."""
    return int(_load().oracle_threads())


def set_threads(n: int) -> None:
    """Use `n` host threads from now on (1: a single-core timing).  Results
    do not depend on it: each output row is one thread's k-ordered sum."""
    _load().oracle_set_threads(int(n))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# binary16 / bfloat16 bit patterns <-> float32

def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 patterns of ``dtype`` ("float16" / "bfloat16") -> exact float32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float32)
    fn = _load().oracle_decode_f16 if dtype == "float16" else _load().oracle_decode_bf16
    fn(_ptr(bits), _ptr(out), bits.size)
    return out


def encode(values: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> uint16 patterns of ``dtype``, round to nearest even."""
    values = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(values.shape, np.uint16)
    fn = _load().oracle_encode_f16 if dtype == "float16" else _load().oracle_encode_bf16
    fn(_ptr(values), _ptr(out), values.size)
    return out


# --------------------------------------------------------------------------
# 8-bit float operands
#
# "Gemm and MatMul Performance Roadmap", the Float8 packing-format item:
# each one-byte pattern of a Float8 format is decoded exactly to float32 and
# the float32 algorithm runs with float32 accumulation.  The two formats
# built here are E4M3FN (1 sign, 4 exponent bits with bias 7, 3 mantissa
# bits; no infinities; S.1111.111 is NaN), E5M2 (1 sign, 5 exponent bits
# with bias 15, 2 mantissa bits; IEEE-style infinities and NaNs), and the two
# "FNUZ" variants the roadmap lists beside them: E4M3FNUZ and E5M2FNUZ have
# the same fields with the exponent bias one larger (8 and 16), no
# infinities, no negative zero, and the one pattern 1.0000.000 (0x80) as NaN.
# Reading where the page is silent: the output is FLOAT (the float32 sums are
# not narrowed), and both operands have the same format.


def decode_fp8(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint8 patterns of an 8-bit float format -> exact float32 values,
    written from the format's fields (decode_fp8_fields), looked up from
    the 256 decoded patterns so that large operands cost one gather."""
    table = decode_fp8_fields(np.arange(256, dtype=np.uint8), dtype)
    return table[np.asarray(bits, dtype=np.uint8)]


def decode_fp8_fields(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint8 patterns of an 8-bit float format -> exact float32 values,
    decoded element by element from the sign, exponent and mantissa fields."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    if dtype == "float8_e4m3fn":
        e, m = (b >> 3) & 0xF, b & 0x7
        mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
        mag = np.where((b & 0x7F) == 0x7F, np.nan, mag)
    elif dtype == "float8_e5m2":
        e, m = (b >> 2) & 0x1F, b & 0x3
        mag = np.where(e == 0, m * 2.0 ** -16, (1.0 + m / 4.0) * np.exp2(e - 15.0))
        mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    elif dtype == "float8_e4m3fnuz":
        e, m = (b >> 3) & 0xF, b & 0x7
        mag = np.where(e == 0, m * 2.0 ** -10, (1.0 + m / 8.0) * np.exp2(e - 8.0))
        mag = np.where(b == 0x80, np.nan, mag)
        sign = np.where(b == 0x80, 1.0, sign)
    elif dtype == "float8_e5m2fnuz":
        e, m = (b >> 2) & 0x1F, b & 0x3
        mag = np.where(e == 0, m * 2.0 ** -17, (1.0 + m / 4.0) * np.exp2(e - 16.0))
        mag = np.where(b == 0x80, np.nan, mag)
        sign = np.where(b == 0x80, 1.0, sign)
    else:
        raise ValueError("not an 8-bit float type: %r" % dtype)
    return (sign * mag).astype(np.float32)


# --------------------------------------------------------------------------
# shape rules

class ShapeError(ValueError):
    """The operand shapes have no MatMul product."""


def output_shape(a_shape, b_shape):
    """Output shape of MatMul(A, B), following the promote / broadcast /
    squeeze rules above.  Raises ShapeError for shapes with no product."""
    a_shape, b_shape = [int(d) for d in a_shape], [int(d) for d in b_shape]
    if len(a_shape) == 0 or len(b_shape) == 0:
        raise ShapeError("rank-0 operand")
    if any(d < 0 for d in a_shape + b_shape):
        raise ShapeError("negative dimension")
    a2 = [1] + a_shape if len(a_shape) == 1 else a_shape
    b2 = b_shape + [1] if len(b_shape) == 1 else b_shape
    m, ka = a2[-2], a2[-1]
    kb, n = b2[-2], b2[-1]
    if ka != kb:
        raise ShapeError("inner dimensions differ: %d vs %d" % (ka, kb))
    batch = _broadcast(a2[:-2], b2[:-2])
    out = list(batch)
    if len(a_shape) > 1:
        out.append(m)
    if len(b_shape) > 1:
        out.append(n)
    return tuple(out)


def _broadcast(a_batch, b_batch):
    """Right-aligned multidirectional broadcast of two batch shapes."""
    r = max(len(a_batch), len(b_batch))
    a = [1] * (r - len(a_batch)) + list(a_batch)
    b = [1] * (r - len(b_batch)) + list(b_batch)
    out = []
    for da, db in zip(a, b):
        if da == db:
            out.append(da)
        elif da == 1:
            out.append(db)
        elif db == 1:
            out.append(da)
        else:
            raise ShapeError("batch dimensions %d and %d do not broadcast" % (da, db))
    return out


# --------------------------------------------------------------------------
# the product

def gemm2d(a: np.ndarray, b: np.ndarray, dtype: str, rows=None):
    """One 2-D product A[M, K] @ B[K, N] with the accumulation rules of
    ``dtype``.  ``rows``: optional list of output rows to compute.  Returns
    (Y, S) with Y in the storage type of ``dtype`` and S = sum |a||b| (float64),
    both [len(rows) or M, N]."""
    lib = _load()
    store = {"float32": np.float32, "float64": np.float64,
             "float16": np.uint16, "bfloat16": np.uint16}[dtype]
    a = np.ascontiguousarray(a, dtype=store)
    b = np.ascontiguousarray(b, dtype=store)
    m, k = a.shape
    k2, n = b.shape
    assert k == k2
    if rows is None:
        rows_arr, nrows, rows_p = None, m, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        assert rows_arr.size == 0 or (rows_arr.min() >= 0 and rows_arr.max() < m)
        nrows, rows_p = rows_arr.size, _ptr(rows_arr)
    y = np.zeros((nrows, n), store)
    s = np.zeros((nrows, n), np.float64)
    if nrows == 0 or n == 0:
        return y, s
    fn = {"float32": lib.oracle_gemm_f32, "float64": lib.oracle_gemm_f64,
          "float16": lib.oracle_gemm_f16, "bfloat16": lib.oracle_gemm_bf16}[dtype]
    fn(m, n, k, _ptr(a), _ptr(b), rows_p, nrows, _ptr(y), _ptr(s))
    return y, s


def matmul(a: np.ndarray, b: np.ndarray, dtype: str):
    """ONNX MatMul of two dense row-major arrays.  Returns (Y, S), both of the
    output shape; Y in the storage type of ``dtype``, S = sum |a||b| per
    output element (float64).  8-bit float operands (uint8 patterns) give a
    float32 Y."""
    if dtype in FP8_DTYPES:
        return matmul(decode_fp8(a, dtype), decode_fp8(b, dtype), "float32")
    if dtype not in DTYPES:
        raise ValueError("unsupported dtype %r" % dtype)
    out_shape = output_shape(a.shape, b.shape)
    store = {"float32": np.float32, "float64": np.float64,
             "float16": np.uint16, "bfloat16": np.uint16}[dtype]
    a2 = a.reshape((1,) + a.shape) if a.ndim == 1 else a
    b2 = b.reshape(b.shape + (1,)) if b.ndim == 1 else b
    m, n = a2.shape[-2], b2.shape[-1]
    batch = _broadcast(a2.shape[:-2], b2.shape[:-2])
    r = len(batch)
    a_batch = [1] * (r - (a2.ndim - 2)) + list(a2.shape[:-2])
    b_batch = [1] * (r - (b2.ndim - 2)) + list(b2.shape[:-2])
    a3 = a2.reshape(a_batch + [m, a2.shape[-1]])
    b3 = b2.reshape(b_batch + [b2.shape[-2], n])
    y = np.zeros(batch + [m, n], store)
    s = np.zeros(batch + [m, n], np.float64)
    for idx in itertools.product(*[range(d) for d in batch]):
        ia = tuple(0 if da == 1 else i for i, da in zip(idx, a_batch))
        ib = tuple(0 if db == 1 else i for i, db in zip(idx, b_batch))
        y[idx], s[idx] = gemm2d(a3[ia], b3[ib], dtype)
    return y.reshape(out_shape), s.reshape(out_shape)


def to_float64(y: np.ndarray, dtype: str) -> np.ndarray:
    """Values of a result array as float64 (16-bit patterns decoded; the
    float32 results of 8-bit float operands as they are)."""
    if dtype in ("float16", "bfloat16"):
        return decode(y, dtype).astype(np.float64)
    return y.astype(np.float64)


# --------------------------------------------------------------------------
# the Gemm operator (rank-2, transA / transB, alpha, beta, broadcast C)
#
# "Gemm and MatMul Performance Roadmap", section "Scope and type matrix":
# Gemm handles rank-2 inputs, alpha, beta, an optional broadcast bias and
# transA / transB, on the same engine as MatMul.  It computes
#     Y = alpha * A' B' + beta * C,   A' = A^T if transA else A,  B' likewise,
# with C broadcast unidirectionally to [M, N] (absent C: no bias term).
# Reading where the page is silent: the epilogue alpha * acc + beta * c is
# evaluated in the accumulator type (float32 for FLOAT, FLOAT16, BFLOAT16;
# float64 for DOUBLE), each operation rounded, and FLOAT16 / BFLOAT16 are
# narrowed once at the end.


def gemm_output_shape(a_shape, b_shape, trans_a, trans_b, c_shape=None):
    """(M, N, K) of Gemm, or ShapeError."""
    if len(a_shape) != 2 or len(b_shape) != 2:
        raise ShapeError("Gemm takes rank-2 A and B")
    if any(int(d) < 0 for d in tuple(a_shape) + tuple(b_shape)):
        raise ShapeError("negative dimension")
    m, ka = (a_shape[1], a_shape[0]) if trans_a else (a_shape[0], a_shape[1])
    kb, n = (b_shape[1], b_shape[0]) if trans_b else (b_shape[0], b_shape[1])
    if ka != kb:
        raise ShapeError("inner dimensions differ: %d vs %d" % (ka, kb))
    if c_shape is not None:
        c = [int(d) for d in c_shape]
        if len(c) > 2:
            raise ShapeError("C has rank > 2")
        c = [1] * (2 - len(c)) + c
        if not (c[0] in (1, m) and c[1] in (1, n)):
            raise ShapeError("C %s does not broadcast to [%d, %d]" % (tuple(c_shape), m, n))
    return int(m), int(n), int(ka)


def _acc2d(a, b, dtype):
    """The accumulator of one 2-D product before narrowing: float32 for
    FLOAT / FLOAT16 / BFLOAT16, float64 for DOUBLE; plus S = sum |a||b|."""
    if dtype in ("float16", "bfloat16"):
        m, k = a.shape
        n = b.shape[1]
        acc = np.zeros((m, n), np.float32)
        s = np.zeros((m, n), np.float64)
        if m and n:
            lib = _load()
            fn = lib.oracle_gemm_f16_acc if dtype == "float16" else lib.oracle_gemm_bf16_acc
            a16 = np.ascontiguousarray(a, np.uint16)
            b16 = np.ascontiguousarray(b, np.uint16)
            fn(m, n, k, _ptr(a16), _ptr(b16), None, m, _ptr(acc), _ptr(s))
        return acc, s
    acc, s = gemm2d(a, b, dtype)
    return acc.astype(np.float64 if dtype == "float64" else np.float32), s


def _wide(dtype):
    return np.float64 if dtype == "float64" else np.float32


def _values(x, dtype):
    """Operand values in the accumulator type (16-bit patterns decoded)."""
    x = np.asarray(x)
    if dtype in ("float16", "bfloat16"):
        return to_float64(x, dtype).astype(np.float32)
    return x.astype(_wide(dtype))


def gemm_op(a, b, dtype, c=None, alpha=1.0, beta=1.0, trans_a=False, trans_b=False,
            residual=None, act="none"):
    """ONNX Gemm, optionally followed by the fused residual and activation
    (see ``fused_epilogue``).  Returns (Y, S) with S the tolerance scale
    L * (|alpha| sum|a||b| + |beta| |c| + |r|) (float64), L the activation's
    Lipschitz constant."""
    m, n, k = gemm_output_shape(a.shape, b.shape, trans_a, trans_b,
                                None if c is None else c.shape)
    ap = np.ascontiguousarray(a.T if trans_a else a)
    bp = np.ascontiguousarray(b.T if trans_b else b)
    wide = _wide(dtype)
    acc, s = _acc2d(ap, bp, dtype)
    y = wide(alpha) * acc
    scale = abs(float(alpha)) * s
    if c is not None:
        cv = _values(c, dtype)
        cb = np.broadcast_to(cv.reshape([1] * (2 - cv.ndim) + list(cv.shape)), (m, n))
        y = y + wide(beta) * cb
        scale = scale + abs(float(beta)) * np.abs(cb.astype(np.float64))
    return fused_epilogue(np.asarray(y, wide), scale, dtype, residual, act)


# --------------------------------------------------------------------------
# the fused epilogue (bias, residual, activation, narrowing)
#
# "Gemm and MatMul Performance Roadmap": the fused-epilogue row of its
# opportunity table (each following elementwise operator fused into the
# product saves one read and one write of the output) and the broadcast /
# fused epilogue item of its plan (bias, residual, activation and output
# conversion in one typed epilogue, no intermediate tensor).  Readings where
# the page is silent: the steps run in the order the page lists them --
# bias, then residual, then activation, then narrowing; the residual has the
# output's shape and type; the activations are ReLU, max(v, 0), and the exact
# GELU, v * Phi(v) = v / 2 * (1 + erf(v / sqrt 2)) = v / 2 * erfc(-v / sqrt 2)
# (the erfc form is the one evaluated); the residual sum is
# rounded in the accumulator type, the activation is evaluated in float64
# and rounded to the accumulator type, and the result is narrowed once.

ACTIVATIONS = ("none", "relu", "gelu")
# max over v of |d/dv (v Phi(v))| = Phi(sqrt 2) + sqrt 2 phi(sqrt 2)
GELU_LIPSCHITZ = 1.12891   # 1.1289041..., rounded up


def activation(v: np.ndarray, act: str) -> np.ndarray:
    """The activation on float64 values (NaN stays NaN)."""
    v = np.asarray(v, np.float64)
    if act == "none":
        return v.copy()
    if act == "relu":
        return np.where(v < 0, 0.0, v)
    if act == "gelu":
        # Phi(v) = (1 + erf(v / sqrt 2)) / 2 = erfc(-v / sqrt 2) / 2; the erfc
        # form keeps its relative accuracy for negative v, where 1 + erf cancels
        erfc = np.vectorize(math.erfc, otypes=[np.float64])
        return 0.5 * v * erfc(-v / math.sqrt(2.0))
    raise ValueError("unknown activation %r" % act)


def fused_epilogue(v, scale, dtype, residual=None, act="none"):
    """From the accumulator-type values v (after alpha and the bias) to the
    stored output: v + r, then the activation, then narrowing.  Returns
    (Y, S) with S widened by |r| and by the activation's Lipschitz constant."""
    wide = _wide(dtype)
    v = np.asarray(v, wide)
    scale = np.asarray(scale, np.float64)
    if residual is not None:
        rv = _values(residual, dtype)
        if rv.shape != v.shape:
            raise ShapeError("residual %s is not the output shape %s" % (rv.shape, v.shape))
        v = (v + rv).astype(wide)
        scale = scale + np.abs(rv.astype(np.float64))
    if act != "none":
        v = activation(v, act).astype(wide)
        if act == "gelu":
            scale = scale * GELU_LIPSCHITZ
    if dtype in ("float16", "bfloat16"):
        return encode(v.astype(np.float32), dtype), scale
    return v, scale


def matmul_acc(a: np.ndarray, b: np.ndarray, dtype: str):
    """MatMul's accumulators before narrowing (float32, or float64 for
    DOUBLE), with the same shape rules and batch loop as ``matmul``."""
    if dtype in FP8_DTYPES:
        return matmul_acc(decode_fp8(a, dtype), decode_fp8(b, dtype), "float32")
    out_shape = output_shape(a.shape, b.shape)
    a2 = a.reshape((1,) + a.shape) if a.ndim == 1 else a
    b2 = b.reshape(b.shape + (1,)) if b.ndim == 1 else b
    m, n = a2.shape[-2], b2.shape[-1]
    batch = _broadcast(a2.shape[:-2], b2.shape[:-2])
    r = len(batch)
    a_batch = [1] * (r - (a2.ndim - 2)) + list(a2.shape[:-2])
    b_batch = [1] * (r - (b2.ndim - 2)) + list(b2.shape[:-2])
    a3 = a2.reshape(a_batch + [m, a2.shape[-1]])
    b3 = b2.reshape(b_batch + [b2.shape[-2], n])
    acc = np.zeros(batch + [m, n], _wide(dtype))
    s = np.zeros(batch + [m, n], np.float64)
    for idx in itertools.product(*[range(d) for d in batch]):
        ia = tuple(0 if da == 1 else i for i, da in zip(idx, a_batch))
        ib = tuple(0 if db == 1 else i for i, db in zip(idx, b_batch))
        acc[idx], s[idx] = _acc2d(a3[ia], b3[ib], dtype)
    return acc.reshape(out_shape), s.reshape(out_shape)


def matmul_fused(a, b, dtype, residual=None, act="none"):
    """MatMul followed by the fused residual and activation.  Returns (Y, S).
    With 8-bit float operands the output (and the residual) is float32."""
    acc, s = matmul_acc(a, b, dtype)
    return fused_epilogue(acc, s, "float32" if dtype in FP8_DTYPES else dtype, residual, act)


# --------------------------------------------------------------------------
# grouped products
#
# "Gemm and MatMul Performance Roadmap": the batch-fusion row of the
# opportunity table (hundreds of tiny or irregular products, where one
# dispatch per product costs more than the product) and the GroupedGemm
# interface of its plan (small products scheduled together).  Reading where
# the page is silent: a group is a list of independent rank-2 products
# Y_i = A_i @ B_i with their own M_i, N_i, K_i, one element type for the
# group, each computed exactly as MatMul computes a rank-2 product.


def grouped(a_list, b_list, dtype):
    """Independent rank-2 products.  Returns ([Y_i], [S_i])."""
    if len(a_list) != len(b_list):
        raise ShapeError("a group needs as many A as B operands")
    ys, ss = [], []
    for a, b in zip(a_list, b_list):
        if np.ndim(a) != 2 or np.ndim(b) != 2:
            raise ShapeError("grouped products are rank-2")
        y, s = matmul(np.asarray(a), np.asarray(b), dtype)
        ys.append(y)
        ss.append(s)
    return ys, ss
