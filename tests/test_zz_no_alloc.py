"""olc_matmul_split_k_static: the split-K product for callers that must not
allocate device memory while they run (a host framework whose memory pool
owns the whole device, a latency-bound serving loop that cannot take
cudaMalloc's implicit synchronisation).  Its partials live in a fixed 4 MiB
device array inside the library instead of a plan-owned cudaMalloc'd
workspace.

The test calls it through the C ABI twice in a row -- the second call sees
whatever the first left in the shared array -- and compares each result with
the oracle on the same inputs, within the parity tolerance tol * sum|a||b|
used by every other GPU test, and with the plan path's split-K.  Around the
second call it checks that nothing was allocated: the device's free memory
and torch's allocated bytes are unchanged.  This file sorts last so that a
run stopping at its first failure has run every other test already; it also
passes on its own in a fresh process (the first call does the per-device
set-up)."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import Plan, binding, synth
from parity import TOL, compare

pytestmark = pytest.mark.gpu


def _entry():
    fn = binding.load().olc_matmul_split_k_static
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.c_int, vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("dtype,shape", [
    ("float16", (32, 131072, 32)),
    ("bfloat16", (48, 20000, 40)),
    ("float32", (33, 9000, 40)),
    ("float64", (16, 4096, 24)),
])
def test_static_split_k_matches_plan_path_twice(dtype, shape):
    m, k, n = shape
    fn = _entry()
    code = binding.DTYPE_CODES[dtype]
    stream = torch.cuda.current_stream()
    for call in range(2):
        a, b = synth.operands((m, k), (k, n), dtype, synth.normal(1.0), synth.normal(0.02),
                              seed=40 + call)
        A, B = a.cuda(), b.cuda()
        y_static = torch.full((m, n), float("nan"), dtype=A.dtype, device="cuda")
        torch.cuda.synchronize()
        free0, used0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        st = fn(code, A.data_ptr(), B.data_ptr(), y_static.data_ptr(), m, n, k,
                stream.cuda_stream)
        assert st == 0, binding.STATUS.get(st, st)
        torch.cuda.synchronize()
        free1, used1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        if call == 1:
            # the first call on a device may load the library's kernel module
            # (and with it the array); every later call allocates nothing
            assert free1 == free0 and used1 == used0, (free0, free1, used0, used1)
        with Plan((m, k), (k, n), dtype) as p:
            p.force("split_k")
            y_plan = torch.empty((m, n), dtype=A.dtype, device="cuda")
            p.execute(A, B, y_plan)
        torch.cuda.synchronize()
        y_ref, s = oracle.gemm2d(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        compare(y_static.cpu(), y_ref, s, dtype)
        ys = oracle.to_float64(synth.to_numpy_storage(y_static.cpu()), dtype)
        yp = oracle.to_float64(synth.to_numpy_storage(y_plan.cpu()), dtype)
        assert not np.isnan(ys).any()
        # two results within tol * S of the oracle are within 2 tol * S of
        # each other
        assert np.all(np.abs(ys - yp) <= 2 * TOL[dtype] * s), "call %d" % call


def test_static_split_k_rejects_oversized_and_bad_arguments():
    fn = _entry()
    A = torch.zeros(2048, 64, device="cuda")
    B = torch.zeros(64, 2048, device="cuda")
    Y = torch.zeros(2048, 2048, device="cuda")
    # 64 x 64 tiles of 32 x 32 = 4096 tiles: more than the array holds
    assert fn(1, A.data_ptr(), B.data_ptr(), Y.data_ptr(), 2048, 2048, 64, None) == 15
    assert fn(7, A.data_ptr(), B.data_ptr(), Y.data_ptr(), 8, 8, 8, None) == 6
    assert fn(1, A.data_ptr(), B.data_ptr(), Y.data_ptr(), -1, 8, 8, None) == 3
    assert fn(1, None, B.data_ptr(), Y.data_ptr(), 8, 8, 8, None) == 1
    assert fn(1, None, None, None, 0, 8, 8, None) == 0          # empty: nothing to do
    Y8 = torch.full((8, 8), 5.0, device="cuda")
    assert fn(1, None, None, Y8.data_ptr(), 8, 8, 0, None) == 0  # K == 0: zeros
    torch.cuda.synchronize()
    assert bool((Y8 == 0).all())
