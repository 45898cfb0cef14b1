"""Failure detection without a GPU fault: a bounded device wait that runs
out is reported as a status and leaves the context usable; host-side errors
come back as statuses before any launch; the multi-rank timing aggregation of
bench.py works across two gloo ranks on the CPU."""

import ctypes
import os

import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import Plan, binding, synth
from parity import compare


def _selftest():
    fn = binding.load().olc_debug_wait_selftest
    fn.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.gpu
def test_bounded_wait_reports_timeout_and_context_survives():
    fn = _selftest()
    assert fn(1_000_000_000, 1, None) == 0                      # the phase completes
    st = fn(2_000_000, 0, None)                                 # nothing arrives: 2 ms limit
    assert binding.STATUS[st] == "OLC_ERR_DEVICE_TIMEOUT"
    assert fn(1_000_000_000, 1, None) == 0                      # error word was cleared
    # the context still runs products correctly after the timeout
    a, b = synth.operands((64, 64), (64, 128), "bfloat16", synth.SMALL_INT, synth.SMALL_INT, 3)
    with Plan(a.shape, b.shape, "bfloat16") as p:
        y = torch.empty(p.output_shape, dtype=torch.bfloat16, device="cuda")
        p.execute_checked(a.cuda(), b.cuda(), y)
    y_ref, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), "bfloat16")
    compare(y.cpu(), y_ref, s, "bfloat16", exact=True)


def test_host_errors_come_back_before_any_launch():
    lib = binding.load()
    with Plan((4, 8), (8, 4), "float32") as p:
        # NULL data pointers for a non-empty product
        assert lib.olc_matmul_execute(p.handle, None, None, None, None) == 1
        assert lib.olc_matmul_execute_checked(p.handle, None, 32, None, 32, None, 0, None) == 8
    assert lib.olc_matmul_execute(None, None, None, None, None) == 1


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs, units = bench.aggregate(1.0 + rank, 10.0 * (rank + 1))
    q.put((rank, secs, units))
    dist.barrier()
    dist.destroy_process_group()


def test_bench_aggregation_two_gloo_ranks():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, secs, units in out:
        assert secs == 2.0 and units == 30.0      # max of the times, sum of the units
