#!/usr/bin/env python
"""Throughput of the GB300 ONNX MatMul library; prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-secondary] [--no-cpu-baseline]

A step is one pass over every product of the workload (default: the BF16
transformer projections [8,2048,4096]x[4096,4096], [8,2048,4096]x[4096,14336]
and [8,2048,14336]x[14336,4096]) with the operands already resident in HBM.
`value` is the whole job's TFLOP/s (GB/s for the bandwidth-bound workloads):
the flops all ranks computed divided by the slowest rank's timed region.
With N > 1 (torchrun), every rank runs its own copy of the workload on its own
GPU (independent problems, no data-path collective; weak scaling).

`--impl reference` times the CPU oracle on a bounded row sample of the same
workload instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MatMul TFLOP/s (BF16/FP16/FP32/FP64) and skinny GB/s, % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dense tensor-core ratio of FP16 to BF16 (equal) and the FP32/FP64 SIMT
# peaks derived from unit counts and the maximum SM clock: 152 SMs x 128 FP32
# lanes x 2 flop x 2.07 GHz, and 152 SMs x 4 FP64 flop per clock x 2.07 GHz
SM_COUNT_GB300 = 152
FP8_OVER_BF16 = 2.0          # dense FP8 / BF16 tensor rate on GB300 (4.5 / 2.25 PFLOP/s nominal)
FP32_LANES_PER_SM = 128
FP64_FLOPS_PER_SM_PER_CLK = 4.0   # ~1.25 TFLOP/s at 2.07 GHz over 152 SMs, FMA = 2 flops


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------
# workload accounting


def _out_shape(a_shape, b_shape):
    a2 = (1,) + tuple(a_shape) if len(a_shape) == 1 else tuple(a_shape)
    b2 = tuple(b_shape) + (1,) if len(b_shape) == 1 else tuple(b_shape)
    import numpy as np
    batch = np.broadcast_shapes(a2[:-2], b2[:-2])
    return batch, a2[-2], a2[-1], b2[-1]


def work_of(a_shape, b_shape, dtype):
    from gemm_matmulplan_broadcast_gb300.synth import ELEMENT_BYTES, output_dtype
    import numpy as np
    batch, m, k, n = _out_shape(a_shape, b_shape)
    items = int(np.prod(batch, dtype=np.int64)) if len(batch) else 1
    eb = ELEMENT_BYTES[dtype]
    flop = 2.0 * m * n * k * items
    byts = (eb * (int(np.prod(a_shape)) + int(np.prod(b_shape))) +
            ELEMENT_BYTES[output_dtype(dtype)] * items * m * n)
    return flop, float(byts)


# --------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # nvidia-smi holds driver locks while it starts; do not time anything
        # until it has written its first sample
        t0 = time.time()
        while time.time() - t0 < 10.0:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                pass
            time.sleep(0.05)
        time.sleep(0.2)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) >= 9:
                    rows.append([c.strip() for c in r])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for i, nm in enumerate(names):
            if any(r[5 + i].lower().startswith("active") for r in rows):
                reasons.append(nm)
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------
# multi-rank aggregation (also exercised by the gloo tests)


def aggregate(local_seconds: float, local_units: float, group=None):
    """(max seconds over ranks, sum of units over ranks)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_seconds, local_units
    backend = dist.get_backend(group)
    dev = "cuda" if backend == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------
# traffic figures from committed ncu summaries


def committed_traffic(kernel_key: str):
    """Per-launch DRAM bytes recorded from an ncu capture, if the kernel's
    source is unchanged since (source hash recorded with the figure)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(kernel_key)
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    if h != ent.get("sha256"):
        return None
    return ent.get("bytes_per_launch")


# --------------------------------------------------------------------------
# our implementation


def build_inputs(workload, device):
    """Per product: (A, B, Y) device tensors and the plan."""
    import torch
    from gemm_matmulplan_broadcast_gb300 import Plan, synth
    items = []
    for prod in workload.products:
        a, b = prod.draw()
        plan = Plan(prod.a_shape, prod.b_shape, prod.dtype)
        A = a.to(device)
        B = b.to(device)
        Y = torch.empty(plan.output_shape, device=device,
                        dtype=synth.TORCH_DTYPES[synth.output_dtype(prod.dtype)])
        flop, byts = work_of(prod.a_shape, prod.b_shape, prod.dtype)
        items.append({"name": prod.name, "plan": plan, "A": A, "B": B, "Y": Y, "a": a, "b": b,
                      "flop": flop, "bytes": byts, "dtype": prod.dtype})
    return items


def rotate_sets(items, min_total_bytes, device):
    """Extra copies of the operands so that consecutive executes of the same
    product touch different memory (inputs larger than L2 in total)."""
    import torch
    for it in items:
        per = it["bytes"]
        n = 1
        while per * n < min_total_bytes and n < 16:
            n += 1
        sets = [(it["A"], it["B"], it["Y"])]
        for _ in range(n - 1):
            sets.append((it["A"].clone(), it["B"].clone(), torch.empty_like(it["Y"])))
        it["sets"] = sets


def time_steps(items, steps, stream, chunk=5):
    """Run `steps` steps; returns (total seconds by the outer events,
    per-product list of per-launch milliseconds, one sample per chunk).

    The steps run in chunks of `chunk`: each product's launches of a chunk
    go back to back (rotating over its operand sets), products in turn, with
    CUDA events only around each product's run of launches.  An event
    between two launches would end the programmatic dependent launch that
    lets a kernel's prologue overlap its predecessor's tail (6-12 us per
    launch on the projections), so events sit only at chunk boundaries;
    taking the products in turn chunk by chunk spreads the clock drift of a
    long run evenly over them."""
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    bounds = [(s0, min(steps, s0 + chunk)) for s0 in range(0, steps, chunk)]
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in bounds] for _ in items]
    with torch.cuda.stream(stream):
        start.record(stream)
        for c, (s0, s1) in enumerate(bounds):
            for i, it in enumerate(items):
                e0, e1 = evs[i][c]
                e0.record(stream)
                for s in range(s0, s1):
                    A, B, Y = it["sets"][s % len(it["sets"])]
                    it["plan"].execute(A, B, Y, stream=stream)
                e1.record(stream)
        end.record(stream)
    end.synchronize()
    total = start.elapsed_time(end) / 1e3
    per = [[evs[i][c][0].elapsed_time(evs[i][c][1]) / (s1 - s0) for c, (s0, s1) in enumerate(bounds)]
           for i in range(len(items))]
    return total, per


def time_e2e(items, steps, stream):
    """End to end through olc_matmul_execute_host: pinned host inputs copied
    in, kernels, result copied out, every step.  The products of a step are
    independent, so each is issued on its own stream (a caller would do the
    same); within a product the library pipelines copies and compute over
    row chunks.  Timed by events on `stream`, which waits for every product
    stream before the end event."""
    import torch
    host = []
    for it in items:
        ah = it["a"].pin_memory()
        bh = it["b"].pin_memory()
        yh = torch.empty(tuple(it["Y"].shape), dtype=it["Y"].dtype).pin_memory()
        host.append((ah, bh, yh))
    h2d = sum(h[0].numel() * h[0].element_size() + h[1].numel() * h[1].element_size()
              for h in host)
    d2h = sum(h[2].numel() * h[2].element_size() for h in host)
    streams = [torch.cuda.Stream() for _ in items]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)

    def one_step():
        fork = torch.cuda.Event()
        fork.record(stream)
        for it, (ah, bh, yh), st in zip(items, host, streams):
            st.wait_event(fork)
            it["plan"].execute_host(ah, bh, yh, it["A"], it["B"], it["Y"], stream=st)
        for st in streams:
            done = torch.cuda.Event()
            done.record(st)
            stream.wait_event(done)

    one_step()
    stream.synchronize()
    start.record(stream)
    for _ in range(steps):
        one_step()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3, h2d, d2h


def cpu_oracle_sample(workload, target_seconds: float, items=None):
    """Time the oracle on a seeded row sample of every product, sized so the
    whole sample takes about `target_seconds`.  Returns (flops, seconds,
    threads, description)."""
    import numpy as np
    import oracle
    from gemm_matmulplan_broadcast_gb300 import synth
    prods = []
    for prod in workload.products:
        if items is not None:
            it = next(x for x in items if x["name"] == prod.name)
            a, b = it["a"], it["b"]
        else:
            a, b = prod.draw()
        batch, m, k, n = _out_shape(prod.a_shape, prod.b_shape)
        if len(batch) and int(np.prod(batch)) == 0 or m * n == 0:
            continue
        an = synth.to_numpy_storage(a)
        bn = synth.to_numpy_storage(b)
        # timing sample: A's rows (all batch items stacked) against one B matrix
        an = an.reshape((1, k) if an.ndim == 1 else (-1, k))
        bn = bn.reshape((k, 1)) if bn.ndim == 1 else bn.reshape((-1, k, n))[0]
        dt = prod.dtype
        if dt in synth.FP8_DTYPES:       # the oracle decodes 8-bit floats, then runs in float32
            an, bn, dt = oracle.decode_fp8(an, dt), oracle.decode_fp8(bn, dt), "float32"
        prods.append((dt, an, np.ascontiguousarray(bn), n, k))
    # size the sample: grow the row count until one pass takes a quarter of
    # the target, then scale to the target
    rng = np.random.default_rng(0)

    def one_pass(rows):
        fl = 0.0
        t0 = time.perf_counter()
        for dt, an, bn, n, k in prods:
            r = min(rows, an.shape[0])
            sel = np.sort(rng.choice(an.shape[0], size=r, replace=False))
            oracle.gemm2d(an, bn, dt, rows=sel)
            fl += 2.0 * r * n * k
        return fl, time.perf_counter() - t0

    max_rows = max(an.shape[0] for _, an, _, _, _ in prods)
    rows = 8
    fl, el = one_pass(rows)
    while el < target_seconds / 4 and rows < max_rows:
        rows = int(min(max_rows, max(rows * 2, rows * (target_seconds / 2) / max(el, 1e-3))))
        fl, el = one_pass(rows)
    if el < target_seconds * 0.6 and rows < max_rows:
        rows = int(min(max_rows, rows * target_seconds / max(el, 1e-3)))
        fl, el = one_pass(rows)
    flops, secs = fl, el
    desc = "%d rows of each of %d products (all N columns, full K), oracle C triple loop" % (
        rows, len(prods))
    return flops, secs, oracle.threads(), desc


def roofline_for(item, ms_per_launch, peaks, long_region: bool):
    """Roofline entry for one product's kernel."""
    dt = item["dtype"]
    algo = item["plan"].algorithm
    if algo in ("skinny_m", "skinny_n", "split_k"):
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        achieved = item["bytes"] / (ms_per_launch / 1e3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak}
    if dt in ("bfloat16", "float16", "float8_e4m3fn", "float8_e5m2"):
        key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
        peak = peaks.get(key, FALLBACK_PEAKS[key])   # fp16 dense rate equals bf16
        if dt.startswith("float8"):
            peak *= FP8_OVER_BF16                    # nominal dense ratio, 4.5 / 2.25 PFLOP/s
        achieved = item["flop"] / (ms_per_launch / 1e3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak}
    clk = peaks.get("sm_max_mhz", 2070.0) * 1e6
    if dt == "float32":
        peak = SM_COUNT_GB300 * FP32_LANES_PER_SM * 2 * clk / 1e12
    else:
        peak = SM_COUNT_GB300 * FP64_FLOPS_PER_SM_PER_CLK * clk / 1e12
    achieved = item["flop"] / (ms_per_launch / 1e3) / 1e12
    return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak}


def kernel_key(item):
    return "%s:%s:%s" % (item["plan"].algorithm, item["dtype"], item["name"])


def measure_workload(workload, steps, warmup, device, peaks, l2_bytes):
    import torch
    items = build_inputs(workload, device)
    rotate_sets(items, 2 * l2_bytes, device)
    stream = torch.cuda.Stream()
    for _ in range(warmup):
        time_steps(items, 1, stream)
    torch.cuda.synchronize()
    return items, stream


def graph_time_per_launch(it, stream, reps=20, launches=None):
    """Per-launch device time of one product, free of host launch gaps:
    `launches` executes (rotating over the operand sets) captured into one
    CUDA graph, the graph replayed `reps` times between CUDA events on the
    capture stream.  Returns the list of per-launch milliseconds, one per
    replay."""
    import torch
    n = launches or max(4, len(it["sets"]))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(3):
            A, B, Y = it["sets"][i % len(it["sets"])]
            it["plan"].execute(A, B, Y, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                A, B, Y = it["sets"][i % len(it["sets"])]
                it["plan"].execute(A, B, Y, stream=stream)
        g.replay()
        stream.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for e0, e1 in evs:
            e0.record(stream)
            g.replay()
            e1.record(stream)
    stream.synchronize()
    out = [e0.elapsed_time(e1) / n for e0, e1 in evs]
    del g
    return out


def measure_secondary(workload, device, peaks, l2):
    """Median per-launch time and roofline of every product of a workload (and
    of each chain stage).  Short kernels are timed through CUDA graphs of
    back-to-back launches so host launch gaps do not count; long ones
    (> 2 ms) with per-launch events."""
    import torch
    from gemm_matmulplan_broadcast_gb300 import Plan
    items = build_inputs(workload, device)
    for ch in workload.chains:
        xs = ch.draw()
        cur_shape = tuple(xs[0].shape)
        cur = xs[0].to(device)
        for j, w in enumerate(xs[1:]):
            plan = Plan(cur_shape, tuple(w.shape), ch.dtype)
            W = w.to(device)
            Y = torch.empty(plan.output_shape, dtype=W.dtype, device=device)
            flop, byts = work_of(cur_shape, tuple(w.shape), ch.dtype)
            items.append({"name": "%s_%d" % (ch.name, j + 1), "plan": plan, "A": cur, "B": W,
                          "Y": Y, "flop": flop, "bytes": byts, "dtype": ch.dtype})
            cur, cur_shape = Y, tuple(Y.shape)
    rotate_sets(items, 2 * l2, device)
    stream = torch.cuda.Stream()
    time_steps(items, 3, stream)
    _, probe = time_steps(items, 1, stream)
    res = []
    for i, it in enumerate(items):
        if it["plan"].launches == 0:
            res.append({"product": it["name"], "algorithm": it["plan"].algorithm,
                        "gpu_launches": 0, "note": "empty output: nothing launched"})
            continue
        if probe[i][0] < 2.0:
            per = graph_time_per_launch(it, stream)
            how = "cuda graph of %d launches x %d replays" % (max(4, len(it["sets"])), len(per))
        else:
            n = int(max(3, min(20, 1000.0 / max(probe[i][0], 1e-3))))
            _, per2 = time_steps([it], n, stream)
            per = per2[0]
            how = "%d launches, events per launch" % n
        ms = statistics.median(per)
        r = roofline_for(it, ms, peaks, False)
        res.append({"product": it["name"], "algorithm": it["plan"].algorithm,
                    "ms_per_launch": ms, "timing": how, "achieved": r["achieved"],
                    "unit": r["unit"], "frac": r["frac"], "bound": r["bound"],
                    "peak": r["peak"]})
    for it in items:
        it["plan"].close()
    return res


def graph_time(fn, nsets, stream, reps=10, launches=None):
    """Per-launch device milliseconds of fn(i) (one launch sequence on
    operand set i % nsets), captured `launches` times into a CUDA graph and
    replayed `reps` times between events on the capture stream."""
    import torch
    n = launches or max(4, nsets)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(3):
            fn(i % nsets)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i % nsets)
        g.replay()
        stream.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for e0, e1 in evs:
            e0.record(stream)
            g.replay()
            e1.record(stream)
    stream.synchronize()
    out = [e0.elapsed_time(e1) / n for e0, e1 in evs]
    del g
    return out


def measure_fused(device, peaks, l2):
    """The fused epilogue on the two transformer projections where it
    belongs: GELU on the up projection [16384, 4096] x [4096, 14336] and a
    residual add on the down projection [16384, 14336] x [14336, 4096]
    (BF16).  Each is timed three ways: the plain product, the product with
    the epilogue fused into its store, and the plain product followed by a
    separate elementwise pass (torch's own kernel, as the unfused
    comparison).  The fusion's saving is one read and one write of the
    output per fused operator."""
    import torch
    import numpy as np
    import torch.nn.functional as F
    from gemm_matmulplan_broadcast_gb300 import Plan, synth
    cases = [("up_gelu", (8, 2048, 4096), (4096, 14336), "gelu", False),
             ("down_residual", (8, 2048, 14336), (14336, 4096), "none", True)]
    out = []
    stream = torch.cuda.Stream()
    for name, a_shape, b_shape, act, resid in cases:
        a, b = synth.operands(a_shape, b_shape, "bfloat16", synth.normal(1.0), synth.normal(0.02), 2)
        plain = Plan(a_shape, b_shape, "bfloat16")
        fused = Plan(a_shape, b_shape, "bfloat16").set_epilogue(act, resid)
        flop, byts = work_of(a_shape, b_shape, "bfloat16")
        y_bytes = 2 * int(np.prod(plain.output_shape))
        nsets = max(2, int(np.ceil(2 * l2 / (byts + y_bytes))))
        sets = []
        for i in range(nsets):
            A = a.to(device) if i == 0 else sets[0][0].clone()
            B = b.to(device) if i == 0 else sets[0][1].clone()
            Y = torch.empty(plain.output_shape, dtype=torch.bfloat16, device=device)
            R = torch.randn(plain.output_shape, dtype=torch.bfloat16, device=device) if resid else None
            sets.append((A, B, Y, R))

        def run_plain(i):
            A, B, Y, _ = sets[i]
            plain.execute(A, B, Y, stream=stream)

        def run_fused(i):
            A, B, Y, R = sets[i]
            fused.execute_fused(A, B, Y, R=R, stream=stream)

        def run_unfused(i):
            A, B, Y, R = sets[i]
            plain.execute(A, B, Y, stream=stream)
            if resid:
                Y.add_(R)
            else:
                Y.copy_(F.gelu(Y))

        # the three variants interleaved over rounds, so that clock and power
        # drift under the power cap does not favour whichever runs first
        samples = {"plain": [], "fused": [], "unfused": []}
        for _ in range(3):
            for label, fn in (("plain", run_plain), ("fused", run_fused), ("unfused", run_unfused)):
                samples[label] += graph_time(fn, nsets, stream, reps=4)
        t = {k: statistics.median(v) for k, v in samples.items()}
        out.append({
            "product": name, "a": list(a_shape), "b": list(b_shape),
            "epilogue": ("residual" if resid else act),
            "ms_plain": t["plain"], "ms_fused": t["fused"], "ms_unfused": t["unfused"],
            "tflops_fused": flop / (t["fused"] * 1e-3) / 1e12,
            "fused_cost_pct": 100.0 * (t["fused"] / t["plain"] - 1.0),
            "unfused_cost_pct": 100.0 * (t["unfused"] / t["plain"] - 1.0),
            "timing": "cuda graph of %d launches x 4 replays x 3 interleaved rounds, %d operand sets" % (max(4, nsets), nsets),
        })
        plain.close()
        fused.close()
        del sets
        torch.cuda.empty_cache()
    return out


def measure_grouped(device, peaks):
    """Hundreds of small irregular products (the pages' batch-fusion case):
    256 members with M, N, K drawn from {16, 32, ..., 256} (seed 7), timed
    as one grouped launch and as one plan execute per member (all captured
    in CUDA graphs, so launch gaps are the GPU's own, not Python's)."""
    import numpy as np
    import torch
    from gemm_matmulplan_broadcast_gb300 import GroupedPlan, Plan, synth
    rng = np.random.default_rng(7)
    shapes = [tuple(int(x) * 16 for x in rng.integers(1, 17, size=3)) for _ in range(256)]
    flop = sum(2.0 * m * n * k for m, n, k in shapes)
    out = []
    stream = torch.cuda.Stream()
    for dtype in ("float16", "float32"):
        tdt = synth.TORCH_DTYPES[dtype]
        As = [torch.randn(m, k, device=device).to(tdt) for m, n, k in shapes]
        Bs = [(torch.randn(k, n, device=device) * 0.1).to(tdt) for m, n, k in shapes]
        Ys = [torch.empty(m, n, dtype=tdt, device=device) for m, n, k in shapes]
        g = GroupedPlan(shapes, dtype)
        ptrs = g.pointer_arrays(As, Bs, Ys)
        plans = [Plan((m, k), (k, n), dtype) for m, n, k in shapes]
        t_group = statistics.median(graph_time(lambda i: g.execute_ptrs(*ptrs, stream=stream),
                                               1, stream, reps=20, launches=4))

        def each(i):
            for p, a, b, y in zip(plans, As, Bs, Ys):
                p.execute(a, b, y, stream=stream)

        t_each = statistics.median(graph_time(each, 1, stream, reps=10, launches=2))
        out.append({"dtype": dtype, "members": len(shapes), "flop": flop,
                    "ms_grouped": t_group, "ms_per_member_launches": t_each,
                    "tflops_grouped": flop / (t_group * 1e-3) / 1e12,
                    "tflops_per_member_launches": flop / (t_each * 1e-3) / 1e12,
                    "speedup": t_each / t_group, "gpu_launches_grouped": 1,
                    "gpu_launches_per_member": len(shapes)})
        g.close()
        for p in plans:
            p.close()
    return out


def measure_alu(stream):
    """The FMA pipes' delivered rate (library probe: independent FMA chains
    on every SM, no memory traffic), beside the peaks derived from unit
    counts and the maximum clock that the FLOAT / DOUBLE rooflines use."""
    from gemm_matmulplan_broadcast_gb300 import binding
    # iterations for about 25-50 ms per launch at the derived peaks
    kinds = [("fp32_ffma2", 0, 800000), ("fp32_ffma", 1, 800000), ("fp64_dfma", 2, 24000),
             ("fp64_dmma", 3, 6000)]
    out = {}
    for name, kind, iters in kinds:
        rates = [binding.alu_rate(kind, iters, stream) for _ in range(3)]
        out[name] = {"tflops": max(rates) / 1e12, "runs": 3, "iters": iters}
    return out


def measure_split_k_curve(device, peaks, l2):
    """The FP16 small-output split-K product [32, K] x [K, 32] as K grows
    (131072 is the named corner): GB/s against K gives the kernel's fixed
    cost per launch (intercept) and its streaming rate (slope)."""
    from gemm_matmulplan_broadcast_gb300 import synth
    prods = tuple(synth.Product("split_k_%d" % k, (32, k), (k, 32), "float16", synth.normal(1.0),
                                synth.normal(0.02), 3) for k in (131072, 262144, 524288, 1048576))
    w = synth.Workload("fp16_split_k_curve", "FP16 [32,K]x[K,32], K = 2^17..2^20, seed 3", prods)
    res = measure_secondary(w, device, peaks, l2)
    # least-squares line t = t0 + bytes / rate over the sizes
    import numpy as np
    x = np.array([2.0 * 32 * int(r["product"].split("_")[-1]) * 2 + 32 * 32 * 2 for r in res])
    t = np.array([r["ms_per_launch"] * 1e-3 for r in res])
    slope, t0 = np.polyfit(x, t, 1)
    return {"points": res, "fit_fixed_us": t0 * 1e6, "fit_stream_gbs": 1.0 / slope / 1e9}


def measure_split_k_static(device, l2):
    """The allocation-free split-K entry point (SIMT split kernel, scratch in
    a fixed device array) on the FP16 corner [32, 131072] x [131072, 32],
    against the plan path's split-K on the same operands: events around 20
    back-to-back calls of each, after warm-up."""
    import ctypes
    import torch
    from gemm_matmulplan_broadcast_gb300 import Plan, binding, synth
    m, k, n = 32, 131072, 32
    a, b = synth.operands((m, k), (k, n), "float16", synth.normal(1.0), synth.normal(0.02), 3)
    A, B = a.to(device), b.to(device)
    Y = torch.empty(m, n, dtype=torch.float16, device=device)
    fn = binding.load().olc_matmul_split_k_static
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.c_int, vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp]
    fn.restype = ctypes.c_int
    stream = torch.cuda.Stream()
    plan = Plan((m, k), (k, n), "float16")

    def static_call():
        st = fn(10, A.data_ptr(), B.data_ptr(), Y.data_ptr(), m, n, k, stream.cuda_stream)
        assert st == 0, st

    def plan_call():
        plan.execute(A, B, Y, stream=stream)

    out = {}
    for label, call in (("static", static_call), ("plan", plan_call)):
        for _ in range(5):
            call()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(20):
            call()
        e1.record(stream)
        e1.synchronize()
        out["ms_" + label] = e0.elapsed_time(e1) / 20
    plan.close()
    byts = 2.0 * (m * k + k * n + m * n)
    out["gbs_static"] = byts / (out["ms_static"] * 1e-3) / 1e9
    out["gbs_plan"] = byts / (out["ms_plan"] * 1e-3) / 1e9
    out["timing"] = "events around 20 back-to-back calls (operands L2-resident)"
    return out


def measure_few_tiles(device, peaks):
    """BF16 products whose 128 x 256 tiles would leave most SMs idle, which
    the general tensor-core path runs as a cluster split-K: [17 | 128, 4096]
    x [4096, 4096] and the long-K small output [64, 8192] x [8192, 512].
    CUDA graphs of back-to-back launches over B copies that exceed L2
    together; the rate is HBM bytes (A + B + Y once) per second against the
    measured copy rate, the bound of these B-streaming products."""
    import torch
    from gemm_matmulplan_broadcast_gb300 import Plan
    stream = torch.cuda.Stream()
    out = []
    g = torch.Generator(device="cpu").manual_seed(3)
    for (m, k, n) in ((17, 4096, 4096), (128, 4096, 4096), (64, 8192, 512)):
        nb = max(2, (300 << 20) // (k * n * 2))
        Bs = [(torch.randn(k, n, generator=g) * 0.02).to(torch.bfloat16).to(device) for _ in range(nb)]
        A = torch.randn(m, k, generator=g).to(torch.bfloat16).to(device)
        Y = torch.empty(m, n, dtype=torch.bfloat16, device=device)
        p = Plan((m, k), (k, n), "bfloat16")
        ms = statistics.median(graph_time(lambda i: p.execute(A, Bs[i % nb], Y, stream=stream), nb, stream,
                                          reps=5, launches=2 * nb))
        byts = (m * k + k * n + m * n) * 2
        out.append({"product": "%dx%dx%d" % (m, k, n), "algorithm": p.algorithm,
                    "workspace_bytes": p.workspace_bytes, "ms_per_launch": ms,
                    "gbs": byts / (ms * 1e-3) / 1e9,
                    "frac": byts / (ms * 1e-3) / 1e9 / peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])})
        p.close()
        del Bs, A, Y
    torch.cuda.empty_cache()
    return out


def measure_unaligned(device, peaks, l2):
    """FLOAT16 / BFLOAT16 products the TMA cannot read in place, on the
    tensor cores: the output projection [16384, 4096] x [4096, 50257] BF16
    (N odd: B is staged into padded rows every call, or once with a
    plan-owned constant B; Y stored by alignment), and the up projection
    [16384, 4096] x [4096, 14336] with A one element into its buffer (A
    staged every call) beside the same product aligned.  CUDA graphs of
    back-to-back launches, the two variants of each pair interleaved over
    three rounds; the operands exceed L2."""
    import torch
    from gemm_matmulplan_broadcast_gb300 import Plan, synth
    stream = torch.cuda.Stream()
    out = []
    # the vocabulary projection
    a, b = synth.operands((16384, 4096), (4096, 50257), "bfloat16", synth.normal(1.0),
                          synth.normal(0.02), 2)
    flop, byts = work_of((16384, 4096), (4096, 50257), "bfloat16")
    A, B = a.to(device), b.to(device)
    Y = torch.empty(16384, 50257, dtype=torch.bfloat16, device=device)
    p = Plan((16384, 4096), (4096, 50257), "bfloat16")
    pc = Plan((16384, 4096), (4096, 50257), "bfloat16")
    pc.set_constant_b(B)
    # the two variants interleaved over rounds (clock drift under load)
    cases = (("vocab_50257_per_call_b", lambda i: p.execute(A, B, Y, stream=stream), p),
             ("vocab_50257_constant_b", lambda i: pc.execute_constant(A, Y, stream=stream), pc))
    samples = {c[0]: [] for c in cases}
    for _ in range(3):
        for label, fn, _plan in cases:
            samples[label] += graph_time(fn, 1, stream, reps=2, launches=2)
    for label, fn, plan in cases:
        ms = statistics.median(samples[label])
        out.append({"product": label, "a": [16384, 4096], "b": [4096, 50257],
                    "algorithm": plan.algorithm, "launches": plan.launches,
                    "ms_per_launch": ms, "tflops": flop / (ms * 1e-3) / 1e12,
                    "frac": flop / (ms * 1e-3) / 1e12 / peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])})
    p.close()
    pc.close()
    del A, B, Y
    torch.cuda.empty_cache()
    # the up projection, aligned and with A one element off
    a, b = synth.operands((8, 2048, 4096), (4096, 14336), "bfloat16", synth.normal(1.0),
                          synth.normal(0.02), 2)
    flop, _ = work_of((8, 2048, 4096), (4096, 14336), "bfloat16")
    abuf = torch.empty(a.numel() + 8, dtype=torch.bfloat16, device=device)
    A_al = abuf[:a.numel()].view(a.shape)
    A_al.copy_(a.to(device))
    abuf2 = torch.empty(a.numel() + 8, dtype=torch.bfloat16, device=device)
    A_off = abuf2[1:1 + a.numel()].view(a.shape)
    A_off.copy_(a.to(device))
    B = b.to(device)
    Y = torch.empty(8, 2048, 14336, dtype=torch.bfloat16, device=device)
    p = Plan((8, 2048, 4096), (4096, 14336), "bfloat16")
    samples = {"up_proj_aligned": [], "up_proj_a_offset_1": []}
    for _ in range(3):
        for label, AA in (("up_proj_aligned", A_al), ("up_proj_a_offset_1", A_off)):
            samples[label] += graph_time(lambda i: p.execute(AA, B, Y, stream=stream), 1, stream,
                                         reps=2, launches=2)
    for label, AA in (("up_proj_aligned", A_al), ("up_proj_a_offset_1", A_off)):
        ms = statistics.median(samples[label])
        out.append({"product": label, "a": [8, 2048, 4096], "b": [4096, 14336],
                    "algorithm": p.algorithm_for(AA, B, Y), "staging_copies": p.staging_copies(AA, B, Y),
                    "ms_per_launch": ms, "tflops": flop / (ms * 1e-3) / 1e12,
                    "frac": flop / (ms * 1e-3) / 1e12 / peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])})
    p.close()
    del abuf, abuf2, B, Y
    torch.cuda.empty_cache()
    return out


def measure_fp8_decode_constant_b(device, peaks):
    """The FP8 few-row products of the decode workload ([1|4|16, 8192] x
    [8192, 28672], E4M3FN) with B owned by the plan (resident weights, set
    once): the tcgen05 few-row kernel streams the plan's transposed copy.
    CUDA graphs of back-to-back launches; two A / Y sets, B 235 MB."""
    import torch
    from gemm_matmulplan_broadcast_gb300 import Plan, synth
    stream = torch.cuda.Stream()
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out = []
    for m in (1, 4, 16):
        a, b = synth.operands((m, 8192), (8192, 28672), "float8_e4m3fn", synth.normal(1.0),
                              synth.normal(0.5), 3)
        p = Plan((m, 8192), (8192, 28672), "float8_e4m3fn")
        p.set_constant_b(b)
        sets = [(a.to(device), torch.empty(m, 28672, device=device)) for _ in range(2)]
        byts = m * 8192 + 8192 * 28672 + 4 * m * 28672
        ms = statistics.median(graph_time(lambda i: p.execute_constant(*sets[i], stream=stream), 2,
                                          stream, reps=10, launches=8))
        gbs = byts / (ms * 1e-3) / 1e9
        out.append({"product": "fp8_rows_%d_constant_b" % m, "algorithm": p.algorithm,
                    "ms_per_launch": ms, "achieved": gbs, "unit": "GB/s", "frac": gbs / hbm,
                    "bound": "hbm", "peak": hbm})
        p.close()
        del sets
    torch.cuda.empty_cache()
    return out


def oracle_single_thread(names):
    """The oracle on one host core over the small named workloads, in full."""
    import oracle
    from gemm_matmulplan_broadcast_gb300 import synth
    n0 = oracle.threads()
    oracle.set_threads(1)
    out = {}
    try:
        for wname in names:
            w = synth.workload(wname)
            fl, secs = 0.0, 0.0
            for prod in w.products:
                a, b = prod.draw()
                an, bn = synth.to_numpy_storage(a), synth.to_numpy_storage(b)
                flop, _ = work_of(prod.a_shape, prod.b_shape, prod.dtype)
                reps = 0
                t0 = time.perf_counter()
                while True:
                    oracle.matmul(an, bn, prod.dtype)
                    reps += 1
                    if time.perf_counter() - t0 > 0.2:
                        break
                secs += (time.perf_counter() - t0) / reps
                fl += flop
            out[wname] = {"gflops": fl / secs / 1e9, "ms_per_pass": secs * 1e3, "threads": 1}
    finally:
        oracle.set_threads(n0)
    return out


def _short(x):
    v = float("%.3g" % x)
    return int(v) if abs(v) >= 100 and v == int(v) else v


def compact_summary(breakdown, secondary):
    """One short entry per named configuration (and the extra workloads),
    kept small so that the end of the JSON line alone carries every figure:
    per product [microseconds per launch, achieved rate, roofline fraction],
    with the rate's unit once per configuration."""
    def short_name(name):
        for pre in ("fp8_proj_", "proj_", "fp8_rows_", "square_"):
            if name.startswith(pre):
                name = name[len(pre):]
        return name.replace("_constant_b", "")

    def rows(lst):
        d = {}
        for r in lst:
            if "achieved" not in r:
                d[short_name(r["product"])] = "empty"
                continue
            d.setdefault("unit", r["unit"])
            d[short_name(r["product"])] = [_short(r["ms_per_launch"] * 1e3), _short(r["achieved"]),
                                           _short(r["frac"])]
        return d
    out = {"fmt": "us/launch,rate,roofline frac", "C3_bf16": rows(breakdown)}
    names = [("C1_fp32", "fp32_64x128x96"), ("C2_fp32", "fp32_broadcast_batch"),
             ("C4_fp16", "fp16_skinny_splitk"), ("C5_fp32", "float32_square_chain"),
             ("C5_fp64", "float64_square_chain"), ("fp8_proj", "fp8_transformer_projection"),
             ("fp8_rows", "fp8_skinny_decode"), ("fp8_rows_const_b", "fp8_rows_constant_b")]
    for key, wname in names:
        if wname in secondary:
            out[key] = rows(secondary[wname])
    if "split_k_curve" in secondary:
        c = secondary["split_k_curve"]
        out["split_k_curve"] = {"fixed_us": _short(c["fit_fixed_us"]), "stream_gbs": _short(c["fit_stream_gbs"]),
                                "gbs": [_short(r["achieved"]) for r in c["points"]]}
    if "split_k_static" in secondary:
        st = secondary["split_k_static"]
        out["split_k_static_us"] = [_short(st["ms_static"] * 1e3), _short(st["ms_plan"] * 1e3)]
    if "unaligned_tc" in secondary:
        out["unaligned_tc"] = {"unit": "TFLOP/s"}
        for r in secondary["unaligned_tc"]:
            out["unaligned_tc"][r["product"].replace("vocab_50257_", "vocab_")] = [
                _short(r["ms_per_launch"] * 1e3), _short(r["tflops"]), _short(r["frac"])]
    if "few_tiles_bf16" in secondary:
        out["few_tiles_bf16"] = {"unit": "GB/s"}
        for r in secondary["few_tiles_bf16"]:
            out["few_tiles_bf16"][r["product"]] = [_short(r["ms_per_launch"] * 1e3), _short(r["gbs"]),
                                                  _short(r["frac"])]
    if "alu_rates" in secondary:
        out["alu_tflops"] = [_short(v["tflops"]) for v in secondary["alu_rates"].values()]
    return out


def run_ours(args):
    import torch
    from gemm_matmulplan_broadcast_gb300 import load, synth
    rank, world, local = dist_setup(args)
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    load()
    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 129 * 1024 * 1024) or 129 * 1024 * 1024

    workload = synth.workload(args.workload)
    items, stream = measure_workload(workload, args.steps, args.warmup, device, peaks, l2)
    flop_step = sum(it["flop"] for it in items)
    byte_step = sum(it["bytes"] for it in items)
    bw_bound = all(it["plan"].algorithm in ("skinny_m", "skinny_n", "split_k") for it in items)

    sampler = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    host_t0 = time.perf_counter()
    total, per = time_steps(items, args.steps, stream)
    host_enqueue_s = time.perf_counter() - host_t0
    clocks = sampler.stop()
    torch.cuda.synchronize()
    barrier()
    secs, units = aggregate(total, (byte_step if bw_bound else flop_step) * args.steps)
    value = units / secs / (1e9 if bw_bound else 1e12)
    unit = "GB/s" if bw_bound else "TFLOP/s"

    # dominant kernel: the product with the largest total time
    means = [statistics.mean(p) for p in per]
    dom = max(range(len(items)), key=lambda i: means[i])
    long_region = total > 1.0
    roof = roofline_for(items[dom], means[dom], peaks, long_region)
    roof["kernel"] = kernel_key(items[dom])
    roof["traffic"] = committed_traffic(kernel_key(items[dom]))
    roof["peak_source"] = peak_src + (" sustained" if (roof["bound"] == "tensor" and long_region)
                                      else " burst" if roof["bound"] == "tensor" else "")
    breakdown = []
    for i, it in enumerate(items):
        r = roofline_for(it, means[i], peaks, long_region)
        breakdown.append({"product": it["name"], "algorithm": it["plan"].algorithm,
                          "ms_per_launch": means[i], "achieved": r["achieved"], "unit": r["unit"],
                          "frac": r["frac"], "bound": r["bound"],
                          "p10_ms": sorted(per[i])[len(per[i]) // 10],
                          "p90_ms": sorted(per[i])[(len(per[i]) * 9) // 10]})

    # end to end through the host-buffer entry point
    e2e_secs, h2d, d2h = time_e2e(items, max(1, min(args.steps, 5)), stream)
    e2e_steps = max(1, min(args.steps, 5))
    e2e_secs_all, e2e_units = aggregate(e2e_secs, (byte_step if bw_bound else flop_step) * e2e_steps)
    e2e = {"value": e2e_units / e2e_secs_all / (1e9 if bw_bound else 1e12), "unit": unit,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}

    secondary = {}
    if not args.no_secondary and args.workload == "bf16_transformer_projection":
        names = ["fp32_64x128x96", "fp32_broadcast_batch", "fp16_skinny_splitk",
                 "float32_square_chain"]
        if not args.no_fp64:
            names.append("float64_square_chain")
        names.append("fp8_transformer_projection")
        names.append("fp8_skinny_decode")
        for wname in names:
            secondary[wname] = measure_secondary(synth.workload(wname), device, peaks, l2)
        secondary["split_k_curve"] = measure_split_k_curve(device, peaks, l2)
        secondary["split_k_static"] = measure_split_k_static(device, l2)
        secondary["unaligned_tc"] = measure_unaligned(device, peaks, l2)
        secondary["few_tiles_bf16"] = measure_few_tiles(device, peaks)
        secondary["fp8_rows_constant_b"] = measure_fp8_decode_constant_b(device, peaks)
        secondary["fused_epilogue"] = measure_fused(device, peaks, l2)
        secondary["grouped_small_products"] = measure_grouped(device, peaks)
        secondary["alu_rates"] = measure_alu(stream)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        fl, cs, cores, desc = cpu_oracle_sample(workload, args.cpu_seconds, items)
        cpu = {"value": fl / cs / (1e12 if not bw_bound else 1.0), "unit": unit if not bw_bound else "flop/s",
               "cores": cores, "kind": "oracle", "sample": desc, "seconds": cs}
        if not args.no_secondary:
            cpu["single_thread"] = oracle_single_thread(["fp32_64x128x96", "fp32_broadcast_batch"])

    launches = sum(it["plan"].launches for it in items) * args.steps
    dtypes = sorted({it["dtype"] for it in items})
    short = {"bfloat16": "bf16", "float16": "f16", "float32": "f32", "float64": "f64",
             "float8_e4m3fn": "e4m3", "float8_e5m2": "e5m2"}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "+".join(short[d] for d in dtypes),
        "data": "synthetic (seeded torch CPU generator per product, A drawn before B in float32, cast to the storage type with RNE)",
        "config": {
            "workload": workload.name,
            "description": workload.description,
            "products": [{"a": list(p.a_shape), "b": list(p.b_shape), "dtype": p.dtype}
                         for p in workload.products],
            "l2": "inputs larger than L2: each product rotates over operand sets totalling "
                  ">= 2x L2 (%d MB)" % (l2 // (1 << 20)),
            "parallelism": "independent replicas per GPU" if world > 1 else "single GPU",
        },
        "roofline": roof,
        "breakdown": breakdown,
        "secondary": secondary,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "host_enqueue_s": host_enqueue_s,
        "gpu": props.name,
        # last, so that a reader keeping only the end of the line keeps it
        "summary": compact_summary(breakdown, secondary),
    }
    if rank == 0:
        print(json.dumps(line, separators=(",", ":")), flush=True)
    for it in items:
        it["plan"].close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# reference arm: the CPU oracle


def run_reference(args):
    from gemm_matmulplan_broadcast_gb300 import synth
    rank, world, _ = dist_setup(args)
    if rank != 0:
        return
    workload = synth.workload(args.workload)
    bw_bound = args.workload == "fp16_skinny_splitk"
    per_step = max(0.5, args.ref_step_seconds)
    # operands drawn once (the same seeded inputs as the GPU arm)
    drawn = []
    for prod in workload.products:
        a, b = prod.draw()
        drawn.append({"name": prod.name, "a": a, "b": b})
    for _ in range(args.warmup):
        cpu_oracle_sample(workload, per_step / 4, drawn)
    flops = secs = 0.0
    cores, desc = 1, ""
    for _ in range(args.steps):
        f, s, cores, desc = cpu_oracle_sample(workload, per_step, drawn)
        flops += f
        secs += s
    value = flops / secs / 1e12
    unit = "TFLOP/s"
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "cpu oracle", "data": "synthetic",
        "config": {"workload": workload.name, "description": workload.description},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    if bw_bound:
        line["note"] = "bandwidth workload reported in TFLOP/s for the CPU oracle"
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="bf16_transformer_projection")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-fp64", action="store_true",
                    help="skip the FP64 square/chain workload (about 10 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
