"""Run one MatMul product a few times, for a profiler or a quick timing.

    python -m gemm_matmulplan_broadcast_gb300.profile_one --a 2048,2048 --b 2048,2048 \\
        --dtype float64 [--reps 3] [--algorithm NAME] [--variant V] [--a-offset E]

Inputs are the seeded synthetic operands (A ~ N(0,1), B ~ N(0,0.02), seed 0)
drawn on the host and copied to the device once; each repetition is one
execute of the same plan, timed with CUDA events on the launching stream.
`--a-offset E` places A E elements into its device buffer (a pointer off a
16-byte boundary).  Prints one line per repetition and the median.
"""

from __future__ import annotations

import argparse
import statistics


def _shape(text: str):
    return tuple(int(x) for x in text.split(",") if x)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--a", required=True, help="A's shape, comma separated")
    ap.add_argument("--b", required=True, help="B's shape, comma separated")
    ap.add_argument("--dtype", default="bfloat16")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--algorithm", default=None)
    ap.add_argument("--variant", type=int, default=None)
    ap.add_argument("--a-offset", type=int, default=0)
    args = ap.parse_args(argv)

    import torch
    from . import Plan, synth

    a_shape, b_shape = _shape(args.a), _shape(args.b)
    a, b = synth.operands(a_shape, b_shape, args.dtype, synth.normal(1.0), synth.normal(0.02), 0)
    if args.a_offset:
        buf = torch.empty(a.numel() + args.a_offset, dtype=a.dtype, device="cuda")
        A = buf[args.a_offset:].view(a.shape)
        A.copy_(a.cuda())
    else:
        A = a.cuda()
    B = b.cuda()
    with Plan(a_shape, b_shape, args.dtype) as p:
        if args.algorithm:
            p.force(args.algorithm)
        if args.variant is not None:
            p.set_tc_variant(args.variant)
        Y = torch.empty(p.output_shape, device="cuda",
                        dtype=synth.TORCH_DTYPES[synth.output_dtype(args.dtype)])
        stream = torch.cuda.current_stream()
        times = []
        for i in range(args.reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            p.execute(A, B, Y, stream=stream)
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
            print("rep %d: %.4f ms (%s)" % (i, times[-1], p.describe()))
        print("median %.4f ms" % statistics.median(times))


if __name__ == "__main__":
    main()
