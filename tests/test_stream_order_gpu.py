"""Stream order across kernels that start early.

The CTA-pair, 1-CTA tensor-core, skinny-N streaming and small-output split-K
kernels are launched so that they may start while the previous kernel in the
stream is finishing, and wait on the device before their first global
access.  Here each product of a chain reads the previous product's output,
with kernels of different kinds back to back on one stream; the outputs must
equal, bit for bit, those of the same chain with the stream synchronised
after every product (every kernel is deterministic).  Each kernel's parity
with the oracle is covered by the other test files."""

import pytest
import torch

from gemm_matmulplan_broadcast_gb300 import Plan, synth

pytestmark = pytest.mark.gpu


def _chain(dtype):
    """The first input and, per step, (plan, B, rows): step i multiplies the
    first `rows` rows of step i-1's output by its B."""
    tdt = synth.TORCH_DTYPES[dtype]
    x0, _ = synth.operands((512, 1024), (1,), dtype, synth.normal(1.0), synth.UNIFORM, seed=21)
    specs = [
        # (rows of the previous output used as A, K = its columns, N, algorithm, tc variant)
        (512, 1024, 512, "general_tc", 2),     # CTA pair
        (32, 512, 32, "split_k", 0),           # small-output split-K (clusters)
        (4, 32, 2048, "skinny_m", 2),          # swapped-operand tensor-core skinny-M
        (4, 2048, 512, "general_tc", 1),       # one CTA per 128 x 256 tile
        (4, 512, 8, "skinny_n", 0),            # register-streaming skinny-N
    ]
    steps = []
    for i, (rows, k, n, algo, variant) in enumerate(specs):
        _, b = synth.operands((1,), (k, n), dtype, synth.UNIFORM, synth.normal(0.05), seed=30 + i)
        p = Plan((rows, k), (k, n), dtype)
        p.force(algo)
        p.set_tc_variant(variant)
        steps.append((p, b.cuda(), rows))
    return x0.cuda().to(tdt), steps


def _run(x0, steps, stream, sync):
    outs = []
    cur = x0
    with torch.cuda.stream(stream):
        for p, b, rows in steps:
            a = cur[:rows]
            y = torch.empty(p.output_shape, dtype=b.dtype, device="cuda")
            p.execute(a, b, y, stream=stream)
            if sync:
                stream.synchronize()
            outs.append(y)
            cur = y
    stream.synchronize()
    return outs


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_chained_products_without_sync_match_synchronised_chain(dtype):
    x0, steps = _chain(dtype)
    assert [p.algorithm for p, _, _ in steps] == [
        "general_tc", "split_k", "skinny_m", "general_tc", "skinny_n"]
    stream = torch.cuda.Stream()
    ref = _run(x0, steps, stream, sync=True)
    for _ in range(3):
        got = _run(x0, steps, stream, sync=False)
        for i, (r, g) in enumerate(zip(ref, got)):
            assert torch.equal(r.view(torch.int16), g.view(torch.int16)), "step %d" % i
    for p, _, _ in steps:
        p.close()


# One plan executed on two streams with no ordering between them: the plan
# orders the executes that use its own device state (workspace or staging
# buffer) across streams, so every output is the product of its own inputs.
# Each case uses such state: split-K partials and counters, the FP8 B
# transposed into the workspace on every call, and staging copies of
# operands with rows that are not 16-byte multiples.
STATE_CASES = [
    ("float16", ((32, 65536), (65536, 32)), "split_k"),
    ("float8_e4m3fn", ((512, 1024), (1024, 512)), "general_tc"),
    ("bfloat16", ((300, 515), (515, 263)), "general_tc"),
]


def _state_inputs(dtype, shapes, n):
    return [synth.operands(shapes[0], shapes[1], dtype, synth.normal(1.0), synth.normal(0.05), 50 + i)
            for i in range(n)]


@pytest.mark.parametrize("dtype,shapes,algo", STATE_CASES, ids=[c[0] for c in STATE_CASES])
def test_executes_on_two_streams_are_ordered_on_plan_state(dtype, shapes, algo):
    import oracle
    from parity import compare
    ins = _state_inputs(dtype, shapes, 4)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    with Plan(shapes[0], shapes[1], dtype) as p:
        assert p.algorithm == algo
        dev = [(a.cuda(), b.cuda()) for a, b in ins]
        a0, b0 = dev[0]
        assert p.workspace_bytes > 0 or p.staging_copies(a0, b0, None) > 0
        ydt = synth.TORCH_DTYPES[synth.output_dtype(dtype)]
        ys = [torch.full(p.output_shape, float("nan"), dtype=ydt, device="cuda") for _ in ins]
        torch.cuda.synchronize()
        for rep in range(2):
            for i, ((A, B), Y) in enumerate(zip(dev, ys)):
                p.execute(A, B, Y, stream=streams[(i + rep) % 2])
            for s in streams:
                s.synchronize()
            for (a, b), Y in zip(ins, ys):
                y_ref, sc = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
                compare(Y.cpu(), y_ref, sc, dtype)


def test_graph_capture_after_an_execute_on_another_stream():
    """A split-K plan executed on one stream, then captured in a CUDA graph on
    another: the capture records no wait on the plan's event (it would tie
    the graph to work outside it), and the replays compute the product."""
    import oracle
    from parity import compare
    dtype, shapes = "float16", ((32, 65536), (65536, 32))
    (a, b), = _state_inputs(dtype, shapes, 1)
    A, B = a.cuda(), b.cuda()
    with Plan(shapes[0], shapes[1], dtype) as p:
        assert p.algorithm == "split_k" and p.workspace_bytes > 0
        Y0 = torch.empty(p.output_shape, dtype=A.dtype, device="cuda")
        first = torch.cuda.Stream()
        p.execute(A, B, Y0, stream=first)
        first.synchronize()
        Y = torch.full(p.output_shape, float("nan"), dtype=A.dtype, device="cuda")
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                p.execute(A, B, Y, stream=cap)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        y_ref, sc = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
        compare(Y.cpu(), y_ref, sc, dtype)
        assert torch.equal(Y, Y0)
