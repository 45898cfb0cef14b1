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
