"""The FMA-pipe probe behind the FLOAT / DOUBLE rooflines: it runs, reports
a positive rate, and stays below twice the peak derived from unit counts
and the maximum clock (152 SMs x 128 FP32 lanes x 2 flop; 152 SMs x 4 FP64
flop per clock) -- a rate far above it would mean the probe lost its work."""

import pytest
import torch

from gemm_matmulplan_broadcast_gb300 import binding

pytestmark = pytest.mark.gpu


def _derived(kind):
    props = torch.cuda.get_device_properties(0)
    clk = 2.07e9
    per_sm = 128 * 2 if kind in (0, 1) else 4
    return props.multi_processor_count * per_sm * clk


@pytest.mark.parametrize("kind,iters", [(0, 20000), (1, 20000), (2, 600), (3, 300)])
def test_alu_probe_rates_are_plausible(kind, iters):
    r = binding.alu_rate(kind, iters)
    assert 0.05 * _derived(kind) < r < 2.0 * _derived(kind), (kind, r, _derived(kind))


def test_alu_probe_rejects_bad_arguments():
    with pytest.raises(binding.OlcError):
        binding.alu_rate(4, 10)
    with pytest.raises(binding.OlcError):
        binding.alu_rate(0, 0)
