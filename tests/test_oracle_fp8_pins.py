"""Pins for the oracle's 8-bit float operands: the decoders against torch's
float8_e4m3fn / float8_e5m2 conversions for all 256 patterns (so a wrong
bias, mantissa width or NaN rule fails), and MatMul of 8-bit operands
against pure-Python integer arithmetic (float32 output, not narrowed)."""

import numpy as np
import pytest
import torch

import oracle
from gemm_matmulplan_broadcast_gb300 import synth
from test_oracle_pins import _brute

U8 = np.arange(256, dtype=np.uint8)


@pytest.mark.parametrize("dtype", oracle.FP8_DTYPES)
def test_decode_all_patterns_match_torch(dtype):
    got = oracle.decode_fp8(U8, dtype).astype(np.float64)
    want = torch.from_numpy(U8.copy()).view(synth.TORCH_DTYPES[dtype]).float().double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_known_values():
    e4 = oracle.decode_fp8(np.array([0x7E, 0x01, 0x38, 0xC0, 0x7F], np.uint8), "float8_e4m3fn")
    assert e4[0] == 448.0 and e4[1] == 2.0 ** -9 and e4[2] == 1.0 and e4[3] == -2.0
    assert np.isnan(e4[4])
    e5 = oracle.decode_fp8(np.array([0x7B, 0x01, 0x3C, 0x7C, 0x7D], np.uint8), "float8_e5m2")
    assert e5[0] == 57344.0 and e5[1] == 2.0 ** -16 and e5[2] == 1.0
    assert np.isinf(e5[3]) and np.isnan(e5[4])


def test_decode_known_values_fnuz():
    # exponent bias one larger than the FN formats, no infinities, no -0, 0x80 the only NaN
    e4 = oracle.decode_fp8(np.array([0x7F, 0x01, 0x40, 0xC0, 0x80, 0x00], np.uint8), "float8_e4m3fnuz")
    assert e4[0] == 240.0 and e4[1] == 2.0 ** -10 and e4[2] == 1.0 and e4[3] == -1.0
    assert np.isnan(e4[4]) and e4[5] == 0.0 and not np.signbit(e4[5])
    assert np.isnan(e4).sum() == 1
    e5 = oracle.decode_fp8(np.array([0x7F, 0x01, 0x40, 0x7C, 0x80, 0xFF], np.uint8), "float8_e5m2fnuz")
    assert e5[0] == 57344.0 and e5[1] == 2.0 ** -17 and e5[2] == 1.0 and e5[3] == 32768.0
    assert np.isnan(e5[4]) and e5[5] == -57344.0
    full4 = oracle.decode_fp8(np.arange(256, dtype=np.uint8), "float8_e4m3fnuz")
    full5 = oracle.decode_fp8(np.arange(256, dtype=np.uint8), "float8_e5m2fnuz")
    assert np.isnan(full4).sum() == 1 and np.isnan(full5).sum() == 1
    assert not np.isinf(full4).any() and not np.isinf(full5).any()


@pytest.mark.parametrize("dtype", oracle.FP8_DTYPES)
def test_fp8_matmul_integer_exact(dtype):
    a, b = synth.operands((2, 5, 40), (40, 7), dtype, synth.SMALL_INT, synth.SMALL_INT, 3)
    y, s = oracle.matmul(synth.to_numpy_storage(a), synth.to_numpy_storage(b), dtype)
    assert y.dtype == np.float32 and y.shape == (2, 5, 7)
    an, bn = a.float().numpy().astype(np.int64), b.float().numpy().astype(np.int64)
    for z in range(2):
        want = np.array(_brute(an[z], bn), dtype=np.float64)
        assert np.array_equal(y[z].astype(np.float64), want)
        assert np.all(s[z] >= np.abs(want))


@pytest.mark.parametrize("dtype", oracle.FP8_DTYPES)
def test_lookup_decode_equals_field_decode(dtype):
    """The oracle decodes large operands by looking up the 256 patterns that
    the field decode produces; both give the same values (NaN where NaN) in
    the input's shape."""
    bits = np.random.default_rng(11).integers(0, 256, (37, 129), dtype=np.uint8)
    got = oracle.decode_fp8(bits, dtype)
    want = oracle.decode_fp8_fields(bits, dtype)
    assert got.shape == bits.shape and got.dtype == np.float32
    assert np.array_equal(got, want, equal_nan=True)
