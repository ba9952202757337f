"""Pins for the oracle's number-format decoders (CPU only).

FP8-E4M3 follows the OCP 8-bit floating point definition (bias 7, max 448,
no infinity, S.1111.111 = NaN), the format the FP8 K/V pages use ("The
Sub-Millisecond Speculative Decoding Meltdown", section "Custom FP8 Quantized
Memory Block Layout").  The oracle's decoder is checked against torch's own
float8_e4m3fn conversion (a library routine) on all 256 codes, and against a
hand-written table of landmark values.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore")


def test_e4m3_all_codes_match_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle_mod.e4m3_to_double(c) for c in range(256)])
    nan_ref = np.isnan(ref)
    assert np.array_equal(nan_ref, np.isnan(mine))
    assert np.array_equal(ref[~nan_ref], mine[~nan_ref])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x80, -0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
    (0x08, 2.0 ** -6), (0x38, 1.0), (0x3C, 1.5), (0x7E, 448.0), (0xFE, -448.0),
    (0x77, 240.0), (0x40, 2.0),
])
def test_e4m3_landmarks(oracle_mod, code, value):
    got = oracle_mod.e4m3_to_double(code)
    assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)


def test_e4m3_nan_codes(oracle_mod):
    assert math.isnan(oracle_mod.e4m3_to_double(0x7F))
    assert math.isnan(oracle_mod.e4m3_to_double(0xFF))


def test_e4m3_values_exact_in_bf16(oracle_mod):
    # every finite E4M3 value is exactly representable in bf16 (3-bit mantissa,
    # exponent range inside bf16's) -- the kernel's in-register decode relies on it
    for c in range(256):
        v = oracle_mod.e4m3_to_double(c)
        if math.isnan(v):
            continue
        assert torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).item() == v


def test_bf16_decode_matches_torch(oracle_mod):
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(4096, generator=g) * 10).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    mine = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(mine, x.to(torch.float64).numpy())
    for special in (0x7F80, 0xFF80):
        assert math.isinf(oracle_mod.bf16_to_double(special))
    assert math.isnan(oracle_mod.bf16_to_double(0x7FC0))
