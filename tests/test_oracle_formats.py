"""Pins for the oracle's storage decoders: library casts and printed format facts."""

import numpy as np
import pytest
import torch

from oracle.formats import bf16_bits_to_f64, e4m3_bits_to_f64


def test_bf16_decoder_matches_torch_on_all_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    want = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = bf16_bits_to_f64(bits.numpy())
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_bits_to_f64(codes.numpy())
    nan = np.isnan(want)
    assert nan.sum() == 2  # S.1111.111 for both signs
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x7E, 448.0), (0xFE, -448.0),
    (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x40, 2.0),
])
def test_e4m3_definition_values(code, value):
    # Bias 7, subnormal step 2^-9, largest finite 448: the OCP E4M3 definition.
    assert e4m3_bits_to_f64(np.array([code], dtype=np.uint8))[0] == value
