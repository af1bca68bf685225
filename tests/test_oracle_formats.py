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


# ---- E4M3 encoder (quantising appended K/V rows)

from oracle.formats import f64_to_e4m3_bits  # noqa: E402


def test_e4m3_encoder_round_trips_every_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3_bits_to_f64(codes)
    finite = ~np.isnan(vals)
    assert np.array_equal(f64_to_e4m3_bits(vals[finite]), codes[finite])
    assert np.all(f64_to_e4m3_bits(np.array([np.nan, -np.nan])) == 0x7F)


def test_e4m3_encoder_is_nearest_by_brute_force():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 60, 2000), rng.uniform(-0.02, 0.02, 2000)])
    x = x[np.abs(x) <= 448]
    got = e4m3_bits_to_f64(f64_to_e4m3_bits(x))
    table = e4m3_bits_to_f64(np.arange(256, dtype=np.uint8))
    table = table[~np.isnan(table)]
    best = np.abs(x[:, None] - table[None, :]).min(axis=1)
    assert np.array_equal(np.abs(got - x), best)


def test_e4m3_encoder_ties_go_to_the_even_code():
    pos = e4m3_bits_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2          # exactly halfway between neighbours
    codes = f64_to_e4m3_bits(mids)
    lower = np.arange(0x7E)
    want = np.where(lower % 2 == 0, lower, lower + 1)
    assert np.array_equal(codes, want.astype(np.uint8))
    assert np.array_equal(f64_to_e4m3_bits(-mids), (want | 0x80).astype(np.uint8))


def test_e4m3_encoder_saturates_and_keeps_zero_sign():
    got = f64_to_e4m3_bits(np.array([448.0, 449.0, 464.0, 1e6, -500.0, 0.0, -0.0]))
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x00, 0x80]


def test_e4m3_encoder_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(11)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * 40
    x = x[x.abs() <= 448]
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f64_to_e4m3_bits(x.double().numpy()), want)
