"""Pins of the oracle's E4M3 table, encoder and per-position quantiser.

Pinned to: the format the page states ("Context Optimization", FP8 KV Cache > How
It Works: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, range +-448, scale =
absmax / 240), hand-worked code values, torch.float8_e4m3fn casts (a library routine
independent of the oracle) and the half-ulp rounding bound.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_format_facts_from_page():
    f = GOLD["e4m3_format"]
    assert f["sign_bits"] + f["exponent_bits"] + f["mantissa_bits"] == 8
    finite = e4m3.E4M3_VALUES[~np.isnan(e4m3.E4M3_VALUES)]
    assert finite.max() == f["range"][1] and finite.min() == f["range"][0]
    # bias 7: exponent field 7 with zero mantissa is exactly 1.0
    assert e4m3.E4M3_VALUES[0b0_0111_000] == 1.0
    assert e4m3.SCALE_DIVISOR == f["scale_divisor"]


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x80, -0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x77, 240.0), (0x7E, 448.0),
    (0xFE, -448.0), (0xB8, -1.0), (0x30, 0.5),
])
def test_hand_worked_codes(code, value):
    got = e4m3.E4M3_VALUES[code]
    assert got == value and np.signbit(got) == np.signbit(value)


def test_nan_codes_and_count():
    assert np.isnan(e4m3.E4M3_VALUES[0x7F]) and np.isnan(e4m3.E4M3_VALUES[0xFF])
    assert np.isnan(e4m3.E4M3_VALUES).sum() == 2
    pos = e4m3.E4M3_VALUES[:0x7F]
    assert np.all(np.diff(pos) > 0)          # strictly increasing magnitudes


def test_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.E4M3_VALUES
    both_nan = np.isnan(vals) & np.isnan(ours)
    assert np.all(both_nan | (vals == ours))


def test_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = e4m3.encode(e4m3.decode(codes))
    assert np.array_equal(back, codes)


def test_encode_matches_torch_cast_on_sweep():
    rng = np.random.default_rng(3)
    y = np.concatenate([
        rng.uniform(-448, 448, 200000), rng.normal(0, 1, 200000), rng.normal(0, 1e-2, 100000),
        # exact midpoints between neighbouring codes exercise ties-to-even
        (e4m3.E4M3_VALUES[1:0x7E] + e4m3.E4M3_VALUES[2:0x7F]) / 2,
        -(e4m3.E4M3_VALUES[1:0x7E] + e4m3.E4M3_VALUES[2:0x7F]) / 2,
    ]).astype(np.float32).astype(np.float64)
    ours = e4m3.encode(y)
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch maps -0.0 to 0x80 too; compare all
    assert np.array_equal(ours, ref)


def test_ties_go_to_even_mantissa():
    # midpoint of 1.0 (0x38, mantissa 0) and 1.125 (0x39, mantissa 1) -> 0x38
    assert e4m3.encode(np.array([1.0625]))[0] == 0x38
    # midpoint of 1.125 (0x39) and 1.25 (0x3A) -> 0x3A (even)
    assert e4m3.encode(np.array([1.1875]))[0] == 0x3A


def test_half_ulp_error_bound():
    rng = np.random.default_rng(5)
    y = rng.uniform(2.0 ** -6, 240.0, 100000).astype(np.float32).astype(np.float64)
    err = np.abs(e4m3.decode(e4m3.encode(y)) - y) / y
    assert err.max() <= 2.0 ** -4 + 1e-15      # normals: relative error <= 2^-(3+1)


def test_sign_of_zero_kept():
    assert e4m3.encode(np.array([-0.0]))[0] == 0x80
    assert e4m3.encode(np.array([-1e-6]))[0] == 0x80
    assert e4m3.encode(np.array([1e-6]))[0] == 0x00


def test_quantise_position_absmax_maps_to_240():
    rng = np.random.default_rng(11)
    x = rng.normal(size=(4, 128)).astype(np.float32).astype(np.float64)
    codes, scale = e4m3.quantise_position(x)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert codes[i] & 0x7F == 0x77              # the absmax element encodes to +-240
    assert scale == np.float32(np.float32(np.abs(x).max()) / np.float32(240.0))
    recon = e4m3.decode(codes) * scale
    assert np.max(np.abs(recon - x)) <= scale * 8.0 + 1e-12   # half-ulp at the top binade


def test_quantise_zero_position():
    codes, scale = e4m3.quantise_position(np.zeros((2, 16)))
    assert scale == 0.0 and not codes.any()
    codes, scale = e4m3.quantise_position(-np.zeros((2, 16)))
    assert scale == 0.0 and not codes.any()


def test_quantise_positions_equals_per_position():
    rng = np.random.default_rng(13)
    x = rng.normal(size=(3, 5, 4, 16)).astype(np.float32).astype(np.float64)
    x[1, 2] = 0.0
    codes, scales = e4m3.quantise_positions(x)
    for a in range(3):
        for b in range(5):
            c1, s1 = e4m3.quantise_position(x[a, b])
            assert s1 == scales[a, b] and np.array_equal(c1, codes[a, b])


def test_fp32_division_is_correctly_rounded():
    rng = np.random.default_rng(17)
    a = rng.uniform(1e-3, 10, 10000).astype(np.float32)
    b = rng.uniform(1e-3, 10, 10000).astype(np.float32)
    ours = e4m3.fl32_div(a, b)
    # reference: numpy's float32 division is IEEE correctly rounded
    assert np.array_equal(ours, (a / b).astype(np.float64))
