"""Pins of the oracle's storage-format codecs (BF16, FP8 E4M3).

The codecs are checked against PyTorch's own converters (independent library
implementations of IEEE/OCP round-to-nearest-even), against the special values
the OCP 8-bit floating point specification fixes (tests/golden), and by
exhaustive enumeration.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e4m3_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "e4m3_special_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                code, value = line.split()
                vals[int(code, 16)] = float(value)
    return vals


def test_e4m3_decode_all_codes_match_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_special_values_from_spec(oracle_mod):
    for code, value in _e4m3_golden().items():
        assert oracle_mod.e4m3_to_f32(np.uint8(code)) == np.float32(value), hex(code)
        assert oracle_mod.f32_to_e4m3(np.float32(value)) == code, hex(code)


def test_e4m3_encode_round_trips_every_finite_value(oracle_mod):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle_mod.e4m3_to_f32(codes)
    back = oracle_mod.f32_to_e4m3(vals)
    assert np.array_equal(back, codes)


def test_e4m3_encode_matches_torch_rne_in_range(oracle_mod):
    rng = np.random.default_rng(1)
    mags = np.concatenate([
        rng.uniform(0, 448, 4000), np.exp2(rng.uniform(-14, 8.8, 4000)),
        rng.uniform(0, 2 ** -6, 2000)]).astype(np.float32)
    mags = mags[mags < 448]
    # every midpoint between neighbouring finite positive values (ties)
    pos = np.sort(oracle_mod.e4m3_to_f32(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((pos[1:].astype(np.float64) + pos[:-1]) / 2).astype(np.float32)
    x = np.concatenate([mags, -mags, mids, -mids, [0.0, -0.0]]).astype(np.float32)
    ours = oracle_mod.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_ties_go_to_even_mantissa(oracle_mod):
    pos = np.sort(oracle_mod.e4m3_to_f32(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((pos[1:].astype(np.float64) + pos[:-1]) / 2).astype(np.float32)
    codes = oracle_mod.f32_to_e4m3(mids)
    assert np.all((codes & 1) == 0)


def test_e4m3_saturates_finite(oracle_mod):
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3.4e38], dtype=np.float32)
    assert np.all(oracle_mod.f32_to_e4m3(x) == 0x7E)
    assert np.all(oracle_mod.f32_to_e4m3(-x) == 0xFE)


def test_e4m3_underflow(oracle_mod):
    sub = 2.0 ** -9
    x = np.array([sub / 2, sub / 2 * 0.999, sub / 2 * 1.001, 1.5 * sub, 2.5 * sub], dtype=np.float32)
    got = oracle_mod.e4m3_to_f32(oracle_mod.f32_to_e4m3(x))
    assert got.tolist() == [0.0, 0.0, sub, 2 * sub, 2 * sub]


def test_bf16_encode_matches_torch(oracle_mod):
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(20000) * 10, np.exp2(rng.uniform(-130, 120, 5000)),
                        [0.0, -0.0, 1.0, 3.4e38, 1e-40, np.inf, -np.inf]]).astype(np.float32)
    # exact ties: 8 significant bits plus a half
    base = rng.integers(128, 256, 2000).astype(np.float32)
    ties = ((base + 0.5) * np.exp2(rng.integers(-20, 20, 2000))).astype(np.float32)
    x = np.concatenate([x, ties, -ties])
    ours = oracle_mod.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_decode_all_patterns(oracle_mod):
    b = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.bf16_to_f32(b)
    ref = (b.astype(np.uint32) << 16).view(np.float32)
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("x", [np.nan])
def test_nan_inputs_are_outside_the_contract_but_stay_nan(oracle_mod, x):
    assert np.isnan(oracle_mod.e4m3_to_f32(oracle_mod.f32_to_e4m3(np.float32(x))))
