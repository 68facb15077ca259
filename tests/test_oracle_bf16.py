"""Pins of the oracle's bf16 conversions against hand-worked values and torch's cast."""

import json
import os

import numpy as np
import pytest

from oracle import bf16_to_f64, f64_to_bf16

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))

CASE_VALUES = {
    "1.0": 1.0,
    "1 + 2^-8 (tie, even down)": 1 + 2.0 ** -8,
    "1 + 3*2^-8 (tie, even up)": 1 + 3 * 2.0 ** -8,
    "1 + 2^-8 + 2^-40 (above the tie)": 1 + 2.0 ** -8 + 2.0 ** -40,
    "-0.0": -0.0,
    "2^-133 (smallest subnormal)": 2.0 ** -133,
    "2^-134 (tie with zero, even down)": 2.0 ** -134,
    "3*2^-134 (tie, even up)": 3 * 2.0 ** -134,
    "2^-126 (smallest normal)": 2.0 ** -126,
    "(2 - 2^-7) * 2^127 (largest finite)": (2 - 2.0 ** -7) * 2.0 ** 127,
    "(2 - 2^-7 + 2^-8) * 2^127 (tie with 2^128, even: inf)": (2 - 2.0 ** -7 + 2.0 ** -8) * 2.0 ** 127,
    "-2.5": -2.5,
}


@pytest.mark.parametrize("name,bits", GOLDEN["bf16_rounding"]["cases"])
def test_hand_worked_rounding(name, bits):
    assert int(f64_to_bf16(CASE_VALUES[name])) == bits


def test_every_pattern_round_trips():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bf16_to_f64(b)
    finite_or_inf = ~np.isnan(v)
    assert np.array_equal(f64_to_bf16(v[finite_or_inf]), b[finite_or_inf])
    assert np.all(f64_to_bf16(v[~finite_or_inf]) == 0x7FC0)


def test_decode_matches_layout():
    # 0x3F80 = sign 0, exponent 127, fraction 0 -> 1.0; 0xC0A0 = -(1 + 2^-2) * 2^2 = -5
    assert bf16_to_f64(np.uint16(0x3F80)) == 1.0
    assert bf16_to_f64(np.uint16(0xC0A0)) == -5.0
    assert bf16_to_f64(np.uint16(0x0001)) == 2.0 ** -133


def test_matches_torch_cast_on_fp32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    f = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),   # subnormal range
        (rng.standard_normal(20000) * 1e38).astype(np.float32),    # near overflow
        rng.integers(-(1 << 20), 1 << 20, 20000).astype(np.float32),
    ])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f64_to_bf16(f.astype(np.float64)), ref)


def test_single_rounding_from_f64():
    # rounding through fp32 first would land on the tie and go to even (0x3F80)
    v = 1 + 2.0 ** -8 + 2.0 ** -40
    assert np.float32(v) == np.float32(1 + 2.0 ** -8)
    assert int(f64_to_bf16(v)) == 0x3F81
