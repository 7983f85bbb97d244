"""Pins for the oracle's number formats: e4m3fn decode/encode and bf16 rounding.

The pins are closed forms of the e4m3fn format (448 from the AstrAI page
"astrai/extension/fp8_state.py", E4M3_MAX), library routines (torch's and,
where installed, ml_dtypes' float8_e4m3fn conversions) and exhaustive checks
over the 256 codes and every midpoint between neighbouring codes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


def test_e4m3_closed_form_values():
    facts = json.load(open(GOLDEN))
    assert oracle.e4m3_decode(0x7E) == facts["e4m3_max"]["value"] == 448.0
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x00) == 0.0
    assert math.copysign(1.0, oracle.e4m3_decode(0x80)) == -1.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9          # smallest subnormal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6          # smallest normal
    assert oracle.e4m3_decode(0x38) == 1.0                # exponent field 7 = bias
    assert oracle.e4m3_decode(0x3C) == 1.5
    assert oracle.e4m3_decode(0x7D) == 416.0
    assert math.isnan(oracle.e4m3_decode(0x7F))
    assert math.isnan(oracle.e4m3_decode(0xFF))
    # no infinities: the exponent-field-15 codes other than 0x7F are finite
    assert all(math.isfinite(oracle.e4m3_decode(c)) for c in range(0x78, 0x7F))


def test_e4m3_decode_matches_torch_for_all_codes():
    table = oracle.e4m3_decode_table()
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(table))
    assert np.array_equal(ref[~nan], table[~nan])
    # signed zeros agree too
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(table[~nan]))


def test_e4m3_decode_matches_ml_dtypes_for_all_codes():
    ml = pytest.importorskip("ml_dtypes")
    ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    table = oracle.e4m3_decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(table))
    assert np.array_equal(ref[~nan], table[~nan])


def test_e4m3_round_trip_all_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_ties_go_to_even_code_at_every_midpoint():
    table = oracle.e4m3_decode_table()
    for c in range(0x7E):
        lo, hi = table[c], table[c + 1]
        mid = (lo + hi) / 2                      # exact in fp32 (needs 5 bits)
        assert np.float32(mid) == mid
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even, hex(c)
        assert oracle.e4m3_encode(-mid) == 0x80 | even
        below = np.nextafter(np.float32(mid), np.float32(0))
        above = np.nextafter(np.float32(mid), np.float32(np.inf))
        assert oracle.e4m3_encode(below) == c
        assert oracle.e4m3_encode(above) == c + 1


def test_e4m3_saturation_and_specials():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(449.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00        # half the smallest subnormal: tie to 0
    assert oracle.e4m3_encode(2.0 ** -10 * 1.0001) == 0x01
    assert oracle.e4m3_encode(1e-30) == 0x00


def test_e4m3_encode_matches_torch_on_dense_sample():
    """torch's fp32 -> float8_e4m3fn cast rounds to nearest even but does not
    saturate, so the sample is clamped to +-448 first."""
    rng = np.random.default_rng(1)
    parts = [rng.standard_normal(20000).astype(np.float32) * s for s in (1e-3, 0.05, 1, 30, 200)]
    # random bit patterns across the whole finite range, clamped
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    parts.append(bits[np.isfinite(bits)])
    v = np.clip(np.concatenate(parts), -448, 448).astype(np.float32)
    ours = oracle.e4m3_encode_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_rounding_closed_forms_and_torch():
    r = oracle.round_to_bf16
    assert r(1.0) == 1.0
    assert r(1 + 2 ** -8) == 1.0                          # tie, even mantissa stays
    assert r(1 + 3 * 2 ** -8) == 1 + 2 ** -6              # tie, odd -> even
    assert r(1 + 2 ** -8 + 2 ** -30) == 1 + 2 ** -7
    assert r(-3.0) == -3.0
    assert r(3.4e38) == math.inf                          # beyond (2-2^-8)*2^127
    assert r(2.0 ** -133) == 2.0 ** -133                  # smallest bf16 subnormal
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(5000) * np.exp(rng.uniform(-20, 20, 5000))).astype(np.float32)
    ours = np.array([r(float(t)) for t in v])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_widening():
    import synth
    v = np.array([0.0, -0.0, 1.0, -2.5, 3.140625, 1e-40, 65504.0], np.float32)
    h = synth.f32_to_bf16_bits(v)
    back = oracle.bf16_to_f32(h)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(back.view(np.uint32), ref.view(np.uint32))
