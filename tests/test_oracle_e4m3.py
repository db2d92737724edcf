"""Pins for the oracle's e4m3 decode table and encoder (CPU only).

The pages fix only the format name ("e4m3", Workers AI post, section 1 "KV cache
quantisation"); the oracle reads it as OCP E4M3.  Each test below pins the oracle
to something other than itself: the format's defining bit fields written as
spot values, torch's float8_e4m3fn conversion (a library routine), and the
rounding rules (nearest, ties to even, saturate instead of overflow).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table():
    return oracle.e4m3_table()


def test_spot_values_from_format_definition():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_format_points.json")))
    tab = _table()
    for p in g["points"]:
        c = int(p["code"], 16)
        v = tab[c]
        assert v == p["value"], (p, v)
        assert math.copysign(1.0, v) == math.copysign(1.0, p["value"])
    for c in g["nan_codes"]:
        assert math.isnan(tab[int(c, 16)])
    assert np.isnan(tab).sum() == 2


def test_table_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = _table()
    both_nan = np.isnan(ref) & np.isnan(tab)
    assert np.all(both_nan | (ref == tab))
    assert np.array_equal(np.isnan(ref), np.isnan(tab))


def test_table_is_monotone_and_symmetric():
    tab = _table()
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(tab[0x80:0xFF], -pos)


def test_encode_decode_roundtrip_all_finite_codes():
    tab = _table()
    finite = [c for c in range(256) if not math.isnan(tab[c])]
    assert len(finite) == 254
    vals = np.array([tab[c] for c in finite], dtype=np.float32)
    enc = oracle.e4m3_encode(vals)
    assert list(enc) == finite


def test_ties_go_to_even_and_neighbours_to_nearest():
    tab = _table()
    for c in range(0, 0x7E):
        lo, hi = tab[c], tab[c + 1]
        mid = np.float32((lo + hi) / 2.0)
        assert float(mid) == (lo + hi) / 2.0  # midpoints are exact in fp32
        even = c if c % 2 == 0 else c + 1
        enc = oracle.e4m3_encode([mid, np.nextafter(mid, np.float32(-1)), np.nextafter(mid, np.float32(1e9)),
                                  -mid])
        assert enc[0] == even, (hex(c), float(mid))
        assert enc[1] == c
        assert enc[2] == c + 1
        assert enc[3] == (even | 0x80)


def test_saturation_nan_and_signed_zero():
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e30, np.inf], dtype=np.float32)
    assert list(oracle.e4m3_encode(big)) == [0x7E] * len(big)
    assert list(oracle.e4m3_encode(-big)) == [0xFE] * len(big)
    assert list(oracle.e4m3_encode([np.nan])) == [0x7F]
    assert list(oracle.e4m3_encode([0.0, -0.0, 1e-30, -1e-30])) == [0x00, 0x80, 0x00, 0x80]
    # half of the smallest subnormal is a tie between 0 (even) and 0x01
    half = np.float32(2.0 ** -10)
    assert list(oracle.e4m3_encode([half, np.nextafter(half, np.float32(1))])) == [0x00, 0x01]


def test_encode_matches_torch_cast_on_in_range_values():
    rng = np.random.default_rng(7)
    # magnitudes spread over the whole e4m3 range, including subnormals
    mag = np.exp2(rng.uniform(-12, 8.8, size=200_000)).astype(np.float32)
    x = (mag * rng.choice([-1, 1], size=mag.shape)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x)
    assert np.array_equal(got, ref)


def test_bf16_to_f32_is_exact_bit_shift():
    bits = np.arange(0, 65536, 257, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    got = oracle.bf16_to_f32(bits)
    same = (got.view(np.uint32) == ref.view(np.uint32))
    assert np.all(same)
