"""Pins of the oracle's FP8 E4M3 codec against the format definition and an
independent implementation (PyTorch's float8_e4m3fn)."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_points.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, value, label = line.split()
            rows.append((int(code, 16), float(value), label))
    return rows


def test_decode_matches_format_definition_points():
    for code, value, label in _golden():
        got = e4m3.decode(np.array([code], dtype=np.uint8))[0]
        if math.isnan(value):
            assert math.isnan(got), label
        else:
            assert got == value and math.copysign(1, got) == math.copysign(1, value), label


def test_decode_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.decode_table()
    np.testing.assert_array_equal(np.isnan(ref), np.isnan(ours))
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(ref[fin], ours[fin])


def test_decode_table_structure():
    t = e4m3.decode_table()
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must be strictly increasing"
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])
    assert pos.max() == e4m3.MAX_FINITE


def test_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes).astype(np.float32)
    np.testing.assert_array_equal(e4m3.encode(vals), codes)


def _all_bf16_finite():
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)]


@pytest.mark.parametrize("scale", [1.0, 5.0 / 448.0, 0.37, 4.25 / 448.0])
def test_encode_matches_torch_rne_over_all_bf16(scale):
    x = _all_bf16_finite()
    inv = np.float32(1.0) / np.float32(scale)
    with np.errstate(over="ignore"):
        prod = (x * inv).astype(np.float32)
    ours = e4m3.quantize(x, scale)
    inrange = np.abs(prod) <= 448.0
    ref = torch.from_numpy(prod[inrange]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours[inrange], ref)
    big = ~inrange
    expect = np.where(np.signbit(prod[big]), 0xFE, 0x7E).astype(np.uint8)
    np.testing.assert_array_equal(ours[big], expect)


def test_encode_brute_force_nearest_even():
    """Brute force over all 256 codes for a sample of values, including exact
    midpoints between neighbouring codes."""
    table = e4m3.decode_table()
    finite = [c for c in range(128) if not math.isnan(table[c])]
    rng = np.random.default_rng(0)
    mids = [(table[c] + table[c + 1]) / 2 for c in range(126)]
    vals = np.concatenate([rng.standard_normal(300) * 50, np.array(mids), -np.array(mids[:40])])
    vals = vals.astype(np.float32)
    got = e4m3.encode(vals)
    for v, g in zip(vals.tolist(), got.tolist()):
        a = abs(v)
        best = min(finite, key=lambda c: (abs(table[c] - a), c & 1))
        if a >= 448:
            best = 0x7E
        if math.copysign(1.0, v) < 0:
            best |= 0x80
        assert g == best, (v, g, best)
