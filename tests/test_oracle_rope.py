"""Pins of the oracle's rotary embedding: closed forms of the table, the
rotation's invariants in float64, the float32 kernel-precision path against
the float64 rotation, and the bf16 rounding against PyTorch."""
import math

import numpy as np
import torch

from oracle import rope


def test_table_closed_forms():
    t = rope.table(10000.0, 4, 101)
    # d = 4: w_0 = 1, w_1 = 10000^(-1/2) = 0.01
    for p in (0, 1, 7, 100):
        np.testing.assert_array_equal(t[p, 0], np.float32([math.cos(p), math.sin(p)]))
    np.testing.assert_array_equal(t[100, 1], np.float32([math.cos(1.0), math.sin(1.0)]))
    # d = 128, theta 500000: w_63 = 500000^(-126/128)
    t2 = rope.table(500000.0, 128, 3)
    w63 = 500000.0 ** (-126 / 128)
    np.testing.assert_array_equal(t2[2, 63], np.float32([math.cos(2 * w63), math.sin(2 * w63)]))


def test_position_zero_is_identity():
    rng = np.random.default_rng(1)
    x = rope.f32_to_bf16_bits(rng.standard_normal((5, 3, 64)).astype(np.float32))
    tab = rope.table(500000.0, 64, 8)
    np.testing.assert_array_equal(rope.apply(x, np.zeros(5, dtype=np.int64), tab), x)


def test_rotate_half_pairing():
    """The reading pairs dimension i with i + d/2: a unit vector on dimension
    i turns towards dimension i + d/2."""
    d, p, i = 16, 3, 2
    x = np.zeros((1, 1, d))
    x[0, 0, i] = 1.0
    y = rope.exact_rotation(x, np.array([p]), 100.0)
    w = 100.0 ** (-2 * i / d)
    expect = np.zeros(d)
    expect[i], expect[i + d // 2] = math.cos(p * w), math.sin(p * w)
    np.testing.assert_allclose(y[0, 0], expect, rtol=0, atol=1e-15)


def test_rotation_preserves_pair_norms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 2, 32))
    pos = rng.integers(0, 40000, 6)
    y = rope.exact_rotation(x, pos, 500000.0)
    n0 = x[..., :16] ** 2 + x[..., 16:] ** 2
    n1 = y[..., :16] ** 2 + y[..., 16:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12, atol=0)


def test_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    ref = None
    for m, n in ((10, 3), (17, 10), (5007, 5000), (32000, 31993)):
        s = float((rope.exact_rotation(q, np.array([m]), 500000.0) * rope.exact_rotation(k, np.array([n]), 500000.0)).sum())
        ref = s if ref is None else ref
        assert abs(s - ref) < 1e-9 * max(1.0, abs(ref)), (m, n, s, ref)


def test_float32_path_within_bf16_rounding_of_exact_rotation():
    rng = np.random.default_rng(4)
    d, n = 128, 64
    x = rope.f32_to_bf16_bits(rng.standard_normal((n, 8, d)).astype(np.float32))
    pos = rng.integers(0, 32768, n)
    got = rope.bf16_bits_to_f32(rope.apply(x, pos, rope.table(500000.0, d, 32768))).astype(np.float64)
    exact = rope.exact_rotation(rope.bf16_bits_to_f32(x), pos, 500000.0)
    # bf16 rounding (unit roundoff 2^-8) plus the float32 table and products
    # (a few 2^-24, scaled by the pair's magnitude)
    pair = np.sqrt(np.concatenate([exact[..., :d // 2] ** 2 + exact[..., d // 2:] ** 2] * 2, axis=-1))
    err = np.abs(got - exact)
    assert np.all(err <= 2.0 ** -8 * np.abs(exact) + 2.0 ** -20 * pair)
    # and mostly well inside it: a sign or pairing mistake would not be
    assert np.median(err / np.maximum(np.abs(exact), 1e-3)) < 2.0 ** -9


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(4096).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 4096),
                           # exact ties between two bf16 values, both parities
                           (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
                           np.float32([0.0, -0.0, 1.0, -3.5, 65504.0])])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(rope.f32_to_bf16_bits(vals), ref)
