"""Rotary position embedding of new K rows (and of Q) before kv_append
(test infrastructure; see the package docstring).

The pages list ``rope`` among the element-wise ops ("Poem ops", the
``ops.elemwise`` row) and RoPE variants among the shared layer blocks
("Write a model in Poem", "Shared building blocks"), with no formula.  The
reading taken is the rotary embedding of the Llama family, whose head
shapes the workloads use:

* frequencies  w_i = theta^(-2i/d),  i = 0 .. d/2-1;
* the angle of a token at position p (its logical index in its working
  set) is p * w_i;
* pairs are (i, i + d/2) ("rotate half"):
      y_i       = x_i cos(p w_i) - x_{i+d/2} sin(p w_i)
      y_{i+d/2} = x_{i+d/2} cos(p w_i) + x_i sin(p w_i)
* V is not rotated.

The rotated rows are stored as bf16, as if the rope op wrote bf16 K and Q
that the append and the attention then read; an e4m3 pool quantises the
rotated bf16 K as kv_append would.

Precision.  The bf16 rounding of the rotated values is an integer decision,
so it is taken in the kernel's precision: the angle table is float64 math
rounded once to float32 (``table``), and each output is two float32
products and a float32 sum or difference, each rounded (``apply``).
``exact_rotation`` is the same rotation in float64 from the angles
themselves; the tests pin ``table``/``apply`` against it and against
closed forms (identity at position 0, norm preservation per pair, the
dependence of <rope(q, m), rope(k, n)> on m - n alone, the pairing of
dimension i with i + d/2).
"""
from __future__ import annotations

import math

import numpy as np


def frequencies(theta: float, head_dim: int) -> np.ndarray:
    """w_i = theta^(-2i/d), float64 [d/2] (the C library's pow; theta is a
    float32 configuration value)."""
    t = float(np.float32(theta))
    return np.array([math.pow(t, -2.0 * i / head_dim) for i in range(head_dim // 2)], dtype=np.float64)


def table(theta: float, head_dim: int, positions: int) -> np.ndarray:
    """float32 [positions, d/2, 2]: (cos, sin) of p * w_i, computed in float64
    (the C library's cos and sin) and rounded once to float32."""
    ang = np.arange(positions, dtype=np.float64)[:, None] * frequencies(theta, head_dim)[None, :]
    return np.stack([np.vectorize(math.cos)(ang), np.vectorize(math.sin)(ang)], axis=-1).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns, nearest with ties to even (finite
    inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def apply(x_bits: np.ndarray, pos: np.ndarray, tab: np.ndarray) -> np.ndarray:
    """Rotate bf16 rows: x_bits uint16 [n, heads, d], pos int [n] ->
    uint16 [n, heads, d] (float32 arithmetic, bf16 result)."""
    x = bf16_bits_to_f32(x_bits)
    half = x.shape[-1] // 2
    cs = tab[np.asarray(pos, dtype=np.int64)]                 # [n, d/2, 2]
    c = cs[:, None, :, 0]
    s = cs[:, None, :, 1]
    x0, x1 = x[..., :half], x[..., half:]
    y0 = (x0 * c).astype(np.float32) - (x1 * s).astype(np.float32)
    y1 = (x1 * c).astype(np.float32) + (x0 * s).astype(np.float32)
    return f32_to_bf16_bits(np.concatenate([y0, y1], axis=-1).astype(np.float32))


def exact_rotation(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """The same rotation in float64 from the angles: x float [n, heads, d]."""
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * frequencies(theta, x.shape[-1])[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x0, x1 = x[..., :half], x[..., half:]
    return np.concatenate([x0 * c - x1 * s, x1 * c + x0 * s], axis=-1)
