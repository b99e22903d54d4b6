"""Q4_0 block quantisation for the oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the CUDA path.

The minfer page "Qwen2 / Qwen2.5 Architecture Support" names Q4_0 beside
Q8_0 as the format of the tied output matmul (section 3) and never defines
it.  The reading used here is the four-bit counterpart of this oracle's
Q8_0 reading, decided in float32 as the quantising side would:

* a block is 32 consecutive elements along the input (K) dimension of one
  weight row;
* ``amax = max |x|`` over the block, ``d = amax / 7`` (float32 division);
* ``c = clamp(round_half_away_from_zero(x / d), -7, 7)`` with a true
  float32 division by the unrounded ``d``; ``c = 0`` where ``d == 0``;
* the stored code is the nibble ``c + 8`` (1..15; 0 is never written), two
  per byte: element ``2j`` in the low nibble of byte ``j``, element
  ``2j + 1`` in the high nibble (16 bytes a block);
* the stored scale is ``float16(d)`` (round to nearest even), so a block
  takes 18 bytes (4.5 bits an element);
* dequantised value ``= float32(scale) * (code - 8)`` (exact in float32: an
  11-bit significand times a 4-bit integer).
"""
from __future__ import annotations

import numpy as np

from .q8_0 import round_half_away_magnitude

QK = 32


def quantize_q4_0(w: np.ndarray):
    """Quantise a float16 matrix ``[rows, K]`` (K a multiple of 32).

    Returns ``(packed, d)``: ``packed`` uint8 ``[rows, K // 2]`` (two codes a
    byte) and ``d`` float16 ``[rows, K // 32]``.
    """
    w = np.asarray(w)
    rows, k = w.shape
    if k % QK:
        raise ValueError(f"K={k} is not a multiple of {QK}")
    x = w.astype(np.float32).reshape(rows, k // QK, QK)
    amax = np.max(np.abs(x), axis=2)                       # float32
    d = (amax / np.float32(7.0)).astype(np.float32)        # float32 division
    safe = np.where(d == 0, np.float32(1.0), d)[:, :, None]
    v = (x / safe).astype(np.float32)                      # float32 division
    c = np.sign(v) * round_half_away_magnitude(np.abs(v))
    c = np.clip(c, -7, 7)
    c = np.where((d == 0)[:, :, None], 0, c)
    codes = (c + 8).astype(np.uint8).reshape(rows, k)
    return pack_nibbles(codes), d.astype(np.float16)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """``[rows, K]`` codes 0..15 -> ``[rows, K // 2]`` bytes, element 2j in
    the low nibble of byte j and element 2j + 1 in the high nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_nibbles`."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    out = np.empty((rows, 2 * half), dtype=np.uint8)
    out[:, 0::2] = packed & 0x0F
    out[:, 1::2] = packed >> 4
    return out


def dequantize_q4_0(packed: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Exact dequantisation to float64: ``float(scale) * (code - 8)``."""
    codes = unpack_nibbles(packed).astype(np.float64) - 8.0
    rows, k = codes.shape
    scale = d.astype(np.float64)[:, :, None]
    return (scale * codes.reshape(rows, k // QK, QK)).reshape(rows, k)
