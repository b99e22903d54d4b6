"""Q8_0 block quantisation for the oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the CUDA path.

The Q8_0 weight format is named (never defined) on the minfer page "Qwen2 /
Qwen2.5 Architecture Support", section 3 (the tied output matmul "is a
n_vocab x n_embd Q4_0/Q8_0 matmul") and section 6 (quant support).  The
reading used here, in float32 as the quantising side decides it:

* a block is 32 consecutive elements along the input (K) dimension of one
  weight row;
* ``amax = max |x|`` over the block, ``d = amax / 127`` (float32 division);
* ``q = clamp(round_half_away_from_zero(x / d), -127, 127)`` with a true
  float32 division by the unrounded ``d``; ``q = 0`` where ``d == 0``;
* the stored scale is ``float16(d)`` (round to nearest even);
* dequantised value ``= float32(scale) * q`` (exact in float32: an 11-bit
  significand times a 7-bit integer).
"""
from __future__ import annotations

import numpy as np

QK = 32


def round_half_away_magnitude(a: np.ndarray) -> np.ndarray:
    """Round non-negative float32 magnitudes to the nearest integer, ties
    upward (so ``sign * result`` rounds half away from zero).

    ``floor(a + 0.5)`` is not this: for ``a = 0.49999997`` (the largest
    float32 below one half) the sum rounds to 1.0 in float32.  Here the
    fractional part ``a - floor(a)`` is exact in float32 (both terms share
    the binade of ``a`` or the floor is zero), so the comparison with one
    half decides the tie exactly."""
    a = np.asarray(a, dtype=np.float32)
    fl = np.floor(a)
    frac = (a - fl).astype(np.float32)
    return fl + (frac >= np.float32(0.5)).astype(np.float32)


def quantize_q8_0(w: np.ndarray):
    """Quantise a float16 matrix ``[rows, K]`` (K a multiple of 32).

    Returns ``(q, d)``: ``q`` int8 ``[rows, K]`` and ``d`` float16
    ``[rows, K // 32]``.
    """
    w = np.asarray(w)
    rows, k = w.shape
    if k % QK:
        raise ValueError(f"K={k} is not a multiple of {QK}")
    x = w.astype(np.float32).reshape(rows, k // QK, QK)
    amax = np.max(np.abs(x), axis=2)                       # float32
    d = (amax / np.float32(127.0)).astype(np.float32)      # float32 division
    safe = np.where(d == 0, np.float32(1.0), d)[:, :, None]
    v = (x / safe).astype(np.float32)                      # float32 division
    r = np.sign(v) * round_half_away_magnitude(np.abs(v))
    r = np.clip(r, -127, 127)
    r = np.where((d == 0)[:, :, None], 0, r)
    q = r.astype(np.int8).reshape(rows, k)
    return q, d.astype(np.float16)


def dequantize_q8_0(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Exact dequantisation to float64: ``float(scale) * q`` per block."""
    rows, k = q.shape
    scale = d.astype(np.float64)[:, :, None]
    return (scale * q.reshape(rows, k // QK, QK).astype(np.float64)).reshape(rows, k)


def q8_0_matmul(x: np.ndarray, wq: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """A product with both operands in Q8_0: ``x @ W^T`` for f32 activation
    rows ``x`` [rows, K] and a Q8_0 weight matrix (``wq`` int8 [out, K],
    ``wd`` float16 [out, K // 32]).

    The minfer page "Qwen2 / Qwen2.5 Architecture Support", section 6, says
    the CPU path runs on Q8_0 activations and the CUDA prefill on an int8
    MMQ product, without further detail.  Reading: each activation row is
    rounded to float32 and quantised to Q8_0 exactly as a weight row is
    (module docstring).  Each 32-block's int8 products are summed exactly,
    that integer is scaled by the two blocks' f16 scales, and the blocks are
    added in order (float64 here)."""
    xq, xd = quantize_q8_0(np.asarray(x, dtype=np.float32))
    rows, k = xq.shape
    nb = k // QK
    xs = xq.reshape(rows, nb, QK).astype(np.int64)
    ws = wq.reshape(wq.shape[0], nb, QK).astype(np.int64)
    out = np.zeros((rows, wq.shape[0]), dtype=np.float64)
    for b in range(nb):
        isum = xs[:, b, :] @ ws[:, b, :].T                      # exact integers
        out += isum.astype(np.float64) * np.outer(xd[:, b].astype(np.float64), wd[:, b].astype(np.float64))
    return out
