"""Second, independent CPU restatement of the MACaQ activation transform.

Test infrastructure (same rules as the rest of ``oracle/``).  It exists only to
cross-check the C oracle bit for bit, so it takes different routes wherever
the definition allows:

* the 32-point Hadamard as whole-array numpy float32 butterflies (reshape to
  pairs at stride h, for h = 1, 2, 4, 8, 16), normalised by
  float32(2 ** -2.5);
* the E8M0 exponent from ``np.frexp`` instead of the fp32 bit fields;
* E2M1 by counting the grid midpoints a magnitude passes (a tie goes up only
  when the lower code is odd), instead of rounding at the binade's spacing.

Follows MACaQ page "What is MACaQ quantization", section "How MACaQ works"
(balance, block Hadamard) and its FAQ "What is W4A4 quantization" (MXFP4).
"""
from __future__ import annotations

import numpy as np

# Midpoints between consecutive E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


def hadamard_blocks_f32(v: np.ndarray) -> np.ndarray:
    """v [..., K] float32, K % 32 == 0 -> blockwise normalised Sylvester H32 . v."""
    shp = v.shape
    x = v.reshape(-1, shp[-1] // 32, 32).astype(np.float32, copy=True)
    for h in (1, 2, 4, 8, 16):
        y = x.reshape(x.shape[0], x.shape[1], 32 // (2 * h), 2, h)
        a = y[:, :, :, 0, :]
        b = y[:, :, :, 1, :]
        x = np.stack((a + b, a - b), axis=3).reshape(x.shape)
    x = x * np.float32(2.0 ** -2.5)
    return x.reshape(shp)


def scale_exponents(amax: np.ndarray) -> np.ndarray:
    _, e = np.frexp(np.asarray(amax, np.float32))   # amax = f * 2^e, f in [0.5, 1)
    se = e.astype(np.int32) - 1 - 2
    se = np.where(np.asarray(amax) == 0, -127, se)
    return np.clip(se, -127, 127).astype(np.int32)


def e2m1_codes(t: np.ndarray) -> np.ndarray:
    t = np.asarray(t, np.float32)
    a = np.abs(t)
    mag = np.zeros(a.shape, np.uint8)
    for c, m in enumerate(_MIDPOINTS):
        up = (a > m) | ((a == m) & (c % 2 == 1))
        mag += up.astype(np.uint8)
    sign = (t.view(np.uint32) >> 31).astype(np.uint8)
    return (sign << 3) | mag


def quantize(x_bits: np.ndarray, f: np.ndarray):
    """bf16 bits [rows, K], factor f [K] -> (codes [rows,K/2], scales [rows,K/32])."""
    x = bf16_bits_to_f32(x_bits)
    rows, K = x.shape
    v = x * np.asarray(f, np.float32)[None, :]
    y = hadamard_blocks_f32(v).reshape(rows, K // 32, 32)
    amax = np.abs(y).max(axis=-1)
    se = scale_exponents(amax)
    t = np.ldexp(y, -se[..., None]).astype(np.float32)
    q = e2m1_codes(t).reshape(rows, K)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    scales = (se + 127).astype(np.uint8)
    return codes, scales
