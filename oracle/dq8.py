"""Plain CPU oracle of the double-quantized absmax of the 4-bit weight-only
layers (the ``bnb.nf4-dq`` and ``bnb.fp4-dq`` options).

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may call it.  It shares no code with the CUDA library.

Source: "Support QLoRA 4-bit finetuning with bitsandbytes" (lit-gpt PR #275)
adds the ``bnb.nf4-dq`` and ``bnb.fp4-dq`` quantize options beside
``bnb.nf4`` / ``bnb.fp4`` and reports their memory and loss in its results
tables; the page does not define them.  They are QLoRA's double
quantization: the fp32 absmax constants of the 64-element blocks (the first
level) are themselves stored in 8 bits.

Reading (every point is listed in the design notes):

* the 4-bit codes are those of the plain format, computed with the exact
  fp32 absmax; only the storage of the absmax changes, and the matmuls use
  the decoded absmax;
* offset = the mean of all the absmax values of the weight, subtracted first
  (the constants are positive; centred, a symmetric code fits them):
  fp32(S / n), S the exactly rounded float64 sum of the n fp32 values, one
  IEEE float64 division and one rounding to fp32;
* d = fp32(c - offset); blocks of 256 consecutive d (the row-major order of
  the absmax array [N, blocks per row]) share a second-level scale
  absmax2 = max |d| (fp32);
* the 8-bit float is FP8 E4M3 (1 sign bit, 4 exponent bits with bias 7, 3
  mantissa bits, exponent 0 subnormal, no infinities, largest finite 448,
  S.1111.111 is NaN); the code of d is the E4M3 value nearest to
  y = fp32(d * s2), s2 = fp32(448 / absmax2) (one IEEE fp32 division per
  block; s2 = 0 for a block of zeros), a tie going to the even code (mantissa
  bit 0 clear, as IEEE rounding does), |y| above 448 saturating to 448, and
  the sign of y kept (so a negative y that rounds to zero gives -0);
* decoding: c' = fp32(fp32(v(q) * f2) + offset), f2 = fp32(absmax2 *
  fp32(1 / 448)): a multiply, as the int8 weights are dequantized.

Parity status: pinned by ``tests/test_dq8_oracle.py`` (the E4M3 values
against fixed anchors and torch's float8_e4m3fn conversion, ties and
saturation, the offset against an exact rational mean, the error bound of
the round trip).
"""
from __future__ import annotations

import math

import numpy as np

BLOCK2 = 256          # absmax values per second-level block
FP8_MAX = 448.0
NAN_CODES = (0x7F, 0xFF)


def e4m3_values() -> np.ndarray:
    """The value of every byte as an E4M3 float (fp32; NaN at 0x7F, 0xFF)."""
    out = np.empty(256, np.float32)
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            out[code] = np.nan
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        out[code] = -mag if s else mag
    return out


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code of every fp32 y (ties to the even code, saturating
    at +-448, the sign of y kept), by comparing against all 127 non-negative
    finite values."""
    y = np.asarray(y, np.float32)
    vals = e4m3_values()[:0x7F].astype(np.float64)         # codes 0x00 .. 0x7E, ascending
    a = np.minimum(np.abs(y.astype(np.float64)), FP8_MAX).reshape(-1, 1)
    dist = np.abs(a - vals.reshape(1, -1))
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best                                     # one or two (a tie) candidates
    codes = np.arange(0x7F)
    even = cand & ((codes & 1) == 0).reshape(1, -1)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    sign = np.signbit(y).reshape(-1).astype(np.uint8) << 7
    return (pick.astype(np.uint8) | sign).reshape(y.shape)


def offset_of(absmax: np.ndarray) -> np.float32:
    """fp32(S / n): S the exactly rounded float64 sum of the values."""
    c = np.asarray(absmax, np.float32).reshape(-1)
    if c.size == 0:
        return np.float32(0.0)
    s = math.fsum(float(x) for x in c)
    return np.float32(s / float(c.size))


def blocks(count: int) -> int:
    return (count + BLOCK2 - 1) // BLOCK2


def quantize(absmax: np.ndarray):
    """(codes u8 with the shape of absmax, absmax2 fp32 [blocks], offset fp32)."""
    c = np.asarray(absmax, np.float32)
    flat = c.reshape(-1)
    n = flat.size
    off = offset_of(flat)
    d = (flat - off).astype(np.float32)                     # one fp32 subtract each
    nb = blocks(n)
    a2 = np.zeros(nb, np.float32)
    q = np.zeros(n, np.uint8)
    for b in range(nb):
        seg = d[b * BLOCK2:(b + 1) * BLOCK2]
        m = np.float32(np.abs(seg).max())
        a2[b] = m
        s2 = np.float32(FP8_MAX) / m if m > 0 else np.float32(0.0)
        y = (seg * np.float32(s2)).astype(np.float32)
        q[b * BLOCK2:(b + 1) * BLOCK2] = e4m3_encode(y)
    return q.reshape(c.shape), a2, off


def dequantize(q: np.ndarray, absmax2: np.ndarray, offset) -> np.ndarray:
    """The decoded absmax values, fp32, with the shape of q."""
    q = np.asarray(q, np.uint8)
    flat = q.reshape(-1)
    v = e4m3_values()[flat]
    inv = np.float32(1.0) / np.float32(FP8_MAX)
    f2 = (np.asarray(absmax2, np.float32) * inv).astype(np.float32)
    f2e = np.repeat(f2, BLOCK2)[:flat.size]
    out = ((v * f2e).astype(np.float32) + np.float32(offset)).astype(np.float32)
    return out.reshape(q.shape)
