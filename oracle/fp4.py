"""Plain CPU oracle of the 4-bit floating-point (FP4) weight-only linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may call it.  It shares no code with the CUDA library.

Source: "Support QLoRA 4-bit finetuning with bitsandbytes" (lit-gpt PR #275):
the PR adds the ``bnb.fp4`` quantize option beside ``bnb.nf4`` for
fine-tuning with frozen 4-bit base weights and 16-bit compute.  The page names
the format but does not define it.

Reading (every point is listed in the design notes):

* the format is E2M1, the 4-bit floating point with 1 sign, 2 exponent and 1
  mantissa bits (exponent bias 1, exponent 0 subnormal): magnitudes 0, 0.5,
  1, 1.5, 2, 3, 4, 6 for the exponent-mantissa bits c = 0..7;
* blocks of 64 consecutive elements of a weight row share one fp32 absmax
  (the storage of the NF4 option), mapped to the largest magnitude 6: the
  levels are E2M1(c) / 6 rounded once to fp32, code 8 s + c carrying the
  sign s;
* the code of x: y = x / absmax as one IEEE fp32 division; c is the
  magnitude level nearest to |y|, decided against the fp32 midpoints of
  adjacent magnitude levels (each the fp32 rounding of the exact mean of two
  fp32 levels), and |y| equal to a midpoint takes the level whose mantissa
  bit is 0 (round half to even, as IEEE rounding does); s = 1 when y < 0
  and c > 0, so zero has the single code 0; an all-zero block has absmax 0
  and codes 0;
* packing, dequantization (fp32(level) * absmax, one fp32 multiply, rounded
  once to the compute dtype) and the matmuls (float64 sums here, one
  rounding of the result) are those of the NF4 option;
* the ``fp4-dq`` variant stores the absmax values in 8 bits; its encoding is
  oracle/dq8.py, and the matmuls here take the decoded values.

Parity status: pinned by ``tests/test_fp4_oracle.py`` (the levels against the
E2M1 bit-field definition, brute-force nearest level, constructed half-way
ties, lossless cases, brute-force float64 matmuls).
"""
from __future__ import annotations

import numpy as np

from . import F16, BF16, F32, round_to, widen

BLOCK = 64
ZERO_CODE = 0
# E2M1 magnitudes of the exponent-mantissa bits 0..7
MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def levels() -> np.ndarray:
    """The 16 levels by code (sign in bit 3), fp32: +-E2M1 / 6."""
    mag = (np.array(MAGNITUDES, np.float64) / 6.0).astype(np.float32)
    return np.concatenate([mag, -mag]).astype(np.float32)


def midpoints() -> np.ndarray:
    """fp32 rounding of the exact mean of adjacent fp32 magnitude levels (7)."""
    m = levels()[:8].astype(np.float64)
    return ((m[:-1] + m[1:]) / 2.0).astype(np.float32)


def tie_goes_up() -> np.ndarray:
    """For each midpoint j: does a value equal to it take the upper level
    j + 1?  Yes when that level's mantissa bit (the low bit of j + 1) is 0."""
    return np.array([((j + 1) & 1) == 0 for j in range(7)])


def padded(K: int) -> int:
    return (K + BLOCK - 1) // BLOCK * BLOCK


def quantize(W: np.ndarray, dtype: str):
    """Blockwise FP4 quantization of a weight W [N, K] stored in ``dtype``.

    Returns (packed uint8 [N, padded(K) / 2], absmax fp32 [N, padded(K) / 64],
    codes uint8 [N, K])."""
    x = widen(W, dtype).astype(np.float32)
    N, K = x.shape
    Kp = padded(K)
    xp = np.zeros((N, Kp), np.float32)
    xp[:, :K] = x
    blocks = xp.reshape(N, Kp // BLOCK, BLOCK)
    absmax = np.abs(blocks).max(axis=2).astype(np.float32)
    safe = np.where(absmax > 0, absmax, np.float32(1.0))
    y = (blocks / safe[:, :, None]).astype(np.float32)     # one fp32 division per element
    y = np.where(absmax[:, :, None] > 0, y, np.float32(0.0))
    a = np.abs(y)[..., None]
    mid, up = midpoints(), tie_goes_up()
    c = ((a > mid) | ((a == mid) & up)).sum(axis=-1).astype(np.uint8)
    codes = np.where((y < 0) & (c > 0), c | 8, c).astype(np.uint8).reshape(N, Kp)
    codes[:, K:] = ZERO_CODE
    packed = ((codes[:, 0::2] << 4) | codes[:, 1::2]).astype(np.uint8)
    return packed, absmax, codes[:, :K].copy()


def unpack(packed: np.ndarray, K: int) -> np.ndarray:
    """Codes [N, K] from the packed rows (even element in the high nibble)."""
    N = packed.shape[0]
    codes = np.empty((N, packed.shape[1] * 2), np.uint8)
    codes[:, 0::2] = packed >> 4
    codes[:, 1::2] = packed & 15
    return codes[:, :K]


def dequantize(packed: np.ndarray, absmax: np.ndarray, K: int, dtype: str) -> np.ndarray:
    """Wdq [N, K] in ``dtype`` storage: fp32(level) * absmax (one fp32
    multiply), rounded once to ``dtype``."""
    codes = unpack(packed, K)
    scale = np.repeat(absmax, BLOCK, axis=1)[:, :K]
    prod = (levels()[codes] * scale).astype(np.float32)
    return round_to(prod.astype(np.float64), dtype)


def forward(A, dtype, packed, absmax, K, bias=None, bias_dtype=None, rows=None):
    """out = round_to(A @ Wdq^T + bias), A [M, K] in the compute dtype (f16
    or bf16), float64 sums.  ``rows``: only these rows of A."""
    if dtype not in (F16, BF16):
        raise ValueError("the compute dtype is f16 or bf16")
    Wdq = dequantize(packed, absmax, K, dtype)
    Ar = A if rows is None else A[rows]
    acc = widen(Ar, dtype) @ widen(Wdq, dtype).T
    if bias is not None:
        acc = acc + widen(bias, bias_dtype)[None, :]
    return dict(Wdq=Wdq, out64=acc, out=round_to(acc, dtype))


def backward_input(G, dtype, packed, absmax, K, rows=None):
    """grad_A = round_to(G @ Wdq), G [M, N] in the compute dtype, float64
    sums (the frozen 4-bit weight has no gradient)."""
    if dtype not in (F16, BF16):
        raise ValueError("the compute dtype is f16 or bf16")
    Wdq = dequantize(packed, absmax, K, dtype)
    Gr = G if rows is None else G[rows]
    acc = widen(Gr, dtype) @ widen(Wdq, dtype)
    return dict(Wdq=Wdq, grad64=acc, grad_A=round_to(acc, dtype))


__all__ = ["BLOCK", "ZERO_CODE", "MAGNITUDES", "levels", "midpoints", "tie_goes_up", "padded", "quantize",
           "unpack", "dequantize", "forward", "backward_input", "F16", "BF16", "F32"]
