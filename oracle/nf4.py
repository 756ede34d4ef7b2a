"""Plain CPU oracle of the 4-bit NormalFloat (NF4) weight-only linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may call it.  It shares no code with the CUDA library.

Source: "Support QLoRA 4-bit finetuning with bitsandbytes" (lit-gpt PR #275):
the PR description adds the ``bnb.nf4`` quantize option for fine-tuning, and
the measurements in its conversation run Llama-2-7B with ``--precision
bf16-true --quantize bnb.nf4``: the frozen base weights are stored in 4 bits
and every matmul runs in the bf16 compute dtype against weights dequantized on
the fly (the conversation attributes the slower training to that
dequantization).  The page names the format but does not define it.

Reading (the published construction of QLoRA's 4-bit NormalFloat, restated;
every point is listed in the design notes):

* levels: 16 values, asymmetric so that zero is exact.  With
  delta = ((1 - 1/30) + (1 - 1/32)) / 2, the 8 positive levels are the
  standard-normal quantiles of the 8 probabilities evenly spaced from delta
  down towards 1/2 (9 points including 1/2, which is dropped), the 7 negative
  levels the negated quantiles of 7 probabilities spaced the same way (8
  points including 1/2), plus 0; all are divided by the largest, so the table
  runs from -1 to 1.  Each level is computed in float64 and rounded once to
  fp32;
* blocks of 64 consecutive elements of a weight row share one fp32 absmax;
* the code of x is the index of the level nearest to x / absmax, decided in
  fp32: x / absmax is one IEEE fp32 division, compared (strictly greater)
  against the 15 midpoints of adjacent levels, each midpoint the fp32 rounding
  of the exact mean of two fp32 levels; an all-zero block has absmax 0 and
  every code is the zero level;
* two codes per byte, the even element of the row in the high nibble; rows
  are padded to a multiple of 64 elements with the zero level;
* dequantization: fp32(level) * absmax as one fp32 multiply, rounded once to
  the compute dtype (bf16 or fp16);
* the matmuls multiply the compute-dtype operands exactly and sum in float64
  here; the result is rounded once to the compute dtype;
* the ``nf4-dq`` variant stores the absmax values themselves in 8 bits; its
  encoding is oracle/dq8.py, and the matmuls here take the decoded values.

Parity status: every function here is pinned by ``tests/test_nf4_oracle.py``
(equal probability mass between levels evaluated with ``math.erf``,
brute-force nearest level on small inputs, lossless special cases, brute-force
float64 matmuls).
"""
from __future__ import annotations

import numpy as np
from scipy.special import ndtri

from . import F16, BF16, F32, round_to, widen

BLOCK = 64
ZERO_CODE = 7
DELTA = ((1.0 - 1.0 / 30.0) + (1.0 - 1.0 / 32.0)) / 2.0


def levels() -> np.ndarray:
    """The 16 NF4 levels, ascending, fp32."""
    pos = ndtri(np.linspace(DELTA, 0.5, 9)[:-1])          # 8 quantiles > 0
    neg = -ndtri(np.linspace(DELTA, 0.5, 8)[:-1])         # 7 quantiles < 0
    v = np.sort(np.concatenate([neg, [0.0], pos]))
    return (v / v.max()).astype(np.float32)


def midpoints(lv: np.ndarray | None = None) -> np.ndarray:
    """fp32 rounding of the exact mean of adjacent fp32 levels (15 values)."""
    lv = levels() if lv is None else lv
    x = lv.astype(np.float64)
    return ((x[:-1] + x[1:]) / 2.0).astype(np.float32)


def padded(K: int) -> int:
    return (K + BLOCK - 1) // BLOCK * BLOCK


def quantize(W: np.ndarray, dtype: str):
    """Blockwise NF4 quantization of a weight W [N, K] stored in ``dtype``.

    Returns (packed uint8 [N, padded(K) / 2], absmax fp32 [N, padded(K) / 64],
    codes uint8 [N, K])."""
    x = widen(W, dtype).astype(np.float32)                 # exact for all three dtypes
    N, K = x.shape
    Kp = padded(K)
    xp = np.zeros((N, Kp), np.float32)
    xp[:, :K] = x
    blocks = xp.reshape(N, Kp // BLOCK, BLOCK)
    absmax = np.abs(blocks).max(axis=2).astype(np.float32)
    safe = np.where(absmax > 0, absmax, np.float32(1.0))
    xn = (blocks / safe[:, :, None]).astype(np.float32)    # one fp32 division per element
    xn = np.where(absmax[:, :, None] > 0, xn, np.float32(0.0))
    mid = midpoints()
    codes = (xn[..., None] > mid).sum(axis=-1).astype(np.uint8).reshape(N, Kp)
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
    prod = (levels()[codes] * scale).astype(np.float32)    # fp32 * fp32 -> fp32 (RNE)
    return round_to(prod.astype(np.float64), dtype)


def forward(A, dtype, packed, absmax, K, bias=None, bias_dtype=None, rows=None):
    """out = round_to(A @ Wdq^T + bias) with A [M, K] in the compute dtype
    (f16 or bf16), float64 sums.  ``rows``: only these rows of A."""
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


__all__ = ["BLOCK", "ZERO_CODE", "DELTA", "levels", "midpoints", "padded", "quantize", "unpack",
           "dequantize", "forward", "backward_input", "F16", "BF16", "F32"]
