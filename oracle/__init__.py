"""Plain CPU oracle of the LLM.int8-style quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this package: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg
of ``bench.py`` may call it.  It shares no code with the CUDA library.

Sources (bitsandbytes PR #33 "Memory efficient backward", the PR description
and the review threads on ``bitsandbytes/autograd/_functions.py``):

* weights are kept as row-major int8 codes ``CB`` with one absmax scale per
  output row ``SCB`` (PR description, "Stores int8 weights in row-major
  format");
* the input is cast to fp16 before the quantization and the result is cast
  back to the input's dtype (PR description, "Cast inputs and outputs of the
  8bit layer to fp16"; commit "cast to half before double_quant");
* outlier columns of A are taken out of the int8 product as ``subA`` and
  multiplied in fp16 against the matching weight rows ``state.subB`` (review
  thread "4. Mixed-precision decomposition matmul");
* the backward rebuilds fp16 weights as ``CB * (SCB / 127)`` with a multiply
  by the reciprocal, never stores them, and multiplies fp16 ``grad_output`` by
  them (PR description, backward bullet; review thread on ``.mul(1/127.0)``);
* ``grad_bias`` is summed from the uncast ``grad_output`` (PR conversation,
  "grad_bias is now computed on natural grad_output before it is cast").

The method is deterministic, so every stage is its definition written out:

* integer stages (fp16 cast, outlier set, row scales, int8 codes, weight codes,
  dequantized fp16 weights, the int32 accumulator) are exact targets;
* the dequantized output and the gradients are computed in float64 and rounded
  once to the storage dtype.

Floating point that decides an integer (a quantization code) is evaluated in
IEEE fp32, the precision the kernels use: ``s = 127 / absmax`` as one fp32
division, ``q = round_half_even(fp32(x) * s)`` as one fp32 multiply.

Readings of points the pages leave open (each is listed in the design notes):

* outlier rule: column ``k`` is an outlier when ``max_m |A16[m, k]| >
  threshold`` (strict), the whole column leaves the int8 product and the row
  scales; a threshold that is not a positive finite number disables the
  decomposition;
* the outlier indices are unique and ascending;
* an all-zero row (after removing outlier columns) has scale 0 and codes 0;
* ``subB`` is built from the dequantized int8 weight (the fp16 weight is not
  kept in memory-efficient mode), with the same formula as the backward;
* the weight is cast to fp16 before its quantization, like the activations;
* the bias is added at its own value (exactly widened), the output is rounded
  once to the input dtype.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(brute force on tiny inputs, closed forms, a lossless special case, the
IEEE-754 definitions of the casts).
"""
from __future__ import annotations

import math

import numpy as np

F16, BF16, F32 = "f16", "bf16", "f32"
DTYPES = (F16, BF16, F32)

# 127 * 127: the product of the two absmax-to-code factors.
_Q2 = 16129.0


# ---------------------------------------------------------------------------
# dtype handling.  Storage convention inside the oracle:
#   f16  -> numpy float16 array
#   bf16 -> numpy uint16 array holding the bf16 bit pattern
#   f32  -> numpy float32 array
# ---------------------------------------------------------------------------

def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored elements."""
    if dtype == F16:
        return np.asarray(x, dtype=np.float16).astype(np.float64)
    if dtype == BF16:
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        with np.errstate(invalid="ignore"):       # NaN patterns stay NaN
            return bits.view(np.float32).astype(np.float64)
    if dtype == F32:
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def _round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values once, to nearest-even, onto the bf16 grid.

    bf16 is IEEE binary32 with the significand cut to 8 bits: exponent range
    of fp32, normal spacing 2**(e-7) in [2**e, 2**(e+1)), subnormal spacing
    2**-133, largest finite (2 - 2**-7) * 2**127.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    ax = np.abs(x)
    # exponent of the binade: 2**e <= |x| < 2**(e+1); clamp to the subnormal step
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    # log2 can be off by one at binade edges: correct it exactly
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, -126.0)
    step = np.ldexp(1.0, (e - 7).astype(np.int64))
    q = np.rint(ax / step) * step          # ax/step is exact (power of 2 scale)
    # Past the largest finite value the nearest-even neighbour is 2**128,
    # which does not exist in the format: overflow to infinity.
    q = np.where(q >= 2.0 ** 128, np.inf, q)
    out[:] = np.where(finite, np.copysign(q, x), x)
    bits32 = out.astype(np.float32).view(np.uint32)   # exact: on the bf16 grid
    return (bits32 >> np.uint32(16)).astype(np.uint16)


def round_to(x64: np.ndarray, dtype: str) -> np.ndarray:
    """One round-to-nearest-even of float64 values into the storage dtype."""
    x64 = np.asarray(x64, dtype=np.float64)
    with np.errstate(over="ignore"):
        if dtype == F16:
            return x64.astype(np.float16)      # numpy: single IEEE RNE rounding
        if dtype == F32:
            return x64.astype(np.float32)      # single IEEE RNE rounding
    if dtype == BF16:
        return _round_to_bf16_bits(x64)
    raise ValueError(dtype)


def cast_f16(x: np.ndarray, dtype: str) -> np.ndarray:
    """Step a1: A16 = fp16_rn(A).  Exact widening, then one RNE rounding."""
    if dtype == F16:
        return np.asarray(x, dtype=np.float16).copy()
    with np.errstate(over="ignore"):              # overflow -> inf is the rule
        return widen(x, dtype).astype(np.float16)


# ---------------------------------------------------------------------------
# forward stages
# ---------------------------------------------------------------------------

def threshold_enabled(threshold: float) -> bool:
    """A threshold that is not a positive finite number turns the
    mixed-precision decomposition off (configs with threshold = inf)."""
    t = float(threshold)
    return math.isfinite(t) and t > 0.0


def column_absmax(A16: np.ndarray) -> np.ndarray:
    """The reduction of step a2: max over the rows of |A16[m, k]| per column
    (float64, exact: the values are fp16; 0 for no rows)."""
    colmax = np.zeros(A16.shape[1], dtype=np.float64)
    for r in range(0, A16.shape[0], 2048):          # row blocks: bounded memory
        colmax = np.maximum(colmax, np.abs(A16[r:r + 2048].astype(np.float64)).max(axis=0))
    return colmax


def outlier_columns_from_absmax(colmax: np.ndarray, threshold: float) -> np.ndarray:
    """The selection of step a2: ascending indices of the columns whose
    absolute maximum exceeds the threshold (taken as an fp32 value)."""
    if not threshold_enabled(threshold):
        return np.zeros(0, dtype=np.int32)
    thr = float(np.float32(threshold))
    return np.nonzero(np.asarray(colmax, dtype=np.float64) > thr)[0].astype(np.int32)


def outlier_columns(A16: np.ndarray, threshold: float) -> np.ndarray:
    """Step a2: ascending unique indices of the columns of A16 holding at least
    one element with |a| > threshold (the threshold taken as an fp32 value)."""
    if not threshold_enabled(threshold) or A16.shape[0] == 0:
        return np.zeros(0, dtype=np.int32)
    return outlier_columns_from_absmax(column_absmax(A16), threshold)


def quantize_rows(A16: np.ndarray, idx: np.ndarray):
    """Step a3: vector-wise (row-wise) absmax int8 quantization of A16 with
    the outlier columns ``idx`` removed.

    Returns (SCA fp32 [M], Aq int8 [M, K], subA fp16 [M, len(idx)]).
    """
    X = A16.astype(np.float32)
    subA = A16[:, idx].copy()
    X[:, idx] = 0.0
    SCA = np.abs(X).max(axis=1) if X.shape[1] else np.zeros(X.shape[0], np.float32)
    SCA = SCA.astype(np.float32)
    Aq = _codes(X, SCA)
    return SCA, Aq, subA


def _codes(X: np.ndarray, absmax: np.ndarray) -> np.ndarray:
    """q = round_half_even(x * (127 / absmax)) in IEEE fp32; absmax 0 -> 0."""
    X = X.astype(np.float32)
    am = absmax.astype(np.float32)
    nz = am > 0
    s = np.zeros_like(am)
    s[nz] = np.float32(127.0) / am[nz]              # one fp32 division per row
    P = X * s[:, None]                              # one fp32 multiply
    q = np.clip(np.rint(P), -127, 127)              # RNE; clip is a no-op
    q[~nz, :] = 0
    return q.astype(np.int8)


def quantize_weight(W: np.ndarray, dtype: str):
    """Step a10: W16 = fp16_rn(W); SCB[n] = max_k |W16[n, k]| (fp32);
    CB[n, k] = round_half_even(fp32(W16) * (127 / SCB[n]))."""
    W16 = cast_f16(W, dtype)
    X = W16.astype(np.float32)
    SCB = (np.abs(X).max(axis=1) if X.shape[1] else np.zeros(X.shape[0])).astype(np.float32)
    return _codes(X, SCB), SCB


def dequant_scale(SCB: np.ndarray) -> np.ndarray:
    """f[n] = SCB[n] * fp32(1/127), one fp32 multiply (multiply, not divide)."""
    return (SCB.astype(np.float32) * np.float32(1.0 / 127.0)).astype(np.float32)


def dequant_weight(CB: np.ndarray, SCB: np.ndarray) -> np.ndarray:
    """Step a9's operand: Wdq[n, k] = fp16_rn(fp32(CB[n, k]) * f[n]).

    Mirrors ``CB.to(fp16).mul_(SCB[:, None] * (1/127))``: the fp32 product is
    rounded to fp32 and then stored into the fp16 tensor."""
    f = dequant_scale(SCB)
    P = CB.astype(np.float32) * f[:, None]          # fp32 multiply, rounded
    return P.astype(np.float16)


def int_gemm(Aq: np.ndarray, CB: np.ndarray) -> np.ndarray:
    """Step a5: Cacc[m, n] = sum_k Aq[m, k] * CB[n, k], exact.

    Every partial sum is an integer below 2**53, so float64 BLAS (any order,
    with or without FMA) returns it exactly."""
    K = Aq.shape[1]
    if K * 127 * 127 >= 2 ** 53:
        raise ValueError("K too large for an exact float64 integer GEMM")
    C = Aq.astype(np.float64) @ CB.astype(np.float64).T
    Ci = C.astype(np.int64)
    if Ci.size and (np.abs(Ci).max() >= 2 ** 31):
        raise OverflowError("int32 accumulator overflow")
    return Ci.astype(np.int32)


def forward(A, dtype, CB, SCB, bias=None, bias_dtype=None, threshold=0.0,
            residual=None, col_absmax=None):
    """Steps a1-a7: the whole quantized forward.

    ``A`` [M, K] in ``dtype`` storage; ``CB`` int8 [N, K]; ``SCB`` fp32 [N];
    ``bias`` [N] in ``bias_dtype`` storage or None; ``residual`` [M, N] in
    ``dtype`` storage or None (added before the single rounding).
    ``col_absmax``: the column maxima of a larger batch that ``A`` is a row
    shard of (token-sharded forward: the outlier set is the whole batch's);
    None takes them over ``A``.

    out = round_to( Cacc * SCA * SCB / 127**2 + subA @ subB^T + bias + residual )
    """
    A16 = cast_f16(A, dtype)
    if col_absmax is None:
        idx = outlier_columns(A16, threshold)
    else:
        idx = outlier_columns_from_absmax(col_absmax, threshold)
    SCA, Aq, subA = quantize_rows(A16, idx)
    Wdq = dequant_weight(CB, SCB)
    subB = Wdq[:, idx]
    Cacc = int_gemm(Aq, CB)
    acc = Cacc.astype(np.float64) * (SCA.astype(np.float64)[:, None]
                                     * SCB.astype(np.float64)[None, :]) / _Q2
    if len(idx):
        acc = acc + subA.astype(np.float64) @ subB.astype(np.float64).T
    if bias is not None:
        acc = acc + widen(bias, bias_dtype)[None, :]
    if residual is not None:
        acc = acc + widen(residual, dtype)
    return dict(A16=A16, idx=idx, SCA=SCA, Aq=Aq, subA=subA, subB=subB,
                Cacc=Cacc, out64=acc, out=round_to(acc, dtype))


def forward_rows(A, dtype, CB, SCB, rows, bias=None, bias_dtype=None,
                 threshold=0.0, residual=None):
    """The forward on a subset of rows, with the outlier set taken over all
    rows of A (rows are independent once the column set is known)."""
    A16 = cast_f16(A, dtype)
    idx = outlier_columns(A16, threshold)
    A16r = A16[rows]
    SCA, Aq, subA = quantize_rows(A16r, idx)
    Wdq = dequant_weight(CB, SCB)
    subB = Wdq[:, idx]
    Cacc = int_gemm(Aq, CB)
    acc = Cacc.astype(np.float64) * (SCA.astype(np.float64)[:, None]
                                     * SCB.astype(np.float64)[None, :]) / _Q2
    if len(idx):
        acc = acc + subA.astype(np.float64) @ subB.astype(np.float64).T
    if bias is not None:
        acc = acc + widen(bias, bias_dtype)[None, :]
    if residual is not None:
        acc = acc + widen(residual, dtype)
    return dict(idx=idx, SCA=SCA, Aq=Aq, subA=subA, Cacc=Cacc, out64=acc,
                out=round_to(acc, dtype))


# ---------------------------------------------------------------------------
# backward stages
# ---------------------------------------------------------------------------

def grad_bias(G, dtype, bias_dtype):
    """Step a8: grad_bias[n] = sum_m G[m, n] of the uncast grad_output,
    in float64, rounded once to the bias dtype."""
    total = np.zeros(G.shape[1], dtype=np.float64)
    for r in range(0, G.shape[0], 2048):            # row blocks: bounded memory
        total += widen(G[r:r + 2048], dtype).sum(axis=0)
    return round_to(total, bias_dtype)


def backward_input(G, dtype, CB, SCB, addend=None, rows=None):
    """Step a9: grad_A = round_to(fp16(G) @ Wdq (+ addend)), float64 sums.

    ``G`` [M, N] in ``dtype`` storage (the layer's output dtype, which is the
    input's dtype); ``addend`` [M, K] in ``dtype`` storage or None (a
    gradient that arrives at the same tensor through another path)."""
    G16 = cast_f16(G if rows is None else G[rows], dtype)
    Wdq = dequant_weight(CB, SCB)
    acc = G16.astype(np.float64) @ Wdq.astype(np.float64)
    if addend is not None:
        acc = acc + widen(addend if rows is None else addend[rows], dtype)
    return dict(G16=G16, Wdq=Wdq, grad64=acc, grad_A=round_to(acc, dtype))


def quantize_cols(X16: np.ndarray):
    """Column-wise (vector-wise along the tokens) absmax int8 quantization of
    a token-major matrix X16 [M, C] (fp16 values): SC[c] = max_m |X16[m, c]|
    (fp32), Xt[c, m] = round_half_even(fp32(X16[m, c]) * (127 / SC[c])),
    returned transposed (C x M), the layout whose rows the weight-gradient
    product contracts.  It is the row-wise quantization of the transpose."""
    Xt = np.ascontiguousarray(X16.T).astype(np.float32)
    SC = (np.abs(Xt).max(axis=1) if Xt.shape[1] else np.zeros(Xt.shape[0])).astype(np.float32)
    return SC, _codes(Xt, SC)


def grad_weight(G, A, dtype):
    """Weight gradient of the trainable-weight mode (has_fp16_weights=True):
    grad_W[n, k] = sum_m G[m, n] A[m, k] with both operands quantized column
    by column (scales per output feature n and per input feature k, taken
    over the tokens), an exact int32 product of the codes, and the dequant
    SCG[n] * SCA[k] / 127^2 in float64, rounded once to ``dtype``.

    ``G`` [M, N] and ``A`` [M, K] in ``dtype`` storage; both are cast to fp16
    first, like every quantized operand of the layer."""
    G16 = cast_f16(G, dtype)
    A16 = cast_f16(A, dtype)
    SCG, Gt = quantize_cols(G16)
    SCA, At = quantize_cols(A16)
    Cacc = int_gemm(Gt, At)
    acc = Cacc.astype(np.float64) * (SCG.astype(np.float64)[:, None] * SCA.astype(np.float64)[None, :]) / _Q2
    return dict(SCG=SCG, Gt=Gt, SCA=SCA, At=At, Cacc=Cacc, grad64=acc, grad_W=round_to(acc, dtype))


# ---------------------------------------------------------------------------
# SiLU between the two layers of the MLP workloads (float64, one rounding)
# ---------------------------------------------------------------------------

def silu(h, dtype):
    x = widen(h, dtype)
    return round_to(x / (1.0 + np.exp(-x)), dtype)


def silu_backward(g, h, dtype):
    x = widen(h, dtype)
    s = 1.0 / (1.0 + np.exp(-x))
    return round_to(widen(g, dtype) * s * (1.0 + x * (1.0 - s)), dtype)
