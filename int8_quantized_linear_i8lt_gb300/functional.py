"""Torch-facing calls of the int8 quantized linear layer.

PyTorch supplies device memory (the caching allocator), the current stream
and autograd; every arithmetic step runs in libi8lt's CUDA kernels.  The
calls fail loudly when the library is missing or the device is not sm_103.

Method: the memory-efficient Linear8bitLt of bitsandbytes PR #33 "Memory
efficient backward" (see include/i8lt.h for the formulas).
"""
from __future__ import annotations

import math
import warnings

import torch

from . import _lib

DTYPE_CODE = {torch.float16: _lib.I8LT_F16, torch.bfloat16: _lib.I8LT_BF16, torch.float32: _lib.I8LT_F32}


class I8LTError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != _lib.I8LT_OK:
        raise I8LTError(f"{what}: {_lib.i8lt_status_string(status)} (status {status})")


def _code(dtype: torch.dtype) -> int:
    try:
        return DTYPE_CODE[dtype]
    except KeyError:
        raise I8LTError(f"unsupported dtype {dtype}") from None


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise I8LTError("libi8lt runs on CUDA tensors only (no CPU path)")


def default_max_outliers(K: int) -> int:
    """Capacity for outlier columns: all K columns, so the capacity can never
    be exceeded (the input of a second MLP layer can hold thousands of
    sporadic outlier columns).  Pass a smaller ``max_outliers`` to shrink the
    workspace (subA and subB are M x cap and N x cap fp16)."""
    return K


def weight_ld(K: int) -> int:
    return _lib.i8lt_weight_ld(K)


def quantize_weight(W: torch.Tensor):
    """W [N, K] (f16 / bf16 / f32, CUDA) -> (CB int8 [N, ld], SCB fp32 [N])."""
    _require_cuda(W)
    W = W.contiguous()
    N, K = W.shape
    CB = torch.empty(N, weight_ld(K), dtype=torch.int8, device=W.device)
    SCB = torch.empty(N, dtype=torch.float32, device=W.device)
    _check(_lib.i8lt_quantize_weight(W.data_ptr(), _code(W.dtype), N, K, CB.data_ptr(), SCB.data_ptr(),
                                     _stream(W)), "i8lt_quantize_weight")
    return CB, SCB


def forward_workspace(M: int, K: int, N: int, max_outliers: int, device) -> torch.Tensor:
    n = _lib.i8lt_forward_workspace_size(M, K, N, max_outliers)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def backward_workspace(M: int, N: int, dtype: torch.dtype, device, K: int | None = None) -> torch.Tensor:
    """Workspace of i8lt_backward_input.  Without ``K``: the fused schedule
    (the fp16 weight is rebuilt tile by tile inside the GEMM, no N x K
    buffer).  With ``K`` it has room for the materialized dequantized weight
    (K_pad x N_pad fp16), which selects the materialized schedule."""
    if K is None:
        n = _lib.i8lt_backward_workspace_size(M, N, _code(dtype))
    else:
        n = _lib.i8lt_backward_workspace_size_dq(M, N, K, _code(dtype))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def forward(A: torch.Tensor, CB: torch.Tensor, SCB: torch.Tensor, K: int, bias: torch.Tensor | None = None,
            threshold: float = 6.0, residual: torch.Tensor | None = None, max_outliers: int | None = None,
            out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
            acc_i32: torch.Tensor | None = None, merge_colmax=None, colmax_ready: bool = False):
    """out [M, N] = int8 linear of A [M, K] (see i8lt_forward).  Returns
    (out, ws); ``ws`` holds the quantized activations and the outlier set.

    ``merge_colmax``: for a token-sharded batch, a callable that receives the
    K column maxima of this call's rows (an int32 view into ``ws``, ordered
    like the magnitudes) and replaces them in place with the maxima over
    all shards, e.g. an all-reduce MAX; the outlier set is then the whole
    batch's (i8lt_forward_colmax / i8lt_forward_from_colmax).
    ``colmax_ready``: the column maxima of A are already in ``ws`` (written
    by the previous layer's forward_silu); only the rest of the forward runs."""
    _require_cuda(A, CB, SCB, bias, residual)
    A = A.contiguous()
    M = A.shape[0]
    if A.shape[1] != K:
        raise I8LTError(f"A has {A.shape[1]} features, the weight {K}")
    N = CB.shape[0]
    cap = _capacity(K, threshold, max_outliers)
    if out is None:
        out = torch.empty(M, N, dtype=A.dtype, device=A.device)
    if ws is None:
        if colmax_ready:
            raise I8LTError("colmax_ready needs the workspace that holds the column maxima")
        ws = forward_workspace(M, K, N, cap, A.device)
    if residual is not None:
        residual = residual.contiguous()
    bias_c = None if bias is None else bias.contiguous()
    args = (_ptr(bias_c), _code(bias_c.dtype) if bias_c is not None else 0, float(threshold),
            _ptr(residual), out.data_ptr(), ws.data_ptr(), ws.numel(), cap)
    if merge_colmax is None and not colmax_ready:
        _check(_lib.i8lt_forward(A.data_ptr(), _code(A.dtype), M, K, CB.data_ptr(), SCB.data_ptr(), N, *args,
                                 acc_i32=_ptr(acc_i32), stream=_stream(A)), "i8lt_forward")
        return out, ws
    if not colmax_ready:
        _check(_lib.i8lt_forward_colmax(A.data_ptr(), _code(A.dtype), M, K, N, ws.data_ptr(), ws.numel(), cap,
                                        stream=_stream(A)), "i8lt_forward_colmax")
    if merge_colmax is not None:
        lay = _lib.i8lt_forward_workspace_layout(M, K, N, cap)
        merge_colmax(ws[lay.colmax:lay.colmax + 4 * K].view(torch.int32))
    _check(_lib.i8lt_forward_from_colmax(A.data_ptr(), _code(A.dtype), M, K, CB.data_ptr(), SCB.data_ptr(), N,
                                         *args, acc_i32=_ptr(acc_i32), stream=_stream(A)),
           "i8lt_forward_from_colmax")
    return out, ws


def _capacity(K: int, threshold: float, max_outliers: int | None) -> int:
    if not (math.isfinite(threshold) and threshold > 0):
        return 0
    return default_max_outliers(K) if max_outliers is None else int(max_outliers)


def colmax_region(ws: torch.Tensor, M: int, K: int, N: int, threshold: float,
                  max_outliers: int | None = None) -> torch.Tensor:
    """The K column maxima of a forward workspace (int32 view)."""
    lay = _lib.i8lt_forward_workspace_layout(M, K, N, _capacity(K, threshold, max_outliers))
    return ws[lay.colmax:lay.colmax + 4 * K].view(torch.int32)


def forward_silu(A: torch.Tensor, CB: torch.Tensor, SCB: torch.Tensor, K: int, bias: torch.Tensor | None = None,
                 threshold: float = 6.0, max_outliers: int | None = None, act_colmax: torch.Tensor | None = None):
    """MLP hidden layer (i8lt_forward_silu): returns (h, silu(h), ws).
    ``act_colmax`` (int32 [N], e.g. ``colmax_region`` of the next layer's
    workspace) receives the column maxima of |fp16(silu(h))|."""
    _require_cuda(A, CB, SCB, bias)
    A = A.contiguous()
    M = A.shape[0]
    if A.shape[1] != K:
        raise I8LTError(f"A has {A.shape[1]} features, the weight {K}")
    N = CB.shape[0]
    cap = _capacity(K, threshold, max_outliers)
    h = torch.empty(M, N, dtype=A.dtype, device=A.device)
    a = torch.empty_like(h)
    if act_colmax is None:
        act_colmax = torch.empty(N, dtype=torch.int32, device=A.device)
    ws = forward_workspace(M, K, N, cap, A.device)
    bias_c = None if bias is None else bias.contiguous()
    _check(_lib.i8lt_forward_silu(A.data_ptr(), _code(A.dtype), M, K, CB.data_ptr(), SCB.data_ptr(), N,
                                  _ptr(bias_c), _code(bias_c.dtype) if bias_c is not None else 0, float(threshold),
                                  None, h.data_ptr(), a.data_ptr(), act_colmax.data_ptr(), ws.data_ptr(), ws.numel(),
                                  cap, stream=_stream(A)), "i8lt_forward_silu")
    return h, a, ws


def allreduce_colmax(group=None):
    """``merge_colmax`` for torch.distributed: an all-reduce MAX of the column
    maxima over ``group`` (one K-sized int32 exchange per forward)."""
    import torch.distributed as dist

    def merge(t: torch.Tensor):
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return merge


def backward_input(G: torch.Tensor, CB: torch.Tensor, SCB: torch.Tensor, K: int, need_grad_A: bool = True,
                   bias_dtype: torch.dtype | None = None, addend: torch.Tensor | None = None,
                   ws: torch.Tensor | None = None, fused: bool = True):
    """(grad_A [M, K] or None, grad_bias [N] or None) from grad_output G [M, N].
    ``fused`` (default): the dequantized weight is rebuilt tile by tile inside
    the GEMM and never stored.  ``fused=False``: it is first written to the
    workspace (K x N fp16) by a memory-bound prepass, then read by a plain
    fp16 GEMM -- more memory, a little faster.  A caller-supplied ``ws``
    decides by its size instead.  Both give the same bits."""
    _require_cuda(G, CB, SCB, addend)
    G = G.contiguous()
    M, N = G.shape
    grad_A = torch.empty(M, K, dtype=G.dtype, device=G.device) if need_grad_A else None
    grad_bias = torch.empty(N, dtype=bias_dtype, device=G.device) if bias_dtype is not None else None
    if ws is None:
        ws = backward_workspace(M, N, G.dtype, G.device, K=None if (fused or not need_grad_A) else K)
    if addend is not None:
        addend = addend.contiguous()
    _check(_lib.i8lt_backward_input(G.data_ptr(), _code(G.dtype), M, N, CB.data_ptr(), SCB.data_ptr(), K,
                                    _ptr(addend), _ptr(grad_A), _ptr(grad_bias),
                                    _code(bias_dtype) if bias_dtype is not None else 0,
                                    ws.data_ptr(), ws.numel(), _stream(G)), "i8lt_backward_input")
    return grad_A, grad_bias


def silu(h: torch.Tensor) -> torch.Tensor:
    _require_cuda(h)
    h = h.contiguous()
    out = torch.empty_like(h)
    _check(_lib.i8lt_silu_forward(h.data_ptr(), _code(h.dtype), h.numel(), out.data_ptr(), _stream(h)),
           "i8lt_silu_forward")
    return out


def silu_backward(g: torch.Tensor, h: torch.Tensor) -> torch.Tensor:
    _require_cuda(g, h)
    g, h = g.contiguous(), h.contiguous()
    out = torch.empty_like(h)
    _check(_lib.i8lt_silu_backward(g.data_ptr(), h.data_ptr(), _code(h.dtype), h.numel(), out.data_ptr(),
                                   _stream(h)), "i8lt_silu_backward")
    return out


def device_status(ws: torch.Tensor):
    """(status code, outlier columns found) of the last call that used ``ws``
    (synchronizes the current stream; clears a recorded error)."""
    r, st, found = _lib.i8lt_read_device_status(ws.data_ptr(), _stream(ws))
    return st, found


# ---------------------------------------------------------------------------
# autograd
# ---------------------------------------------------------------------------

_warned_cast = False


def _warn_cast(dtype):
    global _warned_cast
    if dtype != torch.float16 and not _warned_cast:
        _warned_cast = True
        warnings.warn(f"Linear8bitLt: input of dtype {dtype} is cast to float16 for the int8 "
                      "quantization; the output is cast back to the input's dtype.")


class Int8LinearFunction(torch.autograd.Function):
    """y = int8 linear(x); the weight is frozen (memory-efficient backward:
    grad to the input and the bias only)."""

    @staticmethod
    def forward(ctx, x, CB, SCB, bias, threshold, max_outliers):
        _warn_cast(x.dtype)
        shape = x.shape
        K = shape[-1]
        x2 = x.reshape(-1, K)
        out, _ = forward(x2, CB, SCB, K, bias, threshold, max_outliers=max_outliers)
        ctx.save_for_backward(CB, SCB)
        ctx.K = K
        ctx.x_shape = shape
        ctx.bias_dtype = None if bias is None else bias.dtype
        return out.reshape(*shape[:-1], CB.shape[0])

    @staticmethod
    def backward(ctx, grad_out):
        CB, SCB = ctx.saved_tensors
        need_x = ctx.needs_input_grad[0]
        need_b = ctx.needs_input_grad[3] and ctx.bias_dtype is not None
        G = grad_out.reshape(-1, grad_out.shape[-1])
        gA, gb = backward_input(G, CB, SCB, ctx.K, need_grad_A=need_x,
                                bias_dtype=ctx.bias_dtype if need_b else None)
        if gA is not None:
            gA = gA.reshape(ctx.x_shape)
        return gA, None, None, gb, None, None


def grad_weight(G: torch.Tensor, A: torch.Tensor, out_dtype: torch.dtype | None = None,
                ws: torch.Tensor | None = None) -> torch.Tensor:
    """grad_W [N, K] = G^T A over the tokens, int8 with column-wise scales
    (i8lt_grad_weight); G [M, N], A [M, K]."""
    _require_cuda(G, A)
    G, A = G.contiguous(), A.contiguous()
    M, N = G.shape
    K = A.shape[1]
    if A.shape[0] != M:
        raise I8LTError(f"G has {M} tokens, A {A.shape[0]}")
    out_dtype = out_dtype or G.dtype
    gW = torch.empty(N, K, dtype=out_dtype, device=G.device)
    if ws is None:
        ws = torch.empty(max(_lib.i8lt_grad_weight_workspace_size(M, N, K), 256), dtype=torch.uint8,
                         device=G.device)
    _check(_lib.i8lt_grad_weight(G.data_ptr(), _code(G.dtype), A.data_ptr(), _code(A.dtype), M, N, K, gW.data_ptr(),
                                 _code(out_dtype), ws.data_ptr(), ws.numel(), _stream(G)), "i8lt_grad_weight")
    return gW


class Int8LinearTrainableFunction(torch.autograd.Function):
    """y = int8 linear(x) with a trainable float weight W (bitsandbytes'
    has_fp16_weights=True): every forward quantizes W row-wise (CB, SCB) and
    runs the same int8 forward; the backward gives grad_A through the
    dequantized CB (as the memory-efficient mode does), grad_W through the
    int8 column-wise product (i8lt_grad_weight) and grad_bias."""

    @staticmethod
    def forward(ctx, x, W, bias, threshold, max_outliers):
        _warn_cast(x.dtype)
        shape = x.shape
        K = shape[-1]
        x2 = x.reshape(-1, K)
        CB, SCB = quantize_weight(W)
        out, _ = forward(x2, CB, SCB, K, bias, threshold, max_outliers=max_outliers)
        ctx.save_for_backward(x2, CB, SCB)
        ctx.K = K
        ctx.x_shape = shape
        ctx.w_dtype = W.dtype
        ctx.bias_dtype = None if bias is None else bias.dtype
        return out.reshape(*shape[:-1], CB.shape[0])

    @staticmethod
    def backward(ctx, grad_out):
        x2, CB, SCB = ctx.saved_tensors
        need_x = ctx.needs_input_grad[0]
        need_w = ctx.needs_input_grad[1]
        need_b = ctx.needs_input_grad[2] and ctx.bias_dtype is not None
        G = grad_out.reshape(-1, grad_out.shape[-1])
        gA, gb = backward_input(G, CB, SCB, ctx.K, need_grad_A=need_x,
                                bias_dtype=ctx.bias_dtype if need_b else None)
        gW = grad_weight(G, x2, ctx.w_dtype) if need_w else None
        if gA is not None:
            gA = gA.reshape(ctx.x_shape)
        return gA, gW, gb, None, None


class SiLUFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, h):
        ctx.save_for_backward(h)
        return silu(h)

    @staticmethod
    def backward(ctx, g):
        (h,) = ctx.saved_tensors
        return silu_backward(g, h)


# MLP hidden layer: run the SiLU and fc2's column maxima inside fc1's GEMM
# epilogue (i8lt_forward_silu) instead of as separate passes.  Same bits
# either way.  Off by default: on GB300 the longer epilogue delays the
# GEMM's next tile about as much as the two memory-bound passes it saves
# cost (mlp_7b fc1 alone: 0.765 ms fused against 0.714 ms + 0.03 ms; the
# whole block forward + backward: 2.857 ms against 2.866 ms).
FUSED_SILU = False


class Int8MLPFunction(torch.autograd.Function):
    """y = fc2(silu(fc1(x))) (+ x): the two int8 layers, the SiLU and the
    residual add (fused into fc2's epilogue forward, and into fc1's backward
    as an addend) all in libi8lt kernels."""

    @staticmethod
    def forward(ctx, x, CB1, SCB1, b1, CB2, SCB2, b2, threshold, residual, max_outliers):
        _warn_cast(x.dtype)
        shape = x.shape
        K = shape[-1]
        x2 = x.reshape(-1, K)
        H, N2 = CB1.shape[0], CB2.shape[0]
        M = x2.shape[0]
        res = x2 if residual else None
        if FUSED_SILU:
            # fc1's epilogue applies the SiLU and writes fc2's column maxima
            # into fc2's workspace, so fc2 starts at its outlier index
            ws2 = forward_workspace(M, H, N2, _capacity(H, threshold, max_outliers), x.device)
            h, a, _ = forward_silu(x2, CB1, SCB1, K, b1, threshold, max_outliers=max_outliers,
                                   act_colmax=colmax_region(ws2, M, H, N2, threshold, max_outliers))
            y, _ = forward(a, CB2, SCB2, H, b2, threshold, residual=res, max_outliers=max_outliers, ws=ws2,
                           colmax_ready=True)
        else:
            h, _ = forward(x2, CB1, SCB1, K, b1, threshold, max_outliers=max_outliers)
            a = silu(h)
            y, _ = forward(a, CB2, SCB2, H, b2, threshold, residual=res, max_outliers=max_outliers)
        ctx.save_for_backward(CB1, SCB1, CB2, SCB2, h)
        ctx.K = K
        ctx.H = CB1.shape[0]
        ctx.shape = shape
        ctx.residual = residual
        ctx.b1_dtype = None if b1 is None else b1.dtype
        ctx.b2_dtype = None if b2 is None else b2.dtype
        return y.reshape(*shape[:-1], CB2.shape[0])

    @staticmethod
    def backward(ctx, g):
        CB1, SCB1, CB2, SCB2, h = ctx.saved_tensors
        G = g.reshape(-1, g.shape[-1])
        ga, gb2 = backward_input(G, CB2, SCB2, ctx.H, bias_dtype=ctx.b2_dtype if ctx.needs_input_grad[6] else None)
        gh = silu_backward(ga, h)
        gx, gb1 = backward_input(gh, CB1, SCB1, ctx.K, addend=G if ctx.residual else None,
                                 bias_dtype=ctx.b1_dtype if ctx.needs_input_grad[3] else None)
        return gx.reshape(ctx.shape), None, None, gb1, None, None, gb2, None, None, None


# ---------------------------------------------------------------------------
# 4-bit weight-only layers (QLoRA fine-tuning: frozen 4-bit base weights,
# 16-bit compute; NF4 and FP4 share one storage and one set of matmul
# kernels, see i8lt_nf4_forward / i8lt_fp4_forward in include/i8lt.h)
# ---------------------------------------------------------------------------

FORMATS_4BIT = ("nf4", "fp4")


def _fmt4(fmt: str) -> str:
    if fmt not in FORMATS_4BIT:
        raise I8LTError(f"unknown 4-bit format {fmt!r} (expected one of {FORMATS_4BIT})")
    return fmt


def _fn4(fmt: str, name: str):
    return getattr(_lib, f"i8lt_{_fmt4(fmt)}_{name}")


def levels_4bit(fmt: str = "nf4") -> list[float]:
    """The 16 levels of a 4-bit format, by code."""
    st, lv = _fn4(fmt, "levels")()
    _check(st, f"i8lt_{fmt}_levels")
    return lv


def nf4_levels() -> list[float]:
    return levels_4bit("nf4")


def fp4_levels() -> list[float]:
    return levels_4bit("fp4")


def quantize_4bit(W: torch.Tensor, fmt: str = "nf4"):
    """W [N, K] (f16 / bf16 / f32, CUDA) -> (packed uint8 [N, row_bytes],
    absmax fp32 [N, ceil(K / 64)]) in the 4-bit format ``fmt``."""
    _require_cuda(W)
    W = W.contiguous()
    N, K = W.shape
    packed = torch.empty(N, _lib.i8lt_nf4_row_bytes(K), dtype=torch.uint8, device=W.device)
    absmax = torch.empty(N, _lib.i8lt_nf4_blocks(K), dtype=torch.float32, device=W.device)
    _check(_fn4(fmt, "quantize")(W.data_ptr(), _code(W.dtype), N, K, packed.data_ptr(), absmax.data_ptr(),
                                 _stream(W)), f"i8lt_{fmt}_quantize")
    return packed, absmax


def nf4_quantize(W: torch.Tensor):
    return quantize_4bit(W, "nf4")


def fp4_quantize(W: torch.Tensor):
    return quantize_4bit(W, "fp4")


def dequantize_4bit(packed: torch.Tensor, absmax: torch.Tensor, K: int, dtype: torch.dtype,
                    fmt: str = "nf4") -> torch.Tensor:
    """The dequantized weight [N, K] in ``dtype``."""
    _require_cuda(packed, absmax)
    N = packed.shape[0]
    out = torch.empty(N, K, dtype=dtype, device=packed.device)
    _check(_fn4(fmt, "dequantize")(packed.data_ptr(), absmax.data_ptr(), N, K, out.data_ptr(), _code(dtype),
                                   _stream(packed)), f"i8lt_{fmt}_dequantize")
    return out


def nf4_dequantize(packed: torch.Tensor, absmax: torch.Tensor, K: int, dtype: torch.dtype) -> torch.Tensor:
    return dequantize_4bit(packed, absmax, K, dtype, "nf4")


def fp4_dequantize(packed: torch.Tensor, absmax: torch.Tensor, K: int, dtype: torch.dtype) -> torch.Tensor:
    return dequantize_4bit(packed, absmax, K, dtype, "fp4")


def double_quantize_absmax(absmax: torch.Tensor):
    """The 8-bit storage of a 4-bit weight's absmax values (the ``-dq``
    options): (q uint8 with absmax's shape, absmax2 fp32 [ceil(n / 256)],
    offset fp32 [1]) -- FP8 E4M3 codes of absmax - offset in blocks of 256
    with one fp32 scale each, offset the mean of all the values."""
    _require_cuda(absmax)
    a = absmax.contiguous()
    n = a.numel()
    q = torch.empty(a.shape, dtype=torch.uint8, device=a.device)
    a2 = torch.empty(_lib.i8lt_absmax8_blocks(n), dtype=torch.float32, device=a.device)
    off = torch.empty(1, dtype=torch.float32, device=a.device)
    ws = torch.empty(_lib.i8lt_absmax8_workspace_size(), dtype=torch.uint8, device=a.device)
    _check(_lib.i8lt_absmax8_quantize(a.data_ptr(), n, q.data_ptr(), a2.data_ptr(), off.data_ptr(), ws.data_ptr(),
                                      ws.numel(), _stream(a)), "i8lt_absmax8_quantize")
    return q, a2, off


def dequantize_absmax(q: torch.Tensor, absmax2: torch.Tensor, offset: torch.Tensor,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    """The fp32 absmax values decoded from double_quantize_absmax's storage."""
    _require_cuda(q, absmax2, offset)
    q = q.contiguous()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    _check(_lib.i8lt_absmax8_dequantize(q.data_ptr(), absmax2.data_ptr(), offset.data_ptr(), q.numel(),
                                        out.data_ptr(), _stream(q)), "i8lt_absmax8_dequantize")
    return out


def _nf4_ws(device, ws, K, N, materialized, extra=0):
    """Workspace of the 4-bit matmuls: the status word (and ``extra`` bytes
    of grad_bias partial sums), the weight then decoded inside the GEMM; or
    room for the dequantized weight after them (``materialized``: a prepass
    writes it, a plain 16-bit GEMM reads it; same bits, faster, N * K * 2
    bytes more)."""
    if ws is None:
        n = _lib.i8lt_nf4_workspace_size_dq(K, N) if materialized else _lib.i8lt_nf4_workspace_size()
        ws = torch.empty(n + extra, dtype=torch.uint8, device=device)
    return ws


def forward_4bit(A: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor, K: int,
                 bias: torch.Tensor | None = None, out: torch.Tensor | None = None,
                 ws: torch.Tensor | None = None, materialized: bool = False, fmt: str = "nf4") -> torch.Tensor:
    """out [M, N] = A [M, K] @ Wdq^T (+ bias) in A's dtype (f16 or bf16)."""
    _require_cuda(A, packed, absmax, bias)
    A = A.contiguous()
    M = A.shape[0]
    N = packed.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=A.dtype, device=A.device)
    ws = _nf4_ws(A.device, ws, K, N, materialized)
    _check(_fn4(fmt, "forward")(A.data_ptr(), _code(A.dtype), M, K, packed.data_ptr(), absmax.data_ptr(), N,
                                _ptr(bias), _code(bias.dtype) if bias is not None else 0, out.data_ptr(),
                                ws.data_ptr(), ws.numel(), _stream(A)), f"i8lt_{fmt}_forward")
    return out


def nf4_forward(A, packed, absmax, K, bias=None, out=None, ws=None, materialized=False) -> torch.Tensor:
    return forward_4bit(A, packed, absmax, K, bias, out, ws, materialized, "nf4")


def fp4_forward(A, packed, absmax, K, bias=None, out=None, ws=None, materialized=False) -> torch.Tensor:
    return forward_4bit(A, packed, absmax, K, bias, out, ws, materialized, "fp4")


def backward_input_4bit(G: torch.Tensor, packed: torch.Tensor, absmax: torch.Tensor, K: int,
                        need_grad_A: bool = True, bias_dtype: torch.dtype | None = None,
                        out: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                        materialized: bool = False, fmt: str = "nf4"):
    """(grad_A [M, K] = G [M, N] @ Wdq in G's dtype (f16 or bf16) or None,
    grad_bias [N] in ``bias_dtype`` or None).  grad_bias is reduced inside
    the GEMM (or by a pass of its own when grad_A is not needed)."""
    _require_cuda(G, packed, absmax)
    G = G.contiguous()
    M, N = G.shape
    if need_grad_A and out is None:
        out = torch.empty(M, K, dtype=G.dtype, device=G.device)
    gb = torch.empty(N, dtype=bias_dtype, device=G.device) if bias_dtype is not None else None
    extra = _lib.i8lt_nf4_grad_bias_bytes(M, N) if gb is not None else 0
    ws = _nf4_ws(G.device, ws, K, N, materialized, extra)
    _check(_fn4(fmt, "backward_input")(G.data_ptr(), _code(G.dtype), M, N, packed.data_ptr(), absmax.data_ptr(), K,
                                       _ptr(out) if need_grad_A else None, _ptr(gb),
                                       _code(bias_dtype) if bias_dtype is not None else 0, ws.data_ptr(), ws.numel(),
                                       _stream(G)), f"i8lt_{fmt}_backward_input")
    return (out if need_grad_A else None), gb


def nf4_backward_input(G, packed, absmax, K, out=None, ws=None, materialized=False) -> torch.Tensor:
    """grad_A [M, K] = G [M, N] @ Wdq in G's dtype (f16 or bf16)."""
    return backward_input_4bit(G, packed, absmax, K, out=out, ws=ws, materialized=materialized, fmt="nf4")[0]


def fp4_backward_input(G, packed, absmax, K, out=None, ws=None, materialized=False) -> torch.Tensor:
    return backward_input_4bit(G, packed, absmax, K, out=out, ws=ws, materialized=materialized, fmt="fp4")[0]


class Linear4bitFunction(torch.autograd.Function):
    """y = x @ Wdq^T + bias with the frozen 4-bit weight (format ``fmt``)
    decoded inside the matmuls; gradients to x and to the bias (summed over
    the tokens inside the input-gradient GEMM)."""

    @staticmethod
    def forward(ctx, x, packed, absmax, K, bias, materialized=False, fmt="nf4"):
        shape = x.shape
        x2 = x.reshape(-1, K)
        y = forward_4bit(x2, packed, absmax, K, bias, materialized=materialized, fmt=fmt)
        ctx.save_for_backward(packed, absmax)
        ctx.K, ctx.shape, ctx.materialized, ctx.fmt = K, shape, materialized, fmt
        ctx.bias_dtype = bias.dtype if bias is not None else None
        return y.reshape(*shape[:-1], packed.shape[0])

    @staticmethod
    def backward(ctx, gy):
        packed, absmax = ctx.saved_tensors
        g2 = gy.reshape(-1, packed.shape[0])
        need_x = ctx.needs_input_grad[0]
        need_b = ctx.bias_dtype is not None and ctx.needs_input_grad[4]
        if not (need_x or need_b):
            return None, None, None, None, None, None, None
        gx, gb = backward_input_4bit(g2, packed, absmax, ctx.K, need_grad_A=need_x,
                                     bias_dtype=ctx.bias_dtype if need_b else None,
                                     materialized=ctx.materialized, fmt=ctx.fmt)
        if gx is not None:
            gx = gx.reshape(ctx.shape)
        return gx, None, None, None, gb, None, None


# the NF4 layer's function under its own name
NF4LinearFunction = Linear4bitFunction
