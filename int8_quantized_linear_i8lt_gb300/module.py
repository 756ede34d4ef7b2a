"""nn.Module front ends: Linear8bitLt and the two-layer SiLU MLP.

The int8 weight is never drawn at random (``normal_`` has no int8 kernel, as
the lit-gpt QLoRA PR notes for bnb.int8 training): a layer is built from a
float weight with ``from_float``, or loaded with its CB / SCB buffers.
"""
from __future__ import annotations

import torch

from . import functional as F


class Linear8bitLt(torch.nn.Module):
    """Memory-efficient int8 linear layer (bitsandbytes PR #33): int8
    row-major weight CB with per-row scales SCB, fp16 outlier decomposition
    above ``threshold``, input cast to fp16 and output cast back, backward
    to the input through fp16 weights rebuilt on the fly.  The weight takes
    no gradient; the bias does."""

    def __init__(self, in_features: int, out_features: int, bias: bool = True, threshold: float = 6.0,
                 device=None, bias_dtype: torch.dtype = torch.float16, max_outliers: int | None = None):
        super().__init__()
        self.in_features = in_features
        self.out_features = out_features
        self.threshold = float(threshold)
        self.max_outliers = max_outliers
        ld = F.weight_ld(in_features)
        self.register_buffer("CB", torch.zeros(out_features, ld, dtype=torch.int8, device=device))
        self.register_buffer("SCB", torch.zeros(out_features, dtype=torch.float32, device=device))
        if bias:
            self.bias = torch.nn.Parameter(torch.zeros(out_features, dtype=bias_dtype, device=device))
        else:
            self.register_parameter("bias", None)

    @classmethod
    def from_float(cls, weight: torch.Tensor, bias: torch.Tensor | None = None, threshold: float = 6.0,
                   max_outliers: int | None = None) -> "Linear8bitLt":
        """Quantize a float weight [out, in] on its CUDA device."""
        N, K = weight.shape
        layer = cls(K, N, bias=bias is not None, threshold=threshold, device=weight.device,
                    bias_dtype=bias.dtype if bias is not None else torch.float16, max_outliers=max_outliers)
        CB, SCB = F.quantize_weight(weight)
        layer.CB.copy_(CB)
        layer.SCB.copy_(SCB)
        if bias is not None:
            with torch.no_grad():
                layer.bias.copy_(bias)
        return layer

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return F.Int8LinearFunction.apply(x, self.CB, self.SCB, self.bias, self.threshold, self.max_outliers)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, threshold={self.threshold}")


class Linear8bitLtTrainable(torch.nn.Module):
    """The trainable-weight mode of the same layer (bitsandbytes'
    has_fp16_weights=True): the float weight is a parameter, quantized afresh
    on every forward; its gradient comes from the int8 column-wise product
    G^T A (i8lt_grad_weight)."""

    def __init__(self, in_features: int, out_features: int, bias: bool = True, threshold: float = 6.0,
                 device=None, dtype: torch.dtype = torch.float16, max_outliers: int | None = None):
        super().__init__()
        self.in_features = in_features
        self.out_features = out_features
        self.threshold = float(threshold)
        self.max_outliers = max_outliers
        self.weight = torch.nn.Parameter(torch.empty(out_features, in_features, dtype=dtype, device=device))
        torch.nn.init.kaiming_uniform_(self.weight, a=5 ** 0.5)
        if bias:
            self.bias = torch.nn.Parameter(torch.zeros(out_features, dtype=dtype, device=device))
        else:
            self.register_parameter("bias", None)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return F.Int8LinearTrainableFunction.apply(x, self.weight, self.bias, self.threshold, self.max_outliers)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, threshold={self.threshold}, trainable weight")


class Int8MLP(torch.nn.Module):
    """y = fc2(silu(fc1(x))) (+ x when ``residual``), both layers int8."""

    def __init__(self, fc1: Linear8bitLt, fc2: Linear8bitLt, residual: bool = False):
        super().__init__()
        self.fc1, self.fc2, self.residual = fc1, fc2, residual

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return F.Int8MLPFunction.apply(x, self.fc1.CB, self.fc1.SCB, self.fc1.bias, self.fc2.CB, self.fc2.SCB,
                                       self.fc2.bias, self.fc1.threshold, self.residual, self.fc1.max_outliers)


class Linear4bit(torch.nn.Module):
    """Frozen 4-bit linear layer of QLoRA fine-tuning: the weight is stored
    as packed 4-bit codes (``fmt``: "nf4", 4-bit NormalFloat, or "fp4", the
    E2M1 floating-point format) with one fp32 absmax per 64 elements of a row
    and decoded to the 16-bit compute dtype (the input's: f16 or bf16) inside
    the tensor-core matmuls of the forward and of the input gradient.  The
    weight takes no gradient; the bias does (reduced inside the
    input-gradient GEMM).  ``materialized``: each matmul first writes the
    16-bit weight to a temporary workspace and reads it with a plain GEMM
    (faster, N * K * 2 bytes of transient memory); the results are the same
    bits.  ``double_quant`` (the ``bnb.nf4-dq`` / ``bnb.fp4-dq`` options): the
    absmax values are stored in 8 bits (FP8 E4M3 codes in blocks of 256 with
    an fp32 scale each, around their mean) and decoded by one kernel per
    call."""

    fmt = "nf4"

    def __init__(self, in_features: int, out_features: int, bias: bool = True, device=None,
                 bias_dtype: torch.dtype = torch.bfloat16, materialized: bool = False, fmt: str | None = None,
                 double_quant: bool = False):
        super().__init__()
        from . import _lib
        if fmt is not None:
            self.fmt = F._fmt4(fmt)
        self.in_features = in_features
        self.out_features = out_features
        self.materialized = bool(materialized)
        self.double_quant = bool(double_quant)
        nblk = _lib.i8lt_nf4_blocks(in_features)
        self.register_buffer("packed", torch.zeros(out_features, _lib.i8lt_nf4_row_bytes(in_features),
                                                   dtype=torch.uint8, device=device))
        if self.double_quant:
            self.register_buffer("absmax_q", torch.zeros(out_features, nblk, dtype=torch.uint8, device=device))
            self.register_buffer("absmax2", torch.zeros(_lib.i8lt_absmax8_blocks(out_features * nblk),
                                                        dtype=torch.float32, device=device))
            self.register_buffer("absmax_offset", torch.zeros(1, dtype=torch.float32, device=device))
        else:
            self.register_buffer("absmax", torch.zeros(out_features, nblk, dtype=torch.float32, device=device))
        if bias:
            self.bias = torch.nn.Parameter(torch.zeros(out_features, dtype=bias_dtype, device=device))
        else:
            self.register_parameter("bias", None)

    @classmethod
    def from_float(cls, weight: torch.Tensor, bias: torch.Tensor | None = None,
                   materialized: bool = False, **kw) -> "Linear4bit":
        N, K = weight.shape
        layer = cls(K, N, bias=bias is not None, device=weight.device,
                    bias_dtype=bias.dtype if bias is not None else torch.bfloat16, materialized=materialized, **kw)
        packed, absmax = F.quantize_4bit(weight, layer.fmt)
        layer.packed.copy_(packed)
        if layer.double_quant:
            q, a2, off = F.double_quantize_absmax(absmax)
            layer.absmax_q.copy_(q)
            layer.absmax2.copy_(a2)
            layer.absmax_offset.copy_(off)
        else:
            layer.absmax.copy_(absmax)
        if bias is not None:
            with torch.no_grad():
                layer.bias.copy_(bias)
        return layer

    def decoded_absmax(self) -> torch.Tensor:
        """The fp32 absmax [N, blocks per row] the matmuls use."""
        if self.double_quant:
            return F.dequantize_absmax(self.absmax_q, self.absmax2, self.absmax_offset)
        return self.absmax

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return F.Linear4bitFunction.apply(x, self.packed, self.decoded_absmax(), self.in_features, self.bias,
                                          self.materialized, self.fmt)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, bias={self.bias is not None}, "
                f"fmt={self.fmt}, double_quant={self.double_quant}")


class LinearNF4(Linear4bit):
    """The 4-bit NormalFloat layer (bnb.nf4)."""
    fmt = "nf4"


class LinearFP4(Linear4bit):
    """The 4-bit floating-point (E2M1) layer (bnb.fp4)."""
    fmt = "fp4"
