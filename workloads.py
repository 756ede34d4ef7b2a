"""Seeded synthetic inputs for the int8 quantized linear layer.

This module holds only random-number recipes: no step of the method's
arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle are fed from
here.  Every tensor is drawn on the CPU with its own ``torch.Generator`` seed
(``base + offset``), so that a given (workload, seed) is the same tensor on
every machine; ``device`` only says where the result is copied.

Offsets: activations 0, weight 1, bias 2, grad_output 3, heavy-column
permutation 4; a second layer adds 10 to each.

Heavy ("outlier") columns: ``randperm(K)[:round(frac * K)]`` of the
activation's columns are multiplied by a factor, so that their magnitude
exceeds the outlier threshold, as in the LLM.int8 setting the bitsandbytes
``Linear8bitLt`` layer was built for.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

OFF_A, OFF_W, OFF_BIAS, OFF_G, OFF_HEAVY = 0, 1, 2, 3, 4
OFF_LAYER2 = 10


@dataclass(frozen=True)
class LayerSpec:
    M: int
    K: int
    N: int
    dtype: torch.dtype          # activation / output / grad dtype
    w_std: float
    bias_std: float | None      # None: zero bias
    heavy_frac: float = 0.0
    heavy_factor: float = 1.0
    threshold: float = float("inf")


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    layers: tuple               # tuple[LayerSpec, ...]
    kind: str = "linear"        # "linear": independent layers; "mlp": chained
    residual: bool = False      # mlp: y = L2(silu(L1(x))) + x
    w_dtype: torch.dtype | None = None   # dtype the float weights are drawn in
    extra: dict = field(default_factory=dict)


INF = float("inf")

WORKLOADS = {
    "tiny_mlp": Workload(
        "tiny_mlp",
        "residual MLP on x fp32 (1,600,4): Dense 4->16, SiLU, Dense 16->4, +x; "
        "weights N(0,0.02) fp32, zero bias, no outliers (threshold inf)",
        (LayerSpec(600, 4, 16, torch.float32, 0.02, None),
         LayerSpec(600, 16, 4, torch.float32, 0.02, None)),
        kind="mlp", residual=True, w_dtype=torch.float32),
    "linear_4096": Workload(
        "linear_4096",
        "Linear8bitLt 4096->4096, fp16 A of 2048 tokens N(0,1), 0.1% of the "
        "columns x20, threshold 6; weight N(0,0.02), bias N(0,0.01)",
        (LayerSpec(2048, 4096, 4096, torch.float16, 0.02, 0.01, 0.001, 20.0, 6.0),),
        w_dtype=torch.float16),
    "linear_bf16_4096x11008": Workload(
        "linear_bf16_4096x11008",
        "Linear8bitLt 4096->11008 fed bf16 A of 4096 tokens, 0.5% of the "
        "columns x10, threshold 6; weight N(0,0.02), bias N(0,0.01)",
        (LayerSpec(4096, 4096, 11008, torch.bfloat16, 0.02, 0.01, 0.005, 10.0, 6.0),),
        w_dtype=torch.bfloat16),
    "mlp_7b": Workload(
        "mlp_7b",
        "7B-style MLP 4096->11008 (SiLU) ->4096, fp16, 8192 tokens, 0.1% of "
        "the input columns x20, threshold 6 on both layers",
        (LayerSpec(8192, 4096, 11008, torch.float16, 0.02, 0.01, 0.001, 20.0, 6.0),
         LayerSpec(8192, 11008, 4096, torch.float16, 0.02, 0.01, 0.0, 1.0, 6.0)),
        kind="mlp", w_dtype=torch.float16),
    "proj_8192x28672": Workload(
        "proj_8192x28672",
        "projections 8192->28672 and 28672->8192, fp16 A of 16384 tokens "
        "N(0,1) with 0.2% of the columns x15, threshold 6; weights N(0,0.01), "
        "bias N(0,0.01); each layer fed its own synthetic A",
        (LayerSpec(16384, 8192, 28672, torch.float16, 0.01, 0.01, 0.002, 15.0, 6.0),
         LayerSpec(16384, 28672, 8192, torch.float16, 0.01, 0.01, 0.002, 15.0, 6.0)),
        w_dtype=torch.float16),
}

ORDER = ("tiny_mlp", "linear_4096", "linear_bf16_4096x11008", "mlp_7b",
         "proj_8192x28672")

# The 4-bit NormalFloat weight-only layer of QLoRA fine-tuning (frozen base
# weights, bf16 compute): the Llama-2-7B MLP shapes the QLoRA runs use, with
# the token count of the int8 7B MLP workload.
NF4_WORKLOADS = {
    "qlora_mlp_7b_nf4": Workload(
        "qlora_mlp_7b_nf4",
        "Llama-2-7B-style MLP layers with frozen NF4 weights: 4096->11008 and "
        "11008->4096, bf16 activations of 8192 tokens N(0,1), weights "
        "N(0,0.02) drawn in bf16, no bias; forward and input gradient of each "
        "layer, each fed its own synthetic input",
        (LayerSpec(8192, 4096, 11008, torch.bfloat16, 0.02, None),
         LayerSpec(8192, 11008, 4096, torch.bfloat16, 0.02, None)),
        w_dtype=torch.bfloat16),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std, seed, dtype, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on the CPU, then stored in ``dtype``."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype).to(device)


def heavy_columns(K, frac, seed) -> torch.Tensor:
    n = int(round(frac * K))
    if n == 0:
        return torch.zeros(0, dtype=torch.long)
    return torch.randperm(K, generator=_gen(seed))[:n].sort().values


def activation(spec: LayerSpec, seed: int, device="cpu", rows=None) -> torch.Tensor:
    """A [M, K] ~ N(0,1) with the heavy columns scaled; ``rows`` (optional)
    draws the full matrix and keeps only those rows."""
    x = torch.randn(spec.M, spec.K, generator=_gen(seed + OFF_A), dtype=torch.float32)
    h = heavy_columns(spec.K, spec.heavy_frac, seed + OFF_HEAVY)
    if len(h):
        x[:, h] *= spec.heavy_factor
    if rows is not None:
        x = x[rows]
    return x.to(spec.dtype).to(device)


def layer_tensors(wl: Workload, li: int, seed: int, device="cpu"):
    """Float weight [N, K], bias [N] (or None for a zero bias... returned as
    zeros), grad_output [M, N] of layer ``li``."""
    spec = wl.layers[li]
    base = seed + li * OFF_LAYER2
    wdt = wl.w_dtype or spec.dtype
    W = normal((spec.N, spec.K), spec.w_std, base + OFF_W, wdt, device)
    if spec.bias_std is None:
        b = torch.zeros(spec.N, dtype=wdt, device=device)
    else:
        b = normal((spec.N,), spec.bias_std, base + OFF_BIAS, wdt, device)
    G = normal((spec.M, spec.N), 1.0, base + OFF_G, spec.dtype, device)
    return W, b, G


def layer_input(wl: Workload, li: int, seed: int, device="cpu"):
    """Synthetic input of layer ``li`` (for chained MLPs only layer 0 has
    one: the next layers are fed the previous layer's output)."""
    spec = wl.layers[li]
    return activation(spec, seed + li * OFF_LAYER2, device)


def lossless_case(M, K, N, seed, outlier_cols=(), threshold=6.0, ea_range=(-9, -4), ew_range=(-12, -7)):
    """Inputs on the quantization grid, for an exact check of the method.

    A[m, k] = qa[m, k] * ua[m], W[n, k] = qw[n, k] * uw[n] with integer codes
    |q| <= 127, every row holding a +-127, and power-of-two steps ua, uw.
    The absmax quantization then returns the codes unchanged and its
    dequantization is exact, so the layer must reproduce the fp64 product.
    ``outlier_cols`` get values of magnitude above ``threshold`` (these leave
    the int8 part and go through the fp16 outlier product).
    ``ea_range`` / ``ew_range``: half-open ranges of the exponents of ua / uw.

    Returned as fp16 tensors: (A, W) plus the codes and steps.
    """
    g = _gen(seed)
    qa = torch.randint(-127, 128, (M, K), generator=g)
    qw = torch.randint(-127, 128, (N, K), generator=g)
    # plant +-127 in each row, away from the outlier columns
    keep = [k for k in range(K) if k not in set(outlier_cols)]
    for r in range(M):
        qa[r, keep[int(torch.randint(len(keep), (1,), generator=g))]] = 127 * (1 if r % 2 else -1)
    for r in range(N):
        qw[r, int(torch.randint(K, (1,), generator=g))] = -127 if r % 3 else 127
    ea = torch.randint(ea_range[0], ea_range[1], (M,), generator=g)    # default steps 2^-9 .. 2^-5
    ew = torch.randint(ew_range[0], ew_range[1], (N,), generator=g)    # default 2^-12 .. 2^-8
    ua = torch.pow(2.0, ea.double())
    uw = torch.pow(2.0, ew.double())
    A = qa.double() * ua[:, None]
    W = qw.double() * uw[:, None]
    for j, k in enumerate(outlier_cols):
        # fp16-representable values above the threshold, both signs
        v = torch.randint(1, 64, (M,), generator=g).double() / 4.0 + threshold + 0.25
        sign = torch.where(torch.rand(M, generator=g) < 0.5, -1.0, 1.0).double()
        A[:, k] = v * sign
        # most rows must keep their absmax (127*ua) outside column k: it is
        # already planted in ``keep``
    return dict(A=A.half(), W=W.half(), qa=qa, qw=qw, ua=ua, uw=uw)


def grid_values(shape, qmax, step_exp, seed) -> torch.Tensor:
    """Integers uniform in [-qmax, qmax] times 2**step_exp (float64): values
    that fp16 and bf16 hold exactly while qmax < 256, for inputs whose every
    sum the exact checks can predict."""
    q = torch.randint(-qmax, qmax + 1, tuple(shape), generator=_gen(seed))
    return q.double() * (2.0 ** step_exp)
