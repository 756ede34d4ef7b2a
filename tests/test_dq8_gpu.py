"""GPU parity of the double-quantized absmax (the ``bnb.nf4-dq`` /
``bnb.fp4-dq`` options of "Support QLoRA 4-bit finetuning with bitsandbytes",
lit-gpt PR #275): codes, second-level scales, the offset and the decoded
values bit for bit against oracle/dq8.py, and the 4-bit layers running on the
decoded absmax."""
import numpy as np
import pytest
import torch

import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
import workloads as W
from oracle import dq8 as D
from oracle import nf4 as ON
from oracle import fp4 as OF
import oracle as O
from tests._helpers import assert_tol, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _check_dq(c: np.ndarray):
    """GPU double quantization of the fp32 values c (any shape) equals the
    oracle's bit for bit, and so does the decoding."""
    c = np.ascontiguousarray(c, np.float32)
    q, a2, off = I.double_quantize_absmax(torch.from_numpy(c).to(DEV))
    q_ref, a2_ref, off_ref = D.quantize(c)
    assert to_np(off)[0].view(np.uint32) == np.float32(off_ref).view(np.uint32), (to_np(off)[0], off_ref)
    assert np.array_equal(to_np(a2).view(np.uint32), a2_ref.view(np.uint32))
    assert np.array_equal(to_np(q), q_ref)
    dec = I.dequantize_absmax(q, a2, off)
    dec_ref = D.dequantize(q_ref, a2_ref, off_ref)
    assert np.array_equal(to_np(dec).view(np.uint32), dec_ref.view(np.uint32))
    return q, a2, off, dec


@pytest.mark.parametrize("shape", [(1, 1), (1, 256), (1, 257), (37, 100), (512, 64), (11008, 64)])
def test_absmax8_bit_exact(shape):
    g = np.random.default_rng(shape[0] + shape[1])
    c = np.abs(g.normal(0.02, 0.01, shape)).astype(np.float32)
    _check_dq(c)


def test_absmax8_of_a_quantized_weight():
    """The absmax of the QLoRA 7B MLP's first layer, quantized by the GPU to
    NF4 and equal to the oracle's first level."""
    wl = W.NF4_WORKLOADS["qlora_mlp_7b_nf4"]
    Wf, _, _ = W.layer_tensors(wl, 0, 0)
    packed, absmax = I.nf4_quantize(Wf.to(DEV))
    _, a_ref, _ = ON.quantize(to_np(Wf), O.BF16)
    assert np.array_equal(to_np(absmax).view(np.uint32), a_ref.view(np.uint32))
    _check_dq(a_ref)


def test_absmax8_edge_values():
    """Equal values (every block scale 0), zeros, values over many binades
    with subnormals (the exact sum of the offset), one value."""
    _check_dq(np.full(1000, 0.0371, np.float32))
    _check_dq(np.zeros(300, np.float32))
    g = np.random.default_rng(3)
    spread = np.exp(g.uniform(-100, 20, 5000)).astype(np.float32)
    spread[::17] = np.float32(1e-41)                     # subnormal
    spread[::101] = 0.0
    _check_dq(spread)
    _check_dq(np.array([3.5], np.float32))
    # a sum whose float64 rounding needs the sticky bits: 2^53 + 1 + tiny
    tricky = np.array([2.0 ** 60, 2.0 ** 7, 2.0 ** -40, 3.0], np.float32)
    _check_dq(tricky)


def test_absmax8_empty_and_errors():
    q, a2, off = I.double_quantize_absmax(torch.empty(0, device=DEV))
    assert q.numel() == 0 and a2.numel() == 0 and float(off[0]) == 0.0
    ws = torch.empty(_lib.i8lt_absmax8_workspace_size(), dtype=torch.uint8, device=DEV)
    x = torch.ones(10, device=DEV)
    out = torch.empty(10, dtype=torch.uint8, device=DEV)
    a2 = torch.empty(1, device=DEV)
    off = torch.empty(1, device=DEV)
    assert _lib.i8lt_absmax8_quantize(x.data_ptr(), 10, out.data_ptr(), a2.data_ptr(), off.data_ptr(),
                                      ws.data_ptr(), 16, None) == _lib.I8LT_ERR_WORKSPACE
    assert _lib.i8lt_absmax8_quantize(x.data_ptr(), -1, out.data_ptr(), a2.data_ptr(), off.data_ptr(),
                                      ws.data_ptr(), ws.numel(), None) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_absmax8_quantize(x.data_ptr(), 10, out.data_ptr(), a2.data_ptr(), None,
                                      ws.data_ptr(), ws.numel(), None) == _lib.I8LT_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", ["nf4", "fp4"])
def test_double_quantized_layers(fmt):
    """Linear4bit(double_quant=True): the matmuls run on the decoded absmax
    (bit-identical to the plain entry points given those values) and match
    the oracle's layer on the oracle's decoded absmax."""
    M, K, N = 700, 1024, 768
    g = torch.Generator().manual_seed(21)
    Wf = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    b = (torch.randn(N, generator=g) * 0.01).to(torch.bfloat16)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    G = torch.randn(M, N, generator=g).to(torch.bfloat16)
    layer = I.Linear4bit.from_float(Wf.to(DEV), b.to(DEV), fmt=fmt, double_quant=True)
    assert not hasattr(layer, "absmax") and layer.absmax_q.dtype == torch.uint8
    OM = ON if fmt == "nf4" else OF
    p_ref, a_ref, _ = OM.quantize(to_np(Wf), O.BF16)
    assert np.array_equal(to_np(layer.packed), p_ref)
    q_ref, a2_ref, off_ref = D.quantize(a_ref)
    assert np.array_equal(to_np(layer.absmax_q), q_ref)
    dec_ref = D.dequantize(q_ref, a2_ref, off_ref)
    dec = layer.decoded_absmax()
    assert np.array_equal(to_np(dec).view(np.uint32), dec_ref.view(np.uint32))
    xd = x.to(DEV).requires_grad_(True)
    y = layer(xd)
    assert torch.equal(y, I.forward_4bit(x.to(DEV), layer.packed, dec, K, layer.bias.detach(), fmt=fmt))
    y.backward(G.to(DEV))
    gx, gb = I.backward_input_4bit(G.to(DEV), layer.packed, dec, K, bias_dtype=torch.bfloat16, fmt=fmt)
    assert torch.equal(xd.grad, gx) and torch.equal(layer.bias.grad, gb)
    ref = OM.forward(to_np(x), O.BF16, p_ref, dec_ref, K, bias=to_np(b), bias_dtype=O.BF16)
    assert_tol(O.widen(to_np(y.detach()), O.BF16), ref["out64"], f"{fmt}-dq forward")
    rb = OM.backward_input(to_np(G), O.BF16, p_ref, dec_ref, K)
    assert_tol(O.widen(to_np(xd.grad), O.BF16), rb["grad64"], f"{fmt}-dq grad_A")
