"""The trainable-weight mode (bitsandbytes' has_fp16_weights=True) on the GPU:
the weight gradient through column-wise int8 quantization, checked against
the oracle -- codes, scales and the int32 product bit for bit (read back
from the workspace), grad_W within the tolerance -- and the autograd layer.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build
from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE

from _helpers import ODT, assert_tol, to_np, widen

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _ws_regions(ws, M, N, K):
    """Workspace regions in the order i8lt_grad_weight lays them out (each
    256-byte aligned): status, colmax G, colmax A, scale G, scale A, tile
    chunk maxima G and A, chunk sums G and A, plan, Gt, At."""
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    r_pad = (M + 15) // 16 * 16
    chunks = (r_pad + 1023) // 1024
    tn, tk = (N + 255) // 256, (K + 255) // 256
    sizes = [256, up(N * 4), up(K * 4), up(N * 4), up(K * 4), up(tn * chunks * 4), up(tk * chunks * 4),
             up(N * chunks * 4), up(K * chunks * 4), up(tn * tk * 4), up(N * r_pad * 2), up(K * r_pad * 2)]
    off = np.cumsum([0] + sizes)
    assert off[-1] == _lib.i8lt_grad_weight_workspace_size(M, N, K)
    return dict(scale_g=ws[off[3]:off[3] + 4 * N].view(torch.float32),
                scale_a=ws[off[4]:off[4] + 4 * K].view(torch.float32),
                tsq_g=ws[off[5]:off[5] + 4 * tn * chunks].view(torch.int32).reshape(tn, chunks),
                tsq_a=ws[off[6]:off[6] + 4 * tk * chunks].view(torch.int32).reshape(tk, chunks),
                plan=ws[off[9]:off[9] + 4 * tn * tk].view(torch.int32).reshape(tn, tk),
                gt=ws[off[10]:off[10] + N * r_pad * 2].view(torch.float16).reshape(N, r_pad),
                at=ws[off[11]:off[11] + K * r_pad * 2].view(torch.float16).reshape(K, r_pad))


@pytest.mark.parametrize("M,N,K,dtype", [(300, 520, 1100, torch.float16),    # 2 exact chunks of tokens, ragged
                                         (1025, 257, 72, torch.bfloat16),    # a ragged second chunk
                                         (77, 40, 36, torch.float32),
                                         (4096, 1024, 768, torch.float16)])
def test_grad_weight_matches_the_oracle(M, N, K, dtype):
    spec = W.LayerSpec(M, K, N, dtype, 0.02, 0.01, 0.01, 12.0, 6.0)
    A = W.activation(spec, 41)
    G = W.normal((M, N), 1.0, 42, dtype)
    ws = torch.empty(_lib.i8lt_grad_weight_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    gW = I.grad_weight(G.to(DEV), A.to(DEV), dtype, ws=ws)
    ref = O.grad_weight(to_np(G), to_np(A), ODT[dtype])
    reg = _ws_regions(ws, M, N, K)
    assert np.array_equal(to_np(reg["scale_g"]).view(np.uint32), ref["SCG"].view(np.uint32))
    assert np.array_equal(to_np(reg["scale_a"]).view(np.uint32), ref["SCA"].view(np.uint32))
    gt = to_np(reg["gt"]).astype(np.float32)
    at = to_np(reg["at"]).astype(np.float32)
    assert np.array_equal(gt[:, :M], ref["Gt"].astype(np.float32)) and not np.any(gt[:, M:])
    assert np.array_equal(at[:, :M], ref["At"].astype(np.float32)) and not np.any(at[:, M:])
    # the tolerance rule on the fp32 result; a 16-bit grad_W is that result
    # rounded once (its own rounding of the largest elements -- the heavy
    # input columns -- can exceed 0.02 * mean|ref| by itself)
    gW32 = I.grad_weight(G.to(DEV), A.to(DEV), torch.float32)
    assert_tol(widen(gW32), ref["grad64"], "grad_W")
    assert torch.equal(gW, gW32.to(dtype))


def test_grad_weight_lossless_case_is_exact():
    M, N, K = 512, 96, 64
    case = W.lossless_case(N, M, K, seed=43)
    G = case["A"].t().contiguous()
    A = case["W"].t().contiguous()
    gW = I.grad_weight(G.to(DEV), A.to(DEV), torch.float32)
    exact = G.double().t() @ A.double()
    # the int32 product is exact; the fp32 dequant (SCG * 1/127^2 * SCA * Cacc)
    # adds a few roundings of 2^-24
    rel = ((gW.cpu().double() - exact).abs() / exact.abs().clamp_min(1e-30)).max()
    assert rel < 1e-6, rel


def test_grad_weight_empty_batch_is_zero():
    gW = I.grad_weight(torch.empty(0, 24, dtype=torch.float16, device=DEV),
                       torch.empty(0, 40, dtype=torch.float16, device=DEV))
    assert gW.shape == (24, 40) and not torch.any(gW)


def test_trainable_layer_gradients():
    M, K, N = 640, 512, 384
    spec = W.LayerSpec(M, K, N, torch.float16, 0.02, 0.01, 0.01, 12.0, 6.0)
    x = W.activation(spec, 44).to(DEV)
    layer = I.Linear8bitLtTrainable(K, N, device=DEV)
    with torch.no_grad():
        layer.weight.copy_(W.normal((N, K), 0.02, 45, torch.float16).to(DEV))
        layer.bias.copy_(W.normal((N,), 0.01, 46, torch.float16).to(DEV))
    xr = x.clone().requires_grad_(True)
    y = layer(xr)
    G = W.normal((M, N), 1.0, 47, torch.float16).to(DEV)
    y.backward(G)
    # forward and grad_A: the memory-efficient layer with the weight quantized now
    CB, SCB = I.quantize_weight(layer.weight.detach())
    y_ref, _ = I.forward(x, CB, SCB, K, layer.bias.detach(), 6.0)
    assert torch.equal(y.detach(), y_ref)
    gA_ref, gb_ref = I.backward_input(G, CB, SCB, K, bias_dtype=torch.float16)
    assert torch.equal(xr.grad, gA_ref) and torch.equal(layer.bias.grad, gb_ref)
    # grad_W: the int8 product, within the tolerance of the oracle, and close to the exact G^T x
    ref = O.grad_weight(to_np(G), to_np(x), O.F16)
    assert_tol(widen(layer.weight.grad), ref["grad64"], "grad_W")
    exact = G.double().t() @ x.double()
    rel = (layer.weight.grad.double() - exact).abs().mean() / exact.abs().mean()
    assert rel < 0.02
