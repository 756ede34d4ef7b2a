"""Method-level checks against plain PyTorch with the original float weights.

bitsandbytes PR #33 asked for "a test that tests for minimal difference
between fp16 gradients and int8->fp16 gradients"; its test_modules.py check
(review thread on tests/test_modules.py) runs two int8 layers, backpropagates
(o1 * grad_proj).sum() and compares the input gradient with
grad_proj @ w2 @ w1 of the float weights: every element within 0.05 * scale
(scale = mean |grad_ref|), and at most 0.5% of the elements outside
isclose(atol=0.01 * scale, rtol=0.1).  The same rule is applied here, and to
the forward output against the float linear layer.
"""
import pytest
import torch

import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def page_rule(got, ref, k=0.05):
    got, ref = got.float(), ref.float()
    scale = ref.abs().mean()
    assert torch.allclose(got, ref, rtol=0, atol=k * scale), float((got - ref).abs().max() / scale)
    bad = ~torch.isclose(got, ref, atol=0.01 * scale, rtol=0.1)
    assert bad.sum().item() <= ref.numel() * 0.005, bad.float().mean().item()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("seed", range(3))
def test_two_layer_input_grad_matches_float_weights(dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    dim, hidden = 1024, 4096
    b1 = torch.randn(8, 128, dim, generator=g).to(dtype)
    b1[..., torch.randperm(dim, generator=g)[:4]] *= 20          # outlier features
    w1 = (torch.randn(hidden, dim, generator=g) * 0.02).to(dtype)
    w2 = (torch.randn(dim, hidden, generator=g) * 0.02).to(dtype)
    bias1 = (torch.randn(hidden, generator=g) * 0.01).to(dtype)
    bias2 = (torch.randn(dim, generator=g) * 0.01).to(dtype)
    fc1 = I.Linear8bitLt.from_float(w1.to(DEV), bias1.to(DEV), threshold=6.0)
    fc2 = I.Linear8bitLt.from_float(w2.to(DEV), bias2.to(DEV), threshold=6.0)
    x = b1.to(DEV).requires_grad_(True)
    o1 = fc2(fc1(x))
    grad_proj = torch.randn(o1.shape, generator=g).to(dtype).to(DEV)
    (o1 * grad_proj).sum().backward()
    grad_ref = grad_proj.flatten(2).float() @ w2.to(DEV).float() @ w1.to(DEV).float()
    page_rule(x.grad, grad_ref.reshape(x.shape))
    # forward against the float layers
    ref = (x.detach().float() @ w1.to(DEV).float().t() + bias1.to(DEV).float()) @ w2.to(DEV).float().t() \
        + bias2.to(DEV).float()
    page_rule(o1.detach(), ref)
    # grad_bias of the second layer from the uncast grad_output
    page_rule(fc2.bias.grad, (grad_proj.float()).reshape(-1, dim).sum(0), k=0.02)


def test_weight_is_frozen_and_cast_warning():
    w = torch.randn(64, 32, device=DEV, dtype=torch.float16) * 0.02
    fc = I.Linear8bitLt.from_float(w, torch.zeros(64, device=DEV, dtype=torch.float16))
    assert not any(p.dtype == torch.int8 for p in fc.parameters())
    assert fc.CB.dtype == torch.int8 and not fc.CB.requires_grad
    x = torch.randn(4, 32, device=DEV, dtype=torch.float32, requires_grad=True)
    y = fc(x)
    assert y.dtype == torch.float32
    y.sum().backward()
    assert x.grad is not None and x.grad.dtype == torch.float32
