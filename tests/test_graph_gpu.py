"""The library's calls inside a CUDA graph: every launch and memset goes to
the caller's stream, so a step captured once replays with no host work per
kernel.  Replays give the eager results bit for bit (int8 layer forward and
backward, the 4-bit layer), also after the inputs are overwritten in place."""
import pytest
import torch

import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                                  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


def test_int8_layer_step_replays_bit_exact():
    spec = W.LayerSpec(700, 1100, 520, torch.float16, 0.02, 0.01, 0.01, 20.0, 6.0)
    A = W.activation(spec, 3).to(DEV)
    Wf = W.normal((spec.N, spec.K), 0.02, 4, torch.float16, DEV)
    b = W.normal((spec.N,), 0.01, 5, torch.float16, DEV)
    G = W.normal((spec.M, spec.N), 1.0, 6, torch.float16, DEV)
    CB, SCB = I.quantize_weight(Wf)
    K = spec.K
    ws_f = I.functional.forward_workspace(spec.M, K, spec.N, K, DEV)
    ws_b = I.functional.backward_workspace(spec.M, spec.N, torch.float16, DEV)
    out = torch.empty(spec.M, spec.N, dtype=torch.float16, device=DEV)

    def step():
        I.forward(A, CB, SCB, K, b, 6.0, out=out, ws=ws_f, max_outliers=K)
        return I.backward_input(G, CB, SCB, K, bias_dtype=torch.float16, ws=ws_b)

    g, (gA, gb) = _capture(step)
    ref_out, _ = I.forward(A, CB, SCB, K, b, 6.0, max_outliers=K)
    ref_gA, ref_gb = I.backward_input(G, CB, SCB, K, bias_dtype=torch.float16)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(gA, ref_gA) and torch.equal(gb, ref_gb)
    # new inputs written in place: the replay follows them
    A.copy_(W.activation(spec, 13).to(DEV))
    G.mul_(-0.5)
    g.replay()
    torch.cuda.synchronize()
    ref_out, _ = I.forward(A, CB, SCB, K, b, 6.0, max_outliers=K)
    ref_gA, ref_gb = I.backward_input(G, CB, SCB, K, bias_dtype=torch.float16)
    assert torch.equal(out, ref_out) and torch.equal(gA, ref_gA) and torch.equal(gb, ref_gb)


def test_nf4_layer_replays_bit_exact():
    M, K, N = 600, 1024, 712
    Wf = W.normal((N, K), 0.02, 7, torch.bfloat16, DEV)
    packed, absmax = I.nf4_quantize(Wf)
    A = W.normal((M, K), 1.0, 8, torch.bfloat16, DEV)
    G = W.normal((M, N), 1.0, 9, torch.bfloat16, DEV)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    gA = torch.empty(M, K, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)

    def step():
        I.nf4_forward(A, packed, absmax, K, out=y, ws=ws)
        I.nf4_backward_input(G, packed, absmax, K, out=gA, ws=ws)

    g, _ = _capture(step)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, I.nf4_forward(A, packed, absmax, K))
    assert torch.equal(gA, I.nf4_backward_input(G, packed, absmax, K))
