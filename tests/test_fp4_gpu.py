"""The 4-bit floating-point (FP4, E2M1) weight-only layer on the GPU, through
the C ABI, against the FP4 oracle: levels, packed codes, absmax values and the
dequantized weight bit for bit (ties of the code decision included); the
forward and input-gradient matmuls, which decode the codes inside the
tensor-core pipeline through the level table, within the tolerance rule and
bit for bit on one-hot inputs; and the bias gradient of both 4-bit formats,
reduced inside the input-gradient GEMM."""
import numpy as np
import pytest
import torch

import oracle as O
import oracle.fp4 as OF
import oracle.nf4 as ON
import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build

from _helpers import ODT, assert_tol, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ORACLE = {"nf4": ON, "fp4": OF}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _check_quant(Wf, K, fmt="fp4"):
    packed, absmax = I.quantize_4bit(Wf.to(DEV), fmt)
    p_ref, a_ref, _ = ORACLE[fmt].quantize(to_np(Wf), ODT[Wf.dtype])
    assert np.array_equal(to_np(packed), p_ref), "packed codes differ"
    assert np.array_equal(to_np(absmax).view(np.uint32), a_ref.view(np.uint32)), "absmax differs"
    return packed, absmax, p_ref, a_ref


def test_levels_match_the_oracle():
    got = np.array(I.fp4_levels(), np.float32)
    assert np.array_equal(got.view(np.uint32), OF.levels().view(np.uint32))    # -0 at code 8 included


@pytest.mark.parametrize("N,K,dtype", [(300, 1000, torch.bfloat16), (64, 64, torch.float16),
                                       (257, 4100, torch.float32), (5, 7, torch.bfloat16)])
def test_quantize_and_dequantize_bit_exact(N, K, dtype):
    Wf = W.normal((N, K), 0.02, 3, dtype)
    Wf[1] = 0                                   # an all-zero row
    if K > 64:
        Wf[2, 64:128] = 0                       # an all-zero block
        Wf[3, :64] *= 1000                      # a block of large values
    packed, absmax, p_ref, a_ref = _check_quant(Wf, K)
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        got = I.fp4_dequantize(packed, absmax, K, dt)
        ref = OF.dequantize(p_ref, a_ref, K, ODT[dt])
        assert np.array_equal(to_np(got).view(np.uint8), ref.view(np.uint8)), f"dequantized {dt} differs"


def test_half_way_ties_round_to_even():
    """Weights whose |x / absmax| equals every midpoint exactly (fp32 weights,
    absmax a power of two), one fp32 step either side of it, both signs,
    over many blocks: the codes equal the oracle's (ties to the code whose
    mantissa bit is 0)."""
    mid = OF.midpoints()
    rows = []
    for p in range(-3, 4):
        s = np.float32(2.0 ** p)
        for vals in (mid, np.nextafter(mid, np.float32(2)), np.nextafter(mid, np.float32(-2))):
            r = np.zeros(64, np.float32)
            r[0] = s
            r[1:8] = vals * s
            r[8:15] = -vals * s
            rows.append(r)
    Wt = torch.from_numpy(np.stack(rows))
    packed, absmax, p_ref, _ = _check_quant(Wt, 64)
    codes = OF.unpack(p_ref, 64)
    assert codes[0, 1:8].tolist() == [0, 2, 2, 4, 4, 6, 6]


@pytest.mark.parametrize("M,K,N,dtype,bias", [(600, 1000, 712, torch.bfloat16, True),    # ragged in every dimension
                                              (1, 64, 256, torch.bfloat16, False),
                                              (1100, 2056, 520, torch.float16, True),
                                              (512, 4096, 1024, torch.bfloat16, False)])
def test_forward_and_input_gradient(M, K, N, dtype, bias):
    Wf = W.normal((N, K), 0.02, 5, dtype)
    A = W.normal((M, K), 1.0, 6, dtype)
    G = W.normal((M, N), 1.0, 7, dtype)
    b = W.normal((N,), 0.1, 8, dtype) if bias else None
    packed, absmax, p_ref, a_ref = _check_quant(Wf, K)
    out = I.fp4_forward(A.to(DEV), packed, absmax, K, b.to(DEV) if bias else None)
    ref = OF.forward(to_np(A), ODT[dtype], p_ref, a_ref, K, to_np(b) if bias else None, ODT[dtype])
    assert out.dtype == dtype
    assert_tol(O.widen(to_np(out), ODT[dtype]), ref["out64"], "fp4 forward")
    gA = I.fp4_backward_input(G.to(DEV), packed, absmax, K)
    rb = OF.backward_input(to_np(G), ODT[dtype], p_ref, a_ref, K)
    assert_tol(O.widen(to_np(gA), ODT[dtype]), rb["grad64"], "fp4 grad_A")
    # the materialized schedule (dequantized weight in the workspace) gives the same bits
    assert torch.equal(I.fp4_forward(A.to(DEV), packed, absmax, K, b.to(DEV) if bias else None, materialized=True),
                       out)
    assert torch.equal(I.fp4_backward_input(G.to(DEV), packed, absmax, K, materialized=True), gA)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decoded_weight_inside_the_matmuls_is_bit_exact(dtype):
    """One-hot inputs: every output is a single product 1 * Wdq, so the
    forward returns Wdq^T and the input gradient Wdq -- the FP4 weight
    decoded inside the tensor-core pipeline equals the oracle's dequantized
    weight bit for bit (signed zeros compared as values)."""
    N, K = 712, 1000
    Wf = W.normal((N, K), 0.05, 21, dtype)
    packed, absmax, p_ref, a_ref = _check_quant(Wf, K)
    ref = O.widen(OF.dequantize(p_ref, a_ref, K, ODT[dtype]), ODT[dtype])
    out = I.fp4_forward(torch.eye(K, dtype=dtype, device=DEV), packed, absmax, K)
    assert np.array_equal(O.widen(to_np(out), ODT[dtype]), ref.T)
    gA = I.fp4_backward_input(torch.eye(N, dtype=dtype, device=DEV), packed, absmax, K)
    assert np.array_equal(O.widen(to_np(gA), ODT[dtype]), ref)


@pytest.mark.parametrize("fmt", ["nf4", "fp4"])
@pytest.mark.parametrize("M,K,N,dtype", [(300, 1000, 520, torch.bfloat16),   # ragged 128-token chunks and blocks
                                         (1100, 256, 4104, torch.float16),   # one row tile of the GEMM
                                         (129, 9000, 200, torch.bfloat16)])  # more row tiles than blocks
def test_bias_gradient_of_the_4bit_layers(fmt, M, K, N, dtype):
    """grad_bias of the frozen 4-bit layer: reduced inside the input-gradient
    GEMM (both schedules) or by a pass of its own when grad_A is not asked
    for -- the same bits every way, within the tolerance of the float64 sum,
    and grad_A unchanged by it."""
    Wf = W.normal((N, K), 0.02, 41, dtype)
    G = W.normal((M, N), 1.0, 42, dtype)
    packed, absmax = I.quantize_4bit(Wf.to(DEV), fmt)
    Gd = G.to(DEV)
    gA0, _ = I.backward_input_4bit(Gd, packed, absmax, K, fmt=fmt)
    _lib.i8lt_profile_start(64)
    gA, gb = I.backward_input_4bit(Gd, packed, absmax, K, bias_dtype=torch.float32, fmt=fmt)
    torch.cuda.synchronize()
    _, recs, _ = _lib.i8lt_profile_stop(64)
    assert [n for n, _ in recs] == ["nf4_gemm_bwd", "grad_bias_finalize"]   # no pass of its own over G
    assert torch.equal(gA, gA0)
    gA_m, gb_m = I.backward_input_4bit(Gd, packed, absmax, K, bias_dtype=torch.float32, materialized=True, fmt=fmt)
    _, gb_p = I.backward_input_4bit(Gd, packed, absmax, K, need_grad_A=False, bias_dtype=torch.float32, fmt=fmt)
    assert torch.equal(gA_m, gA)
    assert torch.equal(gb.view(torch.int32), gb_p.view(torch.int32))
    assert torch.equal(gb_m.view(torch.int32), gb_p.view(torch.int32))
    ref = O.widen(to_np(G), ODT[dtype]).sum(0)
    assert_tol(O.widen(to_np(gb), O.F32), ref, f"{fmt} grad_bias")
    # in bf16 output the sum is rounded once
    _, gb16 = I.backward_input_4bit(Gd, packed, absmax, K, bias_dtype=dtype, fmt=fmt)
    assert torch.equal(gb16, gb.to(dtype))


@pytest.mark.parametrize("cls", ["LinearNF4", "LinearFP4"])
def test_module_autograd(cls):
    K, N, M = 512, 384, 300
    Wf = W.normal((N, K), 0.02, 12, torch.bfloat16)
    b = W.normal((N,), 0.1, 13, torch.bfloat16)
    Layer = getattr(I, cls)
    layer = Layer.from_float(Wf.to(DEV), b.to(DEV))
    x = W.normal((2, M // 2, K), 1.0, 14, torch.bfloat16, DEV).requires_grad_(True)
    y = layer(x)
    G = W.normal((2, M // 2, N), 1.0, 15, torch.bfloat16, DEV)
    y.backward(G)
    fmt = layer.fmt
    assert torch.equal(y.reshape(M, N), I.forward_4bit(x.detach().reshape(M, K), layer.packed, layer.absmax, K,
                                                       layer.bias.detach(), fmt=fmt))
    gA, gb = I.backward_input_4bit(G.reshape(M, N), layer.packed, layer.absmax, K, bias_dtype=torch.bfloat16, fmt=fmt)
    assert torch.equal(x.grad.reshape(M, K), gA) and torch.equal(layer.bias.grad, gb)
    assert_tol(O.widen(to_np(layer.bias.grad), O.BF16), G.reshape(M, N).double().sum(0).cpu().numpy(), "bias grad")
    # the bias alone (a frozen input): the pass of its own, the same bits
    layer.bias.grad = None
    layer(x.detach()).backward(G)
    assert torch.equal(layer.bias.grad, gb)
