"""The 4-bit NormalFloat weight-only layer on the GPU, through the C ABI,
against the NF4 oracle: levels, packed codes, absmax values and the
dequantized weight bit for bit; the forward and input-gradient matmuls
(weight decoded inside the tensor-core pipeline) within the tolerance rule,
at sizes spanning several tiles with ragged tails and at the full 7B MLP
shapes on sampled rows."""
import numpy as np
import pytest
import torch

import oracle as O
import oracle.nf4 as ON
import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build

from _helpers import ODT, assert_tol, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _weight(N, K, dtype, seed, std=0.02):
    Wf = W.normal((N, K), std, seed, dtype)
    return Wf


def _check_quant(Wf, K):
    packed, absmax = I.nf4_quantize(Wf.to(DEV))
    p_ref, a_ref, _ = ON.quantize(to_np(Wf), ODT[Wf.dtype])
    assert np.array_equal(to_np(packed), p_ref), "packed codes differ"
    assert np.array_equal(to_np(absmax).view(np.uint32), a_ref.view(np.uint32)), "absmax differs"
    return packed, absmax, p_ref, a_ref


def test_levels_match_the_oracle():
    got = np.array(I.nf4_levels(), np.float32)
    assert np.array_equal(got.view(np.uint32), ON.levels().view(np.uint32))


@pytest.mark.parametrize("N,K,dtype", [(300, 1000, torch.bfloat16), (64, 64, torch.float16),
                                       (257, 4100, torch.float32), (5, 7, torch.bfloat16)])
def test_quantize_and_dequantize_bit_exact(N, K, dtype):
    Wf = _weight(N, K, dtype, 3)
    Wf[1] = 0                                   # an all-zero row
    if K > 64:
        Wf[2, 64:128] = 0                       # an all-zero block
        Wf[3, :64] *= 1000                      # a block of large values
    packed, absmax, p_ref, a_ref = _check_quant(Wf, K)
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        got = I.nf4_dequantize(packed, absmax, K, dt)
        ref = ON.dequantize(p_ref, a_ref, K, ODT[dt])
        assert np.array_equal(to_np(got).view(np.uint8), ref.view(np.uint8)), f"dequantized {dt} differs"


@pytest.mark.parametrize("M,K,N,dtype,bias", [(600, 1000, 712, torch.bfloat16, True),    # ragged in every dimension
                                              (1, 64, 256, torch.bfloat16, False),
                                              (1100, 2056, 520, torch.float16, True),
                                              (512, 4096, 1024, torch.bfloat16, False)])
def test_forward_and_input_gradient(M, K, N, dtype, bias):
    Wf = _weight(N, K, dtype, 5)
    A = W.normal((M, K), 1.0, 6, dtype)
    G = W.normal((M, N), 1.0, 7, dtype)
    b = W.normal((N,), 0.1, 8, dtype) if bias else None
    packed, absmax, p_ref, a_ref = _check_quant(Wf, K)
    out = I.nf4_forward(A.to(DEV), packed, absmax, K, b.to(DEV) if bias else None)
    ref = ON.forward(to_np(A), ODT[dtype], p_ref, a_ref, K, to_np(b) if bias else None, ODT[dtype])
    assert out.dtype == dtype
    assert_tol(O.widen(to_np(out), ODT[dtype]), ref["out64"], "nf4 forward")
    gA = I.nf4_backward_input(G.to(DEV), packed, absmax, K)
    rb = ON.backward_input(to_np(G), ODT[dtype], p_ref, a_ref, K)
    assert_tol(O.widen(to_np(gA), ODT[dtype]), rb["grad64"], "nf4 grad_A")
    # the materialized schedule (dequantized weight in the workspace) gives the same bits
    assert torch.equal(I.nf4_forward(A.to(DEV), packed, absmax, K, b.to(DEV) if bias else None, materialized=True), out)
    assert torch.equal(I.nf4_backward_input(G.to(DEV), packed, absmax, K, materialized=True), gA)


@pytest.mark.parametrize("li", [0, 1])
def test_qlora_7b_layers_sampled_rows(li):
    """The full 8192-token layers of the 7B MLP workload, in the launch
    configuration the benchmark times; the oracle checks 64 sampled rows."""
    wl = W.NF4_WORKLOADS["qlora_mlp_7b_nf4"]
    spec = wl.layers[li]
    Wf, _, G = W.layer_tensors(wl, li, 0)
    A = W.layer_input(wl, li, 0)
    packed, absmax, p_ref, a_ref = _check_quant(Wf, spec.K)
    out = I.nf4_forward(A.to(DEV), packed, absmax, spec.K)
    gA = I.nf4_backward_input(G.to(DEV), packed, absmax, spec.K)
    assert torch.equal(I.nf4_forward(A.to(DEV), packed, absmax, spec.K, materialized=True), out)
    assert torch.equal(I.nf4_backward_input(G.to(DEV), packed, absmax, spec.K, materialized=True), gA)
    rows = np.unique(np.concatenate([[0, spec.M - 1], np.random.default_rng(li).integers(0, spec.M, 62)]))
    dt = ODT[spec.dtype]
    ref = ON.forward(to_np(A), dt, p_ref, a_ref, spec.K, rows=rows)
    assert_tol(O.widen(to_np(out)[rows], dt), ref["out64"], "nf4 forward (sampled rows)")
    rb = ON.backward_input(to_np(G), dt, p_ref, a_ref, spec.K, rows=rows)
    assert_tol(O.widen(to_np(gA)[rows], dt), rb["grad64"], "nf4 grad_A (sampled rows)")


def test_repeat_calls_identical_and_empty_batch():
    K, N = 1024, 768
    Wf = _weight(N, K, torch.bfloat16, 9)
    packed, absmax = I.nf4_quantize(Wf.to(DEV))
    A = W.normal((700, K), 1.0, 10, torch.bfloat16, DEV)
    y0 = I.nf4_forward(A, packed, absmax, K)
    for _ in range(3):
        assert torch.equal(I.nf4_forward(A, packed, absmax, K), y0)
    empty = I.nf4_forward(A[:0], packed, absmax, K)
    assert empty.shape == (0, N)
    assert I.nf4_backward_input(torch.empty(0, N, dtype=torch.bfloat16, device=DEV), packed, absmax, K).shape == (0, K)


def test_fused_matmuls_repeat_bit_identical():
    """The 4-bit matmuls hand the odd CTA's decoded weight tiles to the even
    CTA's MMA the same way as the int8 backward: repeated runs at the 7B MLP's
    first layer (several rounds of pair tiles) must give the same bytes."""
    M, K, N = 8192, 4096, 11008
    Wf = _weight(N, K, torch.bfloat16, 21)
    packed, absmax = I.nf4_quantize(Wf.to(DEV))
    A = W.normal((M, K), 1.0, 22, torch.bfloat16, DEV)
    G = W.normal((M, N), 1.0, 23, torch.bfloat16, DEV)
    y0 = I.nf4_forward(A, packed, absmax, K).clone()
    g0 = I.nf4_backward_input(G, packed, absmax, K).clone()
    for _ in range(7):
        assert torch.equal(I.nf4_forward(A, packed, absmax, K), y0)
        assert torch.equal(I.nf4_backward_input(G, packed, absmax, K), g0)


def test_argument_errors():
    K, N = 100, 64                               # K not a multiple of 8
    Wf = _weight(N, K, torch.bfloat16, 11)
    packed, absmax = I.nf4_quantize(Wf.to(DEV))
    A = torch.zeros(4, K, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    out = torch.empty(4, N, dtype=torch.bfloat16, device=DEV)
    st = _lib.i8lt_nf4_forward(A.data_ptr(), _lib.I8LT_BF16, 4, K, packed.data_ptr(), absmax.data_ptr(), N, None, 0,
                               out.data_ptr(), ws.data_ptr(), 256, None)
    assert st == _lib.I8LT_ERR_INVALID_ARG
    A32 = torch.zeros(4, 96, dtype=torch.float32, device=DEV)
    st = _lib.i8lt_nf4_forward(A32.data_ptr(), _lib.I8LT_F32, 4, 96, packed.data_ptr(), absmax.data_ptr(), N, None,
                               0, out.data_ptr(), ws.data_ptr(), 256, None)
    assert st == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    st = _lib.i8lt_nf4_forward(A.data_ptr(), _lib.I8LT_BF16, 4, 96, packed.data_ptr(), absmax.data_ptr(), N, None,
                               0, out.data_ptr(), ws.data_ptr(), 128, None)
    assert st == _lib.I8LT_ERR_WORKSPACE


def test_module_autograd():
    K, N, M = 512, 384, 300
    Wf = _weight(N, K, torch.bfloat16, 12)
    b = W.normal((N,), 0.1, 13, torch.bfloat16)
    layer = I.LinearNF4.from_float(Wf.to(DEV), b.to(DEV))
    x = W.normal((2, M // 2, K), 1.0, 14, torch.bfloat16, DEV).requires_grad_(True)
    y = layer(x)
    G = W.normal((2, M // 2, N), 1.0, 15, torch.bfloat16, DEV)
    y.backward(G)
    assert torch.equal(y.reshape(M, N), I.nf4_forward(x.detach().reshape(M, K), layer.packed, layer.absmax, K,
                                                      layer.bias.detach()))
    assert torch.equal(x.grad.reshape(M, K), I.nf4_backward_input(G.reshape(M, N), layer.packed, layer.absmax, K))
    ref_gb = G.reshape(M, N).double().sum(0)
    assert torch.allclose(layer.bias.grad.double(), ref_gb, rtol=1e-2, atol=1e-1)
    # the materialized schedule through the module: the same bits
    mat = I.LinearNF4.from_float(Wf.to(DEV), b.to(DEV), materialized=True)
    x2 = x.detach().clone().requires_grad_(True)
    y2 = mat(x2)
    y2.backward(G)
    assert torch.equal(y2, y) and torch.equal(x2.grad, x.grad)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decoded_weight_inside_the_matmuls_is_bit_exact(dtype):
    """With one-hot inputs every output is a single product 1 * Wdq, exact
    in the fp32 accumulator and in the 16-bit output, so the forward returns
    rows of Wdq^T and the input gradient rows of Wdq: the weight decoded
    inside the tensor-core pipeline equals the oracle's dequantized weight
    bit for bit, in both orientations."""
    N, K = 712, 1000                                   # ragged: 256-row tiles and 64-element blocks
    Wf = _weight(N, K, dtype, 21, std=0.05)
    packed, absmax, p_ref, a_ref = _check_quant(Wf, K)
    wdq = ON.dequantize(p_ref, a_ref, K, ODT[dtype])   # [N, K] storage of the oracle
    eye_k = torch.eye(K, dtype=dtype, device=DEV)
    ref = O.widen(wdq, ODT[dtype])                     # values: a zero level may come back as -0
    out = I.nf4_forward(eye_k, packed, absmax, K)      # [K, N] = Wdq^T
    assert np.array_equal(O.widen(to_np(out), ODT[dtype]), ref.T)
    eye_n = torch.eye(N, dtype=dtype, device=DEV)
    gA = I.nf4_backward_input(eye_n, packed, absmax, K)  # [N, K] = Wdq
    assert np.array_equal(O.widen(to_np(gA), ODT[dtype]), ref)


@pytest.mark.parametrize("M,K,N,dtype,bias_dtype", [(1, 8, 8, torch.bfloat16, None),          # smallest legal shape
                                                    (3, 8, 264, torch.float16, torch.float32),  # fp32 bias
                                                    (513, 72, 8, torch.bfloat16, torch.bfloat16)])
def test_small_and_edge_shapes(M, K, N, dtype, bias_dtype):
    Wf = _weight(N, K, dtype, 31)
    A = W.normal((M, K), 1.0, 32, dtype)
    G = W.normal((M, N), 1.0, 33, dtype)
    b = W.normal((N,), 0.1, 34, bias_dtype) if bias_dtype is not None else None
    packed, absmax, p_ref, a_ref = _check_quant(Wf, K)
    out = I.nf4_forward(A.to(DEV), packed, absmax, K, b.to(DEV) if b is not None else None)
    ref = ON.forward(to_np(A), ODT[dtype], p_ref, a_ref, K, to_np(b) if b is not None else None,
                     ODT[bias_dtype] if b is not None else None)
    assert_tol(O.widen(to_np(out), ODT[dtype]), ref["out64"], "nf4 forward")
    gA = I.nf4_backward_input(G.to(DEV), packed, absmax, K)
    rb = ON.backward_input(to_np(G), ODT[dtype], p_ref, a_ref, K)
    assert_tol(O.widen(to_np(gA), ODT[dtype]), rb["grad64"], "nf4 grad_A")
    assert torch.equal(I.nf4_forward(A.to(DEV), packed, absmax, K, b.to(DEV) if b is not None else None,
                                     materialized=True), out)
    assert torch.equal(I.nf4_backward_input(G.to(DEV), packed, absmax, K, materialized=True), gA)
