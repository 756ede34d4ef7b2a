"""GPU parity on the method's degenerate and exact cases, through the C ABI.

The oracle pins these cases on the CPU (tests/test_oracle.py); here the CUDA
path runs them and is compared with the oracle:

* all-zero activation rows: scale 0, codes 0, no NaN (reading: an all-zero
  row has scale 0);
* rows whose only nonzero values sit in outlier columns: the row scale taken
  outside those columns is 0 (bitsandbytes PR #33, "Mixed-precision
  decomposition matmul": the outlier columns leave the int8 product);
* all-zero weight rows: SCB = 0, codes 0, the dequantized weight row is 0;
* exact half-way ties of x * (127 / absmax), which round half to even
  (the rounding reading of the vector-wise quantization);
* the lossless case: activations, weights, bias, residual and grad_output on
  a grid where quantization loses nothing and every fp32 partial sum of the
  kernels is exact.  The outputs and both gradients must then equal the
  oracle's bit for bit, not only within the tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300.build import build

from _helpers import ODT, assert_tol, check_forward_stages, check_weight, gpu_forward, to_np, widen

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    torch.cuda.init()


def _bits(t: torch.Tensor) -> np.ndarray:
    a = to_np(t)
    return a.view(np.uint16) if a.dtype.itemsize == 2 else a.view(np.uint32)


def _backward_both(G, CB, SCB, K, bias_dtype):
    """grad_A and grad_bias through the materialized schedule, and grad_A
    through the fused one (which must give the same bits)."""
    ws_dq = I.functional.backward_workspace(G.shape[0], G.shape[1], G.dtype, DEV, K=K)
    gA, gb = I.backward_input(G, CB, SCB, K, bias_dtype=bias_dtype, ws=ws_dq)
    gA_f, gb_f = I.backward_input(G, CB, SCB, K, bias_dtype=bias_dtype, fused=True)
    assert torch.equal(gA.view(torch.uint8), gA_f.view(torch.uint8)), "fused and materialized grad_A differ"
    assert torch.equal(gb.view(torch.uint8), gb_f.view(torch.uint8))
    return gA, gb


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_zero_rows_outlier_only_rows_and_zero_weight_rows(dtype):
    """Degenerate rows on both sides of the product, in one batch that spans
    several tiles with ragged edges and holds outlier columns."""
    M, K, N = 300, 4096, 520
    # the heavy-column recipes of the fp16 and bf16 workloads at their K (bf16
    # keeps 8 significant bits, so the output's own rounding, 2^-9 relative,
    # stays inside 0.02 mean|ref| only while the largest outputs are within
    # about 10x the mean, as in the workloads)
    hf, hx = (0.001, 20.0) if dtype == torch.float16 else (0.005, 10.0)
    spec = W.LayerSpec(M, K, N, dtype, 0.02, 0.01, hf, hx, 6.0)
    wl = W.Workload("edge", "", (spec,), w_dtype=dtype)
    A = W.activation(spec, 41)
    Wf, b, G = W.layer_tensors(wl, 0, 41)
    heavy = W.heavy_columns(K, spec.heavy_frac, 41 + W.OFF_HEAVY)
    zero_rows = [0, 5, 255, 256, 299]
    only_outlier_rows = [7, 150, 257]
    zero_w_rows = [0, 3, 255, 258, 519]
    A[zero_rows] = 0.0
    keep = torch.zeros(K, dtype=torch.bool)
    keep[heavy] = True
    A[only_outlier_rows] = torch.where(keep, A[only_outlier_rows], torch.zeros((), dtype=dtype))
    Wf[zero_w_rows] = 0.0
    G[zero_rows] = 0.0

    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    assert np.all(SCB_ref[zero_w_rows] == 0) and not np.any(CB_ref[zero_w_rows])
    g = gpu_forward(A.to(DEV), CB, SCB, K, b.to(DEV), 6.0)
    ref = O.forward(to_np(A), ODT[dtype], CB_ref, SCB_ref, to_np(b), ODT[b.dtype], 6.0)
    assert set(heavy.tolist()) <= set(ref["idx"].tolist())
    check_forward_stages(g, ref)
    sca = to_np(g["SCA"])
    assert np.all(sca[zero_rows] == 0) and np.all(sca[only_outlier_rows] == 0)
    aq = to_np(g["Aq"]).astype(np.float32)
    assert not np.any(aq[zero_rows]) and not np.any(aq[only_outlier_rows])
    assert np.all(np.isfinite(widen(g["out"])))
    # a zero row gives exactly the bias; a zero weight row exactly the bias
    # plus nothing (its dequantized row, and so its outlier weights, are 0)
    ob, rb = _bits(g["out"]), ref["out"].view(np.uint16)
    assert np.array_equal(ob[zero_rows], rb[zero_rows])
    assert np.array_equal(ob[:, zero_w_rows], rb[:, zero_w_rows])
    subB = to_np(g["subB"])[:, :len(ref["idx"])].astype(np.float32)
    assert not np.any(subB[zero_w_rows])

    gA, gb = _backward_both(G.to(DEV), CB, SCB, K, b.dtype)
    rbk = O.backward_input(to_np(G), ODT[dtype], CB_ref, SCB_ref)
    assert_tol(widen(gA), rbk["grad64"], "grad_A")
    assert not np.any(widen(gA)[zero_rows]), "zero grad_output rows must give zero grad_A rows"
    assert_tol(widen(gb), O.widen(to_np(G), ODT[dtype]).sum(0), "grad_bias")


def _tie_matrix(rows, K, seed, unit, heavy_col=None, heavy_val=None):
    """fp16-exact rows whose absmax is 127 * 2^j * unit (j = 1, 2; unit a
    power of two) and whose other values are (2i + 1) * 2^(j-1) * unit:
    x * (127 / absmax) = x / (2^j unit) lands exactly half-way between two
    integers."""
    g = torch.Generator().manual_seed(seed)
    A = torch.empty(rows, K, dtype=torch.float64)
    for r in range(rows):
        j = 1 + (r % 2)
        half = 2.0 ** (j - 1)
        odd = torch.randint(-127, 127, (K,), generator=g).double() * 2 + 1      # odd in [-253, 253]
        A[r] = odd * half
        A[r, int(torch.randint(K, (1,), generator=g))] = (127 * 2 ** j) * (1 if r % 3 else -1)
    A *= unit
    if heavy_col is not None:
        A[:, heavy_col] = heavy_val
    return A


@pytest.mark.parametrize("K", [700, 704])    # rows of a multiple of 8 columns: the one-launch quantization
@pytest.mark.parametrize("threshold", [math.inf, 9.0])
def test_round_half_even_ties(threshold, K):
    """Every activation and weight code is an exact .5 tie (except the
    absmax elements): the codes must round half to even on both sides.
    (Activations up to 508 / 64 < 9, weights up to 508 / 4096: the outputs
    stay finite in fp16.)"""
    M, N = 260, 300
    heavy = 11 if math.isfinite(threshold) else None
    A64 = _tie_matrix(M, K, 3, 2.0 ** -6, heavy, 15.5)
    W64 = _tie_matrix(N, K, 4, 2.0 ** -12)
    A, Wf = A64.half(), W64.half()
    assert torch.equal(A.double(), A64) and torch.equal(Wf.double(), W64)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    # the weight codes: the ties broke toward the even integer
    y = W64.numpy() / (SCB_ref.astype(np.float64)[:, None] / 127.0)
    ties = np.abs(y - np.trunc(y)) == 0.5
    assert ties.mean() > 0.99
    assert np.all(CB_ref[ties].astype(np.int64) % 2 == 0)
    g = gpu_forward(A.to(DEV), CB, SCB, K, None, threshold)
    ref = O.forward(to_np(A), O.F16, CB_ref, SCB_ref, threshold=threshold)
    assert ref["idx"].tolist() == ([] if heavy is None else [heavy])
    check_forward_stages(g, ref)
    aq = ref["Aq"].astype(np.int64)
    xa = A64.numpy() / (ref["SCA"].astype(np.float64)[:, None] / 127.0)
    ta = np.abs(xa - np.trunc(xa)) == 0.5
    assert ta.mean() > 0.98 and np.all(aq[ta] % 2 == 0)


def _lossless_inputs(M, K, N, outliers, dtype, seed):
    """Inputs on which the layer is exact on the GPU too.

    ua in 2^-7 .. 2^-5, uw in 2^-10 .. 2^-8, K <= 640, at most 4 outlier
    columns of magnitude <= 22, bias k * 2^-7 with |k| <= 127, residual
    k * 2^-6 with |k| <= 255, grad_output k * 2^-3 with |k| <= 31.  Then
    every term of an output is a multiple of ua * uw, and the bound below
    keeps every fp32 partial sum of the int8 unit, the outlier unit and the
    epilogue under 2^24 such multiples, so each is exact; the same holds for
    the backward (multiples of uw / 8) and the bias gradient (of 2^-3).
    """
    assert K <= 640 and len(outliers) <= 4
    case = W.lossless_case(M, K, N, seed=seed, outlier_cols=outliers, threshold=6.0, ea_range=(-7, -4),
                           ew_range=(-10, -7))
    A64, W64 = case["A"].double(), case["W"].double()
    bias64 = W.grid_values((N,), 127, -7, seed + 1)
    res64 = W.grid_values((M, N), 255, -6, seed + 2)
    G64 = W.grid_values((M, N), 31, -3, seed + 3)
    ua, uw = case["ua"], case["uw"]
    gran = ua[:, None] * uw[None, :]
    bound = (K * 127 * 127 * gran + (A64[:, list(outliers)].abs() @ W64[:, list(outliers)].abs().T)
             + bias64.abs()[None, :] + res64.abs())
    assert bool((bound < 2.0 ** 24 * gran).all())
    gbound = G64.abs() @ W64.abs()
    assert bool((gbound < 2.0 ** 24 * (uw.min() / 8)).all())
    cast = lambda t: t.to(dtype)  # noqa: E731  (exact: every value is on the grid of both 16-bit types)
    for t in (A64, W64, bias64, res64, G64):
        assert torch.equal(cast(t).double(), t)
    return case, cast(A64), cast(W64), cast(bias64), cast(res64), cast(G64)


@pytest.mark.parametrize("outliers", [(), (3,), (0, 17, 400, 639)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_lossless_layer_is_bit_exact(outliers, dtype):
    """The lossless case with bias and residual, over 2 x 3 output tiles with
    ragged edges: out, grad_A and grad_bias equal the oracle bit for bit,
    and the oracle equals the fp64 product of the grid values."""
    M, K, N = 300, 640, 520
    case, A, Wf, bias, res, G = _lossless_inputs(M, K, N, outliers, dtype, 17)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    assert np.array_equal(CB_ref, case["qw"].numpy().astype(np.int8))
    g = gpu_forward(A.to(DEV), CB, SCB, K, bias.to(DEV), 6.0, residual=res.to(DEV))
    dt = ODT[dtype]
    ref = O.forward(to_np(A), dt, CB_ref, SCB_ref, to_np(bias), dt, 6.0, residual=to_np(res))
    assert ref["idx"].tolist() == sorted(outliers)
    exact = A.double().numpy() @ Wf.double().numpy().T + bias.double().numpy()[None, :] + res.double().numpy()
    assert np.array_equal(ref["out64"], exact)
    check_forward_stages(g, ref, out_tol=False)   # the output is checked bit for bit below
    assert np.array_equal(_bits(g["out"]), ref["out"].view(np.uint16)), "lossless forward not bit-exact"

    gA, gb = _backward_both(G.to(DEV), CB, SCB, K, dtype)
    rb = O.backward_input(to_np(G), dt, CB_ref, SCB_ref)
    assert np.array_equal(rb["grad64"], G.double().numpy() @ Wf.double().numpy())
    assert np.array_equal(_bits(gA), rb["grad_A"].view(np.uint16)), "lossless grad_A not bit-exact"
    assert np.array_equal(_bits(gb), O.grad_bias(to_np(G), dt, dt).view(np.uint16)), "grad_bias not bit-exact"


def test_lossless_tiny_mlp_shapes_fp32():
    """The lossless case at the tiny MLP's layer shapes with fp32 input and
    output (K = 4 and 16, N = 16 and 4, below one tile and below one 16-byte
    row of codes): bit-exact output, grad_A and grad_bias."""
    for (M, K, N) in ((600, 4, 16), (600, 16, 4)):
        case, A, Wf, bias, res, G = _lossless_inputs(M, K, N, (), torch.float32, 23)
        CB, SCB = I.quantize_weight(Wf.to(DEV))
        CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
        g = gpu_forward(A.to(DEV), CB, SCB, K, bias.to(DEV), math.inf, residual=res.to(DEV))
        ref = O.forward(to_np(A), O.F32, CB_ref, SCB_ref, to_np(bias), O.F32, math.inf, residual=to_np(res))
        check_forward_stages(g, ref, out_tol=False)
        assert np.array_equal(to_np(g["out"]).view(np.uint32), ref["out"].view(np.uint32))
        gA, gb = _backward_both(G.to(DEV), CB, SCB, K, torch.float32)
        rb = O.backward_input(to_np(G), O.F32, CB_ref, SCB_ref)
        assert np.array_equal(to_np(gA).view(np.uint32), rb["grad_A"].view(np.uint32))
        assert np.array_equal(to_np(gb).view(np.uint32), O.grad_bias(to_np(G), O.F32, O.F32).view(np.uint32))
