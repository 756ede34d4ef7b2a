"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer stages are compared bit for bit: the weight codes CB and scales SCB,
the outlier count and indices, the row scales SCA, the activation codes, the
gathered outlier columns subA / subB and the int32 accumulator.  The
dequantized output and the gradients are compared with the tolerance rule in
``_helpers.assert_tol``.  Small cases run the oracle on every element and
span several tiles, several exact-accumulation chunks and ragged tails; the
full-size workloads check sampled rows.
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

from _helpers import ODT, assert_tol, check_forward_stages, check_wdq, check_weight, gpu_forward, to_np, widen

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    torch.cuda.init()


def _layer(spec, seed, w_dtype=None):
    wl = W.Workload("case", "", (spec,), w_dtype=w_dtype or spec.dtype)
    A = W.activation(spec, seed)
    Wf, b, G = W.layer_tensors(wl, 0, seed)
    return A, Wf, b, G


def run_layer_case(spec, seed=0, rows=None, w_dtype=None, max_outliers=None):
    A, Wf, b, G = _layer(spec, seed, w_dtype)
    K = spec.K
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    g = gpu_forward(A.to(DEV), CB, SCB, K, b.to(DEV), spec.threshold, max_outliers=max_outliers)
    A_np = to_np(A)
    if rows is None:
        ref = O.forward(A_np, ODT[A.dtype], CB_ref, SCB_ref, to_np(b), ODT[b.dtype], spec.threshold)
    else:
        ref = O.forward_rows(A_np, ODT[A.dtype], CB_ref, SCB_ref, rows, to_np(b), ODT[b.dtype], spec.threshold)
    rep = check_forward_stages(g, ref, rows)
    if len(ref["idx"]):
        subB = to_np(g["subB"])[:, :len(ref["idx"])]
        subB_ref = O.dequant_weight(CB_ref, SCB_ref)[:, ref["idx"]]
        assert np.array_equal(subB.view(np.uint16), subB_ref.view(np.uint16))
    # backward to the input and the bias: the materialized schedule (its
    # dequantized weight checked bit for bit), then the fused one, which must
    # give the same bits
    Gd = G.to(DEV)
    ws_dq = I.functional.backward_workspace(spec.M, spec.N, G.dtype, DEV, K=K)
    gA, gb = I.backward_input(Gd, CB, SCB, K, bias_dtype=b.dtype, ws=ws_dq)
    if spec.M > 0:
        check_wdq(ws_dq, spec.M, spec.N, K, G.dtype, CB_ref, SCB_ref)
    del ws_dq
    gA_fused, _ = I.backward_input(Gd, CB, SCB, K, fused=True)
    assert torch.equal(gA_fused.view(torch.uint8), gA.view(torch.uint8)), "fused and materialized grad_A differ"
    del gA_fused, Gd
    rb = O.backward_input(to_np(G), ODT[G.dtype], CB_ref, SCB_ref, rows=rows)
    gA_sel = gA if rows is None else gA[torch.as_tensor(rows, device=DEV)]
    assert_tol(widen(gA_sel), rb["grad64"], "grad_A")
    gsum = np.zeros(spec.N)
    Gn = to_np(G)
    for r in range(0, spec.M, 2048):
        gsum += O.widen(Gn[r:r + 2048], ODT[G.dtype]).sum(0)
    assert_tol(widen(gb), gsum, "grad_bias")
    return g, ref, rep


SMALL = [
    # M, K, N, dtype, heavy fraction, heavy factor, threshold
    (300, 1100, 520, torch.float16, 0.01, 20.0, 6.0),      # 2 exact chunks, 3 x 3 tiles, ragged
    (129, 2112, 257, torch.bfloat16, 0.005, 10.0, 6.0),   # 3 chunks, ragged by one row / column
    (77, 72, 40, torch.float32, 0.0, 1.0, math.inf),      # fp32 input, no outliers
    (256, 4096, 512, torch.float16, 0.002, 15.0, 6.0),    # 4 full chunks, full tiles
    (5, 24, 12, torch.float16, 0.1, 20.0, 6.0),           # tiny, K not a multiple of 16
    (19, 13, 9, torch.float32, 0.0, 1.0, 6.0),            # K, N not multiples of 8 (scalar paths)
    (140, 200, 300, torch.bfloat16, 0.05, 10.0, 6.0),     # many outliers (4 outlier blocks)
    (600, 16, 4, torch.float32, 0.0, 1.0, math.inf),      # the tiny MLP's second layer shape
    # more tiles than CTA pairs in every GEMM: several tiles per pair (both
    # accumulators of the materialized backward, the fused one's single
    # accumulator handed from tile to tile, its split last round)
    (2100, 5120, 264, torch.float16, 0.002, 15.0, 6.0),
    # the longest rows of the one-launch quantization (1024 threads x 4
    # groups of 8) and one group longer, which takes the separate kernels;
    # the weight quantization meets the same boundary
    (200, 32768, 264, torch.float16, 0.001, 15.0, 6.0),
    (200, 32776, 264, torch.bfloat16, 0.001, 15.0, 6.0),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{str(c[3])[6:]}")
def test_layer_small(case):
    M, K, N, dt, hf, hx, thr = case
    spec = W.LayerSpec(M, K, N, dt, 0.02, 0.01, hf, hx, thr)
    run_layer_case(spec, seed=7)


@pytest.mark.parametrize("seed", range(3))
def test_layer_small_seeds(seed):
    """The pages ran every test 10 times for stability; different seeds
    here (ten in the slow run below)."""
    spec = W.LayerSpec(384, 1536, 768, torch.float16, 0.02, 0.01, 0.004, 20.0, 6.0)
    run_layer_case(spec, seed=100 + seed)


def test_exact_int32_beyond_fp32_range():
    """Constant rows make every product +-127^2: |Cacc| = K * 16129 far above
    2^24, where a single fp32 accumulator would round."""
    M, K, N = 130, 3000, 260
    A = torch.ones(M, K, dtype=torch.float16)
    A[1::2] *= -1.0
    A[7, :1500] = -1.0
    Wf = torch.full((N, K), 0.5, dtype=torch.float16)
    Wf[::3] *= -1.0
    g = torch.Generator().manual_seed(3)
    Wf[200:] = torch.where(torch.rand(N - 200, K, generator=g) < 0.5, -0.5, 0.5).half()
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    res = gpu_forward(A.to(DEV), CB, SCB, K, None, math.inf)
    ref = O.forward(to_np(A), O.F16, CB_ref, SCB_ref, threshold=math.inf)
    assert np.abs(ref["Cacc"]).max() == K * 16129 > 2 ** 24
    check_forward_stages(res, ref)


def _chunk_tile_max(codes, k_pad):
    """Per 256-row tile and 1024-column chunk, the largest sum of squared
    codes of one row of the tile in that chunk (zero padding past K)."""
    R, Kc = codes.shape
    q = np.zeros((R, k_pad), np.int64)
    q[:, :Kc] = codes
    nch = (k_pad + 1023) // 1024
    sq = np.stack([(q[:, c * 1024:(c + 1) * 1024] ** 2).sum(1) for c in range(nch)], 1)
    return np.stack([sq[t:t + 256].max(0) for t in range(0, R, 256)])


def _plan(asq, bsq):
    """The accumulation plan by its definition: per tile pair, the largest
    L such that every group of L consecutive chunks (the last one ragged)
    has sum(asq) * sum(bsq) < 2^48, and the fast-conversion bit when every
    such group stays below 2^44."""
    nch = asq.shape[1]
    plan = np.zeros((asq.shape[0], bsq.shape[0]), np.int64)
    for i in range(asq.shape[0]):
        for j in range(bsq.shape[0]):
            for L in range(nch, 0, -1):
                p = [int(asq[i, c:c + L].sum()) * int(bsq[j, c:c + L].sum()) for c in range(0, nch, L)]
                if all(x < 2 ** 48 for x in p) or L == 1:
                    plan[i, j] = L | ((1 << 16) if all(x < 2 ** 44 for x in p) else 0)
                    break
    return plan


def test_accumulation_plan():
    """The GEMM accumulates exactly in fp32 over groups of 1024-deep chunks
    chosen per tile pair from the chunk sums of squared codes (Cauchy-Schwarz
    bounds every partial sum below 2^24).  Row tiles of saturated, ordinary
    and small codes against weight tiles of the same kinds give groups of one
    chunk, of all chunks and in between, fast and slow conversions; the chunk
    maxima and the plan equal their definitions on the oracle's codes and the
    int32 accumulator is exact for every tile pair."""
    M, K, N = 700, 5000, 600
    g = torch.Generator().manual_seed(29)
    A = torch.randn(M, K, generator=g).half()
    A[:256] = 1.0                                   # tile 0: every code 127
    A[512:] = (torch.rand(M - 512, K, generator=g) < 0.01).half() * torch.randn(M - 512, K, generator=g).half()
    Wf = (torch.randn(N, K, generator=g) * 0.02).half()
    Wf[:256] = 0.25                                 # weight tile 0: every code 127
    Wf[512:] = Wf[512:] * (torch.rand(N - 512, K, generator=g) < 0.02).half()
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    res = gpu_forward(A.to(DEV), CB, SCB, K, None, math.inf)
    ref = O.forward(to_np(A), O.F16, CB_ref, SCB_ref, threshold=math.inf)
    check_forward_stages(res, ref)
    k_pad = res["k_pad"]
    asq = _chunk_tile_max(ref["Aq"].astype(np.int64), k_pad)
    bsq = _chunk_tile_max(CB_ref.astype(np.int64), k_pad)
    assert np.array_equal(to_np(res["asq"]).astype(np.int64), asq)
    assert np.array_equal(to_np(res["bsq"]).astype(np.int64), bsq)
    plan = _plan(asq, bsq)
    assert np.array_equal(to_np(res["plan"]).astype(np.int64), plan)
    L, fast = plan & 0xFFFF, plan >> 16
    nch = asq.shape[1]
    assert L.min() == 1 and L.max() == nch and ((L > 1) & (L < nch)).any()
    assert fast.any() and (fast == 0).any()


def test_accumulation_plan_with_outliers():
    """The same mix of accumulation plans with outlier columns.  A tile whose
    int8 reduction is one unit keeps it in the fp32 columns while the outlier
    unit accumulates in the running-sum columns; the other tiles drain between
    their units.  Both kinds run in one launch, with the running-sum columns
    handed between them tile after tile: the int32 accumulator stays exact and
    the output within tolerance."""
    M, K, N = 700, 5000, 600
    g = torch.Generator().manual_seed(31)
    A = torch.randn(M, K, generator=g)
    A[:256] = 1.0                                   # tile 0: every code 127
    A[512:] = (torch.rand(M - 512, K, generator=g) < 0.01) * torch.randn(M - 512, K, generator=g)
    heavy = torch.randperm(K, generator=g)[:6]
    A[:, heavy] *= 20.0                             # outlier columns in every row tile
    A = A.half()
    Wf = (torch.randn(N, K, generator=g) * 0.02).half()
    Wf[:256] = 0.25                                 # weight tile 0: every code 127
    Wf[512:] = Wf[512:] * (torch.rand(N - 512, K, generator=g) < 0.02).half()
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    res = gpu_forward(A.to(DEV), CB, SCB, K, None, 6.0)
    ref = O.forward(to_np(A), O.F16, CB_ref, SCB_ref, threshold=6.0)
    check_forward_stages(res, ref)
    assert len(ref["idx"]) >= 6
    plan = to_np(res["plan"]).astype(np.int64)
    L = plan & 0xFFFF
    nch = (res["k_pad"] + 1023) // 1024
    assert (L >= nch).any() and (L < nch).any()


def test_max_k_accumulator():
    """K at the int32 bound: every product +127^2, |Cacc| = 2147479576."""
    M, K, N = 128, _lib.I8LT_MAX_K, 256
    A = torch.full((M, K), 0.25, dtype=torch.float16, device=DEV)
    Wf = torch.full((N, K), 0.25, dtype=torch.float16, device=DEV)
    Wf[1::2] = -0.25
    CB, SCB = I.quantize_weight(Wf)
    acc = torch.empty(M, N, dtype=torch.int32, device=DEV)
    out, ws = I.forward(A, CB, SCB, K, None, math.inf, acc_i32=acc)
    st, _ = I.device_status(ws)
    assert st == 0
    want = torch.full((N,), K * 16129, dtype=torch.int64)
    want[1::2] *= -1
    assert torch.equal(acc.cpu().long(), want.expand(M, N))
    # out = Cacc * 0.25 * 0.25 / 127^2 = +-K / 16 (finite in fp16)
    assert torch.allclose(out.float().cpu(), want.float().expand(M, N) / 16129 / 16, rtol=1e-3)


def test_empty_batch():
    K, N = 64, 32
    Wf = torch.randn(N, K, dtype=torch.float16, device=DEV)
    CB, SCB = I.quantize_weight(Wf)
    out, ws = I.forward(torch.empty(0, K, dtype=torch.float16, device=DEV), CB, SCB, K, None, 6.0)
    assert out.shape == (0, N)
    gA, gb = I.backward_input(torch.empty(0, N, dtype=torch.float16, device=DEV), CB, SCB, K,
                              bias_dtype=torch.float16)
    assert gA.shape == (0, K)
    assert torch.count_nonzero(gb).item() == 0


def test_outlier_capacity_reported():
    M, K, N = 64, 256, 64
    A = torch.randn(M, K, dtype=torch.float16, device=DEV) * 10        # nearly every column > 1
    Wf = torch.randn(N, K, dtype=torch.float16, device=DEV)
    CB, SCB = I.quantize_weight(Wf)
    out, ws = I.forward(A, CB, SCB, K, None, 1.0, max_outliers=8)
    st, found = I.device_status(ws)
    assert st == _lib.I8LT_ERR_OUTLIER_CAPACITY and found > 8
    st2, _ = I.device_status(ws)          # reading clears it
    assert st2 == 0
    out, ws = I.forward(A, CB, SCB, K, None, 1.0, max_outliers=K)
    assert I.device_status(ws)[0] == 0


def test_residual_and_addend():
    """The fused residual (forward) and addend (backward) equal the oracle's
    single-rounding definitions."""
    M, K, N = 200, 320, 160
    spec = W.LayerSpec(M, K, N, torch.float16, 0.02, 0.01, 0.01, 20.0, 6.0)
    A, Wf, b, G = _layer(spec, 21)
    R = W.normal((M, N), 1.0, 99, torch.float16)
    D = W.normal((M, K), 1.0, 98, torch.float16)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
    g = gpu_forward(A.to(DEV), CB, SCB, K, b.to(DEV), 6.0, residual=R.to(DEV))
    ref = O.forward(to_np(A), O.F16, CB_ref, SCB_ref, to_np(b), O.F16, 6.0, residual=to_np(R))
    check_forward_stages(g, ref)
    gA, _ = I.backward_input(G.to(DEV), CB, SCB, K, addend=D.to(DEV))
    rb = O.backward_input(to_np(G), O.F16, CB_ref, SCB_ref, addend=to_np(D))
    assert_tol(widen(gA), rb["grad64"], "grad_A + addend")


def test_repeat_calls_identical():
    """Same inputs twice (reused workspace): identical bits (no state leaks
    between calls, deterministic reductions)."""
    spec = W.LayerSpec(300, 1100, 520, torch.float16, 0.02, 0.01, 0.01, 20.0, 6.0)
    A, Wf, b, G = _layer(spec, 5)
    A, b, G = A.to(DEV), b.to(DEV), G.to(DEV)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    o1, ws = I.forward(A, CB, SCB, spec.K, b, 6.0)
    o1 = o1.clone()
    o2, _ = I.forward(A, CB, SCB, spec.K, b, 6.0, ws=ws)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    g1, b1 = I.backward_input(G, CB, SCB, spec.K, bias_dtype=b.dtype)
    g2, b2 = I.backward_input(G, CB, SCB, spec.K, bias_dtype=b.dtype)
    assert torch.equal(g1.view(torch.int16), g2.view(torch.int16))
    assert torch.equal(b1.view(torch.int16), b2.view(torch.int16))


@pytest.mark.parametrize("M,N,K,runs", [(4096, 11008, 4096, 12), (8192, 4096, 11008, 12), (16384, 28672, 8192, 20)])
def test_fused_backward_repeats_bit_identical(M, N, K, runs):
    """The odd CTA of a pair hands its converted weight tiles to the even
    CTA's MMA through a cluster-scope release, on the same barrier that the G
    copies complete on.  A hand-over that ordered less would let a stage be
    read before its tile is complete, which shows as runs that differ.
    Repeated runs over several rounds of pair tiles, up to the projection
    workload's first layer, must give the same bytes."""
    g = torch.Generator().manual_seed(7)
    G = torch.randn(M, N, generator=g).half().to(DEV)
    Wf = (torch.randn(N, K, generator=g) * 0.02).half().to(DEV)
    CB, SCB = I.quantize_weight(Wf)
    ref, ref_b = I.backward_input(G, CB, SCB, K, bias_dtype=torch.float16, fused=True)
    ref, ref_b = ref.clone(), ref_b.clone()
    for _ in range(runs - 1):
        gA, gb = I.backward_input(G, CB, SCB, K, bias_dtype=torch.float16, fused=True)
        assert torch.equal(gA.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(gb.view(torch.int16), ref_b.view(torch.int16))


def test_forward_repeats_bit_identical():
    """The forward hands the running-sum columns from one tile's stores to the
    next tile's outlier unit through a barrier of its own.  Repeated forwards
    of the projection workload's first layer (one-unit tiles with outlier
    columns, many tiles per pair) must give the same bytes."""
    spec = W.WORKLOADS["proj_8192x28672"].layers[0]
    wl = W.Workload("case", "", (spec,), w_dtype=spec.dtype)
    A = W.activation(spec, 3).to(DEV)
    Wf, b, _ = W.layer_tensors(wl, 0, 3)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    b = b.to(DEV)
    o0, ws = I.forward(A, CB, SCB, spec.K, b, spec.threshold)
    o0 = o0.clone()
    for _ in range(9):
        o, _ = I.forward(A, CB, SCB, spec.K, b, spec.threshold, ws=ws)
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16))


# ---------------------------------------------------------------------------
# the workloads
# ---------------------------------------------------------------------------

def _rows(M, n=40, seed=0):
    g = np.random.default_rng(seed)
    r = set(g.choice(M, size=min(n, M), replace=False).tolist())
    r |= {0, min(1, M - 1), min(127, M - 1), min(128, M - 1), M - 1}
    return np.array(sorted(r))


# every config over 10 seeds (the pages run their tests 10 times for
# stability), the 16384-token projection over 2 (its oracle rows are sampled)
WORKLOAD_SEEDS = ([("linear_4096", s) for s in range(10)] + [("linear_bf16_4096x11008", s) for s in range(10)]
                  + [("proj_8192x28672", s) for s in range(2)])


@pytest.mark.parametrize("name,base", WORKLOAD_SEEDS, ids=lambda v: str(v))
def test_workload_layers(name, base):
    wl = W.WORKLOADS[name]
    for li, spec in enumerate(wl.layers):
        seed = base + li * W.OFF_LAYER2
        A = W.activation(spec, seed)
        Wf, b, G = W.layer_tensors(wl, li, base)
        K = spec.K
        CB, SCB = I.quantize_weight(Wf.to(DEV))
        CB_ref, SCB_ref = check_weight(CB, SCB, Wf, K)
        del Wf
        g = gpu_forward(A.to(DEV), CB, SCB, K, b.to(DEV), spec.threshold)
        rows = _rows(spec.M, seed=li + 7 * base)
        ref = O.forward_rows(to_np(A), ODT[A.dtype], CB_ref, SCB_ref, rows, to_np(b), ODT[b.dtype],
                             spec.threshold)
        heavy = W.heavy_columns(K, spec.heavy_frac, seed + W.OFF_HEAVY).numpy()
        assert set(heavy.tolist()) <= set(ref["idx"].tolist())
        check_forward_stages(g, ref, rows)
        del g
        gA, gb = I.backward_input(G.to(DEV), CB, SCB, K, bias_dtype=b.dtype)
        rb = O.backward_input(to_np(G), ODT[G.dtype], CB_ref, SCB_ref, rows=rows)
        assert_tol(widen(gA[torch.as_tensor(rows, device=DEV)]), rb["grad64"], f"{name} L{li} grad_A")
        Gn = to_np(G)
        gsum = np.zeros(spec.N)
        for r in range(0, spec.M, 2048):
            gsum += O.widen(Gn[r:r + 2048], ODT[G.dtype]).sum(0)
        assert_tol(widen(gb), gsum, f"{name} L{li} grad_bias")
        del gA, gb, CB, SCB
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name,base", [("tiny_mlp", s) for s in range(10)] + [("mlp_7b", s) for s in range(2)],
                         ids=lambda v: str(v))
def test_workload_mlp(name, base):
    """The chained MLPs: every layer checked against the oracle fed with the
    same input the GPU layer saw (so integer stages stay bit-exact); the
    whole chain against the oracle chain within the tolerance."""
    wl = W.WORKLOADS[name]
    s1, s2 = wl.layers
    x = W.layer_input(wl, 0, base)
    W1, b1, _ = W.layer_tensors(wl, 0, base)
    W2, b2, G = W.layer_tensors(wl, 1, base)
    dt = ODT[x.dtype]
    thr = s1.threshold
    CB1, SCB1 = I.quantize_weight(W1.to(DEV))
    CB2, SCB2 = I.quantize_weight(W2.to(DEV))
    CB1r, SCB1r = check_weight(CB1, SCB1, W1, s1.K)
    CB2r, SCB2r = check_weight(CB2, SCB2, W2, s2.K)
    full = s1.M <= 4096
    rows = None if full else _rows(s1.M, seed=3 + base)
    rsel = (lambda t: t) if full else (lambda t: t[torch.as_tensor(rows, device=DEV)])
    fwd = O.forward if full else (lambda *a, **k: O.forward_rows(a[0], a[1], a[2], a[3], rows, *a[4:], **k))
    xd = x.to(DEV)
    # layer 1
    g1 = gpu_forward(xd, CB1, SCB1, s1.K, b1.to(DEV), thr)
    r1 = fwd(to_np(x), dt, CB1r, SCB1r, to_np(b1), ODT[b1.dtype], thr)
    check_forward_stages(g1, r1, rows)
    h = g1["out"]
    a = I.silu(h)
    assert_tol(widen(rsel(a)), O.widen(O.silu(to_np(rsel(h)), dt), dt), "silu")
    # layer 2 (+ residual x for the tiny MLP)
    res = xd if wl.residual else None
    g2 = gpu_forward(a, CB2, SCB2, s2.K, b2.to(DEV), thr, residual=res)
    r2 = fwd(to_np(a), dt, CB2r, SCB2r, to_np(b2), ODT[b2.dtype], thr,
             residual=to_np(x) if wl.residual else None) if full else O.forward_rows(
        to_np(a), dt, CB2r, SCB2r, rows, to_np(b2), ODT[b2.dtype], thr,
        residual=to_np(x)[rows] if wl.residual else None)
    check_forward_stages(g2, r2, rows)
    # backward chain
    Gd = G.to(DEV)
    ga, gb2 = I.backward_input(Gd, CB2, SCB2, s2.K, bias_dtype=b2.dtype)
    rb2 = O.backward_input(to_np(G), dt, CB2r, SCB2r, rows=rows)
    assert_tol(widen(rsel(ga)), rb2["grad64"], "grad a")
    gh = I.silu_backward(ga, h)
    assert_tol(widen(rsel(gh)), O.widen(O.silu_backward(to_np(rsel(ga)), to_np(rsel(h)), dt), dt), "grad h")
    gx, gb1 = I.backward_input(gh, CB1, SCB1, s1.K, bias_dtype=b1.dtype, addend=Gd if wl.residual else None)
    rb1 = O.backward_input(to_np(gh), dt, CB1r, SCB1r, addend=to_np(G) if wl.residual else None, rows=rows)
    assert_tol(widen(rsel(gx)), rb1["grad64"], "grad x")
    if full:
        # end to end: the oracle chain fed with x only
        e1 = O.forward(to_np(x), dt, CB1r, SCB1r, to_np(b1), ODT[b1.dtype], thr)
        ea = O.silu(e1["out"], dt)
        e2 = O.forward(ea, dt, CB2r, SCB2r, to_np(b2), ODT[b2.dtype], thr,
                       residual=to_np(x) if wl.residual else None)
        assert_tol(widen(g2["out"]), e2["out64"], "mlp out end to end")
        # the autograd module path runs the same kernels: identical bits
        fc1 = I.Linear8bitLt(s1.K, s1.N, threshold=thr, device=DEV, bias_dtype=b1.dtype)
        fc2 = I.Linear8bitLt(s2.K, s2.N, threshold=thr, device=DEV, bias_dtype=b2.dtype)
        for fc, CB, SCB, bb in ((fc1, CB1, SCB1, b1), (fc2, CB2, SCB2, b2)):
            fc.CB.copy_(CB)
            fc.SCB.copy_(SCB)
            with torch.no_grad():
                fc.bias.copy_(bb.to(DEV))
        mlp = I.Int8MLP(fc1, fc2, residual=wl.residual)
        for fused in (False, True):          # SiLU as its own pass, or in fc1's epilogue
            I.functional.FUSED_SILU = fused
            try:
                xr = xd.clone().requires_grad_(True)
                fc1.bias.grad = fc2.bias.grad = None
                y = mlp(xr)
                y.backward(Gd)
            finally:
                I.functional.FUSED_SILU = False
            assert torch.equal(y.detach(), g2["out"])
            assert torch.equal(xr.grad, gx)
            assert torch.equal(fc1.bias.grad, gb1) and torch.equal(fc2.bias.grad, gb2)


@pytest.mark.parametrize("M,K,H,N2,dtype,thr", [(300, 256, 1100, 256, torch.float16, 6.0),
                                                (129, 512, 640, 200, torch.bfloat16, 6.0),
                                                (600, 4, 16, 4, torch.float32, math.inf)])
def test_fused_silu_epilogue_matches_the_unfused_chain(M, K, H, N2, dtype, thr):
    """MLP hidden layer: i8lt_forward_silu's h and silu(h) equal i8lt_forward
    followed by i8lt_silu_forward bit for bit, its column maxima equal
    i8lt_forward_colmax on silu(h), and the next layer run from them equals
    the next layer run on its own."""
    s1 = W.LayerSpec(M, K, H, dtype, 0.05, 0.01, 0.01, 12.0, thr)
    s2 = W.LayerSpec(M, H, N2, dtype, 0.05, 0.01, 0.0, 1.0, thr)
    wl = W.Workload("mlp", "", (s1, s2), kind="mlp", w_dtype=dtype)
    x = W.activation(s1, 21).to(DEV)
    W1, b1, _ = W.layer_tensors(wl, 0, 21)
    W2, b2, _ = W.layer_tensors(wl, 1, 21)
    CB1, SCB1 = I.quantize_weight(W1.to(DEV))
    CB2, SCB2 = I.quantize_weight(W2.to(DEV))
    b1, b2 = b1.to(DEV), b2.to(DEV)
    F = I.functional
    h_ref, _ = I.forward(x, CB1, SCB1, K, b1, thr)
    a_ref = F.silu(h_ref)
    y_ref, _ = I.forward(a_ref, CB2, SCB2, H, b2, thr)
    ws2 = F.forward_workspace(M, H, N2, F._capacity(H, thr, None), x.device)
    colmax = F.colmax_region(ws2, M, H, N2, thr)
    h, a, _ = F.forward_silu(x, CB1, SCB1, K, b1, thr, act_colmax=colmax)
    assert torch.equal(h.view(torch.uint8), h_ref.view(torch.uint8))
    assert torch.equal(a.view(torch.uint8), a_ref.view(torch.uint8))
    ws_chk = F.forward_workspace(M, H, N2, F._capacity(H, thr, None), x.device)
    assert _lib.i8lt_forward_colmax(a.data_ptr(), F.DTYPE_CODE[dtype], M, H, N2, ws_chk.data_ptr(), ws_chk.numel(),
                                    F._capacity(H, thr, None), torch.cuda.current_stream().cuda_stream) == 0
    assert torch.equal(colmax, F.colmax_region(ws_chk, M, H, N2, thr))
    y, _ = I.forward(a, CB2, SCB2, H, b2, thr, ws=ws2, colmax_ready=True)
    assert torch.equal(y.view(torch.uint8), y_ref.view(torch.uint8))


@pytest.mark.parametrize("M,K,N", [(300, 1100, 520),      # ragged chunks of 128 tokens, ragged 64-wide blocks
                                   (1000, 256, 4104),     # one output row tile: every block owned by it
                                   (129, 9000, 200),      # more row tiles than reduction blocks
                                   (2048, 4096, 4096)])   # the fp16 single-layer workload's shape
def test_grad_bias_in_gemm_equals_the_prepass(M, K, N):
    """fp16 grad_output: the backward GEMM reduces grad_bias itself (its
    epilogue warps sum the uncast G in 128-token chunks while the tensor
    cores run) and no prepass reads G.  Both schedules must give the bits
    of the prepass path (taken when grad_A is not requested), which sums in
    the same order, and the result must match the oracle."""
    spec = W.LayerSpec(M, K, N, torch.float16, 0.02, 0.01)
    A, Wf, b, G = _layer(spec, 61)
    Gd = G.to(DEV)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    _lib.i8lt_profile_start(64)
    gA_f, gb_f = I.backward_input(Gd, CB, SCB, K, bias_dtype=torch.float32, fused=True)
    torch.cuda.synchronize()
    _, recs, _ = _lib.i8lt_profile_stop(64)
    names = [n for n, _ in recs]
    assert "gradout_prepass" not in names and names == ["bwd_gemm", "grad_bias_finalize"], names
    _, gb_m = I.backward_input(Gd, CB, SCB, K, bias_dtype=torch.float32, fused=False)
    _lib.i8lt_profile_start(64)
    _, gb_p = I.backward_input(Gd, CB, SCB, K, need_grad_A=False, bias_dtype=torch.float32)
    torch.cuda.synchronize()
    _, recs, _ = _lib.i8lt_profile_stop(64)
    assert [n for n, _ in recs] == ["gradout_prepass", "grad_bias_finalize"]
    assert torch.equal(gb_f.view(torch.int32), gb_p.view(torch.int32)), "in-GEMM grad_bias differs from the prepass"
    assert torch.equal(gb_m.view(torch.int32), gb_p.view(torch.int32))
    Gn = to_np(G)
    assert_tol(widen(gb_f), O.widen(Gn, O.F16).sum(0), "grad_bias")
    # fp32 sums of fp16 values in 128-row chunks: far inside the tolerance
    assert np.abs(widen(gb_f) - O.widen(Gn, O.F16).sum(0)).max() < 1e-3
