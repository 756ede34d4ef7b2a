"""Pins of the NF4 oracle (CPU only): each test checks a property fixed by the
format's construction or by the mathematics, computed by a route the oracle
does not take (``math.erf`` instead of the inverse normal CDF, brute-force
nearest level in float64, pure-Python sums), so that a dropped term, a wrong
sign or index, a swapped nibble or a transposed operand fails one of them."""
import math

import numpy as np
import pytest

import oracle as O
import oracle.nf4 as N


def _phi(x):
    return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def _quantile(p):
    """Standard-normal quantile by bisection on math.erf."""
    lo, hi = -10.0, 10.0
    for _ in range(200):
        mid = (lo + hi) / 2
        lo, hi = (mid, hi) if _phi(mid) < p else (lo, mid)
    return (lo + hi) / 2


def test_levels_shape_and_fixed_points():
    lv = N.levels()
    assert lv.dtype == np.float32 and lv.shape == (16,)
    assert np.all(np.diff(lv) > 0)
    assert lv[0] == -1.0 and lv[15] == 1.0 and lv[N.ZERO_CODE] == 0.0
    assert (lv > 0).sum() == 8 and (lv < 0).sum() == 7


def test_levels_split_the_normal_into_equal_masses():
    """Scaled back by the quantile of delta, consecutive levels from 0 up
    enclose the same normal probability (delta - 1/2) / 8 and from 0 down
    (delta - 1/2) / 7; the outermost levels sit at probabilities delta and
    1 - delta."""
    lv = N.levels().astype(np.float64)
    c = _quantile(N.DELTA)
    p = np.array([_phi(c * v) for v in lv])
    step_pos, step_neg = (N.DELTA - 0.5) / 8, (N.DELTA - 0.5) / 7
    assert p[7] == 0.5
    assert np.allclose(np.diff(p[7:]), step_pos, atol=1e-7)     # 0, then 8 positive levels
    assert np.allclose(np.diff(p[:8]), step_neg, atol=1e-7)     # 7 negative levels, then 0
    assert abs(p[15] - N.DELTA) < 1e-7 and abs(p[0] - (1 - N.DELTA)) < 1e-7


def test_midpoints():
    lv, mid = N.levels(), N.midpoints()
    for i in range(15):
        exact = (float(lv[i]) + float(lv[i + 1])) / 2
        assert lv[i] < mid[i] < lv[i + 1]
        assert abs(float(mid[i]) - exact) <= abs(float(np.spacing(np.float32(exact))))


@pytest.mark.parametrize("dtype", [O.F16, O.BF16, O.F32])
def test_quantize_is_the_nearest_level(dtype):
    rng = np.random.default_rng(5)
    W64 = rng.standard_normal((5, 200)) * np.array([[0.01], [1.0], [30.0], [0.0], [1e-3]])
    W64[4, 64:128] = 0.0                        # an all-zero block inside a row
    W = O.round_to(W64, dtype)
    packed, absmax, codes = N.quantize(W, dtype)
    x = O.widen(W, dtype)
    lv = N.levels().astype(np.float64)
    assert packed.shape == (5, 128) and absmax.shape == (5, 4)
    for n in range(5):
        for k in range(200):
            a = float(np.abs(x[n, (k // 64) * 64:(k // 64 + 1) * 64]).max())
            assert absmax[n, k // 64] == np.float32(a)
            want = N.ZERO_CODE if a == 0 else int(np.argmin(np.abs(x[n, k] / a - lv)))
            if a:
                d = np.sort(np.abs(x[n, k] / a - lv))
                if d[1] - d[0] < 1e-6:              # within rounding of a midpoint: either is nearest
                    continue
            assert codes[n, k] == want, (n, k)
    # a block's absmax element maps to the level of its sign
    for n in range(3):
        for b in range(4):
            seg = x[n, b * 64:min(200, b * 64 + 64)]
            j = int(np.argmax(np.abs(seg)))
            assert codes[n, b * 64 + j] == (15 if seg[j] > 0 else 0)
    assert np.all(codes[3] == N.ZERO_CODE) and np.all(absmax[3] == 0)
    assert np.all(codes[4, 64:128] == N.ZERO_CODE) and absmax[4, 1] == 0


def test_packing_order_and_padding():
    lv = N.levels()
    row = np.zeros((1, 70), np.float32)
    row[0, :4] = [lv[15], lv[0], lv[3], lv[12]]  # absmax 1: codes 15, 0, 3, 12
    packed, absmax, codes = N.quantize(row, O.F32)
    assert absmax[0, 0] == 1.0
    assert packed[0, 0] == 0xF0 and packed[0, 1] == 0x3C
    assert np.all(packed[0, 2:32] == 0x77)          # zeros in the first block
    assert absmax[0, 1] == 0 and np.all(packed[0, 32:] == 0x77)  # 6 zeros + padding
    assert np.array_equal(N.unpack(packed, 70), codes)


def test_dequantize_lossless_cases_and_error_bound():
    lv = N.levels()
    rng = np.random.default_rng(8)
    c = rng.integers(0, 16, size=(3, 128))
    scale = np.array([[1.0], [0.25], [8.0]], np.float32)   # powers of two: products exact
    c[:, 0] = 15                                           # every block's absmax is the scale
    c[:, 64] = 15
    W = (lv[c] * scale).astype(np.float32)
    packed, absmax, codes = N.quantize(W, O.F32)
    assert np.array_equal(codes, c)
    assert np.array_equal(N.dequantize(packed, absmax, 128, O.F32), W)
    # random weights: |Wdq - W| <= half the widest gap * absmax (+ rounding of the dtype)
    Wr = rng.standard_normal((4, 300)).astype(np.float32)
    p, a, _ = N.quantize(Wr, O.F32)
    gap = np.diff(lv.astype(np.float64)).max() / 2
    err = np.abs(N.dequantize(p, a, 300, O.F32).astype(np.float64) - Wr)
    assert np.all(err <= gap * np.repeat(a, 64, axis=1)[:, :300] * (1 + 1e-6))
    # the 16-bit forms are the fp32 form rounded once
    d32 = N.dequantize(p, a, 300, O.F32).astype(np.float64)
    assert np.array_equal(N.dequantize(p, a, 300, O.BF16), O.round_to(d32, O.BF16))
    assert np.array_equal(N.dequantize(p, a, 300, O.F16), O.round_to(d32, O.F16))


@pytest.mark.parametrize("dtype", [O.F16, O.BF16])
def test_matmuls_against_brute_force(dtype):
    rng = np.random.default_rng(11)
    M, K, Nn = 3, 70, 5
    W = O.round_to(rng.standard_normal((Nn, K)) * 0.05, dtype)
    A = O.round_to(rng.standard_normal((M, K)), dtype)
    G = O.round_to(rng.standard_normal((M, Nn)), dtype)
    bias = O.round_to(rng.standard_normal(Nn) * 0.1, dtype)
    packed, absmax, codes = N.quantize(W, dtype)
    fwd = N.forward(A, dtype, packed, absmax, K, bias, dtype)
    bwd = N.backward_input(G, dtype, packed, absmax, K)
    assert np.array_equal(fwd["Wdq"], N.dequantize(packed, absmax, K, dtype))
    assert np.array_equal(bwd["Wdq"], fwd["Wdq"])
    wd = O.widen(fwd["Wdq"], dtype).tolist()
    a = O.widen(A, dtype).tolist()
    g = O.widen(G, dtype).tolist()
    b = O.widen(bias, dtype).tolist()
    for m in range(M):
        for n in range(Nn):
            s = math.fsum(a[m][k] * wd[n][k] for k in range(K)) + b[n]
            assert abs(fwd["out64"][m, n] - s) <= 1e-12 * (1 + abs(s))
        for k in range(K):
            s = math.fsum(g[m][n] * wd[n][k] for n in range(Nn))
            assert abs(bwd["grad64"][m, k] - s) <= 1e-12 * (1 + abs(s))
    assert np.array_equal(fwd["out"], O.round_to(fwd["out64"], dtype))
    with pytest.raises(ValueError):
        N.forward(A, O.F32, packed, absmax, K)
