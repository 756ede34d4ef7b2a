"""Pins of the FP4 (E2M1) oracle, CPU only.  Each test checks a property
fixed by the format's definition or by the mathematics, computed by a route
the oracle does not take: the levels from the sign / exponent / mantissa
bit fields (the oracle holds a table of magnitudes), the code decision by a
brute-force nearest-level search in float64 with ties constructed exactly,
the matmuls by pure-Python sums -- so that a wrong table entry, a flipped
sign bit, a tie sent the wrong way, a swapped nibble or a transposed
operand fails one of them."""
import math
import struct

import numpy as np
import pytest

import oracle as O
import oracle.fp4 as F


def _f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def _e2m1(code: int) -> float:
    """The value of a 4-bit E2M1 pattern s e1 e0 m: exponent bias 1,
    exponent 0 subnormal (m / 2 * 2^0), otherwise 2^(e - 1) (1 + m / 2)."""
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    v = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return -v if s else v


def test_levels_are_e2m1_over_six():
    lv = F.levels()
    assert lv.dtype == np.float32 and lv.shape == (16,)
    for code in range(16):
        want = _f32(_e2m1(code) / 6.0)
        assert float(lv[code]) == want
        assert math.copysign(1.0, float(lv[code])) == (-1.0 if code >= 8 else 1.0)   # code 8 is -0
    assert lv[7] == 1.0 and lv[0] == 0.0 and math.copysign(1.0, lv[8]) == -1.0
    # the largest magnitude is 6, the smallest nonzero 0.5 (subnormal)
    assert max(abs(_e2m1(c)) for c in range(16)) == 6.0 and _e2m1(1) == 0.5


def test_midpoints_and_tie_rule():
    lv, mid, up = F.levels(), F.midpoints(), F.tie_goes_up()
    for j in range(7):
        exact = (float(lv[j]) + float(lv[j + 1])) / 2
        assert lv[j] < mid[j] < lv[j + 1]
        assert abs(float(mid[j]) - exact) <= abs(float(np.spacing(np.float32(exact))))
        # a tie goes to the neighbour whose mantissa bit is 0 (IEEE round half to even)
        even = j if (j & 1) == 0 else j + 1
        assert up[j] == (even == j + 1)


def _brute_codes(x, absmax):
    """Nearest magnitude level of |x / absmax| (fp32 division), searched in
    float64 over all 8 levels; the sign bit for negative x off zero."""
    mags = [_f32(_e2m1(c) / 6.0) for c in range(8)]
    out = []
    for v in x:
        if absmax == 0:
            out.append(0)
            continue
        y = _f32(v / absmax)
        d = [abs(abs(y) - m) for m in mags]
        c = int(np.argmin(d))
        out.append(c | 8 if (y < 0 and c) else c)
    return out


@pytest.mark.parametrize("dtype", [O.F16, O.BF16, O.F32])
def test_quantize_is_the_nearest_level(dtype):
    rng = np.random.default_rng(3)
    W64 = rng.normal(0, 0.02, (7, 200))
    W64[1] = 0.0                                 # an all-zero row
    W64[2, 64:128] *= 1000.0                     # a block of large values
    W = O.round_to(W64, dtype)
    packed, absmax, codes = F.quantize(W, dtype)
    x = O.widen(W, dtype)
    mid = F.midpoints().astype(np.float64)
    for n in range(7):
        for b in range(4):
            blk = x[n, 64 * b:64 * b + 64]
            am = float(np.abs(blk).max()) if blk.size else 0.0
            assert float(absmax[n, b]) == am
            want = _brute_codes(blk, am)
            got = codes[n, 64 * b:64 * b + len(blk)].tolist()
            for i, (g, w) in enumerate(zip(got, want)):
                y = abs(_f32(blk[i] / am)) if am else 0.0
                if np.min(np.abs(mid - y)) < 1e-6:
                    continue                     # next to a midpoint: the tie test pins these
                assert g == w, (n, b, i, blk[i], g, w)
            if am > 0:                           # the block's absmax element is the largest magnitude
                k = int(np.argmax(np.abs(blk)))
                assert got[k] in (7, 15)
    assert not np.any(codes[1]) and not np.any(absmax[1])


def test_half_way_ties_round_to_even():
    """|x / absmax| equal to each midpoint (absmax 1.0, fp32 weights, so the
    division is exact): the code with mantissa bit 0 wins, both signs."""
    mid = F.midpoints()
    row = np.zeros(64, np.float32)
    row[0] = 1.0
    row[1:8] = mid
    row[8:15] = -mid
    _, _, codes = F.quantize(row[None, :], O.F32)
    c = codes[0]
    # the pairs (0, 1), (1, 2), (2, 3), ... tie to 0, 2, 2, 4, 4, 6, 6
    assert c[1:8].tolist() == [0, 2, 2, 4, 4, 6, 6]
    assert c[8:15].tolist() == [0, 10, 10, 12, 12, 14, 14]          # zero keeps the one zero code
    # one fp32 step above a midpoint goes up, one below goes down
    up = np.nextafter(mid, np.float32(2)).astype(np.float32)
    dn = np.nextafter(mid, np.float32(-2)).astype(np.float32)
    row2 = np.zeros(64, np.float32)
    row2[0] = 1.0
    row2[1:8], row2[8:15] = up, dn
    _, _, c2 = F.quantize(row2[None, :], O.F32)
    assert c2[0, 1:8].tolist() == list(range(1, 8)) and c2[0, 8:15].tolist() == list(range(0, 7))


def test_packing_and_padding():
    lv = F.levels()
    row = np.zeros((1, 70), np.float32)
    row[0, 0] = -1.0                              # code 15
    row[0, 1] = 0.0                               # code 0
    row[0, 2] = float(lv[3])                      # code 3 (exact: absmax 1)
    row[0, 3] = -float(lv[4])                     # code 12
    packed, absmax, codes = F.quantize(row, O.F32)
    assert packed.shape == (1, 64)                # 128 padded elements, two per byte
    assert packed[0, 0] == 0xF0 and packed[0, 1] == 0x3C
    assert np.all(packed[0, 35:] == 0)            # padding: the zero code in both nibbles
    assert np.array_equal(F.unpack(packed, 70), codes)


@pytest.mark.parametrize("dtype", [O.BF16, O.F16, O.F32])
def test_dequantize_lossless_and_error_bound(dtype):
    lv = F.levels()
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 16, (5, 128))
    codes[:, 0] = 7                                # every block holds +-1 * absmax
    codes[:, 64] = 15
    scale = 2.0 ** rng.integers(-6, 3, (5, 2))
    x = lv[codes].astype(np.float64) * np.repeat(scale, 64, axis=1)
    W = O.round_to(x, O.F32)
    packed, absmax, _ = F.quantize(W, O.F32)
    back = O.widen(F.dequantize(packed, absmax, 128, dtype), dtype)
    assert np.array_equal(back, O.widen(O.round_to(x, dtype), dtype))
    # generic weights: |x - dq| <= half the widest gap between levels (4/6 to 6/6) times the absmax
    Wg = O.round_to(rng.normal(0, 1, (4, 192)), O.F32)
    pg, ag, _ = F.quantize(Wg, O.F32)
    dq = O.widen(F.dequantize(pg, ag, 192, O.F32), O.F32)
    am = np.repeat(ag.astype(np.float64), 64, axis=1)
    assert np.all(np.abs(dq - O.widen(Wg, O.F32)) <= am * (1.0 / 6.0) * (1 + 1e-6))


def test_matmuls_by_pure_python_sums():
    rng = np.random.default_rng(13)
    M, K, N = 3, 70, 5
    Wq = O.round_to(rng.normal(0, 0.05, (N, K)), O.BF16)
    A = O.round_to(rng.normal(0, 1, (M, K)), O.BF16)
    G = O.round_to(rng.normal(0, 1, (M, N)), O.BF16)
    b = O.round_to(rng.normal(0, 0.1, N), O.BF16)
    packed, absmax, _ = F.quantize(Wq, O.BF16)
    Wdq = O.widen(F.dequantize(packed, absmax, K, O.BF16), O.BF16)
    Aw, Gw, bw = O.widen(A, O.BF16), O.widen(G, O.BF16), O.widen(b, O.BF16)
    r = F.forward(A, O.BF16, packed, absmax, K, b, O.BF16)
    for m in range(M):
        for n in range(N):
            assert r["out64"][m, n] == pytest.approx(math.fsum(Aw[m, k] * Wdq[n, k] for k in range(K)) + bw[n],
                                                     rel=1e-12, abs=1e-14)
    rb = F.backward_input(G, O.BF16, packed, absmax, K)
    for m in range(M):
        for k in range(K):
            assert rb["grad64"][m, k] == pytest.approx(math.fsum(Gw[m, n] * Wdq[n, k] for n in range(N)),
                                                       rel=1e-12, abs=1e-14)
