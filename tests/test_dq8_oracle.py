"""Pins of the double-quantized absmax oracle (oracle/dq8.py), each by a
route the oracle does not take: fixed E4M3 anchors and torch's own
float8_e4m3fn conversion (a library routine), constructed ties, an exact
rational mean, and the error bound of the round trip.

Source: "Support QLoRA 4-bit finetuning with bitsandbytes" (lit-gpt PR #275),
the ``bnb.nf4-dq`` / ``bnb.fp4-dq`` options; the reading is in the oracle's
header."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import dq8 as D

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_e4m3_anchors_and_shape():
    v = D.e4m3_values()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0            # largest finite
    assert v[0x08] == 2.0 ** -6                               # smallest normal
    assert v[0x01] == 2.0 ** -9                               # smallest subnormal
    assert v[0x38] == 1.0 and v[0x40] == 2.0 and v[0x3C] == 1.5 and v[0x37] == 0.9375
    assert v[0x00] == 0.0 and not np.signbit(v[0x00]) and v[0x80] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    pos = v[:0x7F].astype(np.float64)
    assert np.all(np.diff(pos) > 0)                           # ascending, all distinct
    assert np.array_equal(v[0x80:0xFF], -v[:0x7F])            # symmetric


def test_e4m3_values_equal_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    t = codes.view(torch.float8_e4m3fn).float().numpy()
    v = D.e4m3_values()
    finite = ~np.isnan(v)
    assert np.array_equal(np.isnan(t), ~finite)
    assert np.array_equal(t[finite].view(np.uint32), v[finite].view(np.uint32))


def test_e4m3_encode_equals_torch_rounding():
    g = np.random.default_rng(0)
    y = np.concatenate([
        g.uniform(-448, 448, 20000),
        g.uniform(-1, 1, 20000),
        g.uniform(-2.0 ** -5, 2.0 ** -5, 20000),             # subnormals and the smallest normals
        np.ldexp(g.uniform(-1, 1, 5000), g.integers(-12, 9, 5000)),
    ]).astype(np.float32)
    # every midpoint between neighbouring finite values (exact ties), both signs
    pos = D.e4m3_values()[:0x7F].astype(np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    y = np.concatenate([y, mids, -mids, pos.astype(np.float32), -pos.astype(np.float32)[1:]])
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = D.e4m3_encode(y)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (y[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_e4m3_ties_saturation_and_zero_sign():
    enc = D.e4m3_encode
    assert enc(np.float32(1.0625)) == 0x38                    # between 1 (0x38) and 1.125 (0x39): even
    assert enc(np.float32(1.1875)) == 0x3A                    # between 1.125 and 1.25 (0x3A): even
    assert enc(np.float32(1.5 * 2.0 ** -9)) == 0x02           # subnormal tie: 2^-9 (0x01) vs 2^-8 (0x02)
    assert enc(np.float32(0.5 * 2.0 ** -9)) == 0x00           # tie with zero: zero is even
    assert enc(np.float32(448.0)) == 0x7E and enc(np.float32(449.0)) == 0x7E
    assert enc(np.float32(1e30)) == 0x7E and enc(np.float32(-1e30)) == 0xFE
    assert enc(np.float32(-1e-9)) == 0x80 and enc(np.float32(0.0)) == 0x00


def _exact_mean(c):
    return sum((Fraction(float(x)) for x in c), Fraction(0)) / len(c)


@pytest.mark.parametrize("seed", range(4))
def test_offset_is_the_correctly_rounded_mean(seed):
    g = np.random.default_rng(seed)
    c = np.exp(g.normal(-4, 2.5, 3000)).astype(np.float32)   # spread over many binades
    c[::97] = 0.0
    off = D.offset_of(c)
    exact = _exact_mean(c)
    ulp = np.spacing(np.float32(off))
    assert abs(Fraction(float(off)) - exact) <= Fraction(float(ulp)) / 2 * (1 + Fraction(1, 2 ** 28))
    # the sum is exact, so the order of the values does not matter
    assert D.offset_of(g.permutation(c)) == off
    assert D.offset_of(np.array([1, 2, 3, 6], np.float32)) == 3.0


def test_constant_absmax_round_trips_exactly():
    c = np.full((7, 100), 0.0371, np.float32)
    q, a2, off = D.quantize(c)
    assert off == np.float32(0.0371) and np.all(a2 == 0) and np.all(q == 0)
    assert np.array_equal(D.dequantize(q, a2, off), c)


@pytest.mark.parametrize("shape", [(1, 1), (3, 100), (64, 172), (300, 64)])
def test_round_trip_error_bound(shape):
    g = np.random.default_rng(shape[0] * 7 + shape[1])
    c = np.abs(g.normal(0, 0.02, shape)).astype(np.float32) + np.float32(1e-4)
    q, a2, off = D.quantize(c)
    assert q.shape == c.shape and q.dtype == np.uint8 and a2.shape == (D.blocks(c.size),)
    chat = D.dequantize(q, a2, off).reshape(-1).astype(np.float64)
    flat = c.reshape(-1).astype(np.float64)
    d = flat - float(off)
    a2e = np.repeat(a2.astype(np.float64), D.BLOCK2)[:flat.size]
    y = np.where(a2e > 0, np.abs(d) / np.where(a2e > 0, a2e, 1) * 448.0, 0.0)
    bound = (2.0 ** -4 * y + 2.0 ** -10) * a2e / 448.0 * (1 + 2.0 ** -18) + 8 * np.spacing(
        np.maximum(np.abs(flat), abs(float(off))).astype(np.float32)).astype(np.float64)
    err = np.abs(chat - flat)
    assert np.all(err <= bound), float((err / bound).max())
    # the largest |d| of every block takes a code of the largest magnitude (448)
    v = D.e4m3_values()
    for b in range(D.blocks(c.size)):
        seg = slice(b * D.BLOCK2, (b + 1) * D.BLOCK2)
        if a2[b] > 0:
            i = np.argmax(np.abs(d[seg]))
            assert abs(v[q.reshape(-1)[seg][i]]) == 448.0


def test_planted_mistakes_fail_the_pins():
    """A decoding that drops the offset, or an encoder that truncates instead
    of rounding, breaks the round-trip bound or the torch comparison."""
    c = np.abs(np.random.default_rng(5).normal(0.05, 0.01, 512)).astype(np.float32)
    q, a2, off = D.quantize(c)
    wrong = D.dequantize(q, a2, 0.0)
    assert np.abs(wrong - c).max() > 0.01
    y = np.float32([1.12, 3.3, 0.0061])
    trunc = np.array([0x38, 0x45, 0x03], np.uint8)            # truncated codes of the three values
    assert not np.array_equal(D.e4m3_encode(y), trunc)
