"""Randomized properties of the oracles over shapes, scales and dtypes
(hypothesis; skipped where it is not installed).  Each property is fixed by
the method's definition, not by the oracle's code: codes in [-127, 127], the
row maximum at +-127, outlier columns out of the int8 product, the
quantization error bound, int8 part + outlier part = the full product within
that bound; for NF4, the nearest-level rule and the dequantization bound."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")

import oracle as O          # noqa: E402
import oracle.nf4 as N      # noqa: E402

SETTINGS = dict(max_examples=40, deadline=None)


@hyp.given(M=st.integers(1, 9), K=st.integers(1, 70), N_=st.integers(1, 9), scale=st.floats(1e-3, 50.0),
           heavy=st.integers(0, 3), seed=st.integers(0, 2 ** 31 - 1))
@hyp.settings(**SETTINGS)
def test_int8_forward_properties(M, K, N_, scale, heavy, seed):
    rng = np.random.default_rng(seed)
    A = (rng.standard_normal((M, K)) * scale).astype(np.float16)
    cols = rng.choice(K, size=min(heavy, K), replace=False)
    A[:, cols] = (A[:, cols].astype(np.float32) * 40).astype(np.float16)
    W = (rng.standard_normal((N_, K)) * 0.05).astype(np.float16)
    thr = 6.0
    CB, SCB = O.quantize_weight(W, O.F16)
    ref = O.forward(A, O.F16, CB, SCB, threshold=thr)
    idx, SCA, Aq = ref["idx"], ref["SCA"], ref["Aq"]
    A16 = A.astype(np.float64)
    # the outlier set is exactly the columns with some |value| above the threshold
    want = np.nonzero((np.abs(A16) > thr).any(axis=0))[0]
    assert np.array_equal(idx, want)
    assert Aq.min() >= -127 and Aq.max() <= 127 and np.all(Aq[:, idx] == 0)
    X = A16.copy()
    X[:, idx] = 0
    nz = np.abs(X).max(axis=1) > 0
    am = np.argmax(np.abs(X), axis=1)
    assert np.all(np.abs(Aq[np.arange(M), am])[nz] == 127)
    # int8 part + outlier part against the fp64 product of the fp16 inputs
    # with the dequantized weight, within the activation quantization error
    Wdq = O.dequant_weight(CB, SCB).astype(np.float64)
    full = A16 @ Wdq.T
    bound = (SCA.astype(np.float64)[:, None] / 254 * (1 + 2.0 ** -20)) * np.abs(Wdq).sum(axis=1)[None, :]
    int8_part = ref["Cacc"].astype(np.float64) * SCA.astype(np.float64)[:, None] * SCB.astype(np.float64)[None, :] / 16129
    # the weight side of the int8 part is CB * SCB / 127, which Wdq rounds to fp16
    wq = CB.astype(np.float64) * SCB.astype(np.float64)[:, None] / 127
    wbound = np.abs(A16) @ np.abs(Wdq - wq).T
    assert np.all(np.abs(ref["out64"] - full) <= bound + wbound + 1e-9)
    assert np.allclose(int8_part + (ref["subA"].astype(np.float64) @ ref["subB"].astype(np.float64).T
                                    if len(idx) else 0), ref["out64"])


@hyp.given(N_=st.integers(1, 5), K=st.integers(1, 150), scale=st.floats(1e-4, 1e3), seed=st.integers(0, 2 ** 31 - 1),
           dtype=st.sampled_from([O.F16, O.BF16, O.F32]))
@hyp.settings(**SETTINGS)
def test_nf4_quantize_properties(N_, K, scale, seed, dtype):
    rng = np.random.default_rng(seed)
    W = O.round_to(rng.standard_normal((N_, K)) * scale, dtype)
    packed, absmax, codes = N.quantize(W, dtype)
    x = O.widen(W, dtype)
    lv = N.levels().astype(np.float64)
    blk = np.repeat(absmax.astype(np.float64), N.BLOCK, axis=1)[:, :K]
    xn = np.divide(x, blk, out=np.zeros_like(x), where=blk > 0)
    dist = np.abs(xn[..., None] - lv)
    best = dist.min(axis=-1)
    # the chosen level is a nearest one, up to the fp32 rounding of x / absmax
    assert np.all(dist[np.arange(N_)[:, None], np.arange(K)[None, :], codes] <= best + 1e-6)
    assert np.array_equal(N.unpack(packed, K), codes)
    # dequantization error: at most half the widest gap times the block's absmax, plus the dtype's rounding
    for dt in (O.F32, O.BF16):
        d = O.widen(N.dequantize(packed, absmax, K, dt), dt)
        gap = np.diff(lv).max() / 2
        rel = 2.0 ** -8 if dt == O.BF16 else 2.0 ** -23
        assert np.all(np.abs(d - x) <= blk * gap * (1 + 1e-6) + np.abs(d) * rel + 1e-30)
