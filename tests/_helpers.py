"""Shared pieces of the GPU tests: running the CUDA path through the C ABI,
reading its intermediate stages out of the workspace, and the tolerance rule
for floating-point outputs."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib

ODT = {torch.float16: O.F16, torch.bfloat16: O.BF16, torch.float32: O.F32}


def to_np(t: torch.Tensor) -> np.ndarray:
    """Tensor -> oracle storage (bf16 as its uint16 bit pattern)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def widen(t: torch.Tensor) -> np.ndarray:
    return O.widen(to_np(t), ODT[t.dtype])


def tolerance_report(gpu64: np.ndarray, ref64: np.ndarray):
    """The rule for floating-point outputs: every element within
    0.02 * mean|ref|; at most 0.5% of the elements outside
    isclose(atol=0.01 * mean|ref|, rtol=0.1)."""
    scale = float(np.abs(ref64).mean()) if ref64.size else 0.0
    err = np.abs(gpu64 - ref64)
    bad = ~np.isclose(gpu64, ref64, atol=0.01 * scale, rtol=0.1)
    return dict(scale=scale, max_err=float(err.max()) if err.size else 0.0,
                frac_bad=float(bad.mean()) if bad.size else 0.0)


def assert_tol(gpu64, ref64, what=""):
    r = tolerance_report(gpu64, ref64)
    assert np.all(np.isfinite(gpu64)), f"{what}: non-finite values"
    assert r["max_err"] <= 0.02 * r["scale"] + 1e-30, f"{what}: {r}"
    assert r["frac_bad"] <= 0.005, f"{what}: {r}"
    return r


def cap_for(K, threshold, max_outliers=None):
    if not (math.isfinite(threshold) and threshold > 0):
        return 0
    return I.default_max_outliers(K) if max_outliers is None else max_outliers


def gpu_forward(A, CB, SCB, K, bias=None, threshold=6.0, residual=None, max_outliers=None):
    """Run i8lt_forward with the raw int32 accumulator requested; return the
    output and every intermediate stage read back from the workspace."""
    M, N = A.shape[0], CB.shape[0]
    cap = cap_for(K, threshold, max_outliers)
    acc = torch.empty(M, N, dtype=torch.int32, device=A.device)
    out, ws = I.forward(A, CB, SCB, K, bias, threshold, residual=residual, max_outliers=cap, acc_i32=acc)
    st, found = I.device_status(ws)
    lay = _lib.i8lt_forward_workspace_layout(M, K, N, cap)
    nch = (lay.k_pad + 1023) // 1024
    w = ws

    def region(off, nbytes, dtype, shape):
        return w[off:off + nbytes].view(dtype).reshape(shape)

    status = region(lay.status, 16, torch.int32, (4,)).cpu().numpy()
    used = int(status[2]) if cap > 0 else 0
    res = dict(out=out, acc=acc, status=st, found=found, used=used, ws=ws,
               SCA=region(lay.sca, M * 4, torch.float32, (M,)),
               asq=region(lay.asq, (M + 255) // 256 * nch * 4, torch.int32, ((M + 255) // 256, nch)),
               bsq=region(lay.bsq, (N + 255) // 256 * nch * 4, torch.int32, ((N + 255) // 256, nch)),
               plan=region(lay.plan, (M + 255) // 256 * ((N + 255) // 256) * 4, torch.int32,
                           ((M + 255) // 256, (N + 255) // 256)),
               Aq=region(lay.aq, M * lay.k_pad * 2, torch.float16, (M, lay.k_pad)),
               k_pad=lay.k_pad, cap_pad=lay.cap_pad)
    if cap > 0:
        res["idx"] = region(lay.idx, lay.cap_pad * 4, torch.int32, (lay.cap_pad,))
        res["subA"] = region(lay.suba, M * lay.cap_pad * 2, torch.float16, (M, lay.cap_pad))
        res["subB"] = region(lay.subb, N * lay.cap_pad * 2, torch.float16, (N, lay.cap_pad))
    return res


def check_forward_stages(g, ref, rows=None, K=None, out_tol=True):
    """Bit-exact integer stages + tolerance on the output.  ``rows``: the
    GPU rows the oracle result ``ref`` covers (None: all).  ``out_tol``
    False: the caller checks the output itself (bit for bit)."""
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    idx = ref["idx"]
    assert g["status"] == 0, _lib.i8lt_status_string(g["status"])
    assert g["found"] == len(idx)
    if len(idx):
        assert np.array_equal(to_np(g["idx"])[:len(idx)], idx)
        assert np.array_equal(to_np(sel(g["subA"]))[:, :len(idx)].view(np.uint16), ref["subA"].view(np.uint16))
        pad = to_np(sel(g["subA"]))[:, len(idx):(len(idx) + 63) // 64 * 64]
        assert not np.any(pad.astype(np.float32))
    assert np.array_equal(to_np(sel(g["SCA"])).view(np.uint32), ref["SCA"].view(np.uint32))
    Kq = ref["Aq"].shape[1]
    aq = to_np(sel(g["Aq"])).astype(np.float32)
    assert np.array_equal(aq[:, :Kq], ref["Aq"].astype(np.float32)), "int8 codes differ"
    assert not np.any(aq[:, Kq:]), "padding codes not zero"
    assert np.array_equal(to_np(sel(g["acc"])), ref["Cacc"]), "int32 accumulator differs"
    if not out_tol:
        return None
    out = widen(sel(g["out"]))
    return assert_tol(out, ref["out64"], "out")


def check_wdq(ws, M, N, K, dtype, CB_ref, SCB_ref, max_rows=4096):
    """The materialized schedule's dequantized weight, read back from the
    backward workspace (it follows the first i8lt_backward_workspace_size
    bytes): WdqT [K_pad, N_pad] fp16 must equal the oracle's Wdq transposed,
    bit for bit, with zero padding.  At most ``max_rows`` rows k are checked
    (evenly spaced, first and last included)."""
    from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE
    off = _lib.i8lt_backward_workspace_size(M, N, DTYPE_CODE[dtype])
    kp, npad = (K + 15) // 16 * 16, (N + 7) // 8 * 8
    assert ws.numel() >= off + kp * npad * 2
    wdqT = ws[off:off + kp * npad * 2].view(torch.float16).reshape(kp, npad)
    ks = np.unique(np.linspace(0, kp - 1, min(kp, max_rows)).round().astype(np.int64))
    got = wdqT[torch.as_tensor(ks, device=ws.device)].cpu().numpy()
    ref = O.dequant_weight(CB_ref, SCB_ref)          # [N, K] fp16
    inside = ks < K
    assert np.array_equal(got[inside, :N].view(np.uint16), ref[:, ks[inside]].T.view(np.uint16)), "WdqT differs"
    assert not np.any(got[~inside].astype(np.float32)), "WdqT padding rows not zero"
    assert not np.any(got[:, N:].astype(np.float32)), "WdqT padding columns not zero"


def check_weight(CB_gpu, SCB_gpu, W, K):
    CB_ref, SCB_ref = O.quantize_weight(to_np(W), ODT[W.dtype])
    cb = to_np(CB_gpu)
    assert np.array_equal(cb[:, :K], CB_ref)
    assert not np.any(cb[:, K:])
    assert np.array_equal(to_np(SCB_gpu).view(np.uint32), SCB_ref.view(np.uint32))
    return CB_ref, SCB_ref
