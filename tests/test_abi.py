"""Host-side checks of the C ABI (no GPU needed).

The library builds for sm_103a, loads, exports every function that
include/i8lt.h declares, and rejects bad arguments with a status code before
it touches the device.  The pointers passed here are never dereferenced:
every call returns at its argument checks.
"""
import ctypes
import math
import os

import numpy as np
import pytest

from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build


@pytest.fixture(scope="module")
def L():
    build()
    return _lib.load()


def test_exports_every_declared_function(L):
    names = _lib.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_version_and_strings(L):
    assert _lib.i8lt_abi_version() == 4
    for code in range(10):
        assert _lib.i8lt_status_string(code) != "unknown status"
    assert _lib.i8lt_status_string(42) == "unknown status"


@pytest.mark.parametrize("K,ld", [(1, 16), (4, 16), (16, 16), (17, 32), (4096, 4096), (11008, 11008), (-1, -1)])
def test_weight_ld(L, K, ld):
    assert _lib.i8lt_weight_ld(K) == ld


def test_forward_layout(L):
    M, K, N, cap = 600, 4, 16, 0
    lay = _lib.i8lt_forward_workspace_layout(M, K, N, cap)
    assert lay.k_pad == 16 and lay.cap_pad == 0
    M, K, N, cap = 2048, 4096, 4096, 256
    lay = _lib.i8lt_forward_workspace_layout(M, K, N, cap)
    offs = [lay.status, lay.asq, lay.bsq, lay.colmax, lay.mask, lay.idx, lay.sca, lay.plan, lay.aq, lay.suba,
            lay.subb, lay.cbh, lay.total]
    assert offs == sorted(offs)
    assert all(o % 256 == 0 for o in offs)
    nch = (lay.k_pad + 1023) // 1024
    assert lay.bsq - lay.asq >= (M + 255) // 256 * nch * 4
    assert lay.colmax - lay.bsq >= (N + 255) // 256 * nch * 4
    assert lay.plan - lay.sca >= M * 4
    assert lay.aq - lay.plan >= (M + 255) // 256 * ((N + 255) // 256) * 4
    assert lay.suba - lay.aq >= M * lay.k_pad * 2
    assert lay.subb - lay.suba >= M * lay.cap_pad * 2
    assert lay.cbh - lay.subb >= N * lay.cap_pad * 2
    assert lay.total - lay.cbh >= N * lay.k_pad * 2
    assert _lib.i8lt_forward_workspace_size(M, K, N, cap) == lay.total
    # capacity is clamped to K and padded to 64
    assert _lib.i8lt_forward_workspace_layout(8, 40, 8, 1000).cap_pad == 64


FAKE = 1 << 20          # 16-byte aligned, never dereferenced


def fwd(**kw):
    a = dict(A=FAKE, at=0, M=64, K=64, CB=FAKE, SCB=FAKE, N=64, bias=None, bt=0, threshold=6.0, residual=None,
             out=FAKE, ws=FAKE, ws_bytes=1 << 40, max_outliers=16)
    a.update(kw)
    return _lib.i8lt_forward(a["A"], a["at"], a["M"], a["K"], a["CB"], a["SCB"], a["N"], a["bias"], a["bt"],
                             a["threshold"], a["residual"], a["out"], a["ws"], a["ws_bytes"], a["max_outliers"])


def test_forward_argument_errors(L):
    assert fwd(at=3) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert fwd(bias=FAKE, bt=-1) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert fwd(K=0) == _lib.I8LT_ERR_INVALID_ARG
    assert fwd(N=0) == _lib.I8LT_ERR_INVALID_ARG
    assert fwd(M=-1) == _lib.I8LT_ERR_INVALID_ARG
    assert fwd(max_outliers=-1) == _lib.I8LT_ERR_INVALID_ARG
    assert fwd(K=_lib.I8LT_MAX_K + 1) == _lib.I8LT_ERR_K_TOO_LARGE
    assert fwd(CB=None) == _lib.I8LT_ERR_INVALID_ARG
    assert fwd(ws=None) == _lib.I8LT_ERR_INVALID_ARG
    assert fwd(A=None) == _lib.I8LT_ERR_INVALID_ARG
    assert fwd(A=FAKE + 8) == _lib.I8LT_ERR_MISALIGNED
    assert fwd(residual=FAKE + 2) == _lib.I8LT_ERR_MISALIGNED
    assert fwd(ws=FAKE + 16) == _lib.I8LT_ERR_MISALIGNED       # workspace wants 256 bytes
    need = _lib.i8lt_forward_workspace_size(64, 64, 64, 16)
    assert fwd(ws_bytes=need - 1) == _lib.I8LT_ERR_WORKSPACE


def test_sharded_forward_argument_errors(L):
    # step 1 needs no weight; both steps check the workspace like i8lt_forward
    need = _lib.i8lt_forward_workspace_size(64, 64, 64, 16)
    assert _lib.i8lt_forward_colmax(FAKE, 3, 64, 64, 64, FAKE, need, 16) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert _lib.i8lt_forward_colmax(FAKE, 0, 64, 0, 64, FAKE, need, 16) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_forward_colmax(FAKE, 0, 64, 64, 64, FAKE, need - 1, 16) == _lib.I8LT_ERR_WORKSPACE
    assert _lib.i8lt_forward_colmax(FAKE, 0, 64, 64, 64, None, need, 16) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_forward_colmax(FAKE + 4, 0, 64, 64, 64, FAKE, need, 16) == _lib.I8LT_ERR_MISALIGNED
    assert _lib.i8lt_forward_from_colmax(FAKE, 0, 64, 64, None, FAKE, 64, None, 0, 6.0, None, FAKE, FAKE, need,
                                         16) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_forward_from_colmax(FAKE, 0, 64, _lib.I8LT_MAX_K + 1, FAKE, FAKE, 64, None, 0, 6.0, None, FAKE,
                                         FAKE, 1 << 40, 16) == _lib.I8LT_ERR_K_TOO_LARGE


def bwd(**kw):
    a = dict(G=FAKE, gt=0, M=64, N=64, CB=FAKE, SCB=FAKE, K=64, addend=None, grad_A=FAKE, grad_bias=None, bt=0,
             ws=FAKE, ws_bytes=1 << 40)
    a.update(kw)
    return _lib.i8lt_backward_input(a["G"], a["gt"], a["M"], a["N"], a["CB"], a["SCB"], a["K"], a["addend"],
                                    a["grad_A"], a["grad_bias"], a["bt"], a["ws"], a["ws_bytes"])


def test_backward_argument_errors(L):
    assert bwd(gt=9) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert bwd(grad_bias=FAKE, bt=5) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert bwd(K=0) == _lib.I8LT_ERR_INVALID_ARG
    assert bwd(K=_lib.I8LT_MAX_K + 1) == _lib.I8LT_ERR_K_TOO_LARGE
    assert bwd(ws=None) == _lib.I8LT_ERR_WORKSPACE
    assert bwd(G=FAKE + 4) == _lib.I8LT_ERR_MISALIGNED
    assert bwd(grad_A=FAKE, CB=None) == _lib.I8LT_ERR_INVALID_ARG
    need = _lib.i8lt_backward_workspace_size(64, 64, 0)
    assert bwd(ws_bytes=need - 1) == _lib.I8LT_ERR_WORKSPACE
    # bf16 grad_output needs room for its fp16 copy
    assert _lib.i8lt_backward_workspace_size(64, 64, 1) >= need + 64 * 64 * 2


def test_backward_workspace_of_the_materialized_schedule(L):
    # the transient dequantized weight (K_pad x N_pad fp16) follows the fused
    # schedule's workspace
    for M, N, K, gt in [(64, 64, 64, 0), (300, 520, 1100, 1), (7, 13, 5, 2), (0, 8, 8, 0)]:
        lean = _lib.i8lt_backward_workspace_size(M, N, gt)
        dq = _lib.i8lt_backward_workspace_size_dq(M, N, K, gt)
        kp, npad = (K + 15) // 16 * 16, (N + 7) // 8 * 8
        assert dq >= lean + kp * npad * 2
        assert dq - lean < kp * npad * 2 + 256
    assert _lib.i8lt_backward_workspace_size_dq(64, 64, _lib.I8LT_MAX_K + 1, 0) == 0
    assert _lib.i8lt_backward_workspace_size_dq(64, 64, 64, 9) == 0


def test_other_entry_points_argument_errors(L):
    assert _lib.i8lt_quantize_weight(FAKE, 7, 4, 4, FAKE, FAKE, None) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert _lib.i8lt_quantize_weight(FAKE, 0, 4, 0, FAKE, FAKE, None) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_quantize_weight(FAKE + 1, 0, 4, 4, FAKE, FAKE, None) == _lib.I8LT_ERR_MISALIGNED
    assert _lib.i8lt_silu_forward(FAKE, 4, 8, FAKE) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert _lib.i8lt_silu_backward(None, FAKE, 0, 8, FAKE) == _lib.I8LT_ERR_INVALID_ARG
    r, _, _ = _lib.i8lt_read_device_status(None)
    assert r == _lib.I8LT_ERR_INVALID_ARG


def test_debug_wait_timeout_argument_errors(L):
    assert _lib.i8lt_debug_wait_timeout(0, FAKE, 256) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_debug_wait_timeout(3_000_000_000, FAKE, 256) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_debug_wait_timeout(1000, FAKE, 255) == _lib.I8LT_ERR_WORKSPACE
    assert _lib.i8lt_debug_wait_timeout(1000, None, 256) == _lib.I8LT_ERR_WORKSPACE
    assert _lib.i8lt_debug_wait_timeout(1000, FAKE + 16, 256) == _lib.I8LT_ERR_MISALIGNED


def test_valid_call_without_gpu_reports_error_not_crash(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = fwd(ws_bytes=_lib.i8lt_forward_workspace_size(64, 64, 64, 16))
    assert st in (_lib.I8LT_ERR_CUDA, _lib.I8LT_ERR_DEVICE)


def test_max_k_is_the_int32_bound():
    assert _lib.I8LT_MAX_K * 127 * 127 < 2 ** 31 <= (_lib.I8LT_MAX_K + 1) * 127 * 127
    assert math.floor((2 ** 31 - 1) / 16129) == _lib.I8LT_MAX_K


def test_nf4_sizes_and_levels(L):
    assert _lib.i8lt_nf4_row_bytes(0) == 0 and _lib.i8lt_nf4_row_bytes(1) == 32 and _lib.i8lt_nf4_row_bytes(64) == 32
    assert _lib.i8lt_nf4_row_bytes(65) == 64 and _lib.i8lt_nf4_row_bytes(-1) == -1
    assert _lib.i8lt_nf4_blocks(0) == 0 and _lib.i8lt_nf4_blocks(1) == 1 and _lib.i8lt_nf4_blocks(129) == 3
    assert _lib.i8lt_nf4_workspace_size() == 256
    assert _lib.i8lt_nf4_workspace_size_dq(64, 64) == 256 + 64 * 64 * 2
    assert _lib.i8lt_nf4_workspace_size_dq(100, 3) == 256 + 768       # rounded up to 256 bytes
    assert _lib.i8lt_nf4_workspace_size_dq(-1, 8) == 0
    # the levels are computed on the host: no GPU needed
    st, lv = _lib.i8lt_nf4_levels()
    assert st == _lib.I8LT_OK and len(lv) == 16 and lv[0] == -1.0 and lv[7] == 0.0 and lv[15] == 1.0
    assert all(a < b for a, b in zip(lv, lv[1:]))
    # FP4 (E2M1 / 6), by sign-magnitude code; the same host-side computation
    st, lv = _lib.i8lt_fp4_levels()
    assert st == _lib.I8LT_OK and lv[0] == 0.0 and lv[7] == 1.0 and lv[6] == np.float32(4.0 / 6.0)
    assert lv[8:] == [-v for v in lv[:8]] and math.copysign(1.0, lv[8]) == -1.0
    assert all(a < b for a, b in zip(lv[:8], lv[1:8]))
    # grad_bias partial sums of the 4-bit input gradient: 128-token chunks x N fp32, 256-byte aligned
    assert _lib.i8lt_absmax8_blocks(0) == 0 and _lib.i8lt_absmax8_blocks(256) == 1
    assert _lib.i8lt_absmax8_blocks(257) == 2 and _lib.i8lt_absmax8_blocks(-1) == -1
    assert _lib.i8lt_absmax8_workspace_size() == 256 + 256 * 8
    # argument errors come back before any device work
    assert _lib.i8lt_absmax8_quantize(None, -1, None, None, None, None, 0, None) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_absmax8_quantize(None, 0, None, None, 8, None, 0, None) == _lib.I8LT_ERR_WORKSPACE
    assert _lib.i8lt_absmax8_dequantize(None, None, None, 5, None, None) == _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_absmax8_dequantize(None, None, None, 0, None, None) == _lib.I8LT_OK
    assert _lib.i8lt_nf4_grad_bias_bytes(300, 64) == 3 * 64 * 4
    assert _lib.i8lt_nf4_grad_bias_bytes(1, 10) == 256 and _lib.i8lt_nf4_grad_bias_bytes(-1, 10) == 0


def nf4(which, **kw):
    a = dict(X=FAKE, xt=1, M=64, K=64, packed=FAKE, absmax=FAKE, N=64, bias=None, bt=0, out=FAKE, ws=FAKE,
             ws_bytes=256)
    a.update(kw)
    if which == "fwd":
        return _lib.i8lt_nf4_forward(a["X"], a["xt"], a["M"], a["K"], a["packed"], a["absmax"], a["N"], a["bias"],
                                     a["bt"], a["out"], a["ws"], a["ws_bytes"])
    return _lib.i8lt_nf4_backward_input(a["X"], a["xt"], a["M"], a["N"], a["packed"], a["absmax"], a["K"], a["out"],
                                        a.get("gb"), a["bt"], a["ws"], a["ws_bytes"])


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_nf4_argument_errors(L, which):
    assert nf4(which, xt=2) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE      # compute dtype f16 or bf16 only
    assert nf4(which, xt=7) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert nf4(which, K=0) == _lib.I8LT_ERR_INVALID_ARG
    assert nf4(which, N=0) == _lib.I8LT_ERR_INVALID_ARG
    assert nf4(which, M=-1) == _lib.I8LT_ERR_INVALID_ARG
    # the reduction dimension of X must give 16-byte rows
    assert nf4(which, **({"K": 100} if which == "fwd" else {"N": 100})) == _lib.I8LT_ERR_INVALID_ARG
    assert nf4(which, packed=None) == _lib.I8LT_ERR_INVALID_ARG
    assert nf4(which, X=None) == _lib.I8LT_ERR_INVALID_ARG
    assert nf4(which, X=FAKE + 8) == _lib.I8LT_ERR_MISALIGNED
    assert nf4(which, ws=FAKE + 16) == _lib.I8LT_ERR_MISALIGNED
    assert nf4(which, ws_bytes=255) == _lib.I8LT_ERR_WORKSPACE
    if which == "fwd":
        assert nf4(which, bias=FAKE, bt=9) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    else:
        assert nf4(which, gb=FAKE, bt=9) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
        # grad_bias needs room for its partial sums after the status word
        assert nf4(which, gb=FAKE, bt=1, ws_bytes=256) == _lib.I8LT_ERR_WORKSPACE
        assert nf4(which, out=None, gb=None) == _lib.I8LT_ERR_INVALID_ARG   # nothing asked for
        for fn in (_lib.i8lt_fp4_backward_input,):
            assert fn(FAKE, 2, 64, 64, FAKE, FAKE, 64, FAKE, None, 0, FAKE, 256) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert _lib.i8lt_fp4_forward(FAKE, 1, 64, 100, FAKE, FAKE, 64, None, 0, FAKE, FAKE, 256) == \
        _lib.I8LT_ERR_INVALID_ARG
    assert _lib.i8lt_fp4_quantize(FAKE, 5, 4, 4, FAKE, FAKE) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert _lib.i8lt_fp4_dequantize(FAKE, FAKE, 4, 4, FAKE, 3) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert _lib.i8lt_nf4_quantize(FAKE, 5, 4, 4, FAKE, FAKE) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE
    assert _lib.i8lt_nf4_quantize(FAKE, 0, 4, 4, FAKE + 4, FAKE) == _lib.I8LT_ERR_MISALIGNED
    assert _lib.i8lt_nf4_quantize(FAKE, 0, 4, 0, FAKE, FAKE) == _lib.I8LT_OK    # nothing to do
    assert _lib.i8lt_nf4_dequantize(FAKE, FAKE, 4, 4, FAKE, 3) == _lib.I8LT_ERR_UNSUPPORTED_DTYPE


def test_header_compiles_as_c_and_links(L, tmp_path):
    """A C99 program includes include/i8lt.h, links libi8lt.so and runs the
    host-side entry points (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = str(tmp_path / "abi_smoke")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                        os.path.join(root, "tests", "c", "abi_smoke.c"), "-L", libdir, "-li8lt",
                        "-Wl,-rpath," + libdir, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
