"""ctypes binding of libi8lt.so: the C entry points under the same names.

Argument marshalling only: every call goes straight to the CUDA library.
Pointers are Python ints (device addresses), streams are cudaStream_t
handles as ints.  The library must have been built (``build.py``); there is
no fallback of any kind when it is missing.
"""
from __future__ import annotations

import ctypes
import os
import re
from ctypes import POINTER, Structure, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libi8lt.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "i8lt.h")

I8LT_OK = 0
I8LT_ERR_INVALID_ARG = 1
I8LT_ERR_UNSUPPORTED_DTYPE = 2
I8LT_ERR_MISALIGNED = 3
I8LT_ERR_WORKSPACE = 4
I8LT_ERR_K_TOO_LARGE = 5
I8LT_ERR_OUTLIER_CAPACITY = 6
I8LT_ERR_TIMEOUT = 7
I8LT_ERR_CUDA = 8
I8LT_ERR_DEVICE = 9
I8LT_ERR_SCRATCH_LIMIT = 10
I8LT_NOALLOC_SCRATCH_BYTES = 32 << 20

I8LT_F16, I8LT_BF16, I8LT_F32 = 0, 1, 2
I8LT_MAX_K = 133144


class i8lt_fwd_layout(Structure):
    _fields_ = [("status", c_size_t), ("asq", c_size_t), ("bsq", c_size_t), ("colmax", c_size_t),
                ("mask", c_size_t), ("idx", c_size_t), ("sca", c_size_t), ("plan", c_size_t), ("aq", c_size_t),
                ("suba", c_size_t), ("subb", c_size_t), ("cbh", c_size_t), ("total", c_size_t),
                ("k_pad", c_int64), ("cap_pad", c_int64)]


class i8lt_fwd_debug(Structure):
    _fields_ = [("acc_i32", c_void_p)]


class i8lt_kernel_time(Structure):
    _fields_ = [("kernel", c_int), ("ms", c_float)]


KERNELS = ("quantize_weight", "colmax", "outlier_index", "row_quantize", "build_subB", "fwd_gemm",
           "gradout_prepass", "grad_bias_finalize", "bwd_gemm", "silu", "silu_backward", "widen_codes",
           "dequant_weight", "col_quantize", "wgrad_gemm", "unit_plan", "nf4_quantize", "nf4_dequantize",
           "nf4_gemm_fwd", "nf4_gemm_bwd")


# name -> (restype, argtypes); the same names and order as include/i8lt.h
SIGNATURES = {
    "i8lt_abi_version": (c_int, []),
    "i8lt_status_string": (c_char_p, [c_int]),
    "i8lt_weight_ld": (c_int64, [c_int64]),
    "i8lt_quantize_weight": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_void_p]),
    "i8lt_forward_workspace_size": (c_size_t, [c_int64, c_int64, c_int64, c_int64]),
    "i8lt_forward_workspace_layout": (c_int, [c_int64, c_int64, c_int64, c_int64, POINTER(i8lt_fwd_layout)]),
    "i8lt_forward": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64,
                             c_void_p, c_int, c_float, c_void_p, c_void_p,
                             c_void_p, c_size_t, c_int64, POINTER(i8lt_fwd_debug), c_void_p]),
    "i8lt_forward_silu": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64,
                                  c_void_p, c_int, c_float, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_size_t, c_int64, POINTER(i8lt_fwd_debug), c_void_p]),
    "i8lt_forward_colmax": (c_int, [c_void_p, c_int, c_int64, c_int64, c_int64, c_void_p, c_size_t, c_int64,
                                    c_void_p]),
    "i8lt_forward_from_colmax": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64,
                                         c_void_p, c_int, c_float, c_void_p, c_void_p,
                                         c_void_p, c_size_t, c_int64, POINTER(i8lt_fwd_debug), c_void_p]),
    "i8lt_backward_workspace_size": (c_size_t, [c_int64, c_int64, c_int]),
    "i8lt_debug_wait_timeout": (c_int, [c_int64, c_void_p, c_size_t, c_void_p]),
    "i8lt_debug_grid_wait_timeout": (c_int, [c_int64, c_void_p, c_size_t, c_void_p]),
    "i8lt_grad_weight_workspace_size": (c_size_t, [c_int64, c_int64, c_int64]),
    "i8lt_grad_weight": (c_int, [c_void_p, c_int, c_void_p, c_int, c_int64, c_int64, c_int64, c_void_p, c_int,
                                 c_void_p, c_size_t, c_void_p]),
    "i8lt_backward_workspace_size_dq": (c_size_t, [c_int64, c_int64, c_int64, c_int]),
    "i8lt_backward_input": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64,
                                    c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_size_t, c_void_p]),
    "i8lt_backward_input_noalloc": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64,
                                            c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "i8lt_noalloc_read_device_status": (c_int, [POINTER(c_int32), c_void_p]),
    "i8lt_nf4_levels": (c_int, [POINTER(c_float)]),
    "i8lt_fp4_levels": (c_int, [POINTER(c_float)]),
    "i8lt_nf4_row_bytes": (c_int64, [c_int64]),
    "i8lt_nf4_blocks": (c_int64, [c_int64]),
    "i8lt_nf4_quantize": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_void_p]),
    "i8lt_fp4_quantize": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_void_p]),
    "i8lt_nf4_dequantize": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_int, c_void_p]),
    "i8lt_fp4_dequantize": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_int, c_void_p]),
    "i8lt_nf4_workspace_size": (c_size_t, []),
    "i8lt_nf4_workspace_size_dq": (c_size_t, [c_int64, c_int64]),
    "i8lt_nf4_grad_bias_bytes": (c_size_t, [c_int64, c_int64]),
    "i8lt_nf4_forward": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64, c_void_p, c_int,
                                 c_void_p, c_void_p, c_size_t, c_void_p]),
    "i8lt_fp4_forward": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64, c_void_p, c_int,
                                 c_void_p, c_void_p, c_size_t, c_void_p]),
    "i8lt_nf4_backward_input": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64, c_void_p,
                                        c_void_p, c_int, c_void_p, c_size_t, c_void_p]),
    "i8lt_fp4_backward_input": (c_int, [c_void_p, c_int, c_int64, c_int64, c_void_p, c_void_p, c_int64, c_void_p,
                                        c_void_p, c_int, c_void_p, c_size_t, c_void_p]),
    "i8lt_absmax8_blocks": (c_int64, [c_int64]),
    "i8lt_absmax8_workspace_size": (c_size_t, []),
    "i8lt_absmax8_quantize": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                      c_void_p]),
    "i8lt_absmax8_dequantize": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p]),
    "i8lt_silu_forward": (c_int, [c_void_p, c_int, c_int64, c_void_p, c_void_p]),
    "i8lt_silu_backward": (c_int, [c_void_p, c_void_p, c_int, c_int64, c_void_p, c_void_p]),
    "i8lt_profile_start": (c_int, [c_int]),
    "i8lt_profile_stop": (c_int, [POINTER(i8lt_kernel_time), c_int, POINTER(c_int), POINTER(c_int)]),
    "i8lt_kernel_name": (c_char_p, [c_int]),
    "i8lt_gemm_launch_info": (c_int, [c_int, POINTER(c_int), POINTER(c_int), POINTER(c_int)]),
    "i8lt_read_device_status": (c_int, [c_void_p, POINTER(c_int32), POINTER(c_int32), c_void_p]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libi8lt.so (once) and declare every signature."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libi8lt.so is not built ({LIB_PATH} missing); build it with "
                "`python -m int8_quantized_linear_i8lt_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/i8lt.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(i8lt_[a-z_0-9]+)\s*\(", text)))


def _p(x):
    return None if x is None or x == 0 else c_void_p(int(x))


# --- the entry points, same names ------------------------------------------

def i8lt_abi_version() -> int:
    return load().i8lt_abi_version()


def i8lt_status_string(status: int) -> str:
    return load().i8lt_status_string(int(status)).decode()


def i8lt_weight_ld(K: int) -> int:
    return load().i8lt_weight_ld(int(K))


def i8lt_quantize_weight(W, wt, N, K, CB, SCB, stream) -> int:
    return load().i8lt_quantize_weight(_p(W), wt, N, K, _p(CB), _p(SCB), _p(stream))


def i8lt_forward_workspace_size(M, K, N, max_outliers) -> int:
    return load().i8lt_forward_workspace_size(M, K, N, max_outliers)


def i8lt_forward_workspace_layout(M, K, N, max_outliers) -> i8lt_fwd_layout:
    out = i8lt_fwd_layout()
    st = load().i8lt_forward_workspace_layout(M, K, N, max_outliers, ctypes.byref(out))
    if st != I8LT_OK:
        raise ValueError(i8lt_status_string(st))
    return out


def i8lt_forward(A, at, M, K, CB, SCB, N, bias, bt, threshold, residual, out, ws, ws_bytes,
                 max_outliers, acc_i32=None, stream=None) -> int:
    dbg = ctypes.byref(i8lt_fwd_debug(_p(acc_i32))) if acc_i32 else None
    return load().i8lt_forward(_p(A), at, M, K, _p(CB), _p(SCB), N, _p(bias), bt, c_float(threshold),
                               _p(residual), _p(out), _p(ws), ws_bytes, max_outliers, dbg, _p(stream))


def i8lt_forward_silu(A, at, M, K, CB, SCB, N, bias, bt, threshold, residual, out, act, act_colmax, ws, ws_bytes,
                      max_outliers, acc_i32=None, stream=None) -> int:
    dbg = ctypes.byref(i8lt_fwd_debug(_p(acc_i32))) if acc_i32 else None
    return load().i8lt_forward_silu(_p(A), at, M, K, _p(CB), _p(SCB), N, _p(bias), bt, c_float(threshold),
                                    _p(residual), _p(out), _p(act), _p(act_colmax), _p(ws), ws_bytes, max_outliers,
                                    dbg, _p(stream))


def i8lt_forward_colmax(A, at, M, K, N, ws, ws_bytes, max_outliers, stream=None) -> int:
    return load().i8lt_forward_colmax(_p(A), at, M, K, N, _p(ws), ws_bytes, max_outliers, _p(stream))


def i8lt_forward_from_colmax(A, at, M, K, CB, SCB, N, bias, bt, threshold, residual, out, ws, ws_bytes,
                             max_outliers, acc_i32=None, stream=None) -> int:
    dbg = ctypes.byref(i8lt_fwd_debug(_p(acc_i32))) if acc_i32 else None
    return load().i8lt_forward_from_colmax(_p(A), at, M, K, _p(CB), _p(SCB), N, _p(bias), bt, c_float(threshold),
                                           _p(residual), _p(out), _p(ws), ws_bytes, max_outliers, dbg, _p(stream))


def i8lt_grad_weight_workspace_size(M, N, K) -> int:
    return load().i8lt_grad_weight_workspace_size(M, N, K)


def i8lt_grad_weight(G, gt, A, at, M, N, K, grad_W, wt, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_grad_weight(_p(G), gt, _p(A), at, M, N, K, _p(grad_W), wt, _p(ws), ws_bytes, _p(stream))


def i8lt_debug_wait_timeout(limit_ns, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_debug_wait_timeout(limit_ns, _p(ws), ws_bytes, _p(stream))


def i8lt_debug_grid_wait_timeout(limit_ns, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_debug_grid_wait_timeout(limit_ns, _p(ws), ws_bytes, _p(stream))


def i8lt_backward_workspace_size(M, N, gt) -> int:
    return load().i8lt_backward_workspace_size(M, N, gt)


def i8lt_backward_workspace_size_dq(M, N, K, gt) -> int:
    return load().i8lt_backward_workspace_size_dq(M, N, K, gt)


def i8lt_backward_input(G, gt, M, N, CB, SCB, K, addend, grad_A, grad_bias, bt, ws, ws_bytes,
                        stream=None) -> int:
    return load().i8lt_backward_input(_p(G), gt, M, N, _p(CB), _p(SCB), K, _p(addend), _p(grad_A),
                                      _p(grad_bias), bt, _p(ws), ws_bytes, _p(stream))


def i8lt_backward_input_noalloc(G, gt, M, N, CB, SCB, K, addend, grad_A, grad_bias, bt, stream=None) -> int:
    return load().i8lt_backward_input_noalloc(_p(G), gt, M, N, _p(CB), _p(SCB), K, _p(addend), _p(grad_A),
                                              _p(grad_bias), bt, _p(stream))


def i8lt_noalloc_read_device_status(stream=None):
    """-> (return code, status word) of the no-alloc scratch on the current device."""
    st = c_int32(0)
    r = load().i8lt_noalloc_read_device_status(ctypes.byref(st), _p(stream))
    return r, int(st.value)


def i8lt_nf4_levels():
    out = (c_float * 16)()
    st = load().i8lt_nf4_levels(out)
    return st, list(out)


def i8lt_fp4_levels():
    out = (c_float * 16)()
    st = load().i8lt_fp4_levels(out)
    return st, list(out)


def i8lt_nf4_row_bytes(K) -> int:
    return load().i8lt_nf4_row_bytes(int(K))


def i8lt_nf4_blocks(K) -> int:
    return load().i8lt_nf4_blocks(int(K))


def i8lt_nf4_quantize(W, wt, N, K, packed, absmax, stream=None) -> int:
    return load().i8lt_nf4_quantize(_p(W), wt, N, K, _p(packed), _p(absmax), _p(stream))


def i8lt_fp4_quantize(W, wt, N, K, packed, absmax, stream=None) -> int:
    return load().i8lt_fp4_quantize(_p(W), wt, N, K, _p(packed), _p(absmax), _p(stream))


def i8lt_nf4_dequantize(packed, absmax, N, K, out, dt, stream=None) -> int:
    return load().i8lt_nf4_dequantize(_p(packed), _p(absmax), N, K, _p(out), dt, _p(stream))


def i8lt_fp4_dequantize(packed, absmax, N, K, out, dt, stream=None) -> int:
    return load().i8lt_fp4_dequantize(_p(packed), _p(absmax), N, K, _p(out), dt, _p(stream))


def i8lt_nf4_workspace_size() -> int:
    return load().i8lt_nf4_workspace_size()


def i8lt_nf4_workspace_size_dq(K, N) -> int:
    return load().i8lt_nf4_workspace_size_dq(int(K), int(N))


def i8lt_nf4_grad_bias_bytes(M, N) -> int:
    return load().i8lt_nf4_grad_bias_bytes(int(M), int(N))


def i8lt_nf4_forward(A, at, M, K, packed, absmax, N, bias, bt, out, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_nf4_forward(_p(A), at, M, K, _p(packed), _p(absmax), N, _p(bias), bt, _p(out), _p(ws),
                                   ws_bytes, _p(stream))


def i8lt_fp4_forward(A, at, M, K, packed, absmax, N, bias, bt, out, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_fp4_forward(_p(A), at, M, K, _p(packed), _p(absmax), N, _p(bias), bt, _p(out), _p(ws),
                                   ws_bytes, _p(stream))


def i8lt_nf4_backward_input(G, gt, M, N, packed, absmax, K, grad_A, grad_bias, bt, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_nf4_backward_input(_p(G), gt, M, N, _p(packed), _p(absmax), K, _p(grad_A), _p(grad_bias), bt,
                                          _p(ws), ws_bytes, _p(stream))


def i8lt_fp4_backward_input(G, gt, M, N, packed, absmax, K, grad_A, grad_bias, bt, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_fp4_backward_input(_p(G), gt, M, N, _p(packed), _p(absmax), K, _p(grad_A), _p(grad_bias), bt,
                                          _p(ws), ws_bytes, _p(stream))


def i8lt_absmax8_blocks(count) -> int:
    return load().i8lt_absmax8_blocks(int(count))


def i8lt_absmax8_workspace_size() -> int:
    return load().i8lt_absmax8_workspace_size()


def i8lt_absmax8_quantize(absmax, count, q, absmax2, offset, ws, ws_bytes, stream=None) -> int:
    return load().i8lt_absmax8_quantize(_p(absmax), int(count), _p(q), _p(absmax2), _p(offset), _p(ws), ws_bytes,
                                        _p(stream))


def i8lt_absmax8_dequantize(q, absmax2, offset, count, out, stream=None) -> int:
    return load().i8lt_absmax8_dequantize(_p(q), _p(absmax2), _p(offset), int(count), _p(out), _p(stream))


def i8lt_silu_forward(h, dt, n, out, stream=None) -> int:
    return load().i8lt_silu_forward(_p(h), dt, n, _p(out), _p(stream))


def i8lt_silu_backward(g, h, dt, n, out, stream=None) -> int:
    return load().i8lt_silu_backward(_p(g), _p(h), dt, n, _p(out), _p(stream))


def i8lt_read_device_status(ws, stream=None):
    st, found = c_int32(0), c_int32(0)
    r = load().i8lt_read_device_status(_p(ws), ctypes.byref(st), ctypes.byref(found), _p(stream))
    return r, int(st.value), int(found.value)


def i8lt_profile_start(max_launches: int) -> int:
    return load().i8lt_profile_start(int(max_launches))


def i8lt_profile_stop(cap: int = 65536):
    """-> (status, [(kernel name, ms), ...] in launch order, launches counted)"""
    buf = (i8lt_kernel_time * cap)()
    n, launches = c_int(0), c_int(0)
    st = load().i8lt_profile_stop(buf, cap, ctypes.byref(n), ctypes.byref(launches))
    recs = [(i8lt_kernel_name(buf[i].kernel), float(buf[i].ms)) for i in range(n.value)]
    return st, recs, int(launches.value)


def i8lt_kernel_name(kernel: int) -> str:
    return load().i8lt_kernel_name(int(kernel)).decode()


def i8lt_gemm_launch_info(kernel: str):
    """(status, CTAs, threads per CTA, dynamic shared memory) of 'fwd_gemm' / 'bwd_gemm'."""
    k = KERNELS.index(kernel)
    c, t, m = c_int(0), c_int(0), c_int(0)
    st = load().i8lt_gemm_launch_info(k, ctypes.byref(c), ctypes.byref(t), ctypes.byref(m))
    return st, c.value, t.value, m.value
