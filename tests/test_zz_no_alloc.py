"""The backward entry point that allocates nothing on the device.

Some callers cannot call cudaMalloc: a host framework that reserved the GPU's
memory for its own pool at start-up, code running inside another library's
allocator callback, or a loop that must never enter the driver's allocator.
i8lt_backward_input_noalloc serves them with a static scratch array of fixed
size compiled into the library.  This file checks, through the C ABI, that
two calls in a row give the same results as i8lt_backward_input (which takes
a caller-allocated workspace) within the tolerance the parity tests use, and
that a problem larger than the static scratch is refused.  It is collected
last so that a failure here cannot hide failures of the other GPU tests.
"""
import numpy as np
import pytest
import torch

import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build
from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE

from _helpers import assert_tol, widen

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("M,K,N,dtype", [(1000, 1100, 520, torch.float16),     # G used as is
                                         (777, 640, 300, torch.bfloat16),      # G copied to fp16 in scratch
                                         (4096, 4096, 4096, torch.float16)])   # a full-size layer
def test_noalloc_matches_workspace_entry_point(M, K, N, dtype):
    spec = W.LayerSpec(M, K, N, dtype, 0.02, 0.01)
    wl = W.Workload("noalloc", "", (spec,), w_dtype=dtype)
    Wf, b, G = W.layer_tensors(wl, 0, 31)
    Wf, G = Wf.to(DEV), G.to(DEV)
    CB, SCB = I.quantize_weight(Wf)
    ref_A, ref_b = I.backward_input(G, CB, SCB, K, bias_dtype=b.dtype)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        gA = torch.empty(M, K, dtype=dtype, device=DEV)
        gb = torch.empty(N, dtype=b.dtype, device=DEV)
        st = _lib.i8lt_backward_input_noalloc(G.data_ptr(), DTYPE_CODE[dtype], M, N, CB.data_ptr(),
                                              SCB.data_ptr(), K, None, gA.data_ptr(), gb.data_ptr(),
                                              DTYPE_CODE[b.dtype], stream)
        assert st == _lib.I8LT_OK, _lib.i8lt_status_string(st)
        torch.cuda.synchronize()
        assert_tol(widen(gA), widen(ref_A), "grad_A (no-alloc)")
        assert_tol(widen(gb), widen(ref_b), "grad_bias (no-alloc)")


def test_noalloc_refuses_problems_beyond_its_scratch():
    M, N = 8192, 4096                          # bf16 G needs a 64 MiB fp16 copy
    need = _lib.i8lt_backward_workspace_size(M, N, _lib.I8LT_BF16)
    assert need > _lib.I8LT_NOALLOC_SCRATCH_BYTES
    st = _lib.i8lt_backward_input_noalloc(1 << 20, _lib.I8LT_BF16, M, N, 1 << 20, 1 << 20, 64, None, 1 << 20,
                                          None, 0, None)
    assert st == _lib.I8LT_ERR_SCRATCH_LIMIT
