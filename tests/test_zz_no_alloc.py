"""The backward entry point that allocates nothing on the device.

Some callers cannot call cudaMalloc: a host framework that reserved the GPU's
memory for its own pool at start-up, code running inside another library's
allocator callback, or a loop that must never enter the driver's allocator.
i8lt_backward_input_noalloc serves them with a static scratch array of fixed
size compiled into the library.  This file checks, through the C ABI, that
two calls in a row give the same bytes as i8lt_backward_input (which takes a
caller-allocated workspace and runs the same kernels), that the result is
within the parity tolerance of the CPU oracle, that the scratch's status word
reads back clean after each call, that the calls leave the device's free
memory unchanged, and that a problem larger than the static scratch is
refused.  It is collected last so that a failure here cannot hide failures of
the other GPU tests.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build
from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE

from _helpers import ODT, assert_tol, to_np, widen

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
    Wf, Gd = Wf.to(DEV), G.to(DEV)
    CB, SCB = I.quantize_weight(Wf)
    ref_A, ref_b = I.backward_input(Gd, CB, SCB, K, bias_dtype=b.dtype)
    stream = torch.cuda.current_stream().cuda_stream
    outs = [(torch.empty(M, K, dtype=dtype, device=DEV), torch.empty(N, dtype=b.dtype, device=DEV))
            for _ in range(2)]
    torch.cuda.synchronize()
    for i, (gA, gb) in enumerate(outs):
        if i == 1:
            free0 = torch.cuda.mem_get_info()[0]
            alloc0 = torch.cuda.memory_allocated()
        st = _lib.i8lt_backward_input_noalloc(Gd.data_ptr(), DTYPE_CODE[dtype], M, N, CB.data_ptr(),
                                              SCB.data_ptr(), K, None, gA.data_ptr(), gb.data_ptr(),
                                              DTYPE_CODE[b.dtype], stream)
        assert st == _lib.I8LT_OK, _lib.i8lt_status_string(st)
        r, dev_status = _lib.i8lt_noalloc_read_device_status(stream)     # synchronizes the stream
        assert r == _lib.I8LT_OK and dev_status == 0, _lib.i8lt_status_string(dev_status)
        if i == 1:
            # the call took no device memory: neither from torch's pool nor from the driver
            assert torch.cuda.memory_allocated() == alloc0
            assert torch.cuda.mem_get_info()[0] == free0
        # the same kernels on the same inputs: the same bytes as the workspace entry point
        assert torch.equal(gA.view(torch.uint8), ref_A.view(torch.uint8)), "grad_A differs (no-alloc)"
        assert torch.equal(gb.view(torch.uint8), ref_b.view(torch.uint8)), "grad_bias differs (no-alloc)"
    # and once against the CPU oracle (sampled rows of the full-size case)
    CB_ref, SCB_ref = O.quantize_weight(to_np(Wf.cpu()), ODT[dtype])
    rows = np.unique(np.linspace(0, M - 1, min(M, 256)).round().astype(np.int64))
    rb = O.backward_input(to_np(G), ODT[dtype], CB_ref, SCB_ref, rows=rows)
    gA = outs[1][0]
    assert_tol(widen(gA[torch.as_tensor(rows, device=DEV)]), rb["grad64"], "grad_A (no-alloc) vs oracle")
    assert_tol(widen(outs[1][1]), O.widen(to_np(G), ODT[dtype]).sum(0), "grad_bias (no-alloc) vs oracle")


def test_noalloc_refuses_problems_beyond_its_scratch():
    M, N = 8192, 4096                          # bf16 G needs a 64 MiB fp16 copy
    need = _lib.i8lt_backward_workspace_size(M, N, _lib.I8LT_BF16)
    assert need > _lib.I8LT_NOALLOC_SCRATCH_BYTES
    st = _lib.i8lt_backward_input_noalloc(1 << 20, _lib.I8LT_BF16, M, N, 1 << 20, 1 << 20, 64, None, 1 << 20,
                                          None, 0, None)
    assert st == _lib.I8LT_ERR_SCRATCH_LIMIT
