"""The failure path of the device-side waits, exercised without a fault.

Every pipeline wait in the library is bounded: past its limit it writes
I8LT_ERR_TIMEOUT to the workspace status word and the kernel winds down.
i8lt_debug_wait_timeout runs that same wait on a barrier that nothing
completes, with a short limit; the error must come back through
i8lt_read_device_status, and the CUDA context must stay usable (a forward
right after it still matches the oracle).
"""
import time

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build

from _helpers import check_forward_stages, check_weight, gpu_forward, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def test_bounded_wait_reports_timeout_and_the_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _lib.i8lt_debug_wait_timeout(20_000_000, ws.data_ptr(), ws.numel(), stream) == _lib.I8LT_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 2.0
    where = int(ws[12:16].view(torch.int32).item())      # DevStatus: status, found, used, where
    st, _ = I.device_status(ws)
    assert st == _lib.I8LT_ERR_TIMEOUT
    assert where == 9
    assert I.device_status(ws)[0] == 0                    # reading clears the recorded error
    # the context is intact: a layer still matches the oracle
    spec = W.LayerSpec(300, 512, 256, torch.float16, 0.02, 0.01, 0.01, 12.0, 6.0)
    wl = W.Workload("after", "", (spec,), w_dtype=torch.float16)
    A = W.activation(spec, 51)
    Wf, b, _ = W.layer_tensors(wl, 0, 51)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, spec.K)
    g = gpu_forward(A.to(DEV), CB, SCB, spec.K, b.to(DEV), 6.0)
    ref = O.forward(to_np(A), O.F16, CB_ref, SCB_ref, to_np(b), O.F16, 6.0)
    check_forward_stages(g, ref)


def test_grid_wide_wait_reports_timeout_and_the_context_survives():
    """The fused activation quantization's grid-wide wait, one arrival
    short: both blocks give up after the limit, the error (role 7) comes
    back, and a forward that runs the fused kernel right after matches the
    oracle."""
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert _lib.i8lt_debug_grid_wait_timeout(20_000_000, ws.data_ptr(), ws.numel(), stream) == _lib.I8LT_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert 0.015 < elapsed < 2.0
    assert int(ws[64:68].view(torch.int32).item()) == 2  # both blocks arrived once
    where = int(ws[12:16].view(torch.int32).item())
    st, _ = I.device_status(ws)
    assert st == _lib.I8LT_ERR_TIMEOUT and where == 7
    assert I.device_status(ws)[0] == 0
    assert _lib.i8lt_debug_grid_wait_timeout(0, ws.data_ptr(), ws.numel(), stream) == _lib.I8LT_ERR_INVALID_ARG
    spec = W.LayerSpec(700, 1024, 256, torch.float16, 0.02, 0.01, 0.01, 12.0, 6.0)   # fused quantization path
    wl = W.Workload("after", "", (spec,), w_dtype=torch.float16)
    A = W.activation(spec, 52)
    Wf, b, _ = W.layer_tensors(wl, 0, 52)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    CB_ref, SCB_ref = check_weight(CB, SCB, Wf, spec.K)
    g = gpu_forward(A.to(DEV), CB, SCB, spec.K, b.to(DEV), 6.0)
    ref = O.forward(to_np(A), O.F16, CB_ref, SCB_ref, to_np(b), O.F16, 6.0)
    check_forward_stages(g, ref)
