"""Token-sharded forward through the C ABI on one GPU.

The rows of one batch are split into shards with their own workspaces.
i8lt_forward_colmax runs on every shard, the column maxima are combined with
an element-wise maximum (what an all-reduce MAX does across ranks; here the
shards share a GPU, so a torch.maximum stands in for it), and
i8lt_forward_from_colmax finishes every shard.  The shards' rows must equal
i8lt_forward on the whole batch bit for bit: outputs, int32 accumulators and
outlier counts.  The two-rank protocol itself is simulated on CPU ranks in
test_shard_sim.py.
"""
import pytest
import torch

import workloads as W
import int8_quantized_linear_i8lt_gb300 as I
from int8_quantized_linear_i8lt_gb300 import _lib
from int8_quantized_linear_i8lt_gb300.build import build
from int8_quantized_linear_i8lt_gb300.functional import DTYPE_CODE

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("M,K,N,dtype,cuts", [(600, 1100, 520, torch.float16, (0, 250, 600)),
                                              (777, 640, 300, torch.bfloat16, (0, 1, 500, 777)),
                                              (300, 256, 256, torch.float16, (0, 0, 300))])   # an empty shard
def test_sharded_forward_equals_the_whole_batch(M, K, N, dtype, cuts):
    spec = W.LayerSpec(M, K, N, dtype, 0.02, 0.01, 0.01, 10.0, 6.0)
    wl = W.Workload("shard", "", (spec,), w_dtype=dtype)
    A = W.activation(spec, 9).to(DEV)
    col = 7
    A[:, col] = A[:, col].clamp(-1, 1)
    A[M - 1, col] = 8.0                      # an outlier column that only the last shard holds
    Wf, b, _ = W.layer_tensors(wl, 0, 9)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    b = b.to(DEV)
    cap = I.default_max_outliers(K)
    acc_full = torch.empty(M, N, dtype=torch.int32, device=DEV)
    out_full, ws_full = I.forward(A, CB, SCB, K, b, 6.0, max_outliers=cap, acc_i32=acc_full)
    st, found_full = I.device_status(ws_full)
    assert st == 0
    stream = torch.cuda.current_stream().cuda_stream
    at, bt = DTYPE_CODE[dtype], DTYPE_CODE[b.dtype]
    shards = []
    for r0, r1 in zip(cuts[:-1], cuts[1:]):
        Ar = A[r0:r1].contiguous()
        m = r1 - r0
        ws = I.functional.forward_workspace(m, K, N, cap, A.device)
        assert _lib.i8lt_forward_colmax(Ar.data_ptr(), at, m, K, N, ws.data_ptr(), ws.numel(), cap, stream) == 0
        lay = _lib.i8lt_forward_workspace_layout(m, K, N, cap)
        shards.append((r0, r1, Ar, ws, ws[lay.colmax:lay.colmax + 4 * K].view(torch.int32)))
    merged = shards[0][4].clone()
    for sh in shards[1:]:
        merged = torch.maximum(merged, sh[4])
    for sh in shards:
        sh[4].copy_(merged)
    for r0, r1, Ar, ws, _ in shards:
        m = r1 - r0
        out = torch.empty(m, N, dtype=dtype, device=DEV)
        acc = torch.empty(m, N, dtype=torch.int32, device=DEV)
        st = _lib.i8lt_forward_from_colmax(Ar.data_ptr(), at, m, K, CB.data_ptr(), SCB.data_ptr(), N, b.data_ptr(),
                                           bt, 6.0, None, out.data_ptr(), ws.data_ptr(), ws.numel(), cap,
                                           acc_i32=acc.data_ptr() if m else None, stream=stream)
        assert st == 0, _lib.i8lt_status_string(st)
        if m == 0:
            continue
        st, found = I.device_status(ws)
        assert st == 0 and found == found_full
        assert torch.equal(acc, acc_full[r0:r1])
        assert torch.equal(out.view(torch.int16), out_full[r0:r1].view(torch.int16))


def test_merge_hook_of_the_python_forward():
    # with a hook that leaves the maxima alone, the two-step path is the one-step forward
    spec = W.LayerSpec(333, 512, 200, torch.float16, 0.02, 0.01, 0.01, 10.0, 6.0)
    wl = W.Workload("shard", "", (spec,), w_dtype=torch.float16)
    A = W.activation(spec, 3).to(DEV)
    Wf, b, _ = W.layer_tensors(wl, 0, 3)
    CB, SCB = I.quantize_weight(Wf.to(DEV))
    seen = []
    out1, _ = I.forward(A, CB, SCB, spec.K, b.to(DEV), 6.0)
    out2, _ = I.forward(A, CB, SCB, spec.K, b.to(DEV), 6.0, merge_colmax=lambda t: seen.append(t.numel()))
    assert seen == [spec.K]
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
