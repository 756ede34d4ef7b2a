"""Token-sharded forward, simulated on CPU ranks with the oracle.

One batch's rows are split over two gloo ranks.  Each rank takes the column
maxima of |fp16(A)| over its own rows, the ranks combine them with one MAX
all-reduce (the only exchange), and each rank runs the rest of the forward
on its rows with the merged maxima.  The rows of both ranks must equal the
oracle's forward on the whole batch bit for bit; without the exchange a
column that is an outlier only in the other rank's rows would be missed.
The CUDA entry points of the same protocol (i8lt_forward_colmax /
i8lt_forward_from_colmax) are checked on one GPU in test_shard_gpu.py.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

M, K, N = 96, 200, 40
PLANT = (70, 13)          # an outlier that only rank 1's rows hold


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs():
    import oracle as O
    import workloads as W
    spec = W.LayerSpec(M, K, N, torch.float16, 0.02, 0.01, 0.02, 10.0, 6.0)
    wl = W.Workload("shard", "", (spec,), w_dtype=torch.float16)
    A = W.activation(spec, 5)
    A[:, PLANT[1]] = A[:, PLANT[1]].clamp(-1.0, 1.0)
    A[PLANT] = 9.0
    Wf, b, _ = W.layer_tensors(wl, 0, 5)
    CB, SCB = O.quantize_weight(Wf.numpy(), O.F16)
    return A.numpy(), CB, SCB, b.numpy()


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        A, CB, SCB, b = _inputs()
        rows = slice(rank * M // world, (rank + 1) * M // world)
        A_r = A[rows]
        local = torch.from_numpy(O.column_absmax(O.cast_f16(A_r, O.F16)))
        merged = local.clone()
        dist.all_reduce(merged, op=dist.ReduceOp.MAX)
        r = O.forward(A_r, O.F16, CB, SCB, b, O.F16, 6.0, col_absmax=merged.numpy())
        r_local = O.forward(A_r, O.F16, CB, SCB, b, O.F16, 6.0)
        q.put((rank, r["idx"], r["SCA"], r["Aq"], r["Cacc"], r["out"].view(np.uint16), r_local["idx"]))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharded_forward_equals_the_whole_batch():
    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(2)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    A, CB, SCB, b = _inputs()
    full = O.forward(A, O.F16, CB, SCB, b, O.F16, 6.0)
    assert PLANT[1] in full["idx"]
    for rank, idx, SCA, Aq, Cacc, out, idx_local in res:
        rows = slice(rank * M // 2, (rank + 1) * M // 2)
        assert np.array_equal(idx, full["idx"])
        assert np.array_equal(SCA.view(np.uint32), full["SCA"][rows].view(np.uint32))
        assert np.array_equal(Aq, full["Aq"][rows])
        assert np.array_equal(Cacc, full["Cacc"][rows])
        assert np.array_equal(out, full["out"][rows].view(np.uint16))
    # the planted column is an outlier only in rank 1's rows: rank 0 alone misses it
    assert PLANT[1] not in res[0][6] and PLANT[1] in res[1][6]


def test_column_absmax_merge_is_the_whole_batch_reduction():
    import oracle as O
    A, _, _, _ = _inputs()
    A16 = O.cast_f16(A, O.F16)
    parts = [O.column_absmax(A16[i:i + 17]) for i in range(0, M, 17)]
    merged = np.maximum.reduce(parts)
    assert np.array_equal(merged, O.column_absmax(A16))
    assert np.array_equal(O.outlier_columns_from_absmax(merged, 6.0), O.outlier_columns(A16, 6.0))
    assert len(O.outlier_columns_from_absmax(merged, float("inf"))) == 0
    assert np.array_equal(O.column_absmax(A16[:0]), np.zeros(K))


def _fp16_magnitude_bits(colmax64):
    """The library's colmax format: per column the fp16 bit pattern of the
    magnitude (sign cleared), held as int32; integer order = magnitude order."""
    return torch.from_numpy(colmax64.astype(np.float16).view(np.uint16).astype(np.int32))


def _hook_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import oracle as O
    from int8_quantized_linear_i8lt_gb300 import functional as F
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        A, _, _, _ = _inputs()
        rows = slice(rank * M // world, (rank + 1) * M // world)
        local = _fp16_magnitude_bits(O.column_absmax(O.cast_f16(A[rows], O.F16)))
        t = local.clone()
        F.allreduce_colmax()(t)            # the product's merge hook, in place
        q.put((rank, local.numpy(), t.numpy()))
    finally:
        dist.destroy_process_group()


def test_allreduce_colmax_hook_on_two_gloo_ranks():
    """functional.allreduce_colmax, the exchange step of the token-sharded
    forward, run by two gloo ranks on the column maxima of their rows in the
    library's format: every rank ends with the element-wise maximum, which
    is the whole batch's column maxima, and the outlier set read from it is
    the whole batch's."""
    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_hook_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(2)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    A, _, _, _ = _inputs()
    whole = _fp16_magnitude_bits(O.column_absmax(O.cast_f16(A, O.F16))).numpy()
    (_, l0, m0), (_, l1, m1) = res
    assert np.array_equal(m0, np.maximum(l0, l1)) and np.array_equal(m1, m0)
    assert np.array_equal(m0, whole)
    assert not np.array_equal(l0, whole)          # rank 0's rows alone miss the planted outlier
    mags = m0.astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(O.outlier_columns_from_absmax(mags, 6.0), O.outlier_columns(O.cast_f16(A, O.F16), 6.0))
