"""CPU checks of the algorithmic byte counts bench.py divides by time for the
HBM-bound kernels: each is recounted from the shapes of the tensors the
kernel reads and writes."""

import numpy as np

import bench


def test_merge_bytes_from_tensor_shapes():
    T, H, D = 1000, 6, 128
    o_acc, o_part = np.zeros((T, H, D), np.float32), np.zeros((T, H, D), np.float32)
    l_acc, l_part = np.zeros((H, T), np.float32), np.zeros((H, T), np.float32)
    read = o_acc.nbytes + o_part.nbytes + l_acc.nbytes + l_part.nbytes
    write = o_acc.nbytes + l_acc.nbytes
    assert bench.merge_bytes(T, H, D) == read + write


def test_merge_bf16_bytes_from_tensor_shapes():
    T, H, D = 1000, 6, 128
    o_acc, o_part = np.zeros((T, H, D), np.float32), np.zeros((T, H, D), np.float16)   # 2-byte partial
    l_acc, l_part = np.zeros((H, T), np.float32), np.zeros((H, T), np.float32)
    read = o_acc.nbytes + o_part.nbytes + l_acc.nbytes + l_part.nbytes
    write = o_acc.nbytes + l_acc.nbytes
    assert bench.merge_bytes(T, H, D, part_bytes=2) == read + write


def test_tail_zero_bytes_from_tensor_shapes():
    rows_q, rows_kv, end, Hq, Hkv, D = 46077, 46077, 41888, 32, 8, 128
    dq = np.zeros((rows_q, Hq, D), np.float16)   # 2-byte elements like bf16
    dk = np.zeros((rows_kv, Hkv, D), np.float16)
    dv = np.zeros_like(dk)
    assert bench.tail_zero_bytes(rows_q, rows_kv, end, end, Hq, Hkv, D) == dq[end:].nbytes + dk[end:].nbytes + \
        dv[end:].nbytes
    assert bench.tail_zero_bytes(end, end, end, end, Hq, Hkv, D) == 0   # no slack, nothing written


def test_a2a_bytes_from_tensor_shapes():
    T, Hq, Hkv, D = 14632, 16, 4, 128
    q = np.zeros((T, Hq, D), np.float16)
    kv = np.zeros((T, Hkv, D), np.float16)
    assert bench.a2a_move_bytes(T, Hq, D) == 2 * q.nbytes
    # forward moves q, k, v, O; backward q, k, v, O, dO and dQ, dK, dV: each read once and written once
    forward = 2 * (2 * q.nbytes + 2 * kv.nbytes)                       # q, O; k, v
    backward = 2 * (3 * q.nbytes + 2 * kv.nbytes) + 2 * (q.nbytes + 2 * kv.nbytes)   # in: q, O, dO; k, v. out
    step = forward + backward
    assert bench.a2a_step_bytes(T, Hq, Hkv, D) == step


def test_lengths_override_keeps_the_workload_shape_and_renames_it():
    """bench.py --lengths: the named workload's heads, head dimension and cp
    size on other sequence lengths, under a name of its own (so that no
    per-workload record of the named workload applies to it)."""
    import argparse
    a = argparse.Namespace(config="long", lengths="32768")
    w = bench._workload(a)
    assert w.name == "long[32768]" and w.lengths == [32768] and w.T == 32768
    assert (w.Hq, w.Hkv, w.D, w.cp_size) == (32, 8, 128, 4)
    assert bench._kernel_traffic("bwd_kernel", w.name) is None
    a = argparse.Namespace(config="long", lengths=None)
    assert bench._workload(a).name == "long" and bench._workload(a).T == 131072
