"""Host-side caches of the Python binding (no GPU needed).

A DTensor keeps its C descriptor while its slots' addresses and strides are
unchanged, and rebuilds it when a slot is replaced or restrided.  The
workspace-size queries keep their answers per operand set (layouts,
addresses, strides, arguments, device), so a linear called without a
workspace does not plan twice; a changed operand is a new key.  fp32
operands run on the CUDA-core kernel and need no workspace on any device,
so the queries answer 0 here.
"""
import ctypes as C

import torch

import tensor_sharded_linear_gb300 as tsl
from tensor_sharded_linear_gb300 import api


def dt(shape, placements, slots):
    return tsl.DTensor(slots, tsl.DeviceMesh((4,), ("tp",)), placements, shape, torch.float32)


def col_operands():
    x = dt((64, 32), [tsl.Replicate()], [torch.zeros(64, 32)])
    w = dt((32, 128), [tsl.Shard(1)], [torch.zeros(32, 32) for _ in range(4)])
    y = dt((64, 128), [tsl.Shard(1)], [torch.zeros(64, 32) for _ in range(4)])
    return x, w, y


def desc_pointers(d, n):
    return [d.slots[i] or 0 for i in range(n)]


def test_descriptor_reused_while_slots_unchanged(lib):
    _, w, _ = col_operands()
    d1 = w._desc()
    assert w._desc() is d1
    assert desc_pointers(d1, 4) == [t.data_ptr() for t in w.slots]


def test_descriptor_rebuilt_when_a_slot_changes(lib):
    _, w, _ = col_operands()
    d1 = w._desc()
    w.slots[2] = torch.zeros(32, 32)  # another buffer
    d2 = w._desc()
    assert d2 is not d1
    assert desc_pointers(d2, 4) == [t.data_ptr() for t in w.slots]
    # same buffer seen through other strides: a new descriptor with them
    parent = torch.zeros(32, 64)
    w.slots[1] = parent[:, :32]
    d3 = w._desc()
    assert d3 is not d2
    assert [d3.strides[2 + i] for i in range(2)] == [64, 1]


def test_workspace_size_answers_kept_per_operand_set(lib):
    x, w, y = col_operands()
    api._WS_SIZES.clear()
    assert tsl.column_parallel_linear_workspace_bytes(x, [w], [y]) == 0
    assert len(api._WS_SIZES) == 1
    assert tsl.column_parallel_linear_workspace_bytes(x, [w], [y]) == 0
    assert len(api._WS_SIZES) == 1  # answered from the cache
    y.slots[0] = torch.zeros(64, 32)  # a changed operand is a new question
    assert tsl.column_parallel_linear_workspace_bytes(x, [w], [y]) == 0
    assert len(api._WS_SIZES) == 2


def test_cached_answer_matches_a_fresh_query(lib):
    """The memo returns exactly what the library answers for the same operands."""
    x, w, y = col_operands()
    api._WS_SIZES.clear()
    cached = tsl.column_parallel_linear_workspace_bytes(x, [w], [y])
    n = C.c_size_t(99)
    wd, yd = (api.L.DTensorDesc * 1)(w._desc()), (api.L.DTensorDesc * 1)(y._desc())
    assert api.L.load().dt_column_parallel_linear_workspace_size(C.byref(x._desc()), 1, wd, yd, 0,
                                                                 C.byref(n)) == api.L.OK
    assert n.value == cached
