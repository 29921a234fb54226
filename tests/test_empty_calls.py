"""Calls with nothing to compute, through the C ABI on the host (no GPU needed).

With no tokens (or an empty embedding dim) every layer returns DT_OK before
it touches a device: no launch, no device binding, no check of the strides
that torch leaves arbitrary on empty dims.  The slots here are CPU tensors
and the stream is NULL, so a call that reached CUDA would fail.  The same
cases run on the GPU, with their non-empty neighbours (K = 0, an ffn width
of 0), in test_gpu_linear.py and test_gpu_embedding.py.
"""
import ctypes as C

import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import _lib as L
from tensor_sharded_linear_gb300 import api

BF = torch.bfloat16
P = 4
MESH = tsl.DeviceMesh((P,), ("tp",))
MODES = [(tsl.ALL_REDUCE, L.TP_ALL_REDUCE), (tsl.REDUCE_SCATTER, L.TP_REDUCE_SCATTER), (tsl.PARTIAL, L.TP_PARTIAL)]


def zeros(shape, dtype=BF, zero_strides=False):
    """An empty slot may carry any strides: torch.from_numpy of an empty
    array gives all-zero ones."""
    t = torch.zeros(*shape, dtype=dtype)
    return t.as_strided(t.shape, [0] * t.dim()) if zero_strides and t.numel() == 0 else t


def shard(shape, d, mesh=MESH, zero_strides=False):
    slots = []
    for _, s in chunk_bounds(shape[d], mesh.shape[0]):
        z = list(shape)
        z[d] = s
        slots.append(zeros(z, zero_strides=zero_strides))
    return tsl.DTensor(slots, mesh, [tsl.Shard(d)], shape, BF)


def replicate(shape, dtype=BF, mesh=MESH, zero_strides=False):
    return tsl.DTensor([zeros(shape, dtype, zero_strides)], mesh, [tsl.Replicate()], shape, dtype)


def no_launch(lib, call):
    n0 = lib.dt_launch_count()
    st = call()
    assert st == L.OK, lib.dt_last_error().decode()
    assert lib.dt_launch_count() == n0


@pytest.mark.parametrize("zs", [False, True])
def test_column_no_tokens(lib, zs):
    x, w, y = replicate((0, 256), zero_strides=zs), shard((256, 192), 1), shard((0, 192), 1, zero_strides=zs)
    wa, ya = (L.DTensorDesc * 1)(w._desc()), (L.DTensorDesc * 1)(y._desc())
    no_launch(lib, lambda: lib.dt_column_parallel_linear(C.byref(x._desc()), wa, None, ya, 0, None, 0, None, None))


@pytest.mark.parametrize("zs", [False, True])
@pytest.mark.parametrize("mode,cmode", MODES)
def test_row_no_tokens(lib, mode, cmode, zs):
    """REDUCE_SCATTER over no rows gives a group with no output blocks."""
    x, w = shard((0, 256), 1, zero_strides=zs), shard((256, 192), 0)
    y = api._row_out(x, w, 0, mode, None)
    no_launch(lib, lambda: lib.dt_row_parallel_linear(C.byref(x._desc()), C.byref(w._desc()), None,
                                                      C.byref(y._desc()), cmode, 0, None, 0, None, None))


@pytest.mark.parametrize("zs", [False, True])
@pytest.mark.parametrize("mode,cmode", MODES[:2])
def test_mlp_no_tokens_needs_no_workspace(lib, mode, cmode, zs):
    """H of 0 rows takes 0 bytes: a NULL workspace is accepted."""
    x, wg, wu, wd = replicate((0, 256), zero_strides=zs), shard((256, 384), 1), shard((256, 384), 1), shard((384, 192), 0)
    y = api._row_out(x, wd, 0, mode, None)
    need = C.c_size_t(99)
    assert lib.dt_tp_mlp_workspace_size(C.byref(x._desc()), C.byref(wg._desc()), C.byref(wu._desc()),
                                        C.byref(wd._desc()), C.byref(y._desc()), cmode, 0, C.byref(need)) == L.OK
    assert need.value == 0
    no_launch(lib, lambda: lib.dt_tp_mlp(C.byref(x._desc()), C.byref(wg._desc()), C.byref(wu._desc()),
                                         C.byref(wd._desc()), C.byref(y._desc()), cmode, 0, None, 0, None, None))


@pytest.mark.parametrize("ids_shape,dim", [((2, 0), 512), ((0,), 4096), ((3, 5), 0)])
def test_embedding_nothing_to_gather(lib, ids_shape, dim):
    mesh = tsl.DeviceMesh((8,), ("tp",))
    table = shard((100, dim), 1, mesh)
    ids = replicate(ids_shape, torch.int32, mesh, zero_strides=True)
    out = tsl.DTensor.empty(mesh, [tsl.Replicate()], ids_shape + (dim,), BF, device="cpu")
    no_launch(lib, lambda: lib.dt_tp_embedding(C.byref(ids._desc()), C.byref(table._desc()), C.byref(out._desc()), 0,
                                               None, None))


def test_embedding_empty_vocabulary_refused(lib):
    """A table of no rows with tokens to gather: refused before any launch
    (every id would be out of range, and the slots hold no memory)."""
    mesh = tsl.DeviceMesh((8,), ("tp",))
    table = shard((0, 512), 1, mesh, zero_strides=True)
    ids = replicate((2, 3), torch.int32, mesh)
    out = tsl.DTensor.empty(mesh, [tsl.Replicate()], (2, 3, 512), BF, device="cpu")
    n0 = lib.dt_launch_count()
    st = lib.dt_tp_embedding(C.byref(ids._desc()), C.byref(table._desc()), C.byref(out._desc()), 0, None, None)
    assert st == L.ERR_SHAPE and b"no rows" in lib.dt_last_error()
    assert lib.dt_launch_count() == n0
