"""Guard bands around every output: the kernels write their outputs and
nothing else.

Each output slot is a view inside a larger device buffer filled with a
sentinel byte: 4 KiB before and after it, and, where the view's row pitch is
wider than its rows, the gap at the end of every row.  After the call every
byte outside the view's elements must still hold the sentinel.  This stands
in for a memory checker on the paths most exposed to an off-by-one: ragged
GEMM tiles in every row mode (masked stores, REDUCE_SCATTER row routing),
split-tail launches (partials and counters in the workspace, which is
guarded too), the MLP's H in its workspace, uneven realigned redistribute
copies (both copy kernels' shapes), materialised replicas, and embedding
rows zero-filled for out-of-range ids.  Every result is also checked
against the oracle.
"""
import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import linear as olin
from oracle import placement as opl
from oracle import redistribute as ord_
from oracle.embedding import tp_embedding as oracle_embedding
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import dtensor_from_locals, to_dev, to_host
from test_gpu_linear import check_bf16, check_fp32, col_dtensor, mesh1, row_dtensor, w64, x_rep, x_shard

pytestmark = pytest.mark.gpu

SENTINEL = 0xA5
BAND = 4096
ESIZE = {torch.bfloat16: 2, torch.float32: 4, torch.int32: 4}


class Guarded:
    """A [rows, cols] (or 1-D) view in a sentinel-filled buffer, row pitch
    cols + pad elements, BAND bytes of sentinel on both sides."""

    def __init__(self, shape, dtype, pad=0):
        self.shape, self.dtype, self.pad = tuple(shape), dtype, pad
        e = ESIZE[dtype]
        rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
        cols = shape[-1]
        self.rows, self.cols, self.pitch = rows, cols, cols + pad
        nbytes = rows * self.pitch * e
        self.buf = torch.full((BAND + nbytes + BAND,), SENTINEL, dtype=torch.uint8, device="cuda")
        flat = self.buf[BAND:BAND + nbytes].view(dtype)
        v = flat.view(rows, self.pitch)[:, :cols]
        self.view = v.view(shape) if len(shape) != 2 else v  # a view of the buffer, never a copy
        if len(shape) == 1:
            self.view = flat[:cols]

    def check(self, what):
        host = self.buf.cpu().numpy()
        e = ESIZE[self.dtype]
        mask = np.ones(host.shape, dtype=bool)
        inner = mask[BAND:BAND + self.rows * self.pitch * e].reshape(self.rows, self.pitch * e)
        inner[:, :self.cols * e] = False
        bad = np.nonzero(mask & (host != SENTINEL))[0]
        assert bad.size == 0, f"{what}: {bad.size} guard bytes overwritten, first at offset {int(bad[0]) - BAND}"


def guarded_like(mesh, placements, gshape, dtype, pad=0, materialize=False):
    """An empty DTensor whose slots are guarded views; returns (dtensor, guards)."""
    probe = tsl.DTensor.empty(mesh, placements, gshape, dtype, materialize_replicas=materialize)
    guards = [Guarded(tuple(t.shape), dtype, pad) for t in probe.slots]
    return tsl.DTensor([g.view for g in guards], mesh, placements, gshape, dtype, materialize), guards


def guarded_workspace(nbytes):
    """A workspace of nbytes (256-byte aligned) between two sentinel bands."""
    buf = torch.full((BAND + nbytes + BAND,), SENTINEL, dtype=torch.uint8, device="cuda")
    return buf, buf[BAND:BAND + nbytes]


def check_workspace_guard(buf, nbytes, what):
    host = buf.cpu().numpy()
    assert (host[:BAND] == SENTINEL).all() and (host[BAND + nbytes:] == SENTINEL).all(), f"{what}: workspace guard"


@pytest.mark.parametrize("pad", [0, 8, 3])
def test_column_ragged_tiles(lib, pad):
    """M, N and K off the tile grid; output pitch padded (aligned and not)."""
    M, K, N, p = 300, 200, 4 * 264 + 8, 4
    x = workloads.randn_bf16((M, K), 901)
    w = workloads.randn_bf16((K, N), 902, (1.0 / K) ** 0.5)
    xd, wd = x_rep(x, p), col_dtensor(w, p)
    y, guards = guarded_like(mesh1(p), [tsl.Shard(1)], (M, N), torch.float32, pad)
    tsl.column_parallel_linear(xd, wd, out=y)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for i, g in enumerate(guards):
        g.check(f"shard {i}")
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"shard {i}")


@pytest.mark.parametrize("mode", [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER, tsl.PARTIAL])
def test_row_modes_ragged(lib, mode):
    M, K, N, p = 517, 4 * 200, 8 * 41, 4
    x = workloads.randn_bf16((M, K), 911)
    w = workloads.randn_bf16((K, N), 912, (1.0 / K) ** 0.5)
    xd, wd = x_shard(x, p), row_dtensor(w, p)
    pl = {tsl.ALL_REDUCE: tsl.Replicate(), tsl.REDUCE_SCATTER: tsl.Shard(0), tsl.PARTIAL: tsl.Partial()}[mode]
    y, guards = guarded_like(mesh1(p), [pl], (M, N), torch.bfloat16, pad=8)
    tsl.row_parallel_linear(xd, wd, mode=mode, out=y)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for i, g in enumerate(guards):
        g.check(f"{mode} out {i}")
    omode = {tsl.ALL_REDUCE: olin.ALL_REDUCE, tsl.REDUCE_SCATTER: olin.REDUCE_SCATTER, tsl.PARTIAL: olin.PARTIAL}[mode]
    expect = olin.row_parallel([w64(x[:, o:o + s]) for o, s in chunk_bounds(K, p)],
                               [w64(w[o:o + s]) for o, s in chunk_bounds(K, p)], None, omode, parts=p)
    for i, e in enumerate(expect):
        got = to_host(y.slots[i], "bf16")
        assert got.shape == e.shape
        assert (np.abs(w64(got) - e) <= 2e-3 + 2.0 ** -8 * np.abs(e)).all(), f"{mode} out {i}"


def test_split_tail_outputs_and_workspace(lib):
    """A split column launch: outputs and the workspace's neighbours untouched."""
    M, K, N, p = 300, 12000, 4 * 520, 4
    x = workloads.randn_bf16((M, K), 921)
    w = workloads.randn_bf16((K, N), 922, (1.0 / K) ** 0.5)
    xd, wd = x_rep(x, p), col_dtensor(w, p)
    y, guards = guarded_like(mesh1(p), [tsl.Shard(1)], (M, N), torch.float32, pad=4)
    need = tsl.column_parallel_linear_workspace_bytes(xd, [wd], [y])
    assert need > 0
    buf, ws = guarded_workspace(need)
    for _ in range(2):
        tsl.column_parallel_linear(xd, wd, out=y, workspace=ws)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    check_workspace_guard(buf, need, "split column")
    for i, g in enumerate(guards):
        g.check(f"shard {i}")
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"shard {i}")


def test_mlp_workspace_and_output(lib):
    """H and the down projection's split scratch stay inside the MLP's workspace."""
    M, K, F, N, p = 512, 256, 8 * 1024, 2560, 8
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=930)
    wd = workloads.randn_bf16((F, N), 934, (1.0 / F) ** 0.5)
    xd, wgd, wud, wdd = x_rep(x, p), col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    y, guards = guarded_like(mesh1(p), [tsl.Replicate()], (M, N), torch.float32, pad=4)
    need = tsl.tp_mlp_workspace_bytes(xd, wgd, wud, wdd, y)
    buf, ws = guarded_workspace(need)
    tsl.tp_mlp(xd, wgd, wud, wdd, out=y, workspace=ws)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    check_workspace_guard(buf, need, "mlp")
    guards[0].check("mlp output")
    cols = chunk_bounds(F, p)
    (expect,), _ = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols],
                               [w64(wd[o:o + s]) for o, s in cols])
    check_fp32(to_host(y.slots[0], "fp32"), expect, "mlp")


@pytest.mark.parametrize("gshape", [(8191, 8190), (1031, 2049)])
def test_uneven_redistribute_copies(lib, gshape):
    """Every sweep transition on an uneven shape into guarded, padded slots."""
    mesh = (2, 4)
    g = workloads.redistribute_global(gshape)
    for sp, dp in [([opl.Shard(0), opl.Shard(0)], [opl.Shard(0), opl.Shard(1)]),
                   ([opl.Shard(0), opl.Shard(1)], [opl.Shard(0), opl.Shard(0)]),
                   ([opl.Shard(0), opl.Shard(1)], [opl.Shard(0), opl.Replicate()]),
                   ([opl.Shard(0), opl.Replicate()], [opl.Shard(0), opl.Shard(1)]),
                   ([opl.Shard(0), opl.Partial()], [opl.Shard(0), opl.Shard(0)])]:
        src, dst = opl.Layout(mesh, sp, gshape), opl.Layout(mesh, dp, gshape)
        if isinstance(sp[1], opl.Partial):
            loc = [workloads.redistribute_partials(src.local_shape(s), 1, seed=310 + s)[0] for s in range(src.nslots)]
        else:
            loc = ord_.distribute(g, src, "bf16")
        d = dtensor_from_locals(loc, src, "bf16")
        out, guards = guarded_like(tsl.DeviceMesh(mesh), [lib_pl(p) for p in dp], gshape, torch.bfloat16, pad=3)
        tsl.redistribute(d, out)
        torch.cuda.synchronize()
        for i, gd in enumerate(guards):
            gd.check(f"{sp} -> {dp} slot {i}")
        for i, (t, e) in enumerate(zip(out.slots, ord_.redistribute(loc, src, dst, "bf16"))):
            np.testing.assert_array_equal(to_host(t, "bf16"), e, err_msg=f"{sp} -> {dp} slot {i}")


def lib_pl(p):
    if isinstance(p, opl.Shard):
        return tsl.Shard(p.dim)
    if isinstance(p, opl.Replicate):
        return tsl.Replicate()
    return tsl.Partial()


def test_materialised_replicas(lib):
    gshape, mesh = (1025, 3000), (2, 4)
    src = opl.Layout(mesh, [opl.Shard(0), opl.Shard(1)], gshape)
    dst = opl.Layout(mesh, [opl.Shard(0), opl.Replicate()], gshape, True)
    loc = ord_.distribute(workloads.redistribute_global(gshape), src, "bf16")
    d = dtensor_from_locals(loc, src, "bf16")
    out, guards = guarded_like(tsl.DeviceMesh(mesh), [tsl.Shard(0), tsl.Replicate()], gshape, torch.bfloat16, pad=5,
                               materialize=True)
    tsl.redistribute(d, out)
    torch.cuda.synchronize()
    for i, gd in enumerate(guards):
        gd.check(f"replica {i}")
    for i, (t, e) in enumerate(zip(out.slots, ord_.redistribute(loc, src, dst, "bf16"))):
        np.testing.assert_array_equal(to_host(t, "bf16"), e, err_msg=f"replica {i}")


def test_embedding_out_of_range_ids(lib):
    table, ids = workloads.embedding_inputs(vocab=500, dim=520, ids_shape=(3, 50), seed_base=940)
    ids = ids.copy()
    ids[0, 0], ids[2, 49], ids[1, 7] = 500, -1, 1 << 30
    p = 8
    mesh = mesh1(p)
    shards = [np.ascontiguousarray(table[:, o:o + s]) for o, s in chunk_bounds(520, p)]
    tdt = tsl.DTensor([to_dev(s, "bf16") for s in shards], mesh, [tsl.Shard(1)], table.shape, torch.bfloat16)
    idt = tsl.DTensor([to_dev(ids, "int32")], mesh, [tsl.Replicate()], ids.shape, torch.int32)
    out, guards = guarded_like(mesh, [tsl.Replicate()], ids.shape + (520,), torch.bfloat16, pad=6)
    tsl.read_device_status(clear=True)
    tsl.tp_embedding(idt, tdt, out=out)
    status = tsl.read_device_status(clear=True)
    assert status & tsl._lib.DEV_ERR_INDEX
    guards[0].check("embedding")
    expect, bad = oracle_embedding(ids, shards, 520)
    assert bad
    np.testing.assert_array_equal(to_host(out.slots[0], "bf16"), expect)
