"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol ``include/dt.h`` declares, answers layout queries like the oracle, and
rejects bad calls on the host before any launch."""
import ctypes as C
import os
import random
import re

import pytest

from oracle import placement as opl
from tensor_sharded_linear_gb300 import _lib as L

from test_oracle_placement import random_layout

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dt.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^DT_API\s+[\w\s\*]+?\b(dt_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(L.EXPORTS)


def abi_layout(lay: opl.Layout, dtype=L.BF16):
    a = L.Layout()
    a.mesh_ndim = len(lay.mesh_shape)
    for m, s in enumerate(lay.mesh_shape):
        a.mesh_shape[m] = s
    for m, p in enumerate(lay.placements):
        if isinstance(p, opl.Shard):
            a.placements[m].kind, a.placements[m].dim = L.SHARD, p.dim
        elif isinstance(p, opl.Replicate):
            a.placements[m].kind = L.REPLICATE
        else:
            a.placements[m].kind = L.PARTIAL
    a.ndim = len(lay.gshape)
    for d, s in enumerate(lay.gshape):
        a.gshape[d] = s
    a.dtype = dtype
    a.materialize_replicas = int(lay.materialize_replicas)
    return a


def test_layout_queries_match_oracle(lib):
    rng = random.Random(3)
    for _ in range(400):
        lay = random_layout(rng)
        a = abi_layout(lay)
        n = C.c_int32()
        assert lib.dt_layout_nslots(C.byref(a), C.byref(n)) == L.OK
        assert n.value == lay.nslots
        for r in range(opl.mesh_size(lay.mesh_shape)):
            s = C.c_int32()
            assert lib.dt_layout_slot_of_rank(C.byref(a), r, C.byref(s)) == L.OK
            assert s.value == lay.slot_of_rank(r)
        for s in range(lay.nslots):
            ls = (C.c_int64 * 4)()
            go = (C.c_int64 * 4)()
            assert lib.dt_layout_slot_box(C.byref(a), s, ls, go) == L.OK
            box = lay.box(s)
            nd = len(lay.gshape)
            assert tuple(ls[:nd]) == tuple(sz for _, sz in box)
            assert tuple(go[:nd]) == tuple(o for o, _ in box)


def test_malformed_layouts_are_rejected(lib):
    a = abi_layout(opl.Layout((2, 2), [opl.Shard(0), opl.Replicate()], (4, 4)))
    a.placements[0].dim = 5
    n = C.c_int32()
    assert lib.dt_layout_nslots(C.byref(a), C.byref(n)) == L.ERR_INVALID_ARG
    assert b"Shard(5)" in lib.dt_last_error()
    a = abi_layout(opl.Layout((2,), [opl.Shard(0)], (4,)))
    a.mesh_shape[0] = 0
    assert lib.dt_layout_nslots(C.byref(a), C.byref(n)) == L.ERR_INVALID_ARG
    a = abi_layout(opl.Layout((2,), [opl.Shard(0)], (4,)))
    a.dtype = 9
    assert lib.dt_layout_nslots(C.byref(a), C.byref(n)) == L.ERR_INVALID_ARG
    s = C.c_int32()
    a = abi_layout(opl.Layout((2,), [opl.Shard(0)], (4,)))
    assert lib.dt_layout_slot_of_rank(C.byref(a), 2, C.byref(s)) == L.ERR_INVALID_ARG


_FAKE = 0x7F0000000000  # never dereferenced: every call below fails on the host


def fake_desc(lay: opl.Layout, dtype=L.BF16):
    d = L.DTensorDesc()
    d.layout = abi_layout(lay, dtype)
    d.nslots = lay.nslots
    ptrs = (C.c_void_p * lay.nslots)(*[_FAKE + 4096 * i for i in range(lay.nslots)])
    d.slots = C.cast(ptrs, C.POINTER(C.c_void_p))
    d.strides = None
    d._keep = ptrs
    return d


def test_host_rejections_before_launch(lib):
    mesh = (4,)
    R, S0, S1, P = opl.Replicate(), opl.Shard(0), opl.Shard(1), opl.Partial()
    # Shard -> Partial is not defined
    src = fake_desc(opl.Layout(mesh, [S0], (8, 8)))
    dst = fake_desc(opl.Layout(mesh, [P], (8, 8)))
    assert lib.dt_redistribute(C.byref(src), C.byref(dst), None, None) == L.ERR_UNSUPPORTED
    # global shapes must agree
    dst = fake_desc(opl.Layout(mesh, [R], (8, 9)))
    assert lib.dt_redistribute(C.byref(src), C.byref(dst), None, None) == L.ERR_SHAPE
    # wrong slot count
    bad = fake_desc(opl.Layout(mesh, [S0], (8, 8)))
    bad.nslots = 3
    assert lib.dt_redistribute(C.byref(bad), C.byref(src), None, None) == L.ERR_INVALID_ARG
    # a batch is checked pair by pair before anything launches; the error names the pair
    ok_s = fake_desc(opl.Layout(mesh, [S0], (8, 8)))
    ok_d = fake_desc(opl.Layout(mesh, [S1], (8, 8)))
    srcs = (L.DTensorDesc * 2)(ok_s, src)
    dsts = (L.DTensorDesc * 2)(ok_d, fake_desc(opl.Layout(mesh, [P], (8, 8))))
    assert lib.dt_redistribute_batch(2, srcs, dsts, None, None) == L.ERR_UNSUPPORTED
    assert lib.dt_last_error().startswith(b"pair 1:")
    assert lib.dt_redistribute_batch(0, None, None, None, None) == L.OK
    assert lib.dt_redistribute_batch(-1, srcs, dsts, None, None) == L.ERR_INVALID_ARG
    assert lib.dt_redistribute_batch(1, None, dsts, None, None) == L.ERR_INVALID_ARG
    # column-parallel input must be Replicate on tp (DTorch check_placement)
    x = fake_desc(opl.Layout(mesh, [S1], (16, 32)))
    w = fake_desc(opl.Layout(mesh, [S1], (32, 64)))
    y = fake_desc(opl.Layout(mesh, [S1], (16, 64)))
    assert lib.dt_column_parallel_linear(C.byref(x), C.byref(w), None, C.byref(y), 0, None, 0, None, None) == L.ERR_PLACEMENT
    assert b"Replicate" in lib.dt_last_error()
    # row-parallel input must be Shard(-1) on tp
    xr = fake_desc(opl.Layout(mesh, [R], (16, 32)))
    wr = fake_desc(opl.Layout(mesh, [S0], (32, 64)))
    yr = fake_desc(opl.Layout(mesh, [R], (16, 64)))
    assert lib.dt_row_parallel_linear(C.byref(xr), C.byref(wr), None, C.byref(yr), L.TP_ALL_REDUCE, 0, None, 0,
                                      None, None) == L.ERR_PLACEMENT
    # REDUCE_SCATTER output must be Shard(0)
    xs = fake_desc(opl.Layout(mesh, [S1], (16, 32)))
    assert lib.dt_row_parallel_linear(C.byref(xs), C.byref(wr), None, C.byref(yr), L.TP_REDUCE_SCATTER, 0, None, 0,
                                      None, None) == L.ERR_PLACEMENT
    # shape mismatch: w rows != x cols
    w_bad = fake_desc(opl.Layout(mesh, [S0], (31, 64)))
    assert lib.dt_row_parallel_linear(C.byref(xs), C.byref(w_bad), None, C.byref(yr), L.TP_ALL_REDUCE, 0, None, 0,
                                      None, None) == L.ERR_SHAPE
    # bad mode
    assert lib.dt_row_parallel_linear(C.byref(xs), C.byref(wr), None, C.byref(yr), 7, 0, None, 0, None, None) \
        == L.ERR_INVALID_ARG
    # embedding: table must be Shard(1) on tp
    ids = fake_desc(opl.Layout(mesh, [R], (2, 3)), L.INT32)
    table = fake_desc(opl.Layout(mesh, [S0], (100, 16)))
    out = fake_desc(opl.Layout(mesh, [R], (2, 3, 16)))
    assert lib.dt_tp_embedding(C.byref(ids), C.byref(table), C.byref(out), 0, None, None) == L.ERR_PLACEMENT


def test_gemm_dimensions_beyond_32_bits_are_refused(lib):
    """The GEMM's M, N and coordinates are 32-bit on the device: an
    activation with 2^31 rows (32 GB in bf16, so it fits a GB300) is refused
    on the host before anything launches, not truncated."""
    mesh = (4,)
    R, S1 = opl.Replicate(), opl.Shard(1)
    big = 1 << 31
    x = fake_desc(opl.Layout(mesh, [R], (big, 8)))
    w = fake_desc(opl.Layout(mesh, [S1], (8, 64)))
    y = fake_desc(opl.Layout(mesh, [S1], (big, 64)))
    assert lib.dt_column_parallel_linear(C.byref(x), C.byref(w), None, C.byref(y), 0, None, 0, None, None) == L.ERR_CAPACITY
    assert b"2^31" in lib.dt_last_error()
    # row-parallel with K = 2^31 (x Shard(-1), w Shard(0) on tp)
    S0 = opl.Shard(0)
    xr = fake_desc(opl.Layout(mesh, [S1], (8, big)))
    wr = fake_desc(opl.Layout(mesh, [S0], (big, 64)))
    yr = fake_desc(opl.Layout(mesh, [R], (8, 64)))
    assert lib.dt_row_parallel_linear(C.byref(xr), C.byref(wr), None, C.byref(yr), L.TP_ALL_REDUCE, 0, None, 0,
                                      None, None) == L.ERR_CAPACITY
    assert b"2^31" in lib.dt_last_error()


def test_status_strings(lib):
    for s in range(8):
        assert lib.dt_status_string(s)
    assert lib.dt_version() >= 100


def test_workspace_queries_on_host(lib):
    """The linears' workspace queries check their operands as the calls do,
    before anything touches a device; the CUDA-core path (fp32) needs no
    workspace on any device; a bf16 problem's answer depends on the device's
    CTA pairs, so without a CUDA device it is DT_ERR_CUDA."""
    import torch
    mesh = (4,)
    R, S0, S1 = opl.Replicate(), opl.Shard(0), opl.Shard(1)
    n = C.c_size_t(123)
    # column: x Replicate, w Shard(1), y Shard(-1)
    x = fake_desc(opl.Layout(mesh, [R], (512, 256)))
    w = fake_desc(opl.Layout(mesh, [S1], (256, 1024)))
    y = fake_desc(opl.Layout(mesh, [S1], (512, 1024)))
    assert lib.dt_column_parallel_linear_workspace_size(C.byref(x), 1, C.byref(w), C.byref(y), 0, None) \
        == L.ERR_INVALID_ARG
    assert lib.dt_column_parallel_linear_workspace_size(C.byref(x), 0, C.byref(w), C.byref(y), 0, C.byref(n)) \
        == L.ERR_INVALID_ARG
    bad_x = fake_desc(opl.Layout(mesh, [S1], (512, 256)))
    assert lib.dt_column_parallel_linear_workspace_size(C.byref(bad_x), 1, C.byref(w), C.byref(y), 0,
                                                        C.byref(n)) == L.ERR_PLACEMENT
    # fp32 operands run on the CUDA-core kernel: no workspace, on any device
    x32 = fake_desc(opl.Layout(mesh, [R], (512, 256)), L.FP32)
    w32 = fake_desc(opl.Layout(mesh, [S1], (256, 1024)), L.FP32)
    y32 = fake_desc(opl.Layout(mesh, [S1], (512, 1024)), L.FP32)
    assert lib.dt_column_parallel_linear_workspace_size(C.byref(x32), 1, C.byref(w32), C.byref(y32), 0,
                                                        C.byref(n)) == L.OK
    assert n.value == 0
    # row: x Shard(-1), w Shard(0), y per mode
    xr = fake_desc(opl.Layout(mesh, [S1], (512, 1024)))
    wr = fake_desc(opl.Layout(mesh, [S0], (1024, 256)))
    yr = fake_desc(opl.Layout(mesh, [R], (512, 256)))
    ys = fake_desc(opl.Layout(mesh, [S0], (512, 256)))
    assert lib.dt_row_parallel_linear_workspace_size(C.byref(xr), C.byref(wr), C.byref(ys), L.TP_ALL_REDUCE, 0,
                                                     C.byref(n)) == L.ERR_PLACEMENT
    assert lib.dt_row_parallel_linear_workspace_size(C.byref(xr), C.byref(wr), C.byref(yr), 9, 0, C.byref(n)) \
        == L.ERR_INVALID_ARG
    # MLP: bf16 only
    mlp = [fake_desc(opl.Layout(mesh, [R], (512, 256)), L.FP32), fake_desc(opl.Layout(mesh, [S1], (256, 1024))),
           fake_desc(opl.Layout(mesh, [S1], (256, 1024))), fake_desc(opl.Layout(mesh, [S0], (1024, 256))),
           fake_desc(opl.Layout(mesh, [R], (512, 256)))]
    assert lib.dt_tp_mlp_workspace_size(*[C.byref(d) for d in mlp], L.TP_ALL_REDUCE, 0, C.byref(n)) \
        == L.ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert lib.dt_column_parallel_linear_workspace_size(C.byref(x), 1, C.byref(w), C.byref(y), 0,
                                                            C.byref(n)) == L.ERR_CUDA
        assert b"CUDA device" in lib.dt_last_error()
        assert lib.dt_row_parallel_linear_workspace_size(C.byref(xr), C.byref(wr), C.byref(yr), L.TP_ALL_REDUCE, 0,
                                                         C.byref(n)) == L.ERR_CUDA


def test_linear_workspace_alignment_checked_first(lib):
    """A workspace must be 256-byte aligned; a misaligned one is refused before
    any operand is read or anything launches."""
    mesh = (4,)
    R, S1 = opl.Replicate(), opl.Shard(1)
    x = fake_desc(opl.Layout(mesh, [R], (16, 32)))
    w = fake_desc(opl.Layout(mesh, [S1], (32, 64)))
    y = fake_desc(opl.Layout(mesh, [S1], (16, 64)))
    assert lib.dt_column_parallel_linear(C.byref(x), C.byref(w), None, C.byref(y), 0, _FAKE + 16, 1 << 20, None,
                                         None) == L.ERR_ALIGNMENT
    xr = fake_desc(opl.Layout(mesh, [S1], (16, 32)))
    wr = fake_desc(opl.Layout(mesh, [opl.Shard(0)], (32, 64)))
    yr = fake_desc(opl.Layout(mesh, [R], (16, 64)))
    assert lib.dt_row_parallel_linear(C.byref(xr), C.byref(wr), None, C.byref(yr), L.TP_ALL_REDUCE, 0, _FAKE + 8,
                                      1 << 20, None, None) == L.ERR_ALIGNMENT


def test_mlp_workspace_checked_before_launch(lib):
    """dt_tp_mlp needs at least H's bytes of 256-byte aligned workspace; a
    missing, short or misaligned one is refused on the host."""
    mesh = (4,)
    R, S0, S1 = opl.Replicate(), opl.Shard(0), opl.Shard(1)
    descs = [fake_desc(opl.Layout(mesh, [R], (512, 256))), fake_desc(opl.Layout(mesh, [S1], (256, 1024))),
             fake_desc(opl.Layout(mesh, [S1], (256, 1024))), fake_desc(opl.Layout(mesh, [S0], (1024, 256))),
             fake_desc(opl.Layout(mesh, [R], (512, 256)))]
    args = [C.byref(d) for d in descs] + [L.TP_ALL_REDUCE, 0]
    h_bytes = 512 * 1024 * 2
    assert lib.dt_tp_mlp(*args, None, 0, None, None) == L.ERR_INVALID_ARG
    assert str(h_bytes).encode() in lib.dt_last_error()
    assert lib.dt_tp_mlp(*args, _FAKE, h_bytes - 256, None, None) == L.ERR_INVALID_ARG
    assert lib.dt_tp_mlp(*args, _FAKE + 128, h_bytes, None, None) == L.ERR_ALIGNMENT
