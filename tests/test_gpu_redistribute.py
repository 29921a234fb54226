"""GPU parity of dt_redistribute against the oracle: bit-exact, every element.

Covers every transition kind (Shard(a) <-> Shard(b), Shard <-> Replicate,
Partial -> Replicate / Shard, Replicate -> Partial, Partial -> Partial) on
random small meshes and shapes with ragged and empty shards, materialised
replicas, strided (view) slots, fp32 / bf16 / int32 data, the worked 2x2
example, and the full-size 8192 x 8192 and 8191 x 8190 sweep on a (2, 4)
mesh with the launch configuration the benchmark times.
"""
import random

import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import bf16
from oracle import placement as opl
from oracle import redistribute as ord_
from tensor_sharded_linear_gb300 import workloads

from helpers import (dtensor_from_locals, lib_placements, locals_of, random_placements, random_values,
                     sweep_transitions, to_dev)

pytestmark = pytest.mark.gpu

R, P = opl.Replicate(), opl.Partial()


def S(d):
    return opl.Shard(d)


def run_pair(src_locals, src: opl.Layout, dst: opl.Layout, dtype: str):
    expect = ord_.redistribute(src_locals, src, dst, dtype)
    dsrc = dtensor_from_locals(src_locals, src, dtype)
    out = dsrc.redistribute(lib_placements(dst.placements), materialize_replicas=dst.materialize_replicas)
    torch.cuda.synchronize()
    got = locals_of(out, dtype)
    assert len(got) == len(expect)
    for s, (g, e) in enumerate(zip(got, expect)):
        assert g.shape == e.shape, (s, g.shape, e.shape)
        np.testing.assert_array_equal(g, e, err_msg=f"slot {s}: {src.placements} -> {dst.placements}")


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("dtype", ["bf16", "fp32", "int32"])
def test_random_transitions(lib, seed, dtype):
    rng = random.Random(seed * 7 + len(dtype))
    nrng = np.random.default_rng(seed)
    for _ in range(12):
        nm = rng.randint(1, 3)
        mesh = tuple(rng.randint(1, 4) for _ in range(nm))
        nd = rng.randint(1, 3)
        gshape = tuple(rng.choice([1, 2, 3, 5, 7, 9, 16, 33, 70]) for _ in range(nd))
        allow_p = dtype != "int32"
        src = opl.Layout(mesh, random_placements(rng, nm, nd, allow_p), gshape, rng.random() < 0.25)
        dst = opl.Layout(mesh, random_placements(rng, nm, nd, allow_p), gshape, rng.random() < 0.25)
        src_locals = [random_values(src.local_shape(s), dtype, nrng) for s in range(src.nslots)]
        if src.materialize_replicas:  # replicas must agree: copy coordinate-0 values
            for s in range(src.nslots):
                c = list(src.slot_coords(s))
                for m, p in enumerate(src.placements):
                    if isinstance(p, opl.Replicate):
                        c[m] = 0
                src_locals[s] = src_locals[src.slot_of_coords(c)]
        try:
            ord_.redistribute(src_locals, src, dst, dtype)
        except NotImplementedError:
            continue
        run_pair(src_locals, src, dst, dtype)


def test_worked_2x2_example(lib):
    g = workloads.arange_f32((4, 4))
    a = opl.Layout((2, 2), [S(0), R], (4, 4))
    b = opl.Layout((2, 2), [R, S(1)], (4, 4))
    la = ord_.distribute(g, a, "fp32")
    run_pair(la, a, b, "fp32")
    lb = ord_.redistribute(la, a, b, "fp32")
    run_pair(lb, b, a, "fp32")
    # distribute_tensor on the device reproduces the printed per-rank values
    mesh = tsl.DeviceMesh((2, 2), ("dp", "tp"))
    d = tsl.DTensor.distribute_tensor(torch.arange(16, dtype=torch.float32, device="cuda").reshape(4, 4), mesh,
                                      [tsl.Shard(0), tsl.Replicate()])
    assert d.to_local(0).tolist() == [[0, 1, 2, 3], [4, 5, 6, 7]]
    assert d.to_local(3).tolist() == [[8, 9, 10, 11], [12, 13, 14, 15]]


def test_strided_view_slots(lib):
    """Slots that are column views of one parent buffer (non-unit row pitch)."""
    nrng = np.random.default_rng(4)
    gshape = (37, 52)
    src = opl.Layout((4,), [S(1)], gshape)
    dst = opl.Layout((4,), [S(0)], gshape)
    g = bf16.round_rne(nrng.standard_normal(gshape))
    parent = to_dev(g, "bf16")
    views = [parent[:, o:o + s] for o, s in opl.chunk_bounds(52, 4)]
    d = tsl.DTensor(views, tsl.DeviceMesh((4,)), [tsl.Shard(1)], gshape, torch.bfloat16)
    out = d.redistribute([tsl.Shard(0)])
    expect = ord_.redistribute(ord_.distribute(g, src, "bf16"), src, dst, "bf16")
    for t, e in zip(out.slots, expect):
        np.testing.assert_array_equal(t.cpu().view(torch.int16).numpy().view(np.uint16), e)


def test_empty_shards_and_tiny(lib):
    nrng = np.random.default_rng(5)
    for gshape, mesh in [((3, 5), (4,)), ((1,), (3,)), ((0, 4), (2,)), ((5, 1), (2, 3))]:
        for sp, dp in [([S(0)] * len(mesh), [R] * len(mesh)), ([R] * len(mesh), [S(len(gshape) - 1)] * len(mesh))]:
            src = opl.Layout(mesh, sp, gshape)
            dst = opl.Layout(mesh, dp, gshape)
            src_locals = [random_values(src.local_shape(s), "bf16", nrng) for s in range(src.nslots)]
            run_pair(src_locals, src, dst, "bf16")


@pytest.mark.parametrize("gshape", [(256, 320), (1000, 1030), (8192, 8192), (8191, 8190)])
def test_sweep_transitions(lib, gshape):
    mesh = workloads.REDISTRIBUTE["mesh"]
    g = workloads.redistribute_global(gshape)
    for name, sp, dp in sweep_transitions():
        src = opl.Layout(mesh, sp, gshape)
        dst = opl.Layout(mesh, dp, gshape)
        if any(isinstance(p, opl.Partial) for p in sp):
            src_locals = []
            for s in range(src.nslots):
                src_locals.append(workloads.redistribute_partials(src.local_shape(s), 1, seed=310 + s)[0])
        else:
            src_locals = ord_.distribute(g, src, "bf16")
        run_pair(src_locals, src, dst, "bf16")


@pytest.mark.parametrize("op", ["avg", "max"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_partial_avg_max_random(lib, op, dtype):
    """Partial(avg) / Partial(max) sources and destinations on random small
    layouts, bit-exact against the oracle."""
    rng = random.Random({"avg": 11, "max": 23}[op] + {"bf16": 0, "fp32": 100}[dtype])
    nrng = np.random.default_rng(17)
    done = 0
    for _ in range(60):
        nm = rng.randint(1, 3)
        mesh = tuple(rng.randint(1, 4) for _ in range(nm))
        nd = rng.randint(1, 3)
        gshape = tuple(rng.choice([1, 3, 7, 16, 33, 70]) for _ in range(nd))

        def pls():
            out = []
            for _ in range(nm):
                r = rng.random()
                out.append(S(rng.randrange(nd)) if r < 0.4 else (R if r < 0.65 else opl.Partial(op)))
            return out
        src = opl.Layout(mesh, pls(), gshape)
        dst = opl.Layout(mesh, pls(), gshape)
        src_locals = [random_values(src.local_shape(s), dtype, nrng) for s in range(src.nslots)]
        try:
            ord_.redistribute(src_locals, src, dst, dtype)
        except NotImplementedError:
            continue
        run_pair(src_locals, src, dst, dtype)
        done += 1
    assert done >= 10


@pytest.mark.parametrize("op", ["avg", "max"])
def test_partial_avg_max_full_size(lib, op):
    gshape = workloads.REDISTRIBUTE["shape"]
    mesh = workloads.REDISTRIBUTE["mesh"]
    for dp in ([S(0), R], [S(0), S(0)]):
        src = opl.Layout(mesh, [S(0), opl.Partial(op)], gshape)
        dst = opl.Layout(mesh, dp, gshape)
        src_locals = [workloads.redistribute_partials(src.local_shape(s), 1, seed=410 + s)[0] for s in range(src.nslots)]
        run_pair(src_locals, src, dst, "bf16")


@pytest.mark.parametrize("op", ["sum", "avg", "max"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_many_partial_sources(lib, op, dtype):
    """Partial on every dim of a (2, 3, 4) and a (4, 4, 4) mesh: 24 and 64
    sources per element, past the vector path's 16, still in rank order."""
    nrng = np.random.default_rng(31)
    for mesh, gshape in [((2, 3, 4), (37, 70)), ((4, 4, 4), (9, 33))]:
        src = opl.Layout(mesh, [opl.Partial(op)] * 3, gshape)
        for dp in ([R, R, R], [S(1), R, S(0)]):
            dst = opl.Layout(mesh, dp, gshape)
            src_locals = [random_values(src.local_shape(s), dtype, nrng) for s in range(src.nslots)]
            run_pair(src_locals, src, dst, dtype)


@pytest.mark.parametrize("gshape", [(8192, 8192), (8191, 8190), (70, 33)])
def test_materialised_replicas(lib, gshape):
    """Shard -> Replicate and Replicate -> Replicate with a copy per rank
    (each source box is read once and written to every replica), and back."""
    mesh = workloads.REDISTRIBUTE["mesh"]
    g = workloads.redistribute_global(gshape)
    for sp, dp, smat, dmat in (([S(0), S(0)], [S(0), R], False, True), ([S(0), S(1)], [S(0), R], False, True),
                               ([S(0), R], [R, R], True, True), ([S(0), R], [S(0), S(1)], True, False)):
        src = opl.Layout(mesh, sp, gshape, smat)
        dst = opl.Layout(mesh, dp, gshape, dmat)
        run_pair(ord_.distribute(g, src, "bf16"), src, dst, "bf16")


def test_materialised_replicas_strided_views(lib):
    """Replica slots with different strides are written by separate tasks."""
    gshape = (40, 52)
    g = bf16.round_rne(np.random.default_rng(8).standard_normal(gshape))
    mesh = tsl.DeviceMesh((4,))
    src = tsl.DTensor([to_dev(np.ascontiguousarray(g[o:o + s]), "bf16") for o, s in opl.chunk_bounds(40, 4)], mesh,
                      [tsl.Shard(0)], gshape, torch.bfloat16)
    parent = torch.zeros((40, 2 * 52), dtype=torch.bfloat16, device="cuda")
    slots = [torch.empty(gshape, dtype=torch.bfloat16, device="cuda"), parent[:, :52],
             torch.empty(gshape, dtype=torch.bfloat16, device="cuda"), parent[:, 52:]]
    dst = tsl.DTensor(slots, mesh, [tsl.Replicate()], gshape, torch.bfloat16, materialize_replicas=True)
    tsl.redistribute(src, dst)
    torch.cuda.synchronize()
    for t in dst.slots:
        np.testing.assert_array_equal(t.cpu().view(torch.int16).numpy().view(np.uint16), g)
