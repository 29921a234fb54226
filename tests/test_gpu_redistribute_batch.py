"""GPU parity of dt_redistribute_batch against the oracle: bit-exact, every element.

The batch runs n independent redistributes in as few launches as the
parameter block holds.  Covered: the benchmark's full-size sweep (copies,
sums, ragged 8191 x 8190) as one call with its launch count, batches of
random layouts mixing meshes, shapes, dtypes and reduce ops, and batches
large enough to spill into several launches of each kind.
"""
import random

import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import placement as opl
from oracle import redistribute as ord_
from tensor_sharded_linear_gb300 import _lib as L
from tensor_sharded_linear_gb300 import workloads

from helpers import (TORCH_DTYPE, dtensor_from_locals, lib_placements, locals_of, random_placements, random_values,
                     sweep_transitions, to_dev)

pytestmark = pytest.mark.gpu


def make_pair(src_locals, src: opl.Layout, dst: opl.Layout, dtype: str):
    dsrc = dtensor_from_locals(src_locals, src, dtype)
    ddst = tsl.DTensor.empty(dsrc.mesh, lib_placements(dst.placements), dst.gshape, TORCH_DTYPE[dtype],
                             dst.materialize_replicas, device="cuda")
    # poison the outputs so a box the batch skips cannot match by accident
    for t in ddst.slots:
        t.view(torch.uint8).fill_(0xA5)
    return dsrc, ddst


def check(ddst, dtype, expect, what):
    got = locals_of(ddst, dtype)
    assert len(got) == len(expect)
    for s, (g, e) in enumerate(zip(got, expect)):
        assert g.shape == e.shape, (what, s, g.shape, e.shape)
        np.testing.assert_array_equal(g, e, err_msg=f"{what}, slot {s}")


def sweep_pairs(gshape):
    mesh = workloads.REDISTRIBUTE["mesh"]
    g = workloads.redistribute_global(gshape)
    out = []
    for name, sp, dp in sweep_transitions():
        src = opl.Layout(mesh, sp, gshape)
        dst = opl.Layout(mesh, dp, gshape)
        if any(isinstance(p, opl.Partial) for p in sp):
            src_locals = [workloads.redistribute_partials(src.local_shape(s), 1, seed=510 + s)[0]
                          for s in range(src.nslots)]
        else:
            src_locals = ord_.distribute(g, src, "bf16")
        out.append((f"{name} {gshape}", src_locals, src, dst))
    return out


def run_batch(cases, dtypes):
    pairs, expects = [], []
    for (what, src_locals, src, dst), dtype in zip(cases, dtypes):
        expects.append(ord_.redistribute(src_locals, src, dst, dtype))
        pairs.append(make_pair(src_locals, src, dst, dtype))
    lib = L.load()
    n0 = lib.dt_launch_count()
    tsl.redistribute_batch(pairs)
    launches = lib.dt_launch_count() - n0
    torch.cuda.synchronize()
    for (what, *_), (_, d), e, dtype in zip(cases, pairs, expects, dtypes):
        check(d, dtype, e, what)
    return launches


@pytest.mark.parametrize("gshapes", [[(256, 320)], [(8192, 8192), (8191, 8190)]])
def test_sweep_as_one_batch(lib, gshapes):
    """Every transition of the sweep, at each shape, in one call: one copy
    launch and one reduction launch when the parameter block holds them."""
    cases = [c for gs in gshapes for c in sweep_pairs(gs)]
    launches = run_batch(cases, ["bf16"] * len(cases))
    # at two shapes the 12 copy pairs need 72 slots a side and 192 boxes, the
    # 4 reduction pairs 20 + 32 slots and 80 partial references: one launch each
    assert launches == 2, launches


@pytest.mark.parametrize("seed", range(4))
def test_random_mixed_batches(lib, seed):
    rng = random.Random(900 + seed)
    nrng = np.random.default_rng(900 + seed)
    cases, dtypes = [], []
    while len(cases) < 24:
        dtype = rng.choice(["bf16", "fp32", "int32"])
        nm = rng.randint(1, 3)
        mesh = tuple(rng.randint(1, 4) for _ in range(nm))
        nd = rng.randint(1, 3)
        gshape = tuple(rng.choice([1, 2, 3, 5, 7, 9, 16, 33, 70]) for _ in range(nd))
        allow_p = dtype != "int32"
        sp = random_placements(rng, nm, nd, allow_p)
        dp = random_placements(rng, nm, nd, allow_p)
        if allow_p and rng.random() < 0.4:  # some avg / max reductions in the same batch
            op = rng.choice(["avg", "max"])
            sp = [opl.Partial(op) if isinstance(p, opl.Partial) else p for p in sp]
            dp = [opl.Partial(op) if isinstance(p, opl.Partial) else p for p in dp]
        src = opl.Layout(mesh, sp, gshape, rng.random() < 0.25)
        dst = opl.Layout(mesh, dp, gshape, rng.random() < 0.25)
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
        cases.append((f"case {len(cases)}: {src.placements} -> {dst.placements} {gshape}", src_locals, src, dst))
        dtypes.append(dtype)
    run_batch(cases, dtypes)


def test_batch_spills_into_several_launches(lib):
    """40 pairs on a 64-slot mesh: the slot tables overflow many times; each
    kind of work still lands, bit-exact."""
    nrng = np.random.default_rng(77)
    mesh = (4, 16)
    cases = []
    for i in range(40):
        gshape = (64 + i, 48 + 3 * i)
        if i % 3 == 2:
            sp, dp = [opl.Shard(0), opl.Partial()], [opl.Shard(1), opl.Replicate()]
        else:
            sp, dp = [opl.Shard(0), opl.Shard(1)], [opl.Shard(1), opl.Shard(0)]
        src = opl.Layout(mesh, sp, gshape)
        dst = opl.Layout(mesh, dp, gshape)
        src_locals = [random_values(src.local_shape(s), "fp32", nrng) for s in range(src.nslots)]
        cases.append((f"pair {i}", src_locals, src, dst))
    launches = run_batch(cases, ["fp32"] * len(cases))
    assert launches > 2, launches


def test_empty_batch_and_empty_pairs(lib):
    tsl.redistribute_batch([])
    nrng = np.random.default_rng(3)
    cases = []
    for gshape in [(0, 4), (3, 0), (5, 7)]:
        src = opl.Layout((2,), [opl.Shard(0)], gshape)
        dst = opl.Layout((2,), [opl.Replicate()], gshape)
        cases.append((str(gshape), [random_values(src.local_shape(s), "bf16", nrng) for s in range(2)], src, dst))
    run_batch(cases, ["bf16"] * 3)


def test_repeated_calls_replay_the_plan(lib):
    """A repeated call with the same operands replays its recorded launches:
    new source data each time, every result bit-exact, batch and single call,
    before and after dt_clear_cache."""
    mesh = (2, 4)
    gshape = (130, 70)
    cases = [("S0->S1", [opl.Shard(0), opl.Shard(0)], [opl.Shard(0), opl.Shard(1)]),
             ("P->S0", [opl.Shard(0), opl.Partial()], [opl.Shard(0), opl.Shard(0)])]
    layouts = [(opl.Layout(mesh, sp, gshape), opl.Layout(mesh, dp, gshape)) for _, sp, dp in cases]
    nrng = np.random.default_rng(61)
    first = [make_pair([random_values(src.local_shape(s), "bf16", nrng) for s in range(src.nslots)], src, dst, "bf16")
             for src, dst in layouts]
    lib_ = L.load()
    for rnd in range(4):
        if rnd == 2:
            assert lib_.dt_clear_cache() == L.OK
        locals_ = []
        for (dsrc, _), (src, _) in zip(first, layouts):  # fresh data in the same buffers
            loc = [random_values(src.local_shape(s), "bf16", nrng) for s in range(src.nslots)]
            for t, a in zip(dsrc.slots, loc):
                t.copy_(to_dev(a, "bf16"))
            locals_.append(loc)
        if rnd % 2 == 0:
            tsl.redistribute_batch(first)
        else:
            for dsrc, ddst in first:
                tsl.redistribute(dsrc, ddst)
        torch.cuda.synchronize()
        for (_, ddst), (src, dst), loc in zip(first, layouts, locals_):
            check(ddst, "bf16", ord_.redistribute(loc, src, dst, "bf16"), f"round {rnd}")
