"""GPU parity of the bulk (TMA) copy kernel against the oracle: bit-exact.

Copy launches whose every row starts on a 16-byte boundary in source and
destination and is a multiple of 16 bytes long run on the bulk-copy engine
(global -> shared -> global, no thread touching the data); the others run
on the warp-per-segment copy kernel.  The cases reach every branch of the
bulk kernel: rows packed several to a work item and long rows cut into
segments, bf16 / fp32 / int32, three- and four-dimensional boxes whose rows
wrap the outer indices inside one work item, slots that are views of
parent buffers at 16-byte aligned offsets with padded pitches, batches of
several pairs, copies to materialised replicas (one staged row stored to
every replica), and a launch that mixes an aligned and an unaligned pair (it
takes the other kernel).  The same cases run with the bulk kernel turned
off (DT_RD_BULK=0, in a child process).
"""
import os
import random
import subprocess
import sys

import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import placement as opl
from oracle import redistribute as ord_

from helpers import dtensor_from_locals, lib_placements, locals_of, random_values, to_dev, to_host

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
R = opl.Replicate()
TD = {"bf16": torch.bfloat16, "fp32": torch.float32, "int32": torch.int32}


def S(d):
    return opl.Shard(d)


def run(src_locals, src: opl.Layout, dst: opl.Layout, dtype: str):
    expect = ord_.redistribute(src_locals, src, dst, dtype)
    out = dtensor_from_locals(src_locals, src, dtype).redistribute(lib_placements(dst.placements),
                                                                    materialize_replicas=dst.materialize_replicas)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    got = locals_of(out, dtype)
    for s, (g, e) in enumerate(zip(got, expect)):
        assert g.shape == e.shape
        np.testing.assert_array_equal(g, e, err_msg=f"{src.placements} -> {dst.placements} {src.gshape}: slot {s}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32", "int32"])
@pytest.mark.parametrize("gshape", [(64, 1024), (40, 4096), (12, 24576), (5, 40960)])
def test_aligned_shard_moves(lib, dtype, gshape):
    """Rows of 0.5 to 160 KB, all 16-byte aligned: packed and segmented items."""
    nrng = np.random.default_rng(sum(gshape))
    for mesh, pairs in [((4,), [([S(0)], [S(1)]), ([S(1)], [S(0)]), ([S(1)], [R]), ([R], [S(1)]), ([S(0)], [R])]),
                        ((2, 4), [([S(0), S(1)], [S(1), S(0)]), ([S(0), S(0)], [S(0), S(1)]),
                                  ([S(1), S(1)], [R, R]), ([R, S(1)], [S(0), S(1)])])]:
        for sp, dp in pairs:
            src, dst = opl.Layout(mesh, sp, gshape), opl.Layout(mesh, dp, gshape)
            g = random_values(gshape, dtype, nrng)
            run(ord_.distribute(g, src, dtype), src, dst, dtype)


@pytest.mark.parametrize("gshape,sp,dp", [
    ((6, 40, 512), [S(1), S(2)], [S(2), S(1)]),
    ((3, 7, 11, 256), [S(1), S(3)], [S(3), S(0)]),
    ((4, 32, 1024), [S(0), S(1)], [R, S(0)]),
    ((2, 6, 3, 4096), [S(2), R], [S(1), S(3)]),
])
def test_higher_rank_boxes(lib, gshape, sp, dp):
    """Boxes whose rows wrap two outer indices inside one work item."""
    nrng = np.random.default_rng(len(gshape))
    src, dst = opl.Layout((2, 2), sp, gshape), opl.Layout((2, 2), dp, gshape)
    g = random_values(gshape, "bf16", nrng)
    run(ord_.distribute(g, src, "bf16"), src, dst, "bf16")


@pytest.mark.parametrize("offset,pad", [(0, 0), (8, 8), (64, 24), (3, 5)])
def test_views_in_parent_buffers(lib, offset, pad):
    """Slots are views of parent buffers `offset` elements in, with `pad`
    spare elements per row: (8, 8) and (64, 24) keep every row 16-byte
    aligned (bulk kernel), (3, 5) does not (the other kernel)."""
    nrng = np.random.default_rng(offset + pad)
    gshape = (300, 2048)
    src, dst = opl.Layout((4,), [S(0)], gshape), opl.Layout((4,), [S(1)], gshape)
    g = random_values(gshape, "bf16", nrng)
    locals_ = ord_.distribute(g, src, "bf16")

    def view(shape):
        rows, cols = shape
        pitch = cols + pad
        parent = torch.zeros(rows * pitch + offset + 16, dtype=torch.bfloat16, device="cuda")
        return parent[offset:offset + rows * pitch].view(rows, pitch)[:, :cols]

    ins = []
    for a in locals_:
        v = view(a.shape)
        v.copy_(to_dev(a, "bf16"))
        ins.append(v)
    outs = [view(dst.local_shape(s)) for s in range(dst.nslots)]
    d = tsl.DTensor(ins, tsl.DeviceMesh((4,)), [tsl.Shard(0)], gshape, torch.bfloat16)
    out = tsl.DTensor(outs, tsl.DeviceMesh((4,)), [tsl.Shard(1)], gshape, torch.bfloat16)
    tsl.redistribute(d, out)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for s, (t, e) in enumerate(zip(out.slots, ord_.redistribute(locals_, src, dst, "bf16"))):
        np.testing.assert_array_equal(to_host(t, "bf16"), e, err_msg=f"slot {s}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("gshape", [(64, 1024), (12, 24576), (40, 2056)])
def test_materialised_replicas(lib, dtype, gshape):
    """Copies to a materialised Replicate layout (a slot per rank): each
    source row is staged once and stored to every replica.  Rows packed
    several to an item, long rows cut into segments, and (40, 2056) whose
    S(1) shards are 514 elements: bf16 rows of 1028 bytes are not 16-byte
    multiples (the other kernel), fp32 rows of 2056 bytes are."""
    nrng = np.random.default_rng(sum(gshape) + len(dtype))
    mesh = (2, 4)
    for sp, dp, smat, dmat in (([S(0), S(0)], [S(0), R], False, True), ([S(0), S(1)], [R, R], False, True),
                               ([S(0), R], [R, R], True, True), ([R, S(1)], [S(0), R], False, True)):
        src, dst = opl.Layout(mesh, sp, gshape, smat), opl.Layout(mesh, dp, gshape, dmat)
        g = random_values(gshape, dtype, nrng)
        run(ord_.distribute(g, src, dtype), src, dst, dtype)


@pytest.mark.parametrize("shift", [8, 4])
def test_replicas_at_any_distance(lib, shift):
    """Materialised replicas that are views of one parent buffer, `shift`
    elements apart from 16-byte boundaries: 8 bf16 (16 bytes) keeps every
    replica a multiple of 16 bytes from the first (bulk kernel), 4 (8 bytes)
    does not (the other kernel).  Bit-exact either way."""
    gshape = (64, 2048)
    g = random_values(gshape, "bf16", np.random.default_rng(shift))
    src_l = opl.Layout((4,), [S(0)], gshape)
    locals_ = ord_.distribute(g, src_l, "bf16")
    src = dtensor_from_locals(locals_, src_l, "bf16")
    n = gshape[0] * gshape[1]
    parent = torch.zeros(4 * n + 4 * shift + 64, dtype=torch.bfloat16, device="cuda")
    # replica k starts k * (n + shift) elements in: 16-byte aligned for k = 0
    slots = [parent[k * (n + shift):k * (n + shift) + n].view(gshape) for k in range(4)]
    dst = tsl.DTensor(slots, tsl.DeviceMesh((4,)), [tsl.Replicate()], gshape, torch.bfloat16,
                      materialize_replicas=True)
    tsl.redistribute(src, dst)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for k, t in enumerate(dst.slots):
        np.testing.assert_array_equal(to_host(t, "bf16"), g, err_msg=f"shift {shift} replica {k}")


def test_batches(lib):
    """Several aligned pairs in one launch; then the same with one unaligned pair added."""
    rng = random.Random(3)
    nrng = np.random.default_rng(3)
    for extra in (False, True):
        pairs, expects = [], []
        shapes = [(rng.choice([16, 64, 128]), rng.choice([1024, 4096, 8192, 20480])) for _ in range(5)]
        if extra:
            shapes.append((33, 1030))  # 1030 / 2 = 515-element shards: rows at every alignment
        for gshape in shapes:
            mesh = (2, 2)
            sp = [S(0), rng.choice([S(0), S(1), R])]
            dp = [rng.choice([S(0), R]), rng.choice([S(1), S(0)])]
            src, dst = opl.Layout(mesh, sp, gshape), opl.Layout(mesh, dp, gshape)
            loc = ord_.distribute(random_values(gshape, "bf16", nrng), src, "bf16")
            a = dtensor_from_locals(loc, src, "bf16")
            b = tsl.DTensor.empty(tsl.DeviceMesh(mesh), lib_placements(dp), gshape, torch.bfloat16)
            pairs.append((a, b))
            expects.append(ord_.redistribute(loc, src, dst, "bf16"))
        tsl.redistribute_batch(pairs)
        torch.cuda.synchronize()
        assert tsl.read_device_status() == 0
        for i, ((_, b), e) in enumerate(zip(pairs, expects)):
            for s, (t, x) in enumerate(zip(locals_of(b, "bf16"), e)):
                np.testing.assert_array_equal(t, x, err_msg=f"extra={extra} pair {i} slot {s}")


CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_gpu_redistribute_bulk as T
for dt in ("bf16", "fp32", "int32"):
    for g in [(64, 1024), (40, 4096), (12, 24576), (5, 40960)]:
        T.test_aligned_shard_moves(None, dt, g)
for args in [((6, 40, 512), [T.S(1), T.S(2)], [T.S(2), T.S(1)]), ((3, 7, 11, 256), [T.S(1), T.S(3)], [T.S(3), T.S(0)])]:
    T.test_higher_rank_boxes(None, *args)
for off, pad in ((8, 8), (3, 5)):
    T.test_views_in_parent_buffers(None, off, pad)
T.test_batches(None)
for dt in ("bf16", "fp32"):
    for g in [(64, 1024), (12, 24576), (40, 2056)]:
        T.test_materialised_replicas(None, dt, g)
for shift in (8, 4):
    T.test_replicas_at_any_distance(None, shift)
print("OK")
"""


def test_warp_copy_kernel_on_the_same_cases(lib):
    env = dict(os.environ, DT_RD_BULK="0")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "OK" in r.stdout
