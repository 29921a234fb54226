"""Pins for the oracle's placement arithmetic (CPU only).

Pinned against: the per-rank values printed by the Hyper-Parallel DTensor API
for ``distribute_tensor`` (tests/golden/distribute_tensor_2x2.txt), the shape
examples printed there (tests/golden/shape_examples.txt), ``torch.chunk``
(the library routine the wineandchord reference shards with), numpy's
row-major ``unravel_index``, and the coverage invariant stated by the
wineandchord page (every shard covers each global index exactly once).
"""
import os
import random

import numpy as np
import pytest
import torch

from oracle import placement as pl
from oracle import redistribute as rd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_placements(text):
    out = []
    for tok in text.split(","):
        tok = tok.strip()
        if tok == "R":
            out.append(pl.Replicate())
        elif tok.startswith("S"):
            out.append(pl.Shard(int(tok[1:])))
        elif tok == "P":
            out.append(pl.Partial())
    return out


def check_printed_distribute(placement=pl, redistribute=rd):
    rows = {}
    with open(os.path.join(GOLDEN, "distribute_tensor_2x2.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rank, body = line.split(":")
            rows[int(rank)] = np.array([[float(v) for v in r.split()] for r in body.split(";")], dtype=np.float32)
    g = np.arange(16, dtype=np.float32).reshape(4, 4)
    lay = placement.Layout((2, 2), [placement.Shard(0), placement.Replicate()], (4, 4))
    locals_ = redistribute.distribute(g, lay, "fp32")
    for rank, expect in rows.items():
        np.testing.assert_array_equal(locals_[lay.slot_of_rank(rank)], expect)


def test_printed_distribute_tensor_values():
    check_printed_distribute()


def test_printed_shape_examples():
    with open(os.path.join(GOLDEN, "shape_examples.txt")) as f:
        lines = [l for l in f if l.strip() and not l.startswith("#")]
    assert len(lines) == 3
    for line in lines:
        name, mesh, pls, gshape, lshape, _src = [t.strip() for t in line.split("|")]
        mesh = tuple(int(v) for v in mesh.split(","))
        pls = _parse_placements(pls)
        gshape = tuple(int(v) for v in gshape.split(","))
        lshape = tuple(int(v) for v in lshape.split(","))
        lay = pl.Layout(mesh, pls, gshape)
        for s in range(lay.nslots):
            assert lay.local_shape(s) == lshape, name
        assert pl.global_shape_from_local(lshape, mesh, lay.placements) == gshape, name


def check_chunk_matches_torch(placement=pl):
    for n in range(1, 41):
        for p in range(1, 10):
            chunks = torch.chunk(torch.arange(n), p)
            expect = [(int(c[0]), len(c)) for c in chunks]
            got = placement.chunk_bounds(n, p)
            assert len(got) == p
            assert got[:len(expect)] == expect, (n, p)
            # the missing trailing chunks are empty
            assert all(s == 0 for _, s in got[len(expect):]), (n, p)


def test_chunk_matches_torch_chunk():
    check_chunk_matches_torch()


def test_rank_order_is_row_major():
    for shape in [(2, 2), (2, 4), (3, 1, 2), (4,), (2, 3, 2)]:
        for r in range(int(np.prod(shape))):
            assert pl.rank_coords(shape, r) == tuple(int(v) for v in np.unravel_index(r, shape))
            assert pl.coords_rank(shape, pl.rank_coords(shape, r)) == r


def random_layout(rng, max_mesh_dims=3, max_rank=3, max_extent=9, allow_partial=True):
    nm = rng.randint(1, max_mesh_dims)
    mesh = tuple(rng.randint(1, 4) for _ in range(nm))
    nd = rng.randint(1, max_rank)
    gshape = tuple(rng.randint(0 if rng.random() < 0.1 else 1, max_extent) for _ in range(nd))
    pls = []
    for _ in range(nm):
        r = rng.random()
        if r < 0.45:
            pls.append(pl.Shard(rng.randrange(-nd, nd)))
        elif r < 0.8 or not allow_partial:
            pls.append(pl.Replicate())
        else:
            pls.append(pl.Partial())
    return pl.Layout(mesh, pls, gshape, materialize_replicas=rng.random() < 0.3)


def torch_chunk_block(index_tensor, layout, coords):
    """Independent block model: apply torch.chunk mesh dim by mesh dim."""
    t = index_tensor
    for m, p in enumerate(layout.placements):
        if isinstance(p, pl.Shard):
            chunks = torch.chunk(t, layout.mesh_shape[m], dim=p.dim) if t.shape[p.dim] > 0 else ()
            if coords[m] < len(chunks):
                t = chunks[coords[m]]
            else:
                shape = list(t.shape)
                shape[p.dim] = 0
                t = t.new_empty(shape)
    return t


def check_boxes_against_torch_chunk(placement=pl, trials=300):
    rng = random.Random(7)
    for _ in range(trials):
        lay = random_layout(rng)
        n = int(np.prod(lay.gshape))
        idx = torch.arange(n).reshape(lay.gshape) if n else torch.empty(lay.gshape, dtype=torch.int64)
        for coords in lay.all_coords():
            block = torch_chunk_block(idx, lay, coords)
            box = lay.box_of_coords(coords)
            assert tuple(block.shape) == tuple(s for _, s in box), (lay.placements, coords)
            if block.numel():
                sl = tuple(slice(o, o + s) for o, s in box)
                assert torch.equal(block, idx[sl])


def test_boxes_match_nested_torch_chunk():
    check_boxes_against_torch_chunk()


def test_coverage_each_index_once_per_partial_coordinate():
    rng = random.Random(11)
    for _ in range(300):
        lay = random_layout(rng)
        pdims = lay.partial_dims()
        counts = {}
        for slot in range(lay.nslots):
            c = lay.slot_coords(slot)
            key = tuple(c[m] for m in pdims)
            cnt = counts.setdefault(key, np.zeros(lay.gshape, dtype=np.int64))
            sl = tuple(slice(o, o + s) for o, s in lay.box(slot))
            if lay.materialize_replicas:
                # count one replica only: Replicate coordinates must be 0
                if any(c[m] != 0 for m, p in enumerate(lay.placements) if isinstance(p, pl.Replicate)):
                    continue
            cnt[sl] += 1
        for key, cnt in counts.items():
            assert (cnt == 1).all(), (lay.mesh_shape, lay.placements, lay.gshape, key)


def test_slot_count_and_replica_sharing():
    lay = pl.Layout((2, 4), [pl.Shard(0), pl.Replicate()], (8, 8))
    assert lay.nslots == 2
    assert {lay.slot_of_rank(r) for r in range(4)} == {0}
    assert {lay.slot_of_rank(r) for r in range(4, 8)} == {1}
    mat = pl.Layout((2, 4), [pl.Shard(0), pl.Replicate()], (8, 8), materialize_replicas=True)
    assert mat.nslots == 8 and [mat.slot_of_rank(r) for r in range(8)] == list(range(8))


def test_uneven_workload_chunks():
    # [8191, 8190] on (dp=2, tp=4) with dp Shard(0) and tp Shard(0) / Shard(1)
    lay0 = pl.Layout((2, 4), [pl.Shard(0), pl.Shard(0)], (8191, 8190))
    rows = [lay0.local_shape(s)[0] for s in range(8)]
    assert rows == [1024, 1024, 1024, 1024, 1024, 1024, 1024, 1023]
    lay1 = pl.Layout((2, 4), [pl.Shard(0), pl.Shard(1)], (8191, 8190))
    assert [lay1.local_shape(s) for s in range(4)] == [(4096, 2048)] * 3 + [(4096, 2046)]
    assert [lay1.local_shape(s)[0] for s in range(4, 8)] == [4095] * 4


@pytest.mark.parametrize("bad", ["floor", "reverse"])
def test_planted_chunk_mistake_is_caught(monkeypatch, bad):
    """A plausible error in the split rule must fail a pin."""
    orig = pl.chunk_bounds

    def floor_split(n, p):
        c = n // p
        return [(j * c, c if j < p - 1 else n - j * c) for j in range(p)]

    def reversed_split(n, p):
        return list(reversed(orig(n, p)))

    monkeypatch.setattr(pl, "chunk_bounds", floor_split if bad == "floor" else reversed_split)
    with pytest.raises(AssertionError):
        check_chunk_matches_torch()
        check_boxes_against_torch_chunk(trials=100)
