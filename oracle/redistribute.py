"""redistribute(): any placement -> any placement on the same mesh.

Oracle -- test infrastructure only.

The plain definition: the locals of the source describe one global tensor
(Hyper-Parallel DTensor API, ``full_tensor``: gather everything, clearing
Partial); the destination's locals are that global tensor's blocks under the
destination placements (``distribute_tensor``).  ``redistribute`` is the
composition (``redistribute``: build the destination layout, then move the
data; ``reduce_partial``: Partial -> Replicate by an all-reduce).

Storage types: bf16 tensors are numpy ``uint16`` bit patterns, fp32 tensors
``float32``, int32 tensors ``int32``.

Readings where the pages are silent (listed in the design notes):
* Partial(sum) order and precision.  For every element the partial values
  are added in ascending row-major order of their Partial-dim coordinates
  (rank order), sequentially in fp32 (bf16 widened exactly), and a bf16
  result is rounded once, nearest-even, at the end.  The first partial value
  is taken as is (it is not added to a zero, which would turn -0 into +0).
* A mesh dim that is Partial in both source and destination is left
  unreduced: each of its coordinates keeps its own partial value.
* Replicate -> Partial: coordinate 0 of that mesh dim keeps the value, the
  other coordinates hold zeros, so the partial values still sum to the
  tensor.  Shard -> Partial is not defined here (``NotImplementedError``).
* Partial(avg): the rank-order fp32 sum, then one correctly rounded fp32
  division by the number of partial values, then (bf16) one rounding.
  Partial(max): rank order, a = v if v > a else a, first value as is.
  Replicate -> Partial(avg / max): every coordinate keeps the value (it is
  its own average and maximum).  A layout reduces all its Partial dims with
  one op.
* Materialised replicas are read at Replicate coordinate 0.
"""
from __future__ import annotations

from itertools import product

import numpy as np

from . import bf16
from .placement import Layout, Partial, Replicate, Shard

_ACC = {"bf16": np.float32, "fp32": np.float32, "int32": np.int64}
_STORE = {"bf16": np.uint16, "fp32": np.float32, "int32": np.int32}


def _widen(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16.widen(a)
    if dtype == "fp32":
        return np.asarray(a, dtype=np.float32)
    return np.asarray(a, dtype=np.int64)


def _narrow(acc: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16.round_rne(acc)
    if dtype == "fp32":
        return acc.astype(np.float32)
    return acc.astype(np.int32)


def _sl(box):
    return tuple(slice(o, o + s) for o, s in box)


def distribute(global_arr: np.ndarray, layout: Layout, dtype: str) -> list[np.ndarray]:
    """Slice a global tensor into the slots of ``layout`` (``distribute_tensor``).

    Partial mesh dims follow the Replicate -> Partial reading: coordinate 0
    keeps the block, other coordinates get zeros.
    """
    g = np.asarray(global_arr)
    assert g.shape == layout.gshape, (g.shape, layout.gshape)
    out = []
    for slot in range(layout.nslots):
        coords = layout.slot_coords(slot)
        block = np.array(g[_sl(layout.box_of_coords(coords))], dtype=_STORE[dtype], copy=True)
        zero_dims = [m for m in layout.partial_dims() if layout.placements[m].op == "sum"]
        if any(coords[m] != 0 for m in zero_dims):
            block[...] = 0
        out.append(block)
    return out


def partial_op(layout: Layout) -> str:
    ops = {layout.placements[m].op for m in layout.partial_dims()}
    if len(ops) > 1:
        raise NotImplementedError("one reduce op per layout")
    return ops.pop() if ops else "sum"


def to_global(locals_: list[np.ndarray], layout: Layout, dtype: str, keep=None) -> np.ndarray:
    """The global tensor that the slots of ``layout`` describe (``full_tensor``).

    ``keep`` maps a Partial mesh dim to a fixed coordinate: that dim is not
    summed over (used for Partial -> Partial moves).
    """
    keep = dict(keep or {})
    nm = len(layout.mesh_shape)
    op = partial_op(layout)
    sum_dims = [m for m in layout.partial_dims() if m not in keep]
    count = 1
    for m in sum_dims:
        count *= layout.mesh_shape[m]
    shard_dims = [m for m, p in enumerate(layout.placements) if isinstance(p, Shard)]
    acc = np.zeros(layout.gshape, dtype=_ACC[dtype])
    seen = np.zeros(layout.gshape, dtype=bool)
    # Outer loop: Partial coordinates in row-major (rank) order.  Inner loop:
    # every shard block.  Each element therefore receives its partial values
    # in rank order, one per Partial coordinate.
    for pc in product(*[range(layout.mesh_shape[m]) for m in sum_dims]):
        for sc in product(*[range(layout.mesh_shape[m]) for m in shard_dims]):
            coords = [0] * nm
            for m, c in zip(sum_dims, pc):
                coords[m] = c
            for m, c in zip(shard_dims, sc):
                coords[m] = c
            for m, c in keep.items():
                coords[m] = c
            box = layout.box_of_coords(coords)
            if any(s == 0 for _, s in box):
                continue
            local = locals_[layout.slot_of_coords(coords)]
            assert local.shape == tuple(s for _, s in box), (local.shape, box)
            val = _widen(local, dtype)
            sl = _sl(box)
            first = ~seen[sl]
            # first contribution is assigned, later ones are combined
            if op == "max":
                acc[sl] = np.where(first, val, np.where(val > acc[sl], val, acc[sl]))
            else:
                acc[sl] = np.where(first, val, acc[sl] + val)
            seen[sl] = True
    assert seen.all() or acc.size == 0, "coverage: some global index has no owner"
    if op == "avg" and sum_dims:
        if dtype == "int32":
            raise NotImplementedError("Partial(avg) of int32")
        acc = (acc.astype(np.float32) / np.float32(count)).astype(np.float32)
    return _narrow(acc, dtype)


def redistribute(src_locals, src: Layout, dst: Layout, dtype: str) -> list[np.ndarray]:
    """Move data from ``src`` placements to ``dst`` placements (``redistribute``)."""
    if src.mesh_shape != dst.mesh_shape or src.gshape != dst.gshape:
        raise ValueError("redistribute keeps the mesh and the global shape")
    nm = len(src.mesh_shape)
    kept = [m for m in range(nm)
            if isinstance(src.placements[m], Partial) and isinstance(dst.placements[m], Partial)]
    for m in kept:
        if src.placements[m].op != dst.placements[m].op:
            raise NotImplementedError("a kept Partial dim cannot change its reduce op")
    zero_rule = []
    for m in range(nm):
        if isinstance(dst.placements[m], Partial) and m not in kept:
            if isinstance(src.placements[m], Replicate):
                if dst.placements[m].op == "sum":
                    zero_rule.append(m)
            else:
                raise NotImplementedError("Shard -> Partial is not defined")
    cache = {}
    out = []
    for slot in range(dst.nslots):
        coords = dst.slot_coords(slot)
        box = dst.box_of_coords(coords)
        shape = tuple(s for _, s in box)
        if any(coords[m] != 0 for m in zero_rule):
            out.append(np.zeros(shape, dtype=_STORE[dtype]))
            continue
        key = tuple(coords[m] for m in kept)
        if key not in cache:
            cache[key] = to_global(src_locals, src, dtype, keep={m: coords[m] for m in kept})
        out.append(np.array(cache[key][_sl(box)], copy=True))
    return out
