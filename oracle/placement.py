"""Placement arithmetic: mesh coordinates, block split, slots and boxes.

Oracle -- test infrastructure only.

Sources
-------
* Hyper-Parallel DTensor API, ``distribute_tensor`` example: on a (2, 2)
  mesh named ("dp", "tp") with placements [Shard(0), Replicate()], ranks 0
  and 1 get rows 0-1 of arange(16).reshape(4, 4) and ranks 2 and 3 get rows
  2-3.  So ranks are numbered row-major over the mesh (the last mesh dim
  varies fastest) and a Shard on mesh dim 0 splits rows in rank-coordinate
  order.
* Hyper-Parallel DTensor API, placement-type table: Shard(dim) splits the
  tensor along ``dim``; Replicate() keeps a full copy on that mesh dim;
  Partial(reduce_op) holds a pending reduction.
* Hyper-Parallel DTensor API, ``shape`` property: a local (4, 8) shard split
  in 2 along dim 0 has global shape (8, 8).
* Model parallelism (wineandchord), "Tensor-parallel linear layers": shards
  are made with ``torch.chunk`` and every shard covers each global index
  exactly once.

Readings where the pages are silent (listed in the design notes):
* Uneven split.  ``torch.chunk`` semantics: chunk width c = ceil(n / p);
  part j covers [j*c, min((j+1)*c, n)), which is empty for trailing parts
  when p*c overshoots n.  Empty parts are kept so every rank has a shard.
* Two mesh dims sharding the same tensor dim nest in mesh-dim order: the
  outer mesh dim splits first, the inner one splits that block.
* Replicate storage.  Ranks that differ only in Replicate coordinates hold
  identical values and by default share one stored "slot"; with
  ``materialize_replicas`` every rank has its own slot.
"""
from __future__ import annotations

from dataclasses import dataclass
from itertools import product
from typing import Sequence


@dataclass(frozen=True)
class Shard:
    dim: int


@dataclass(frozen=True)
class Replicate:
    pass


@dataclass(frozen=True)
class Partial:
    """A pending reduction across this mesh dim: op is "sum" (the default),
    "avg" or "max" (Hyper-Parallel DTensor API: Partial(reduce_op))."""
    op: str = "sum"


def chunk_bounds(n: int, parts: int) -> list[tuple[int, int]]:
    """(offset, size) of each of ``parts`` torch.chunk-style blocks of [0, n).

    Width c = ceil(n / parts); block j starts at min(j*c, n) and holds
    max(0, min(c, n - j*c)) elements.
    """
    if parts <= 0:
        raise ValueError("parts must be positive")
    c = -(-n // parts) if n > 0 else 0
    out = []
    for j in range(parts):
        start = min(j * c, n)
        size = max(0, min(c, n - j * c))
        out.append((start, size))
    return out


def rank_coords(mesh_shape: Sequence[int], rank: int) -> tuple[int, ...]:
    """Row-major coordinates of ``rank`` (last mesh dim fastest)."""
    coords = []
    for extent in reversed(mesh_shape):
        coords.append(rank % extent)
        rank //= extent
    return tuple(reversed(coords))


def coords_rank(mesh_shape: Sequence[int], coords: Sequence[int]) -> int:
    r = 0
    for extent, c in zip(mesh_shape, coords):
        r = r * extent + c
    return r


def mesh_size(mesh_shape: Sequence[int]) -> int:
    n = 1
    for e in mesh_shape:
        n *= e
    return n


class Layout:
    """A global tensor's distribution over a logical device mesh.

    ``placements[m]`` is the placement on mesh dim ``m``.  Negative Shard
    dims are normalised against the tensor rank (the DTorch guide uses
    ``Shard(-1)`` / ``Shard(input.dim() - 1)`` for the row-parallel input).
    """

    def __init__(self, mesh_shape, placements, gshape, materialize_replicas=False):
        self.mesh_shape = tuple(int(e) for e in mesh_shape)
        self.gshape = tuple(int(s) for s in gshape)
        nd = len(self.gshape)
        pls = []
        for p in placements:
            if isinstance(p, Shard):
                d = p.dim + nd if p.dim < 0 else p.dim
                if not 0 <= d < nd:
                    raise ValueError(f"shard dim {p.dim} out of range for rank {nd}")
                pls.append(Shard(d))
            elif isinstance(p, (Replicate, Partial)):
                pls.append(p)
            else:
                raise TypeError(p)
        if len(pls) != len(self.mesh_shape):
            raise ValueError("one placement per mesh dim")
        self.placements = tuple(pls)
        self.materialize_replicas = bool(materialize_replicas)

    # -- slots ---------------------------------------------------------
    def distinct_dims(self) -> list[int]:
        """Mesh dims whose coordinate selects different stored data."""
        if self.materialize_replicas:
            return list(range(len(self.mesh_shape)))
        return [m for m, p in enumerate(self.placements) if not isinstance(p, Replicate)]

    @property
    def nslots(self) -> int:
        n = 1
        for m in self.distinct_dims():
            n *= self.mesh_shape[m]
        return n

    def slot_of_coords(self, coords) -> int:
        s = 0
        for m in self.distinct_dims():
            s = s * self.mesh_shape[m] + coords[m]
        return s

    def slot_of_rank(self, rank: int) -> int:
        return self.slot_of_coords(rank_coords(self.mesh_shape, rank))

    def slot_coords(self, slot: int) -> tuple[int, ...]:
        """Representative coordinates of a slot: 0 on the shared (Replicate) dims."""
        coords = [0] * len(self.mesh_shape)
        for m in reversed(self.distinct_dims()):
            coords[m] = slot % self.mesh_shape[m]
            slot //= self.mesh_shape[m]
        return tuple(coords)

    # -- boxes ---------------------------------------------------------
    def box_of_coords(self, coords) -> tuple[tuple[int, int], ...]:
        """Per tensor dim (global offset, size) of the block held at ``coords``."""
        box = [(0, n) for n in self.gshape]
        for m, p in enumerate(self.placements):
            if isinstance(p, Shard):
                off, size = box[p.dim]
                sub_off, sub_size = chunk_bounds(size, self.mesh_shape[m])[coords[m]]
                box[p.dim] = (off + sub_off, sub_size)
        return tuple(box)

    def box(self, slot: int):
        return self.box_of_coords(self.slot_coords(slot))

    def local_shape(self, slot: int) -> tuple[int, ...]:
        return tuple(s for _, s in self.box(slot))

    def partial_dims(self) -> list[int]:
        return [m for m, p in enumerate(self.placements) if isinstance(p, Partial)]

    def all_coords(self):
        return product(*[range(e) for e in self.mesh_shape])


def global_shape_from_local(local_shape, mesh_shape, placements):
    """The ``shape`` property rule for even shards: local extent times the
    number of parts along every sharded dim (Hyper-Parallel DTensor API,
    ``shape``)."""
    g = list(local_shape)
    for m, p in enumerate(placements):
        if isinstance(p, Shard):
            g[p.dim] *= mesh_shape[m]
    return tuple(g)
