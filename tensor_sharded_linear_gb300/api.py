"""DTensor-style Python API over libdt (argument marshalling only).

Every rank of the mesh is a logical shard on ONE GPU: a ``DTensor`` holds one
torch device tensor per stored slot (ranks that differ only in Replicate
coordinates share a slot unless ``materialize_replicas`` is set).  Every
operation runs in libdt's CUDA kernels on the current torch stream; PyTorch
only allocates device memory.

Names follow the pages: DeviceMesh, Shard / Replicate / Partial,
``distribute_tensor``, ``from_local``, ``to_local``, ``redistribute``,
``reduce_partial``, ``full_tensor`` (Hyper-Parallel DTensor API);
``redistribute_by_dict(..., default_placement_mode="keep")``,
ColumnParallelLinear, RowParallelLinear(WithReplicateOutput),
ReplicateParallelLinear, EmbeddingWithReplicateOutput (DTorch guide);
ALL_REDUCE / REDUCE_SCATTER modes (nanotron tutorial, 5.1).
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import _lib as L

ALL_REDUCE = "ALL_REDUCE"
REDUCE_SCATTER = "REDUCE_SCATTER"
PARTIAL = "PARTIAL"
_MODES = {PARTIAL: L.TP_PARTIAL, ALL_REDUCE: L.TP_ALL_REDUCE, REDUCE_SCATTER: L.TP_REDUCE_SCATTER}

_DT = {torch.bfloat16: L.BF16, torch.float32: L.FP32, torch.int32: L.INT32}
_TORCH = {v: k for k, v in _DT.items()}


# ---------------------------------------------------------------- placements

@dataclass(frozen=True)
class Shard:
    dim: int


@dataclass(frozen=True)
class Replicate:
    pass


@dataclass(frozen=True)
class Partial:
    reduce_op: str = "sum"


class DeviceMesh:
    """A logical N-D grid of ranks with named dims (all on one GPU)."""

    def __init__(self, shape: Sequence[int], dim_names: Optional[Sequence[str]] = None, device="cuda"):
        self.shape = tuple(int(s) for s in shape)
        self.dim_names = tuple(dim_names) if dim_names is not None else tuple(f"d{i}" for i in range(len(self.shape)))
        if len(self.dim_names) != len(self.shape):
            raise ValueError("one name per mesh dim")
        self.device = torch.device(device)

    @property
    def ndim(self) -> int:
        return len(self.shape)

    @property
    def size(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n

    def dim_name_index(self, name) -> Optional[int]:
        """Index of a named dim, or None when the mesh has no such dim (then no TP)."""
        if name is None:
            return None
        if isinstance(name, int):
            return name
        return self.dim_names.index(name) if name in self.dim_names else None

    def __eq__(self, other):
        return isinstance(other, DeviceMesh) and self.shape == other.shape

    def __hash__(self):
        return hash(self.shape)


def init_device_mesh(device_type, mesh_shape, mesh_dim_names=None) -> DeviceMesh:
    return DeviceMesh(mesh_shape, mesh_dim_names, device=device_type)


def _layout(mesh: DeviceMesh, placements, gshape, dtype, materialize) -> L.Layout:
    lay = L.Layout()
    lay.mesh_ndim = mesh.ndim
    for m, s in enumerate(mesh.shape):
        lay.mesh_shape[m] = s
    if len(placements) != mesh.ndim:
        raise ValueError("one placement per mesh dim")
    for m, p in enumerate(placements):
        if isinstance(p, Shard):
            lay.placements[m].kind, lay.placements[m].dim = L.SHARD, p.dim
        elif isinstance(p, Replicate):
            lay.placements[m].kind = L.REPLICATE
        elif isinstance(p, Partial):
            ops = {"sum": L.SUM, "avg": L.AVG, "max": L.MAX}
            if p.reduce_op not in ops:
                raise ValueError(f"Partial reduce op {p.reduce_op!r}: one of sum, avg, max")
            lay.placements[m].kind, lay.placements[m].op = L.PARTIAL, ops[p.reduce_op]
        else:
            raise TypeError(p)
    lay.ndim = len(gshape)
    for d, s in enumerate(gshape):
        lay.gshape[d] = int(s)
    lay.dtype = _DT[dtype]
    lay.materialize_replicas = 1 if materialize else 0
    return lay


def _stream_handle() -> int:
    return torch.cuda.current_stream().cuda_stream


# ---------------------------------------------------------------- DTensor

class DTensor:
    """A global tensor distributed over a logical mesh, one device tensor per slot."""

    def __init__(self, slots: Sequence[torch.Tensor], mesh: DeviceMesh, placements, gshape, dtype,
                 materialize_replicas: bool = False):
        self.mesh = mesh
        self.placements = tuple(placements)
        self.gshape = tuple(int(s) for s in gshape)
        self.dtype = dtype
        self.materialize_replicas = bool(materialize_replicas)
        self._layout = _layout(mesh, self.placements, self.gshape, dtype, materialize_replicas)
        n = C.c_int32()
        L.check(L.load().dt_layout_nslots(C.byref(self._layout), C.byref(n)), "layout")
        if len(slots) != n.value:
            raise ValueError(f"{len(slots)} slots given, the layout has {n.value}")
        for s, t in enumerate(slots):
            if tuple(t.shape) != self.slot_shape(s):
                raise ValueError(f"slot {s} has shape {tuple(t.shape)}, expected {self.slot_shape(s)}")
            if t.dtype != dtype:
                raise ValueError("slot dtype")
        self.slots = list(slots)
        self._layout_key = bytes(self._layout)

    # -- layout queries (host only)
    @property
    def nslots(self) -> int:
        return len(self.slots)

    def slot_box(self, slot: int):
        ls = (C.c_int64 * L.MAX_TENSOR_DIMS)()
        go = (C.c_int64 * L.MAX_TENSOR_DIMS)()
        L.check(L.load().dt_layout_slot_box(C.byref(self._layout), slot, ls, go), "slot_box")
        nd = len(self.gshape)
        return tuple(ls[:nd]), tuple(go[:nd])

    def slot_shape(self, slot: int):
        return self.slot_box(slot)[0]

    def slot_of_rank(self, rank: int) -> int:
        s = C.c_int32()
        L.check(L.load().dt_layout_slot_of_rank(C.byref(self._layout), rank, C.byref(s)), "slot_of_rank")
        return s.value

    @property
    def shape(self):
        return self.gshape

    @property
    def device_mesh(self):
        return self.mesh

    def local_shape(self, rank: int = 0):
        return self.slot_shape(self.slot_of_rank(rank))

    def to_local(self, rank: int = 0) -> torch.Tensor:
        return self.slots[self.slot_of_rank(rank)]

    # -- construction
    @staticmethod
    def empty(mesh: DeviceMesh, placements, gshape, dtype=torch.bfloat16, materialize_replicas=False,
              device=None) -> "DTensor":
        device = mesh.device if device is None else device
        lay = _layout(mesh, tuple(placements), gshape, dtype, materialize_replicas)
        n = C.c_int32()
        L.check(L.load().dt_layout_nslots(C.byref(lay), C.byref(n)), "layout")
        shapes = []
        for s in range(n.value):
            ls = (C.c_int64 * L.MAX_TENSOR_DIMS)()
            L.check(L.load().dt_layout_slot_box(C.byref(lay), s, ls, None), "slot_box")
            shapes.append(tuple(ls[:len(gshape)]))
        slots = [torch.empty(sh, dtype=dtype, device=device) for sh in shapes]
        return DTensor(slots, mesh, placements, gshape, dtype, materialize_replicas)

    @staticmethod
    def from_local(slots, mesh: DeviceMesh, placements, gshape=None, materialize_replicas=False) -> "DTensor":
        """Wrap existing per-slot tensors (no data movement)."""
        slots = list(slots) if isinstance(slots, (list, tuple)) else [slots]
        dtype = slots[0].dtype
        if gshape is None:
            g = list(slots[0].shape)
            for m, p in enumerate(placements):
                if isinstance(p, Shard):
                    g[p.dim] *= mesh.shape[m]
            gshape = g
        return DTensor(slots, mesh, placements, gshape, dtype, materialize_replicas)

    @staticmethod
    def distribute_tensor(tensor: torch.Tensor, mesh: DeviceMesh, placements, materialize_replicas=False) -> "DTensor":
        """Slice a full device tensor into the slots of ``placements``."""
        src = DTensor([tensor.contiguous()], mesh, [Replicate()] * mesh.ndim, tuple(tensor.shape), tensor.dtype)
        return src.redistribute(placements, materialize_replicas=materialize_replicas)

    # -- data movement
    def redistribute(self, placements, materialize_replicas=None, out: "DTensor" = None) -> "DTensor":
        if materialize_replicas is None:
            materialize_replicas = self.materialize_replicas
        if out is None:
            out = DTensor.empty(self.mesh, placements, self.gshape, self.dtype, materialize_replicas,
                                device=self.slots[0].device if self.slots else None)
        redistribute(self, out)
        return out

    def redistribute_by_dict(self, placements_dict, default_placement_mode="keep") -> "DTensor":
        """Change only the named mesh dims; keep the others (DTorch guide)."""
        if default_placement_mode != "keep":
            raise ValueError("only default_placement_mode='keep'")
        pls = list(self.placements)
        for key, p in placements_dict.items():
            m = self.mesh.dim_name_index(key)
            if m is None:
                continue
            pls[m] = p
        return self.redistribute(pls)

    def check_placement(self, mesh_dim, expect) -> bool:
        m = self.mesh.dim_name_index(mesh_dim)
        p = self.placements[m]
        if isinstance(expect, Shard) and isinstance(p, Shard):
            nd = len(self.gshape)
            return (expect.dim % nd) == (p.dim % nd)
        return p == expect

    def reduce_partial(self) -> "DTensor":
        return self.redistribute([Replicate() if isinstance(p, Partial) else p for p in self.placements])

    def full_tensor(self) -> torch.Tensor:
        return self.redistribute([Replicate()] * self.mesh.ndim, materialize_replicas=False).slots[0]

    def dim(self) -> int:
        return len(self.gshape)

    # -- ABI descriptor
    def _key(self):
        """What the descriptor is made of: each slot's address and strides."""
        return tuple((t.data_ptr() if t.numel() else 0, t.stride()) for t in self.slots)

    def _desc(self):
        """The C descriptor (dt_dtensor) of this tensor.  Built once and kept
        while the slots' addresses and strides stay the same."""
        key = self._key()
        cached = getattr(self, "_desc_cache", None)
        if cached is not None and cached[0] == key:
            return cached[1]
        n = max(1, self.nslots)
        ptrs = (C.c_void_p * n)(*[p or None for p, _ in key])
        strides = (C.c_int64 * max(1, self.nslots * len(self.gshape)))(*[d for _, st in key for d in st])
        desc = L.DTensorDesc()
        desc.layout = self._layout
        desc.nslots = self.nslots
        desc.slots = C.cast(ptrs, C.POINTER(C.c_void_p))
        desc.strides = C.cast(strides, C.POINTER(C.c_int64))
        desc._keep = (ptrs, strides)  # keep the arrays alive with the descriptor
        self._desc_cache = (key, desc)
        return desc

    def __repr__(self):
        return f"DTensor(gshape={self.gshape}, placements={self.placements}, mesh={self.mesh.shape}, slots={self.nslots})"


def _empty_desc():
    d = L.DTensorDesc()
    d.nslots = 0
    return d


# ---------------------------------------------------------------- operations

def redistribute(src: DTensor, dst: DTensor) -> None:
    """dt_redistribute into preallocated ``dst``."""
    L.check(L.load().dt_redistribute(C.byref(src._desc()), C.byref(dst._desc()), None, _stream_handle()),
            "redistribute")


def redistribute_batch(pairs: Sequence[tuple]) -> None:
    """dt_redistribute_batch: every (src, dst) pair in as few launches as fit
    (one for the copies, one for the Partial reductions)."""
    n = len(pairs)
    if n == 0:
        return
    # the descriptors own the slot/stride arrays the copies below point at
    sdescs = [s._desc() for s, _ in pairs]
    ddescs = [d._desc() for _, d in pairs]
    sd = (L.DTensorDesc * n)(*sdescs)
    dd = (L.DTensorDesc * n)(*ddescs)
    L.check(L.load().dt_redistribute_batch(n, sd, dd, None, _stream_handle()), "redistribute_batch")
    del sdescs, ddescs


def read_device_status(clear: bool = True) -> int:
    """Synchronise and read the library's device status word (DT_DEV_* bits)."""
    torch.cuda.synchronize()
    v = C.c_int32()
    L.check(L.load().dt_read_device_status(C.byref(v), 1 if clear else 0), "read_device_status")
    return v.value


def _tp_index(mesh: DeviceMesh, tp_dim) -> int:
    m = mesh.dim_name_index(tp_dim)
    return -1 if m is None else m


def _col_out(x: DTensor, w: DTensor, tp: int, out_dtype, output: str = "shard") -> DTensor:
    """Output of a column layer: Shard(-1) on tp, or Replicate with
    output="replicate" (all tokens either way, also for a token-sharded x)."""
    nd = len(x.gshape)
    pls = list(x.placements)
    if tp >= 0:
        pls[tp] = Replicate() if output == "replicate" else Shard(nd - 1)
    return DTensor.empty(x.mesh, pls, x.gshape[:-1] + (w.gshape[1],), out_dtype or x.dtype,
                         device=x.slots[0].device)


def _ws_args(workspace: Optional[torch.Tensor]):
    """(pointer, bytes) of a workspace tensor, or (None, 0)."""
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


_WS_SIZES: dict = {}


def _op_key(op, tensors, *args):
    """Everything a workspace size depends on: the operands' layouts,
    addresses and strides, the call's other arguments and the device."""
    return (op, tensors[0].slots[0].device if tensors[0].slots else None,
            tuple((t._layout_key, t._key()) for t in tensors), args)


def _ws_size(key, query):
    """A workspace-size query's answer, kept per operand set (see _op_key)."""
    v = _WS_SIZES.get(key)
    if v is None:
        if len(_WS_SIZES) >= 256:
            _WS_SIZES.clear()
        v = _WS_SIZES[key] = query()
    return v


def _workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    """Device memory for a call's workspace (None when it needs none).  Torch
    allocates it: the library itself allocates nothing."""
    return torch.empty(nbytes, dtype=torch.uint8, device=device) if nbytes > 0 else None


def column_parallel_linear_workspace_bytes(x: DTensor, ws: Sequence[DTensor], ys: Sequence[DTensor],
                                           tp_dim="tp") -> int:
    """dt_column_parallel_linear_workspace_size for the weights ``ws`` and outputs ``ys``."""
    n = len(ws)
    tp = _tp_index(x.mesh, tp_dim)

    def query():
        wdescs, ydescs = [w._desc() for w in ws], [y._desc() for y in ys]
        wd, yd = (L.DTensorDesc * n)(*wdescs), (L.DTensorDesc * n)(*ydescs)
        out = C.c_size_t()
        L.check(L.load().dt_column_parallel_linear_workspace_size(C.byref(x._desc()), n, wd, yd, tp, C.byref(out)),
                "column_parallel_linear_workspace_size")
        return out.value

    return _ws_size(_op_key("column", [x, *ws, *ys], n, tp), query)


def column_parallel_linear(x: DTensor, w: DTensor, bias: Optional[DTensor] = None, tp_dim="tp",
                           out_dtype=None, out: Optional[DTensor] = None, output: str = "shard",
                           workspace: Optional[torch.Tensor] = None) -> DTensor:
    """Y_i = X W_i (+ b_i).

    x Replicate on tp, or Shard(0) on tp (sequence-parallel entry: the token
    shards are read in place, no gathered copy is made).  The output is
    Shard(-1) on tp, or Replicate with output="replicate" (each shard writes
    its column block of the one Replicate tensor).  ``workspace`` (a device
    tensor of at least ``column_parallel_linear_workspace_bytes``) lets the
    GEMM split its last wave; without one a workspace of that size is taken
    from torch's allocator."""
    return column_parallel_linear_multi(x, [w], [bias] if bias is not None else None, tp_dim, out_dtype,
                                        [out] if out is not None else None, output, workspace)[0]


def column_parallel_linear_multi(x: DTensor, ws: Sequence[DTensor], biases=None, tp_dim="tp", out_dtype=None,
                                 outs=None, output: str = "shard", workspace: Optional[torch.Tensor] = None):
    """Several column-parallel linears sharing x, in one launch (fused q/k/v)."""
    tp = _tp_index(x.mesh, tp_dim)
    ys = list(outs) if outs is not None else [_col_out(x, w, tp, out_dtype, output) for w in ws]
    n = len(ws)
    if workspace is None:
        workspace = _workspace(column_parallel_linear_workspace_bytes(x, ws, ys, tp_dim), x.slots[0].device)
    # the descriptors own the slot/stride arrays the copies below point at
    wdescs = [w._desc() for w in ws]
    ydescs = [y._desc() for y in ys]
    bdescs = [(b._desc() if b is not None else _empty_desc()) for b in biases] if biases is not None else None
    wd = (L.DTensorDesc * n)(*wdescs)
    yd = (L.DTensorDesc * n)(*ydescs)
    bd = (L.DTensorDesc * n)(*bdescs) if bdescs is not None else None
    L.check(L.load().dt_column_parallel_linear_multi(C.byref(x._desc()), n, wd, bd, yd, tp, *_ws_args(workspace),
                                                     None, _stream_handle()), "column_parallel_linear_multi")
    del wdescs, ydescs, bdescs
    return ys


def _row_out(x: DTensor, w: DTensor, tp: int, mode: str, out_dtype) -> DTensor:
    pls = list(x.placements)
    if tp >= 0:
        pls[tp] = {ALL_REDUCE: Replicate(), REDUCE_SCATTER: Shard(0), PARTIAL: Partial()}[mode]
    return DTensor.empty(x.mesh, pls, x.gshape[:-1] + (w.gshape[1],), out_dtype or x.dtype,
                         device=x.slots[0].device)


def row_parallel_linear_workspace_bytes(x: DTensor, w: DTensor, y: DTensor, mode: str = ALL_REDUCE,
                                        tp_dim="tp") -> int:
    """dt_row_parallel_linear_workspace_size."""
    tp = _tp_index(x.mesh, tp_dim)

    def query():
        out = C.c_size_t()
        L.check(L.load().dt_row_parallel_linear_workspace_size(C.byref(x._desc()), C.byref(w._desc()),
                                                               C.byref(y._desc()), _MODES[mode], tp, C.byref(out)),
                "row_parallel_linear_workspace_size")
        return out.value

    return _ws_size(_op_key("row", [x, w, y], mode, tp), query)


def row_parallel_linear(x: DTensor, w: DTensor, bias: Optional[DTensor] = None, mode: str = ALL_REDUCE,
                        tp_dim="tp", out_dtype=None, out: Optional[DTensor] = None,
                        workspace: Optional[torch.Tensor] = None) -> DTensor:
    """Y = sum_i X_i W_i (+ b once): Replicate / Shard(0) / Partial on tp per ``mode``."""
    tp = _tp_index(x.mesh, tp_dim)
    y = out if out is not None else _row_out(x, w, tp, mode, out_dtype)
    if workspace is None:
        workspace = _workspace(row_parallel_linear_workspace_bytes(x, w, y, mode, tp_dim), x.slots[0].device)
    b = bias._desc() if bias is not None else None
    L.check(L.load().dt_row_parallel_linear(C.byref(x._desc()), C.byref(w._desc()),
                                            C.byref(b) if b is not None else None, C.byref(y._desc()),
                                            _MODES[mode], tp, *_ws_args(workspace), None, _stream_handle()),
            "row_parallel_linear")
    return y


def tp_mlp_workspace_bytes(x: DTensor, w_gate: DTensor, w_up: DTensor, w_down: DTensor, y: DTensor,
                           mode: str = ALL_REDUCE, tp_dim="tp") -> int:
    """dt_tp_mlp_workspace_size: H plus the split tail's scratch."""
    tp = _tp_index(x.mesh, tp_dim)

    def query():
        n = C.c_size_t()
        L.check(L.load().dt_tp_mlp_workspace_size(C.byref(x._desc()), C.byref(w_gate._desc()), C.byref(w_up._desc()),
                                                  C.byref(w_down._desc()), C.byref(y._desc()), _MODES[mode], tp,
                                                  C.byref(n)), "tp_mlp_workspace_size")
        return n.value

    return _ws_size(_op_key("mlp", [x, w_gate, w_up, w_down, y], mode, tp), query)


def tp_mlp_output(x: DTensor, w_down: DTensor, mode: str = ALL_REDUCE, tp_dim="tp", out_dtype=None) -> DTensor:
    """An empty output of ``tp_mlp`` for ``mode``."""
    return _row_out(x, w_down, _tp_index(x.mesh, tp_dim), mode, out_dtype)


def tp_mlp(x: DTensor, w_gate: DTensor, w_up: DTensor, w_down: DTensor, mode: str = ALL_REDUCE, tp_dim="tp",
           out_dtype=None, out: Optional[DTensor] = None, workspace: Optional[torch.Tensor] = None) -> DTensor:
    """H = bf16(SiLU(X Wg_i) * (X Wu_i)), then the row-parallel down projection."""
    tp = _tp_index(x.mesh, tp_dim)
    y = out if out is not None else _row_out(x, w_down, tp, mode, out_dtype)
    if workspace is None:
        workspace = _workspace(tp_mlp_workspace_bytes(x, w_gate, w_up, w_down, y, mode, tp_dim), x.slots[0].device)
    L.check(L.load().dt_tp_mlp(C.byref(x._desc()), C.byref(w_gate._desc()), C.byref(w_up._desc()),
                               C.byref(w_down._desc()), C.byref(y._desc()), _MODES[mode], tp, *_ws_args(workspace),
                               None, _stream_handle()), "tp_mlp")
    return y


def cuda_core_gemm_count() -> int:
    """dt_cuda_core_gemm_count: CUDA-core GEMM launches so far in this process."""
    return int(L.load().dt_cuda_core_gemm_count())


def mlp_hidden_view(x: DTensor, w_gate: DTensor, workspace: torch.Tensor, tp_dim="tp") -> torch.Tensor:
    """The [M, F] bf16 H block that ``tp_mlp`` wrote for a single-slot x."""
    rows = 1
    for s in x.slots[0].shape[:-1]:
        rows *= s
    F = w_gate.gshape[1]
    return workspace[: rows * F * 2].view(torch.bfloat16).view(rows, F)


def tp_embedding(ids: DTensor, table: DTensor, tp_dim="tp", out: Optional[DTensor] = None) -> DTensor:
    """EmbeddingWithReplicateOutput: gather into a Replicate [.., dim] output."""
    tp = _tp_index(ids.mesh, tp_dim)
    if out is None:
        out = DTensor.empty(ids.mesh, [Replicate()] * ids.mesh.ndim, ids.gshape + (table.gshape[1],), table.dtype,
                            device=table.slots[0].device)
    L.check(L.load().dt_tp_embedding(C.byref(ids._desc()), C.byref(table._desc()), C.byref(out._desc()), tp, None,
                                     _stream_handle()), "tp_embedding")
    return out


def tp_attention_projections(x: DTensor, wq: DTensor, wk: DTensor, wv: DTensor, wo: DTensor,
                             mode: str = REDUCE_SCATTER, tp_dim="tp", out_dtype=None):
    """q/k/v column-parallel in one launch, then o row-parallel on q's Shard(-1) output."""
    q, k, v = column_parallel_linear_multi(x, [wq, wk, wv], tp_dim=tp_dim)
    o = row_parallel_linear(q, wo, mode=mode, tp_dim=tp_dim, out_dtype=out_dtype)
    return o, q, k, v


# ---------------------------------------------------------------- DTorch-style layers

class Linear:
    """Tensor-parallel linear holding distributed [in, out] weights (DTorch ``Linear``).

    ``tp_shard_type`` "col": weight Shard(1) on tp, bias Shard(0), input must be
    Replicate on tp.  "row": weight Shard(0), bias Replicate (added once), input
    must be Shard(-1).  ``tp_dim=None`` (or a name the mesh lacks) means no TP.
    """

    input_placement = None
    output_placement = None

    def __init__(self, weight: torch.Tensor, bias: Optional[torch.Tensor], mesh: DeviceMesh, *, tp_dim="tp",
                 tp_shard_type=None):
        self.mesh = mesh
        self.tp_dim = mesh.dim_name_index(tp_dim)
        self.tp_shard_type = tp_shard_type
        wpl = [Replicate()] * mesh.ndim
        bpl = [Replicate()] * mesh.ndim
        if self.tp_dim is not None:
            wpl[self.tp_dim] = Shard(0) if tp_shard_type == "row" else Shard(1)
            bpl[self.tp_dim] = Replicate() if tp_shard_type == "row" else Shard(0)
        self.weight = DTensor.distribute_tensor(weight, mesh, wpl)
        self.bias = DTensor.distribute_tensor(bias, mesh, bpl) if bias is not None else None

    def redistribute_input(self, x: DTensor) -> DTensor:
        if self.tp_dim is not None and self.input_placement is not None:
            x = x.redistribute_by_dict({self.tp_dim: self.input_placement})
        if self.tp_dim is not None:
            expect = Shard(x.dim() - 1) if self.tp_shard_type == "row" else Replicate()
            if not x.check_placement(self.tp_dim, expect):
                raise L.DtError(L.ERR_PLACEMENT, f"input placement {x.placements} breaks the {self.tp_shard_type} rule")
        return x

    def redistribute_output(self, y: DTensor) -> DTensor:
        if self.tp_dim is not None and self.output_placement is not None:
            y = y.redistribute_by_dict({self.tp_dim: self.output_placement})
        return y

    def forward(self, x: DTensor) -> DTensor:
        tp = -1 if self.tp_dim is None else self.tp_dim
        if self.tp_shard_type == "row":
            return row_parallel_linear(x, self.weight, self.bias, mode=PARTIAL, tp_dim=tp)
        return column_parallel_linear(x, self.weight, self.bias, tp_dim=tp)

    def __call__(self, x: DTensor) -> DTensor:
        return self.redistribute_output(self.forward(self.redistribute_input(x)))


class ColumnParallelLinear(Linear):
    def __init__(self, weight, bias, mesh, tp_dim="tp"):
        super().__init__(weight, bias, mesh, tp_dim=tp_dim, tp_shard_type="col")


class ColumnParallelLinearWithReplicateOutput(ColumnParallelLinear):
    """Column linear whose output is Replicate on tp: fused, every shard's GEMM
    writes its column block of the Replicate output (no separate all-gather)."""

    def forward(self, x: DTensor) -> DTensor:
        if self.tp_dim is None:
            return super().forward(x)
        return column_parallel_linear(x, self.weight, self.bias, tp_dim=self.tp_dim, output="replicate")


class ColumnParallelLinearWithReplicateInputOutput(ColumnParallelLinearWithReplicateOutput):
    """Input converted to Replicate on tp, output Replicate.  A token-sharded
    (Shard(0)) input is consumed in place by the GEMM instead of being
    gathered first; any other placement is redistributed to Replicate."""

    def redistribute_input(self, x: DTensor) -> DTensor:
        if self.tp_dim is not None and x.placements[self.tp_dim] == Shard(0):
            return x
        if self.tp_dim is not None:
            x = x.redistribute_by_dict({self.tp_dim: Replicate()})
        return super().redistribute_input(x)


class RowParallelLinear(Linear):
    def __init__(self, weight, bias, mesh, tp_dim="tp"):
        super().__init__(weight, bias, mesh, tp_dim=tp_dim, tp_shard_type="row")


class RowParallelLinearWithReplicateOutput(RowParallelLinear):
    """Partial -> Replicate fused into the GEMM accumulator (ALL_REDUCE)."""

    def forward(self, x: DTensor) -> DTensor:
        if self.tp_dim is None:
            return super().forward(x)
        return row_parallel_linear(x, self.weight, self.bias, mode=ALL_REDUCE, tp_dim=self.tp_dim)


class ReplicateParallelLinear(Linear):
    def __init__(self, weight, bias, mesh):
        super().__init__(weight, bias, mesh, tp_dim=None)


class EmbeddingWithReplicateOutput:
    """Table Shard(1) on tp; ids Replicate; output Replicate (DTorch guide)."""

    def __init__(self, weight: torch.Tensor, mesh: DeviceMesh, tp_dim="tp"):
        self.mesh = mesh
        self.tp_dim = mesh.dim_name_index(tp_dim)
        pl = [Replicate()] * mesh.ndim
        if self.tp_dim is not None:
            pl[self.tp_dim] = Shard(1)
        self.weight = DTensor.distribute_tensor(weight, mesh, pl)

    def __call__(self, ids: DTensor) -> DTensor:
        return tp_embedding(ids, self.weight, tp_dim=-1 if self.tp_dim is None else self.tp_dim)
