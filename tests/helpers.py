"""Conversions between the oracle's numpy storage and torch device tensors."""
import numpy as np
import torch

from oracle import bf16
from oracle import placement as opl
import tensor_sharded_linear_gb300 as tsl


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    if dtype == "fp32":
        return torch.from_numpy(a.astype(np.float32)).cuda()
    return torch.from_numpy(a.astype(np.int32)).cuda()


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp32":
        return t.numpy().astype(np.float32)
    return t.numpy().astype(np.int32)


TORCH_DTYPE = {"bf16": torch.bfloat16, "fp32": torch.float32, "int32": torch.int32}


def oracle_placements(pls):
    out = []
    for p in pls:
        if isinstance(p, tsl.Shard):
            out.append(opl.Shard(p.dim))
        elif isinstance(p, tsl.Replicate):
            out.append(opl.Replicate())
        else:
            out.append(opl.Partial(p.reduce_op))
    return out


def lib_placements(pls):
    out = []
    for p in pls:
        if isinstance(p, opl.Shard):
            out.append(tsl.Shard(p.dim))
        elif isinstance(p, opl.Replicate):
            out.append(tsl.Replicate())
        else:
            out.append(tsl.Partial(p.op))
    return out


def dtensor_from_locals(locals_, layout: opl.Layout, dtype: str) -> "tsl.DTensor":
    mesh = tsl.DeviceMesh(layout.mesh_shape)
    slots = [to_dev(a, dtype) for a in locals_]
    return tsl.DTensor(slots, mesh, lib_placements(layout.placements), layout.gshape, TORCH_DTYPE[dtype],
                       layout.materialize_replicas)


def locals_of(dt: "tsl.DTensor", dtype: str):
    return [to_host(t, dtype) for t in dt.slots]


# ---- seeded layouts and values shared by the redistribute parity tests

def random_values(shape, dtype, rng):
    if dtype == "bf16":
        return bf16.round_rne(rng.standard_normal(shape) * 10.0 ** rng.integers(-2, 3))
    if dtype == "fp32":
        return (rng.standard_normal(shape) * 10.0 ** rng.integers(-2, 3)).astype(np.float32)
    return rng.integers(-2 ** 31, 2 ** 31 - 1, size=shape, dtype=np.int64).astype(np.int32)


def random_placements(rng, nm, nd, allow_partial=True):
    out = []
    for _ in range(nm):
        r = rng.random()
        if r < 0.5:
            out.append(opl.Shard(rng.randrange(nd)))
        elif r < 0.8 or not allow_partial:
            out.append(opl.Replicate())
        else:
            out.append(opl.Partial())
    return out


def sweep_transitions():
    """The benchmark's redistribute sweep on a (dp=2, tp=4) mesh; dp kept Shard(0)."""
    return [
        ("S0->S1", [opl.Shard(0), opl.Shard(0)], [opl.Shard(0), opl.Shard(1)]),
        ("S1->S0", [opl.Shard(0), opl.Shard(1)], [opl.Shard(0), opl.Shard(0)]),
        ("S0->R", [opl.Shard(0), opl.Shard(0)], [opl.Shard(0), opl.Replicate()]),
        ("S1->R", [opl.Shard(0), opl.Shard(1)], [opl.Shard(0), opl.Replicate()]),
        ("R->S0", [opl.Shard(0), opl.Replicate()], [opl.Shard(0), opl.Shard(0)]),
        ("R->S1", [opl.Shard(0), opl.Replicate()], [opl.Shard(0), opl.Shard(1)]),
        ("P->R", [opl.Shard(0), opl.Partial()], [opl.Shard(0), opl.Replicate()]),
        ("P->S0", [opl.Shard(0), opl.Partial()], [opl.Shard(0), opl.Shard(0)]),
    ]
