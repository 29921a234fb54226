"""Conversions between the oracle's numpy storage and torch device tensors."""
import numpy as np
import torch

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
