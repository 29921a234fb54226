"""GPU parity of dt_tp_embedding against the oracle: bit-exact, every element."""
import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle.embedding import tp_embedding as oracle_embedding
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import to_dev, to_host

pytestmark = pytest.mark.gpu


def run(table, ids, parts, dtype="bf16", materialize=False):
    vocab, dim = table.shape
    mesh = tsl.DeviceMesh((parts,), ("tp",))
    shards = [np.ascontiguousarray(table[:, o:o + s]) for o, s in chunk_bounds(dim, parts)]
    tdt = tsl.DTensor([to_dev(s, dtype) for s in shards], mesh, [tsl.Shard(1)], (vocab, dim),
                      torch.bfloat16 if dtype == "bf16" else torch.float32)
    idt = tsl.DTensor([to_dev(ids, "int32")], mesh, [tsl.Replicate()], ids.shape, torch.int32)
    out = tsl.DTensor.empty(mesh, [tsl.Replicate()], ids.shape + (dim,),
                            torch.bfloat16 if dtype == "bf16" else torch.float32, materialize_replicas=materialize)
    for t in out.slots:
        t.fill_(7)
    tsl.read_device_status(clear=True)
    tsl.tp_embedding(idt, tdt, out=out)
    status = tsl.read_device_status(clear=True)
    expect, bad = oracle_embedding(ids, shards, dim)
    for t in out.slots:
        np.testing.assert_array_equal(to_host(t, dtype), expect)
    return status, bad


@pytest.mark.parametrize("dim,parts", [(512, 8), (70, 8), (64, 4), (33, 4), (4096, 8)])
def test_small_tables(lib, dim, parts):
    table, ids = workloads.embedding_inputs(vocab=1000, dim=dim, ids_shape=(3, 37), seed_base=700 + dim)
    status, bad = run(table, ids, parts)
    assert status == 0 and not bad


def test_fp32_and_materialised_output(lib):
    rng = np.random.default_rng(2)
    table = rng.standard_normal((300, 40)).astype(np.float32)
    ids = rng.integers(0, 300, size=(5, 7)).astype(np.int32)
    status, _ = run(table, ids, 4, dtype="fp32", materialize=True)
    assert status == 0


@pytest.mark.parametrize("dim", [64, 4096])  # 4096 over 8: 1 KiB rows (one row per warp at 18 tokens)
def test_out_of_range_ids_set_status(lib, dim):
    table, ids = workloads.embedding_inputs(vocab=100, dim=dim, ids_shape=(2, 9), seed_base=760)
    ids = ids.copy()
    ids[0, 3] = 100
    ids[1, 0] = -5
    status, bad = run(table, ids, 8)
    assert bad and status & tsl._lib.DEV_ERR_INDEX


def test_full_size_config(lib):
    """table [128256, 4096] bf16 N(0, 0.02^2) in 8 shards, ids [4, 4096]: every element."""
    table, ids = workloads.embedding_inputs()
    status, bad = run(table, ids, workloads.EMBEDDING["parts"])
    assert status == 0 and not bad


def test_out_of_range_ids_two_rows_in_flight(lib):
    """16384 tokens x 8 shards of 1 KiB rows: more items than warps, so each warp
    copies its rows two at a time, and some of those rows have bad ids."""
    table, ids = workloads.embedding_inputs(vocab=1000, dim=4096, ids_shape=(4, 4096), seed_base=780)
    ids = ids.copy()
    rng = np.random.default_rng(781)
    flat = ids.reshape(-1)
    pos = rng.choice(flat.size, 64, replace=False)
    flat[pos[:32]] = 1000 + rng.integers(0, 50, 32)
    flat[pos[32:]] = -1 - rng.integers(0, 50, 32)
    status, bad = run(table, ids, 8)
    assert bad and status & tsl._lib.DEV_ERR_INDEX


def test_no_tokens(lib):
    """Empty ids: OK, no launch, an empty output."""
    table, _ = workloads.embedding_inputs(vocab=100, dim=512, ids_shape=(1, 1), seed_base=790)
    n0 = lib.dt_launch_count()
    status, bad = run(table, np.zeros((2, 0), dtype=np.int32), 8)
    assert status == 0 and not bad
    assert lib.dt_launch_count() == n0
