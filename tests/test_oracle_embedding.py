"""Pins for the oracle's embedding gather (CPU only).

The gather is a pure copy, so with every shard concatenated back along the
embedding dim it must equal ``torch.nn.functional.embedding`` (a library
routine) bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle.embedding import tp_embedding
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads


@pytest.mark.parametrize("dim,parts", [(64, 8), (70, 8), (33, 4), (5, 8), (16, 1)])
def test_matches_library_embedding(dim, parts):
    table, ids = workloads.embedding_inputs(vocab=257, dim=dim, ids_shape=(3, 19), seed_base=900 + dim)
    shards = [np.ascontiguousarray(table[:, o:o + s]) for o, s in chunk_bounds(dim, parts)]
    out, bad = tp_embedding(ids, shards, dim)
    assert not bad
    ref = torch.nn.functional.embedding(torch.from_numpy(ids.astype(np.int64)),
                                        torch.from_numpy(table.view(np.int16))).numpy().view(np.uint16)
    np.testing.assert_array_equal(out, ref)


def test_out_of_range_ids_give_zero_rows():
    table, ids = workloads.embedding_inputs(vocab=50, dim=16, ids_shape=(2, 5), seed_base=990)
    ids = ids.copy()
    ids[0, 1] = 50
    ids[1, 3] = -1
    shards = [np.ascontiguousarray(table[:, o:o + s]) for o, s in chunk_bounds(16, 4)]
    out, bad = tp_embedding(ids, shards, 16)
    assert bad
    assert not out[0, 1].any() and not out[1, 3].any()
    np.testing.assert_array_equal(out[0, 0], table[ids[0, 0]])
