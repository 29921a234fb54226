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


def test_no_tokens_and_no_vocabulary():
    """Empty ids give an empty [.., dim] output and no index error; with an
    empty vocabulary every id is out of range, so every row is zero."""
    table, _ = workloads.embedding_inputs(vocab=40, dim=12, ids_shape=(1, 1), seed_base=995)
    shards = [np.ascontiguousarray(table[:, o:o + s]) for o, s in chunk_bounds(12, 4)]
    out, bad = tp_embedding(np.zeros((2, 0), dtype=np.int32), shards, 12)
    assert out.shape == (2, 0, 12) and not bad
    empty = [np.zeros((0, s), dtype=table.dtype) for _, s in chunk_bounds(12, 4)]
    out, bad = tp_embedding(np.array([[0, 3]], dtype=np.int32), empty, 12)
    assert bad and out.shape == (1, 2, 12) and not out.any()
