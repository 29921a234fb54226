"""EmbeddingWithReplicateOutput gather (oracle; test infrastructure only).

Source: DTorch user guide -- Module parallel, section 2 (tensor parallel):
``nn.EmbeddingWithReplicateOutput`` keeps the table Shard(1) on tp (each
rank holds a slice of the embedding dim for every vocabulary row), the
token ids must be Replicate on tp, and the output is made Replicate by an
all-gather along the embedding dim.

So, for token t and shard i with column block [o_i, o_i + d_i):
    out[t, o_i : o_i + d_i] = table_i[id_t, :]
which is a pure copy.  Reading for ids outside [0, vocab) (pages silent):
that token's output row is all zeros and the call reports an index error.
"""
from __future__ import annotations

import numpy as np

from .placement import chunk_bounds


def tp_embedding(ids: np.ndarray, table_shards, dim: int):
    """Return (out, bad) with out[..., dim] assembled from the shards.

    ``table_shards[i]`` is [vocab, d_i] with d_i from the torch.chunk split of
    ``dim``; ``bad`` is True when some id was out of range.
    """
    ids = np.asarray(ids)
    parts = len(table_shards)
    vocab = table_shards[0].shape[0]
    out = np.zeros(ids.shape + (dim,), dtype=table_shards[0].dtype)
    valid = (ids >= 0) & (ids < vocab)
    for i, (o, d) in enumerate(chunk_bounds(dim, parts)):
        t = table_shards[i]
        assert t.shape == (vocab, d)
        block = out[..., o:o + d]             # zeros where the id is invalid
        block[valid] = t[ids[valid]]          # row gather of the valid ids
    return out, bool((~valid).any())
