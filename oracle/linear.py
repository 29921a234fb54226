"""Tensor-parallel linears in fp64 (oracle; test infrastructure only).

Sources
-------
* Model parallelism (wineandchord), "Tensor Parallel": for Y = X W,
  column parallel splits W by output columns, W = [W_1 .. W_P] and
  Y_i = X W_i; row parallel splits X by its last dim and W by rows and sums,
  Y = sum_i X_i W_i.  "Tensor-parallel linear layers" uses the [in, out]
  weight convention, ``torch.chunk`` shards, and checks both against the
  dense X W on x[3, 8], W[8, 12], 4 parts.
* DTorch user guide -- Module parallel, section 3: column bias is sharded
  like the output features; row bias is Partial() on tp, so the reduced
  output carries the bias exactly once.  The column layer's input must be
  Replicate on tp, the row layer's input Shard(-1).
* nanotron tutorial ch. 5, section 5.1: the row layer's output is either
  all-reduced (ALL_REDUCE: every rank gets the full output) or
  reduce-scattered (REDUCE_SCATTER: each rank keeps a block of rows); the
  Llama attention is q/k/v column + o row, the MLP likewise.

Arithmetic: inputs are widened exactly to fp64 (bf16 -> fp64, fp32 -> fp64)
and every product is computed in fp64 with ``numpy.matmul`` (a library
primitive used as one step).  Where the method stores an intermediate in
bf16 (the MLP's H and the attention's q feeding o), the oracle rounds that
intermediate once, nearest-even, from its fp64 value.
"""
from __future__ import annotations

import numpy as np

from . import bf16
from .placement import chunk_bounds

ALL_REDUCE = "all_reduce"
REDUCE_SCATTER = "reduce_scatter"
PARTIAL = "partial"


def as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to fp64."""
    if dtype == "bf16":
        return bf16.widen64(a)
    return np.asarray(a, dtype=np.float64)


def column_parallel(x, w_shards, bias_shards=None):
    """Y_i = X W_i (+ b_i) for every column shard i; fp64 in, fp64 out.

    ``x`` is [..., K] (Replicate on tp), ``w_shards[i]`` is [K, N_i].
    """
    ys = []
    for i, w in enumerate(w_shards):
        y = np.matmul(x, w)
        if bias_shards is not None and bias_shards[i] is not None:
            y = y + bias_shards[i]
        ys.append(y)
    return ys


def column_parallel_seq(x_token_shards, w_shards, bias_shards=None):
    """Sequence-parallel column entry (nanotron tutorial 5.1, REDUCE_SCATTER
    mode of TensorParallelColumnLinear): the input arrives sharded over tokens
    (dim 0); it is all-gathered, then every column shard is applied to all
    tokens.  Returns the Shard(-1) outputs with all tokens."""
    x = np.concatenate(list(x_token_shards), axis=0)
    return column_parallel(x, w_shards, bias_shards)


def column_parallel_replicate(x, w_shards, bias_shards=None):
    """ColumnParallelLinearWithReplicateOutput (DTorch guide, section 3): the
    Shard(-1) outputs gathered into one Replicate tensor along features."""
    return np.concatenate(column_parallel(x, w_shards, bias_shards), axis=-1)


def row_sum(x_shards, w_shards):
    """sum_i X_i W_i in fp64, terms added in rank order."""
    y = None
    for xi, wi in zip(x_shards, w_shards):
        t = np.matmul(xi, wi)
        y = t if y is None else y + t
    return y


def row_parallel(x_shards, w_shards, bias=None, mode=ALL_REDUCE, parts=None):
    """Row-parallel linear.  Returns the list of output locals for ``mode``.

    ALL_REDUCE     -> [Y]                   (Replicate; one stored copy)
    REDUCE_SCATTER -> [Y rows of block j]   (Shard(0), torch.chunk row blocks)
    PARTIAL        -> [X_i W_i]             (Partial; bias added to part 0 only,
                                             so the parts sum to Y + b)
    """
    p = len(w_shards) if parts is None else parts
    if mode == PARTIAL:
        outs = [np.matmul(xi, wi) for xi, wi in zip(x_shards, w_shards)]
        if bias is not None:
            outs[0] = outs[0] + bias
        return outs
    y = row_sum(x_shards, w_shards)
    if bias is not None:
        y = y + bias
    if mode == ALL_REDUCE:
        return [y]
    if mode == REDUCE_SCATTER:
        return [y[o:o + s] for o, s in chunk_bounds(y.shape[0], p)]
    raise ValueError(mode)


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g)), fp64."""
    return g / (1.0 + np.exp(-g))


def mlp_hidden(x, wg_shards, wu_shards):
    """H_i = bf16(SiLU(X Wg_i) * (X Wu_i)) for every shard; returns bf16 bits.

    Llama-style gated MLP on column-parallel gate/up projections (nanotron
    tutorial 5.1: the MLP follows the attention's column/row pattern).
    """
    hs = []
    for wg, wu in zip(wg_shards, wu_shards):
        h = silu(np.matmul(x, wg)) * np.matmul(x, wu)
        hs.append(bf16.round_rne(h))
    return hs


def tp_mlp(x, wg_shards, wu_shards, wd_shards, mode=ALL_REDUCE):
    """Column gate/up -> SiLU*mul (bf16 H) -> row down projection.

    Returns (outputs for ``mode``, H shards as bf16 bits).
    """
    hs = mlp_hidden(x, wg_shards, wu_shards)
    h64 = [bf16.widen64(h) for h in hs]
    return row_parallel(h64, wd_shards, None, mode), hs


def attention_projections(x, wq_shards, wk_shards, wv_shards, wo_shards, mode=REDUCE_SCATTER):
    """q/k/v column-parallel, then o row-parallel on q's Shard(-1) output.

    The attention itself is not part of the path; q's bf16 output stands in
    for the attention output that feeds o.  Returns
    (o outputs for ``mode``, q, k, v shards as bf16 bits).
    """
    q = [bf16.round_rne(y) for y in column_parallel(x, wq_shards)]
    k = [bf16.round_rne(y) for y in column_parallel(x, wk_shards)]
    v = [bf16.round_rne(y) for y in column_parallel(x, wv_shards)]
    o = row_parallel([bf16.widen64(qi) for qi in q], wo_shards, None, mode)
    return o, q, k, v
