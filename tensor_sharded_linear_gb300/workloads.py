"""Seeded synthetic inputs for the tensor-parallel workloads.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle
take their inputs from here, so the two sides see the same bytes.

Recipe
------
* Every tensor is drawn from its own ``torch.Generator`` on the CPU, seeded
  with ``seed``; normal draws are ``torch.randn`` scaled by ``std``, then
  converted with ``Tensor.to(torch.bfloat16)`` (round to nearest even) where
  the workload is bf16.  bf16 tensors are returned as numpy ``uint16`` bit
  patterns, fp32 as ``float32``, ids as ``int32``.
* Large tensors are drawn in row blocks of at most 64 Mi elements from the
  same generator, so host memory stays bounded; the stream of numbers is a
  fixed function of (shape, seed).
* Seeds: the worked example uses seed 0 for x and W, as the page does; the
  other workloads use ``100 * workload + k`` for their k-th tensor.
"""
from __future__ import annotations

import numpy as np
import torch

_BLOCK = 64 * 1024 * 1024


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _rows_per_block(shape) -> int:
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    return max(1, _BLOCK // max(inner, 1))


def randn_f32(shape, seed: int, std: float = 1.0) -> np.ndarray:
    g = _gen(seed)
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.float32)
    if out.size == 0:
        return out
    rb = _rows_per_block(shape)
    for r0 in range(0, shape[0], rb):
        r1 = min(shape[0], r0 + rb)
        t = torch.randn((r1 - r0,) + shape[1:], generator=g, dtype=torch.float32)
        if std != 1.0:
            t = t * std
        out[r0:r1] = t.numpy()
    return out


def randn_bf16(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0, std^2) draws (torch CPU RNE conversion)."""
    g = _gen(seed)
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if out.size == 0:
        return out
    rb = _rows_per_block(shape)
    for r0 in range(0, shape[0], rb):
        r1 = min(shape[0], r0 + rb)
        t = torch.randn((r1 - r0,) + shape[1:], generator=g, dtype=torch.float32)
        if std != 1.0:
            t = t * std
        out[r0:r1] = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


def randint_i32(shape, low: int, high: int, seed: int) -> np.ndarray:
    g = _gen(seed)
    t = torch.randint(int(low), int(high), tuple(int(s) for s in shape), generator=g, dtype=torch.int64)
    return t.numpy().astype(np.int32)


def arange_f32(shape) -> np.ndarray:
    n = int(np.prod(shape))
    return np.arange(n, dtype=np.float32).reshape(shape)


# -- the workloads, by name and size ---------------------------------------

WORKED_EXAMPLE = dict(x=(3, 8), w=(8, 12), parts=4, mesh=(2, 2), square=(4, 4))
EMBEDDING = dict(vocab=128256, dim=4096, parts=8, ids=(4, 4096), std=0.02)
REDISTRIBUTE = dict(shape=(8192, 8192), uneven=(8191, 8190), mesh=(2, 4), partials=4)
MLP = dict(tokens=4096, hidden=4096, ffn=11008, parts=8)
ATTENTION = dict(tokens=8192, hidden=4096, parts=4)


def worked_example():
    """x[3, 8] and W[8, 12] ([in, out]), fp32 N(0, 1), both from seed 0.

    The page seeds the global torch RNG with 0 and draws x then W; the same
    stream is reproduced here with one generator.
    """
    g = _gen(0)
    x = torch.randn(3, 8, generator=g)
    w = torch.randn(8, 12, generator=g)
    return x.numpy().copy(), w.numpy().copy()


def embedding_inputs(vocab=None, dim=None, ids_shape=None, seed_base=200):
    vocab = EMBEDDING["vocab"] if vocab is None else vocab
    dim = EMBEDDING["dim"] if dim is None else dim
    ids_shape = EMBEDDING["ids"] if ids_shape is None else ids_shape
    table = randn_bf16((vocab, dim), seed_base + 0, EMBEDDING["std"])
    ids = randint_i32(ids_shape, 0, vocab, seed_base + 1)
    return table, ids


def redistribute_global(shape=None, seed=300):
    shape = REDISTRIBUTE["shape"] if shape is None else shape
    return randn_bf16(shape, seed)


def redistribute_partials(local_shape, count, seed=310):
    """``count`` independent N(0, 1) partial slots of ``local_shape``."""
    return [randn_bf16(local_shape, seed + k) for k in range(count)]


def mlp_inputs(tokens=None, hidden=None, ffn=None, seed_base=400):
    tokens = MLP["tokens"] if tokens is None else tokens
    hidden = MLP["hidden"] if hidden is None else hidden
    ffn = MLP["ffn"] if ffn is None else ffn
    x = randn_bf16((tokens, hidden), seed_base + 0)
    wg = randn_bf16((hidden, ffn), seed_base + 1, (1.0 / hidden) ** 0.5)
    wu = randn_bf16((hidden, ffn), seed_base + 2, (1.0 / hidden) ** 0.5)
    wd = randn_bf16((ffn, hidden), seed_base + 3, (1.0 / ffn) ** 0.5)
    return x, wg, wu, wd


def attention_inputs(tokens=None, hidden=None, seed_base=500):
    tokens = ATTENTION["tokens"] if tokens is None else tokens
    hidden = ATTENTION["hidden"] if hidden is None else hidden
    std = (1.0 / hidden) ** 0.5
    x = randn_bf16((tokens, hidden), seed_base + 0)
    ws = [randn_bf16((hidden, hidden), seed_base + 1 + k, std) for k in range(4)]
    return (x, *ws)
