"""Seeded random cases of the tensor-parallel linears against the fp64 oracle.

Each case draws M, K, N and the part count P, so shards are ragged
(torch.chunk, empty tails included), tiles are ragged in M, N and K, and
TMA's out-of-bounds fill is exercised; bias on or off, bf16 and fp32
outputs, weights stored [in, out] or as [out, in] views, and every
row-parallel mode; token-sharded inputs into fused column layers (the
sequence-parallel entry).  K a multiple of 8 keeps bf16 row pitches 16-byte
aligned (the tcgen05 path); other K give pitches TMA cannot read, which the
calls copy to padded pitches in their workspace (the Python API passes the
queried size) and run on the tcgen05 path too; the CUDA-core kernel is
tested in test_gpu_linear.py.  Tolerances as in the other linear tests.
"""
import random

import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import linear as olin
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import to_dev, to_host
from test_gpu_linear import OMODE, check_bf16, check_fp32, col_dtensor, mesh1, row_dtensor, w64, x_rep, x_shard

pytestmark = pytest.mark.gpu


def draw(rng, aligned):
    M = rng.choice([1, 7, 129, 256, 300, 513, 700])
    K = rng.choice([8, 64, 136, 512, 1000, 1368]) if aligned else rng.choice([5, 37, 130, 301])
    N = rng.choice([8, 40, 264, 520, 1032]) if aligned else rng.choice([9, 77, 303])
    P = rng.choice([1, 2, 3, 4, 8])
    return M, K, N, P


@pytest.mark.parametrize("seed", range(48))
def test_column_fuzz(lib, seed):
    rng = random.Random(3000 + seed)
    aligned = seed % 4 != 3
    M, K, N, P = draw(rng, aligned)
    x = workloads.randn_bf16((M, K), 3100 + seed)
    w = workloads.randn_bf16((K, N), 3200 + seed, (1.0 / K) ** 0.5)
    use_bias = rng.random() < 0.5
    kmajor = aligned and rng.random() < 0.3
    cols = chunk_bounds(N, P)
    bd = None
    if use_bias:
        b = workloads.randn_bf16((N,), 3300 + seed, 0.5)
        bd = tsl.DTensor([to_dev(np.ascontiguousarray(b[o:o + s]), "bf16") for o, s in cols], mesh1(P),
                         [tsl.Shard(0)], (N,), torch.bfloat16)
    xd, wd = x_rep(x, P), col_dtensor(w, P, k_major=kmajor)
    y32 = tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32)
    y16 = tsl.column_parallel_linear(xd, wd, bd)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in cols],
                                  [w64(b[o:o + s]) for o, s in cols] if use_bias else None)
    what = f"M={M} K={K} N={N} P={P} bias={use_bias} kmajor={kmajor}"
    for i, e in enumerate(expect):
        f = to_host(y32.slots[i], "fp32")
        check_fp32(f, e, f"{what} shard {i}")
        check_bf16(to_host(y16.slots[i], "bf16"), f, e, f"{what} shard {i}")


@pytest.mark.parametrize("seed", range(48))
def test_row_fuzz(lib, seed):
    rng = random.Random(4000 + seed)
    aligned = seed % 4 != 3
    M, K, N, P = draw(rng, aligned)
    mode = [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER, tsl.PARTIAL][seed % 3]
    x = workloads.randn_bf16((M, K), 4100 + seed)
    w = workloads.randn_bf16((K, N), 4200 + seed, (1.0 / K) ** 0.5)
    use_bias = mode != tsl.PARTIAL and rng.random() < 0.5
    kmajor = aligned and rng.random() < 0.3
    bd = None
    if use_bias:
        b = workloads.randn_bf16((N,), 4300 + seed, 0.5)
        bd = tsl.DTensor([to_dev(b, "bf16")], mesh1(P), [tsl.Replicate()], (N,), torch.bfloat16)
    xd, wd = x_shard(x, P), row_dtensor(w, P, k_major=kmajor)
    y32 = tsl.row_parallel_linear(xd, wd, bd, mode=mode, out_dtype=torch.float32)
    y16 = tsl.row_parallel_linear(xd, wd, bd, mode=mode)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    omode = OMODE[mode]
    rows = chunk_bounds(K, P)
    expect = olin.row_parallel([w64(x[:, o:o + s]) for o, s in rows], [w64(w[o:o + s]) for o, s in rows],
                               w64(b) if use_bias else None, omode, parts=P)
    what = f"M={M} K={K} N={N} P={P} mode={mode} bias={use_bias} kmajor={kmajor}"
    assert len(expect) == len(y32.slots)
    for i, e in enumerate(expect):
        f = to_host(y32.slots[i], "fp32")
        check_fp32(f, e, f"{what} out {i}")
        check_bf16(to_host(y16.slots[i], "bf16"), f, e, f"{what} out {i}")


@pytest.mark.parametrize("seed", range(24))
def test_mlp_fuzz(lib, seed):
    rng = random.Random(5000 + seed)
    M = rng.choice([1, 100, 256, 333])
    K = rng.choice([64, 136, 256])
    P = rng.choice([1, 2, 4, 8])
    F = P * rng.choice([8, 64, 96, 136])
    N = rng.choice([8, 200, 384])
    mode = [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER, tsl.PARTIAL][seed % 3]
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=5100 + 10 * seed)
    wd = workloads.randn_bf16((F, N), 5200 + seed, (1.0 / F) ** 0.5)
    xd = x_rep(x, P)
    y = tsl.tp_mlp(xd, col_dtensor(wg, P), col_dtensor(wu, P), row_dtensor(wd, P), mode=mode,
                   out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    cols = chunk_bounds(F, P)
    expect, _ = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols],
                            [w64(wd[o:o + s]) for o, s in cols], OMODE[mode])
    what = f"M={M} K={K} F={F} N={N} P={P} mode={mode}"
    assert len(expect) == len(y.slots)
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"{what} out {i}")


def x_tokens(x_bits, p):
    """[T, K] bf16, Shard(0) over p (token shards)."""
    slots = [to_dev(np.ascontiguousarray(x_bits[o:o + s]), "bf16") for o, s in chunk_bounds(x_bits.shape[0], p)]
    return tsl.DTensor(slots, mesh1(p), [tsl.Shard(0)], x_bits.shape, torch.bfloat16)


@pytest.mark.parametrize("seed", range(24))
def test_column_variants_fuzz(lib, seed):
    """Sequence-parallel entry (token-sharded x), Replicate output, and
    several weights sharing x in one launch, on random shapes."""
    rng = random.Random(6000 + seed)
    aligned = seed % 4 != 3
    M, K, N, P = draw(rng, aligned)
    seq = rng.random() < 0.5
    x = workloads.randn_bf16((M, K), 6100 + seed)
    xd = x_tokens(x, P) if seq else x_rep(x, P)
    cols = chunk_bounds(N, P)
    xs = [w64(x[o:o + s]) for o, s in chunk_bounds(M, P)]
    what = f"M={M} K={K} N={N} P={P} seq={seq}"
    if seed % 2 == 0:
        w = workloads.randn_bf16((K, N), 6200 + seed, (1.0 / K) ** 0.5)
        y = tsl.column_parallel_linear(xd, col_dtensor(w, P), out_dtype=torch.float32, output="replicate")
        torch.cuda.synchronize()
        assert tsl.read_device_status() == 0
        expect = olin.column_parallel_replicate(w64(x), [w64(w[:, o:o + s]) for o, s in cols])
        check_fp32(to_host(y.slots[0], "fp32"), expect, f"{what} replicate output")
    else:
        ws = [workloads.randn_bf16((K, N), 6300 + 3 * seed + j, (1.0 / K) ** 0.5) for j in range(3)]
        ys = tsl.column_parallel_linear_multi(xd, [col_dtensor(w, P) for w in ws], out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert tsl.read_device_status() == 0
        for j, w in enumerate(ws):
            shards = [w64(w[:, o:o + s]) for o, s in cols]
            expect = olin.column_parallel_seq(xs, shards) if seq else olin.column_parallel(w64(x), shards)
            for i, e in enumerate(expect):
                check_fp32(to_host(ys[j].slots[i], "fp32"), e, f"{what} weight {j} shard {i}")


@pytest.mark.parametrize("seed", range(16))
def test_sequence_parallel_fuzz(lib, seed):
    """Token-sharded x (Shard(0)) into 1 to 3 fused column layers: each token
    shard is one block of the GEMM's rows, read in place.  Token counts give
    one or several M tiles per shard, equal or not (the launch orders its
    tiles as row blocks of one GEMM when every shard has the same M tiles)."""
    rng = random.Random(6000 + seed)
    P = rng.choice([2, 3, 4, 8])
    T = rng.choice([5, 300, 1030, 1300, 2100, 2600])
    K = rng.choice([64, 136, 512, 1368])
    N = rng.choice([40, 264, 520, 1032])
    nw = rng.choice([1, 2, 3])
    x = workloads.randn_bf16((T, K), 6100 + seed)
    ws = [workloads.randn_bf16((K, N), 6200 + 10 * seed + j, (1.0 / K) ** 0.5) for j in range(nw)]
    toks = chunk_bounds(T, P)
    xd = tsl.DTensor([to_dev(np.ascontiguousarray(x[o:o + s]), "bf16") for o, s in toks], mesh1(P),
                     [tsl.Shard(0)], x.shape, torch.bfloat16)
    wds = [col_dtensor(w, P) for w in ws]
    outs = [tsl.DTensor.empty(mesh1(P), [tsl.Shard(1)], (T, N), torch.float32) for _ in ws]
    tsl.column_parallel_linear_multi(xd, wds, outs=outs)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    xs = [w64(x[o:o + s]) for o, s in toks]
    cols = chunk_bounds(N, P)
    for j, w in enumerate(ws):
        expect = olin.column_parallel_seq(xs, [w64(w[:, o:o + s]) for o, s in cols])
        for i, e in enumerate(expect):
            check_fp32(to_host(outs[j].slots[i], "fp32"), e, f"T={T} K={K} N={N} P={P} weight {j} shard {i}")
