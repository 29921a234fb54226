"""GPU parity of the GEMM's split tail against the fp64 oracle.

When the last wave of 256 x 256 tiles would leave CTA pairs idle and the
tiles are long in K, the tail tiles' K iterations are divided over every pair; each piece writes an
fp32 partial accumulator and the piece that completes a tile's count adds
them in K order and runs the epilogue.  The shapes below have fewer tiles
than the 76 pairs a GB300 holds and enough K for the split to pay:
column (bias, ragged M/N/K, fp32 and bf16 outputs), row-parallel in every
output mode, the gated MLP (gate/up end to end, down on the oracle's H)
and fused q/k/v.  The scratch is the caller's workspace (the Python API
takes one of the queried size from torch's allocator): the queries report
the library's rule, a call without enough workspace runs every tile whole,
and a split call allocates no device memory.  Also: the split result is
bit-identical from launch to launch (the partials are added in a fixed
order and the counters are zeroed before every launch), two streams split
concurrently with separate workspaces, and the unsplit schedule
(DT_GEMM_SPLIT=0, in a child process) agrees with the oracle on the same
shapes.  Tolerances as in the other linear tests (the MLP output: the
relative Frobenius bound, for the reason its test gives).
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import linear as olin
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import to_dev, to_host
from test_gpu_linear import (REL_FRO_TOL, check_bf16, check_bf16_pair, check_fp32, col_dtensor, mesh1, row_dtensor,
                             w64, x_rep, x_shard)

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def ceil_div(a, b):
    return -(-a // b)


PAIRS = 76  # CTA pairs resident on a GB300 (152 SMs)


def split_expected(tiles, kiters, dual=False, pairs=PAIRS):
    """The library's rule: a pair's share of the tail's K iterations plus
    the split's fixed cost (40 iterations) is shorter than a tile, and no
    tail tile has more than 8 pieces (the finishing warp reads them all).
    `dual` (the gated MLP) does not change the rule."""
    rem = tiles % pairs
    share_min = rem * kiters // pairs
    if rem == 0 or share_min < 8:
        return False
    np_ = ceil_div(kiters, share_min) + 1
    return np_ <= 8 and rem * kiters / pairs + 40 <= kiters


def r256(n):
    return (n + 255) // 256 * 256


def split_bytes(tiles, kiters, dual=False, pairs=PAIRS):
    """Workspace of one split launch: an fp32 [2, 128, 256] partial per piece
    (the tail tiles plus one per pair boundary inside the tail) and 8
    counters per tail tile, each region 256-byte aligned."""
    if not split_expected(tiles, kiters, dual, pairs):
        return 0
    rem = tiles % pairs
    return r256((rem + pairs - 1) * 2 * 128 * 256 * 4) + r256(8 * rem * 4)


def device_pairs():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def no_workspace():
    """An empty device tensor: its data pointer is NULL, so the call gets no workspace."""
    return torch.empty(0, dtype=torch.uint8, device="cuda")


def column_case(seed=11):
    M, K, N, p = 300, 12000, 4 * 520, 4
    assert split_expected(ceil_div(M, 256) * p * ceil_div(N // p, 256), ceil_div(K, 64))
    x = workloads.randn_bf16((M, K), seed)
    w = workloads.randn_bf16((K, N), seed + 1, (1.0 / K) ** 0.5)
    b = workloads.randn_bf16((N,), seed + 2, 0.5)
    bd = tsl.DTensor([to_dev(np.ascontiguousarray(b[o:o + s]), "bf16") for o, s in chunk_bounds(N, p)], mesh1(p),
                     [tsl.Shard(0)], (N,), torch.bfloat16)
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)],
                                  [w64(b[o:o + s]) for o, s in chunk_bounds(N, p)])
    return x_rep(x, p), col_dtensor(w, p), bd, expect


def test_column_split(lib):
    xd, wd, bd, expect = column_case()
    y32 = tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32)
    y16 = tsl.column_parallel_linear(xd, wd, bd)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for i, e in enumerate(expect):
        f = to_host(y32.slots[i], "fp32")
        check_fp32(f, e, f"shard {i}")
        check_bf16(to_host(y16.slots[i], "bf16"), f, e, f"shard {i}")


@pytest.mark.parametrize("mode", [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER, tsl.PARTIAL])
def test_row_split(lib, mode):
    """ALL_REDUCE and REDUCE_SCATTER split (one group, 4 K segments); the
    PARTIAL launch (one group per shard) is too short to split and runs
    whole, checked all the same."""
    M, K, N, p = 700, 4 * 2000, 1304, 4  # 1304 = 5 x 256 + 24: ragged, with a TMA-compatible pitch
    tiles = ceil_div(M, 256) * ceil_div(N, 256) * (p if mode == tsl.PARTIAL else 1)
    kiters = ceil_div(K // p, 64) * (1 if mode == tsl.PARTIAL else p)
    assert split_expected(tiles, kiters) == (mode != tsl.PARTIAL)
    x = workloads.randn_bf16((M, K), 41)
    w = workloads.randn_bf16((K, N), 42, (1.0 / K) ** 0.5)
    b = workloads.randn_bf16((N,), 43, 0.5)
    bd = tsl.DTensor([to_dev(b, "bf16")], mesh1(p), [tsl.Replicate()], (N,), torch.bfloat16)
    xd, wd = x_shard(x, p), row_dtensor(w, p)
    y32 = tsl.row_parallel_linear(xd, wd, bd, mode=mode, out_dtype=torch.float32)
    y16 = tsl.row_parallel_linear(xd, wd, bd, mode=mode)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    omode = {tsl.ALL_REDUCE: olin.ALL_REDUCE, tsl.REDUCE_SCATTER: olin.REDUCE_SCATTER, tsl.PARTIAL: olin.PARTIAL}[mode]
    expect = olin.row_parallel([w64(x[:, o:o + s]) for o, s in chunk_bounds(K, p)],
                               [w64(w[o:o + s]) for o, s in chunk_bounds(K, p)], w64(b), omode, parts=p)
    for i, e in enumerate(expect):
        f = to_host(y32.slots[i], "fp32")
        check_fp32(f, e, f"{mode} out {i}")
        check_bf16(to_host(y16.slots[i], "bf16"), f, e, f"{mode} out {i}")


MLP_SPLIT_SHAPES = [
    (256, 10000, 8 * 600, 384, 8),  # 40 dual tiles, 157 K iterations: 3 pieces per tail tile
    (256, 8000, 5 * 600, 384, 5),   # 25 dual tiles, 125 K iterations: 5 pieces per tail tile
]


@pytest.mark.parametrize("M,K,F,N,p", MLP_SPLIT_SHAPES)
def test_mlp_split(lib, M, K, F, N, p):
    """The fused MLP with its gated gate/up GEMM split (each shard's last
    tile 88 columns of gate and up; 600 = 4 x 128 + 88).  The split GEMM's output, H, is checked per element; the
    MLP output with the relative Frobenius bound.  (Its max-abs error also
    carries H's bf16 rounding: where the kernel's fp32 SiLU(g)*u and the
    oracle's fp64 one round to neighbouring bf16 values, each such element
    moves outputs by one bf16 ulp of H times a weight, which at this K can
    pass 2e-3 on a few outputs with either schedule.  The down GEMM's split
    is test_mlp_down_split, on the oracle's H.)"""
    assert split_expected(ceil_div(M, 256) * p * ceil_div(F // p, 128), ceil_div(K, 64), dual=True)
    x, wg, wu, wd = workloads.mlp_inputs(M, K, F, seed_base=700)
    wd = workloads.randn_bf16((F, N), 704, (1.0 / F) ** 0.5)
    xd = x_rep(x, p)
    wgd, wud, wdd = col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    y = tsl.tp_mlp_output(xd, wdd, mode=tsl.ALL_REDUCE, out_dtype=torch.float32)
    ws = torch.empty(tsl.tp_mlp_workspace_bytes(xd, wgd, wud, wdd, y), dtype=torch.uint8, device="cuda")
    y = tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, out=y, workspace=ws)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    cols = chunk_bounds(F, p)
    expect, hs = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols],
                             [w64(wd[o:o + s]) for o, s in cols], olin.ALL_REDUCE)
    check_bf16_pair(to_host(tsl.api.mlp_hidden_view(xd, col_dtensor(wg, p), ws), "bf16"),
                    np.concatenate(hs, axis=-1), "H")
    got = to_host(y.slots[0], "fp32").astype(np.float64)
    assert np.isfinite(got).all()
    fro = np.linalg.norm(got - expect[0]) / np.linalg.norm(expect[0])
    assert fro <= REL_FRO_TOL, fro


def test_mlp_down_split(lib):
    """The MLP's down projection split (20 tiles, 8 segments of 16 K
    iterations), fed the oracle's own bf16 H: ALL_REDUCE of H_i Wd_i."""
    M, K, F, N, p = 512, 256, 8 * 1024, 2560, 8
    assert split_expected(ceil_div(M, 256) * ceil_div(N, 256), p * ceil_div(F // p, 64))
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=720)
    wd = workloads.randn_bf16((F, N), 724, (1.0 / F) ** 0.5)
    cols = chunk_bounds(F, p)
    hs = olin.mlp_hidden(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols])
    h = np.concatenate(hs, axis=-1)
    y = tsl.row_parallel_linear(x_shard(h, p), row_dtensor(wd, p), mode=tsl.ALL_REDUCE, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    expect = olin.row_parallel([w64(hi) for hi in hs], [w64(wd[o:o + s]) for o, s in cols], None, olin.ALL_REDUCE)
    check_fp32(to_host(y.slots[0], "fp32"), expect[0], "down projection")


def test_qkv_split(lib):
    """Fused q/k/v: 3 weights x 4 shards, 24 tiles of 128 K iterations."""
    T, K, N, p = 512, 8192, 1024, 4
    assert split_expected(ceil_div(T, 256) * 3 * p * ceil_div(N // p, 256), ceil_div(K, 64))
    x = workloads.randn_bf16((T, K), 751)
    ws = [workloads.randn_bf16((K, N), 752 + j, (1.0 / K) ** 0.5) for j in range(3)]
    ys = tsl.column_parallel_linear_multi(x_rep(x, p), [col_dtensor(w, p) for w in ws], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for j, w in enumerate(ws):
        expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
        for i in range(p):
            check_fp32(to_host(ys[j].slots[i], "fp32"), expect[i], f"weight {j} shard {i}")


def test_split_is_deterministic(lib):
    """Ten launches of one split GEMM (one workspace) give the same bits:
    fixed summation order, and the counters are zeroed before every launch."""
    xd, wd, bd, expect = column_case(seed=21)
    out = tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32)
    first = [t.clone() for t in out.slots]
    for _ in range(10):
        tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32, out=out)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for a, b in zip(first, out.slots):
        assert torch.equal(a, b)
    for i, e in enumerate(expect):
        check_fp32(to_host(out.slots[i], "fp32"), e, f"shard {i}")


def test_split_on_two_streams(lib):
    """Two streams run split GEMMs at the same time, each with its own workspace."""
    cases = [column_case(seed=31), column_case(seed=41)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    torch.cuda.synchronize()
    for (xd, wd, bd, _), s in zip(cases, streams):
        with torch.cuda.stream(s):
            outs.append(tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32))
    for _ in range(3):  # interleave more launches on both
        for (xd, wd, bd, _), s, o in zip(cases, streams, outs):
            with torch.cuda.stream(s):
                tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32, out=o)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for (_, _, _, expect), o in zip(cases, outs):
        for i, e in enumerate(expect):
            check_fp32(to_host(o.slots[i], "fp32"), e, f"shard {i}")


def test_workspace_queries_follow_the_rule(lib):
    """The size queries report the split rule's bytes (0 where a launch
    does not split), and the MLP's query adds H's 256-byte aligned blocks."""
    pairs = device_pairs()
    xd, wd, _, _ = column_case()
    ys = [tsl.DTensor.empty(xd.mesh, [tsl.Shard(1)], (300, wd.gshape[1]), torch.float32)]
    assert tsl.column_parallel_linear_workspace_bytes(xd, [wd], ys) == split_bytes(2 * 4 * 3, 188, pairs=pairs)
    M, K, N, p = 700, 4 * 2000, 1304, 4  # 1304 = 5 x 256 + 24: ragged, with a TMA-compatible pitch
    xr, wr = x_shard(workloads.randn_bf16((M, K), 41), p), row_dtensor(workloads.randn_bf16((K, N), 42), p)
    for mode, tiles, kiters in ((tsl.ALL_REDUCE, 3 * 6, 4 * 32), (tsl.REDUCE_SCATTER, 3 * 6, 4 * 32),
                                (tsl.PARTIAL, 4 * 3 * 6, 32)):
        y = tsl.api._row_out(xr, wr, 0, mode, torch.float32)
        assert tsl.row_parallel_linear_workspace_bytes(xr, wr, y, mode) == split_bytes(tiles, kiters, pairs=pairs), mode
    M, K, F, N, p = 256, 10000, 8 * 600, 384, 8
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=700)
    wd = workloads.randn_bf16((F, N), 704, (1.0 / F) ** 0.5)
    xm, wgd, wud, wdd = x_rep(x, p), col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    y = tsl.tp_mlp_output(xm, wdd)
    h_bytes = r256(M * F * 2)
    up = split_bytes(p * ceil_div(F // p, 128), ceil_div(K, 64), dual=True, pairs=pairs)
    down = split_bytes(ceil_div(N, 256), p * ceil_div(F // p, 64), pairs=pairs)
    assert tsl.tp_mlp_workspace_bytes(xm, wgd, wud, wdd, y) == h_bytes + max(up, down)


def test_split_needs_the_workspace(lib):
    """No workspace, or one 256 bytes short: every tile whole (both give the
    same bits, within tolerance); the queried size: the split schedule,
    whose fp32 sums run in another order, so some output bits differ."""
    xd, wd, bd, expect = column_case(seed=51)
    need = tsl.column_parallel_linear_workspace_bytes(xd, [wd], [tsl.api._col_out(xd, wd, 0, torch.float32)])
    assert need > 0
    runs = {}
    for name, ws in (("none", no_workspace()),
                     ("short", torch.empty(need - 256, dtype=torch.uint8, device="cuda")),
                     ("full", torch.empty(need, dtype=torch.uint8, device="cuda"))):
        runs[name] = tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    for name, y in runs.items():
        for i, e in enumerate(expect):
            check_fp32(to_host(y.slots[i], "fp32"), e, f"{name} shard {i}")
    assert all(torch.equal(a, b) for a, b in zip(runs["none"].slots, runs["short"].slots))
    assert not all(torch.equal(a, b) for a, b in zip(runs["none"].slots, runs["full"].slots))


def test_split_call_allocates_nothing(lib):
    """With the caller's workspace, a split launch on a stream the library
    has never seen leaves the device's free memory unchanged."""
    xd, wd, bd, expect = column_case(seed=61)
    y = tsl.api._col_out(xd, wd, 0, torch.float32)
    ws = torch.empty(tsl.column_parallel_linear_workspace_bytes(xd, [wd], [y]), dtype=torch.uint8, device="cuda")
    tsl.column_parallel_linear(xd, wd, bd, out=y, workspace=ws)  # loads the kernels, plans, encodes descriptors
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            tsl.column_parallel_linear(xd, wd, bd, out=y, workspace=ws)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert tsl.read_device_status() == 0
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"shard {i}")


CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_gpu_split_tail as T
T.test_column_split(None)
T.test_row_split(None, T.tsl.ALL_REDUCE)
for shape in T.MLP_SPLIT_SHAPES:
    T.test_mlp_split(None, *shape)
T.test_mlp_down_split(None)
print("OK")
"""


def test_unsplit_schedule_agrees(lib):
    """The same shapes with every tile whole (DT_GEMM_SPLIT=0)."""
    env = dict(os.environ, DT_GEMM_SPLIT="0")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "OK" in r.stdout
