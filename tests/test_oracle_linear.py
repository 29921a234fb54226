"""Pins for the oracle's linears (CPU only).

Pinned by: the wineandchord worked example (x[3, 8] @ W[8, 12], 4 parts,
seed 0: column and row parallel both equal the dense product, output shape
(3, 12)), with the dense product computed by brute-force scalar loops;
closed forms of SiLU; ``scipy.special.expit`` as a library routine for the
sigmoid; and identities between the modes (Partial parts sum to the
ALL_REDUCE result, REDUCE_SCATTER blocks concatenate to it, the row bias
appears once).
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import expit

from oracle import bf16
from oracle import linear as ol
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads


def brute_matmul(a, b):
    n, k = a.shape
    k2, m = b.shape
    assert k == k2
    out = np.zeros((n, m))
    for i in range(n):
        for j in range(m):
            s = 0.0
            for t in range(k):
                s += float(a[i, t]) * float(b[t, j])
            out[i, j] = s
    return out


def col_shards(w, p):
    return [w[:, o:o + s] for o, s in chunk_bounds(w.shape[1], p)]


def row_shards(w, p):
    return [w[o:o + s] for o, s in chunk_bounds(w.shape[0], p)]


def x_shards(x, p):
    return [x[:, o:o + s] for o, s in chunk_bounds(x.shape[1], p)]


def check_worked_example(linear=ol):
    x, w = workloads.worked_example()
    x64, w64 = x.astype(np.float64), w.astype(np.float64)
    dense = brute_matmul(x64, w64)
    col = np.concatenate(linear.column_parallel(x64, col_shards(w64, 4)), axis=-1)
    row = linear.row_parallel(x_shards(x64, 4), row_shards(w64, 4), mode=linear.ALL_REDUCE)[0]
    assert col.shape == (3, 12) and row.shape == (3, 12)
    np.testing.assert_allclose(col, dense, rtol=0, atol=1e-12)
    np.testing.assert_allclose(row, dense, rtol=0, atol=1e-12)
    return x, w, col, row


def test_worked_example_equals_dense():
    check_worked_example()


def test_worked_example_fp32_assert_close():
    """The page compares fp32 torch results with assert_close defaults."""
    x, w, col, row = check_worked_example()
    dense32 = torch.from_numpy(x) @ torch.from_numpy(w)
    torch.testing.assert_close(torch.from_numpy(col.astype(np.float32)), dense32)
    torch.testing.assert_close(torch.from_numpy(row.astype(np.float32)), dense32)


def test_worked_example_inputs_are_the_seed0_stream():
    torch.manual_seed(0)
    x_ref, w_ref = torch.randn(3, 8), torch.randn(8, 12)
    x, w = workloads.worked_example()
    np.testing.assert_array_equal(x, x_ref.numpy())
    np.testing.assert_array_equal(w, w_ref.numpy())


@pytest.mark.parametrize("p", [1, 2, 3, 4, 5, 7])
def test_uneven_shards_equal_dense(p):
    rng = np.random.default_rng(p)
    x = rng.standard_normal((5, 11))
    w = rng.standard_normal((11, 13))
    dense = brute_matmul(x, w)
    col = np.concatenate(ol.column_parallel(x, col_shards(w, p)), axis=-1)
    row = ol.row_parallel(x_shards(x, p), row_shards(w, p), mode=ol.ALL_REDUCE)[0]
    np.testing.assert_allclose(col, dense, atol=1e-12, rtol=0)
    np.testing.assert_allclose(row, dense, atol=1e-12, rtol=0)


def test_modes_and_bias_once():
    rng = np.random.default_rng(4)
    p = 4
    x = rng.standard_normal((10, 12))
    w = rng.standard_normal((12, 6))
    b = rng.standard_normal(6)
    xs, ws = x_shards(x, p), row_shards(w, p)
    full = ol.row_parallel(xs, ws, b, ol.ALL_REDUCE)[0]
    np.testing.assert_allclose(full, brute_matmul(x, w) + b, atol=1e-12, rtol=0)
    parts = ol.row_parallel(xs, ws, b, ol.PARTIAL)
    np.testing.assert_allclose(sum(parts), full, atol=1e-12, rtol=0)
    blocks = ol.row_parallel(xs, ws, b, ol.REDUCE_SCATTER)
    assert [blk.shape[0] for blk in blocks] == [3, 3, 3, 1]
    np.testing.assert_array_equal(np.concatenate(blocks, axis=0), full)
    # column bias goes with its shard
    bs = [b[o:o + s] for o, s in chunk_bounds(6, 3)]
    cols = ol.column_parallel(x, col_shards(brute_matmul(np.eye(12), w), 3), bs)
    np.testing.assert_allclose(np.concatenate(cols, -1), brute_matmul(x, w) + b, atol=1e-12, rtol=0)


def test_silu_closed_forms():
    g = np.linspace(-30, 30, 601)
    s = ol.silu(g)
    assert ol.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(s - ol.silu(-g), g, atol=1e-12, rtol=0)    # x*sig(x) + x*sig(-x)... = x
    np.testing.assert_allclose(s, g * expit(g), atol=1e-14, rtol=1e-14)
    assert abs(ol.silu(np.array([50.0]))[0] - 50.0) < 1e-15 * 50
    assert abs(ol.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16


def test_mlp_hidden_brute_force():
    rng = np.random.default_rng(6)
    x = bf16.widen64(bf16.round_rne(rng.standard_normal((4, 16))))
    wg = bf16.widen64(bf16.round_rne(rng.standard_normal((16, 10)) / 4))
    wu = bf16.widen64(bf16.round_rne(rng.standard_normal((16, 10)) / 4))
    wd = bf16.widen64(bf16.round_rne(rng.standard_normal((10, 16)) / 4))
    p = 2
    (y,), hs = ol.tp_mlp(x, col_shards(wg, p), col_shards(wu, p), row_shards(wd, p), ol.ALL_REDUCE)
    g = brute_matmul(x, wg)
    u = brute_matmul(x, wu)
    h = np.empty_like(g)
    for i in range(h.shape[0]):
        for j in range(h.shape[1]):
            h[i, j] = g[i, j] / (1.0 + math.exp(-g[i, j])) * u[i, j]
    hb = bf16.round_rne(h)
    np.testing.assert_array_equal(np.concatenate(hs, -1), hb)
    np.testing.assert_allclose(y, brute_matmul(bf16.widen64(hb), wd), atol=1e-12, rtol=0)


def test_attention_projections_reduce_scatter():
    rng = np.random.default_rng(8)
    p = 4
    x = bf16.widen64(bf16.round_rne(rng.standard_normal((12, 16))))
    ws = [bf16.widen64(bf16.round_rne(rng.standard_normal((16, 16)) / 4)) for _ in range(4)]
    o, q, k, v = ol.attention_projections(x, *[col_shards(w, p) for w in ws[:3]], row_shards(ws[3], p))
    qf = bf16.round_rne(brute_matmul(x, ws[0]))
    np.testing.assert_array_equal(np.concatenate(q, -1), qf)
    np.testing.assert_array_equal(np.concatenate(v, -1), bf16.round_rne(brute_matmul(x, ws[2])))
    dense_o = brute_matmul(bf16.widen64(qf), ws[3])
    assert [blk.shape[0] for blk in o] == [3, 3, 3, 3]
    np.testing.assert_allclose(np.concatenate(o, 0), dense_o, atol=1e-12, rtol=0)


@pytest.mark.parametrize("bad", ["drop_last", "transpose", "sign"])
def test_planted_linear_mistakes_are_caught(monkeypatch, bad):
    if bad == "drop_last":
        monkeypatch.setattr(ol, "row_sum", lambda xs, ws: sum(np.matmul(a, b) for a, b in zip(xs[:-1], ws[:-1])))
    elif bad == "transpose":
        orig = ol.column_parallel
        monkeypatch.setattr(ol, "column_parallel",
                            lambda x, ws, b=None: orig(x, [w[::-1] for w in ws], b))
    else:
        monkeypatch.setattr(ol, "row_sum", lambda xs, ws: -sum(np.matmul(a, b) for a, b in zip(xs, ws)))
    with pytest.raises(AssertionError):
        check_worked_example()


def test_sequence_parallel_entry_and_replicate_output():
    """The gathered-token column entry equals the column linear on the full
    input, and the Replicate output equals the dense product (brute force)."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((11, 6))
    w = rng.standard_normal((6, 10))
    p = 4
    xs = [x[o:o + s] for o, s in chunk_bounds(11, p)]
    seq = ol.column_parallel_seq(xs, col_shards(w, p))
    dense = brute_matmul(x, w)
    np.testing.assert_allclose(np.concatenate(seq, -1), dense, atol=1e-12, rtol=0)
    assert all(y.shape[0] == 11 for y in seq)
    np.testing.assert_allclose(ol.column_parallel_replicate(x, col_shards(w, p)), dense, atol=1e-12, rtol=0)


def test_mlp_modes_agree():
    """The MLP's PARTIAL parts sum to its ALL_REDUCE output, and its
    REDUCE_SCATTER row blocks (torch.chunk of the tokens) tile it; that
    output is the brute-force product of the bf16 H and the down weight."""
    rng = np.random.default_rng(14)
    p = 3
    x = bf16.widen64(bf16.round_rne(rng.standard_normal((7, 12))))
    wg = bf16.widen64(bf16.round_rne(rng.standard_normal((12, 9)) / 4))
    wu = bf16.widen64(bf16.round_rne(rng.standard_normal((12, 9)) / 4))
    wd = bf16.widen64(bf16.round_rne(rng.standard_normal((9, 5)) / 4))
    args = (x, col_shards(wg, p), col_shards(wu, p), row_shards(wd, p))
    (full,), hs = ol.tp_mlp(*args, ol.ALL_REDUCE)
    np.testing.assert_allclose(full, brute_matmul(bf16.widen64(np.concatenate(hs, -1)), wd), atol=1e-12, rtol=0)
    parts, _ = ol.tp_mlp(*args, ol.PARTIAL)
    assert len(parts) == p
    np.testing.assert_allclose(sum(parts), full, atol=1e-12, rtol=0)
    for i, (o, s) in enumerate(chunk_bounds(9, p)):  # part i is H_i times its rows of the down weight
        np.testing.assert_allclose(parts[i], brute_matmul(bf16.widen64(hs[i]), wd[o:o + s]), atol=1e-12, rtol=0)
    blocks, _ = ol.tp_mlp(*args, ol.REDUCE_SCATTER)
    assert [b.shape[0] for b in blocks] == [3, 3, 1]
    np.testing.assert_array_equal(np.concatenate(blocks, 0), full)


def test_degenerate_sizes():
    """Closed forms of the empty cases: with K = 0 the product is the zero
    matrix, so a row layer's output is its bias (PARTIAL: on part 0 only) and
    a column layer's is its bias shards; an MLP with no ffn columns gives 0;
    no tokens give empty outputs of the right widths."""
    rng = np.random.default_rng(16)
    M, N, p = 5, 7, 3
    b = rng.standard_normal(N)
    xs = [np.zeros((M, 0)) for _ in range(p)]
    ws = [np.zeros((0, N)) for _ in range(p)]
    (y,) = ol.row_parallel(xs, ws, b, ol.ALL_REDUCE)
    np.testing.assert_array_equal(y, np.broadcast_to(b, (M, N)))
    parts = ol.row_parallel(xs, ws, b, ol.PARTIAL)
    np.testing.assert_array_equal(parts[0], np.broadcast_to(b, (M, N)))
    assert all(not q.any() for q in parts[1:])
    blocks = ol.row_parallel(xs, ws, b, ol.REDUCE_SCATTER, parts=p)
    assert [blk.shape for blk in blocks] == [(2, N), (2, N), (1, N)]
    np.testing.assert_array_equal(np.concatenate(blocks, 0), np.broadcast_to(b, (M, N)))
    bs = [b[o:o + s] for o, s in chunk_bounds(N, p)]
    cols = ol.column_parallel(np.zeros((M, 0)), [np.zeros((0, s)) for _, s in chunk_bounds(N, p)], bs)
    np.testing.assert_array_equal(np.concatenate(cols, -1), np.broadcast_to(b, (M, N)))
    x = rng.standard_normal((M, 4))
    (ym,), hs = ol.tp_mlp(x, [np.zeros((4, 0))] * p, [np.zeros((4, 0))] * p, [np.zeros((0, N))] * p, ol.ALL_REDUCE)
    assert ym.shape == (M, N) and not ym.any() and all(h.size == 0 for h in hs)
    cols = ol.column_parallel(np.zeros((0, 4)), col_shards(rng.standard_normal((4, N)), p))
    assert [c.shape for c in cols] == [(0, s) for _, s in chunk_bounds(N, p)]
