"""GPU parity of the layers and moves built beside the hot path:

* the sequence-parallel column entry (nanotron 5.1's REDUCE_SCATTER-mode
  column layer: x sharded over tokens, all-gathered, then the column GEMM) --
  the token shards are read in place by the GEMM;
* ColumnParallelLinearWithReplicateOutput / ...InputOutput (DTorch guide,
  section 3) -- each shard's GEMM writes its column block of the Replicate
  output;
* the Ulysses layout move, Shard(2) -> Shard(1) of [N, H, L, E] (DTorch
  guide, section 2, context parallel) -- a 4-D redistribute, bit-exact.
"""
import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import bf16
from oracle import linear as olin
from oracle import placement as opl
from oracle import redistribute as ord_
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import dtensor_from_locals, lib_placements, locals_of, to_dev, to_host
from test_gpu_linear import check_bf16_pair, check_fp32, col_dtensor, mesh1, w64

pytestmark = pytest.mark.gpu


def x_tokens(x_bits, p):
    """[T, K] bf16, Shard(0) over p (token shards)."""
    slots = [to_dev(np.ascontiguousarray(x_bits[o:o + s]), "bf16") for o, s in chunk_bounds(x_bits.shape[0], p)]
    return tsl.DTensor(slots, mesh1(p), [tsl.Shard(0)], x_bits.shape, torch.bfloat16)


@pytest.mark.parametrize("T,K,N,p", [
    (384, 256, 1056, 4), (301, 200, 8 * 136, 8), (1024, 512, 512, 4),
    (1300, 256, 520, 4),  # two M tiles per token shard, the second ragged: row blocks
    (1030, 256, 520, 4),  # shards of 258, 258, 258, 256 rows: 2, 2, 2, 1 M tiles, no row blocks
])
def test_sequence_parallel_column_entry(lib, T, K, N, p):
    x = workloads.randn_bf16((T, K), 91)
    w = workloads.randn_bf16((K, N), 92, (1.0 / K) ** 0.5)
    y = tsl.column_parallel_linear(x_tokens(x, p), col_dtensor(w, p), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    assert y.placements == (tsl.Shard(1),) and y.gshape == (T, N)
    xs = [w64(x[o:o + s]) for o, s in chunk_bounds(T, p)]
    expect = olin.column_parallel_seq(xs, [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
    for i in range(p):
        got = to_host(y.slots[i], "fp32")
        assert got.shape[0] == T
        check_fp32(got, expect[i], f"shard {i}")


@pytest.mark.parametrize("seq_input", [False, True])
def test_column_replicate_output(lib, seq_input):
    T, K, N, p = 300, 256, 1056, 4
    x = workloads.randn_bf16((T, K), 93)
    w = workloads.randn_bf16((K, N), 94, (1.0 / K) ** 0.5)
    b = workloads.randn_bf16((N,), 95, 0.5)
    xd = x_tokens(x, p) if seq_input else tsl.DTensor([to_dev(x, "bf16")], mesh1(p), [tsl.Replicate()], x.shape,
                                                       torch.bfloat16)
    bd = tsl.DTensor([to_dev(np.ascontiguousarray(b[o:o + s]), "bf16") for o, s in chunk_bounds(N, p)], mesh1(p),
                     [tsl.Shard(0)], (N,), torch.bfloat16)
    y = tsl.column_parallel_linear(xd, col_dtensor(w, p), bd, out_dtype=torch.float32, output="replicate")
    torch.cuda.synchronize()
    assert y.placements == (tsl.Replicate(),) and len(y.slots) == 1
    expect = olin.column_parallel_replicate(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)],
                                            [w64(b[o:o + s]) for o, s in chunk_bounds(N, p)])
    check_fp32(to_host(y.slots[0], "fp32"), expect, "replicate output")


def test_replicate_input_output_layer_takes_token_shards_in_place(lib):
    T, K, N, p = 256, 128, 512, 4
    x = workloads.randn_bf16((T, K), 96)
    w = workloads.randn_bf16((K, N), 97, (1.0 / K) ** 0.5)
    mesh = mesh1(p)
    layer = tsl.ColumnParallelLinearWithReplicateInputOutput(to_dev(w, "bf16"), None, mesh)
    launches = tsl._lib.load().dt_launch_count()
    y = layer(x_tokens(x, p))
    torch.cuda.synchronize()
    # one GEMM launch: no separate gather of x and no separate gather of y
    assert tsl._lib.load().dt_launch_count() - launches == 1
    expect = olin.column_parallel_replicate(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
    g = bf16.widen64(to_host(y.slots[0], "bf16"))
    assert (np.abs(g - expect) <= 2e-3 + 2.0 ** -8 * np.abs(expect)).all()


def test_sequence_parallel_qkv_full_size(lib):
    """Attention projections entered sequence-parallel: X [8192, 4096] Shard(0)
    over 4, q/k/v in one launch; sampled rows against the oracle."""
    cfg = workloads.ATTENTION
    p = cfg["parts"]
    x, wq, wk, wv, _ = workloads.attention_inputs()
    xd = x_tokens(x, p)
    q, k, v = tsl.column_parallel_linear_multi(xd, [col_dtensor(w, p) for w in (wq, wk, wv)])
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    rows = np.array(sorted({0, 2047, 2048, 5000, 8191} | set(np.random.default_rng(3).choice(8192, 24).tolist())))
    H = cfg["hidden"]
    cols = chunk_bounds(H, p)
    for name, got, w in (("q", q, wq), ("k", k, wk), ("v", v, wv)):
        ref = olin.column_parallel(w64(x[rows]), [w64(w[:, a:a + s]) for a, s in cols])
        g = np.concatenate([to_host(t, "bf16") for t in got.slots], axis=-1)[rows]
        check_bf16_pair(g, bf16.round_rne(np.concatenate(ref, axis=-1)), f"{name} sampled rows")


@pytest.mark.parametrize("shape,p", [((2, 32, 512, 128), 4), ((1, 6, 37, 5), 3), ((2, 8, 4096, 128), 4)])
def test_ulysses_move(lib, shape, p):
    """Sequence-sharded Q/K/V (Shard(2) on a cp mesh dim) to head-sharded
    (Shard(1)): the all-to-all of Ulysses context parallelism."""
    g = workloads.randn_bf16(shape, 98)
    src = opl.Layout((p,), [opl.Shard(2)], shape)
    dst = opl.Layout((p,), [opl.Shard(1)], shape)
    locals_ = ord_.distribute(g, src, "bf16")
    d = dtensor_from_locals(locals_, src, "bf16")
    out = d.redistribute(lib_placements(dst.placements))
    torch.cuda.synchronize()
    for s, (got, exp) in enumerate(zip(locals_of(out, "bf16"), ord_.redistribute(locals_, src, dst, "bf16"))):
        np.testing.assert_array_equal(got, exp, err_msg=f"slot {s}")
    back = out.redistribute([tsl.Shard(2)])
    for got, exp in zip(locals_of(back, "bf16"), locals_):
        np.testing.assert_array_equal(got, exp)
