"""Full-size workloads, in the launch configuration the benchmark times,
checked on sampled output rows that the fp64 oracle computes one by one, and
on properties that hold at any size (finite outputs; the bf16 output is the
round-to-nearest-even of the fp32 output everywhere)."""
import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import bf16
from oracle import linear as olin
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import to_dev, to_host
from test_gpu_linear import check_bf16_pair, check_fp32, col_dtensor, mesh1, row_dtensor, w64, x_rep

pytestmark = pytest.mark.gpu


def sample_rows(m, k=40, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(m, size=k, replace=False).tolist()) | {0, 127, 128, m - 1}
    return np.array(sorted(rows))


def test_mlp_full_size(lib):
    """X [4096, 4096]; gate/up [4096, 11008] Shard(1) over 8; down [11008, 4096] Shard(0); ALL_REDUCE."""
    cfg = workloads.MLP
    p = cfg["parts"]
    x, wg, wu, wd = workloads.mlp_inputs()
    xd = x_rep(x, p)
    wgd, wud, wdd = col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    ws = torch.empty(tsl.tp_mlp_workspace_bytes(xd, wgd), dtype=torch.uint8, device="cuda")
    y32 = tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, out_dtype=torch.float32, workspace=ws)
    y16 = tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, workspace=ws)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    f = to_host(y32.slots[0], "fp32")
    assert np.isfinite(f).all()
    np.testing.assert_array_equal(to_host(y16.slots[0], "bf16"), bf16.round_rne(f))
    rows = sample_rows(cfg["tokens"])
    cols = chunk_bounds(cfg["ffn"], p)
    (expect,), _ = olin.tp_mlp(w64(x[rows]), [w64(wg[:, o:o + s]) for o, s in cols],
                               [w64(wu[:, o:o + s]) for o, s in cols], [w64(wd[o:o + s]) for o, s in cols])
    check_fp32(f[rows], expect, "mlp sampled rows")


def test_attention_full_size(lib):
    """X [8192, 4096]; q/k/v/o [4096, 4096] over 4; o REDUCE_SCATTER to 4 x [2048, 4096]."""
    cfg = workloads.ATTENTION
    p = cfg["parts"]
    x, wq, wk, wv, wo = workloads.attention_inputs()
    xd = x_rep(x, p)
    o, q, k, v = tsl.tp_attention_projections(xd, col_dtensor(wq, p), col_dtensor(wk, p), col_dtensor(wv, p),
                                              row_dtensor(wo, p), mode=tsl.REDUCE_SCATTER, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    rows = sample_rows(cfg["tokens"], seed=1)
    H = cfg["hidden"]
    cols = chunk_bounds(H, p)
    eo, eq, ek, ev = olin.attention_projections(w64(x[rows]), *[[w64(w[:, a:a + s]) for a, s in cols]
                                                                for w in (wq, wk, wv)],
                                                [w64(wo[a:a + s]) for a, s in cols], olin.ALL_REDUCE)
    blocks = chunk_bounds(cfg["tokens"], p)
    got = np.concatenate([to_host(t, "fp32") for t in o.slots], axis=0)
    assert got.shape == (cfg["tokens"], H) and [t.shape[0] for t in o.slots] == [s for _, s in blocks]
    check_fp32(got[rows], eo[0], "o sampled rows")
    for name, got_t, ref in (("q", q, eq), ("k", k, ek), ("v", v, ev)):
        g = np.concatenate([to_host(t, "bf16") for t in got_t.slots], axis=-1)[rows]
        check_bf16_pair(g, np.concatenate(ref, axis=-1), f"{name} sampled rows")
