"""Full-size workloads, in the launch configuration the benchmark times
(the library's default workspaces, so the down projection splits its last
wave), against the fp64 oracle.

The sampled variants check rows that the oracle computes one by one; the
full variants compare every element.  The MLP and the attention are two
linears with a bf16 intermediate (H; q) between them.  Where the kernel's
fp32 value of an intermediate and the oracle's fp64 value fall on opposite
sides of a bf16 rounding point, the two roundings differ by one ulp, which
then moves a whole row of the second linear's output by up to ulp * |w|.
So every element is checked stage by stage: the intermediate against the
oracle's own bf16 rounding (check_bf16_pair), the second linear against the
oracle applied to the kernel's intermediate (the linear tolerance,
check_fp32), and the end-to-end output against the oracle in relative
Frobenius norm (plus the max-abs bound on the sampled rows)."""
import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import bf16
from oracle import linear as olin
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import to_host
from test_gpu_linear import REL_FRO_TOL, check_bf16_pair, check_fp32, col_dtensor, row_dtensor, w64, x_rep

pytestmark = pytest.mark.gpu


def sample_rows(m, k=40, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(m, size=k, replace=False).tolist()) | {0, 127, 128, m - 1}
    return np.array(sorted(rows))


def rel_fro(got, expect):
    return float(np.linalg.norm(got.astype(np.float64) - expect) / np.linalg.norm(expect))


def run_mlp():
    cfg = workloads.MLP
    p = cfg["parts"]
    x, wg, wu, wd = workloads.mlp_inputs()
    xd = x_rep(x, p)
    wgd, wud, wdd = col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    y32 = tsl.tp_mlp_output(xd, wdd, mode=tsl.ALL_REDUCE, out_dtype=torch.float32)
    ws = torch.empty(tsl.tp_mlp_workspace_bytes(xd, wgd, wud, wdd, y32), dtype=torch.uint8, device="cuda")
    tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, out=y32, workspace=ws)
    h = to_host(tsl.api.mlp_hidden_view(xd, wgd, ws), "bf16")
    y16 = tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, workspace=ws)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    f = to_host(y32.slots[0], "fp32")
    assert np.isfinite(f).all()
    np.testing.assert_array_equal(to_host(y16.slots[0], "bf16"), bf16.round_rne(f))
    return cfg, p, (x, wg, wu, wd), h, f


def test_mlp_full_size(lib):
    """X [4096, 4096]; gate/up [4096, 11008] Shard(1) over 8; down [11008, 4096] Shard(0); ALL_REDUCE.
    Sampled rows end to end."""
    cfg, p, (x, wg, wu, wd), _, f = run_mlp()
    rows = sample_rows(cfg["tokens"])
    cols = chunk_bounds(cfg["ffn"], p)
    (expect,), _ = olin.tp_mlp(w64(x[rows]), [w64(wg[:, o:o + s]) for o, s in cols],
                               [w64(wu[:, o:o + s]) for o, s in cols], [w64(wd[o:o + s]) for o, s in cols])
    check_fp32(f[rows], expect, "mlp sampled rows")


def test_mlp_full_size_every_element(lib):
    """The same launch, every element: H, the down projection on the kernel's H, and Y end to end."""
    cfg, p, (x, wg, wu, wd), h, f = run_mlp()
    cols = chunk_bounds(cfg["ffn"], p)
    wds = [w64(wd[o:o + s]) for o, s in cols]
    (expect,), hs = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols],
                                [w64(wu[:, o:o + s]) for o, s in cols], wds)
    check_bf16_pair(h, np.concatenate(hs, axis=-1), "H, every element")
    (down,) = olin.row_parallel([w64(h[:, o:o + s]) for o, s in cols], wds, None, olin.ALL_REDUCE)
    check_fp32(f, down, "down projection on the kernel's H, every element")
    assert rel_fro(f, expect) <= REL_FRO_TOL, "end to end"


def run_attention():
    cfg = workloads.ATTENTION
    p = cfg["parts"]
    x, wq, wk, wv, wo = workloads.attention_inputs()
    xd = x_rep(x, p)
    o, q, k, v = tsl.tp_attention_projections(xd, col_dtensor(wq, p), col_dtensor(wk, p), col_dtensor(wv, p),
                                              row_dtensor(wo, p), mode=tsl.REDUCE_SCATTER, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    blocks = chunk_bounds(cfg["tokens"], p)
    assert [t.shape[0] for t in o.slots] == [s for _, s in blocks]
    got_o = np.concatenate([to_host(t, "fp32") for t in o.slots], axis=0)
    assert got_o.shape == (cfg["tokens"], cfg["hidden"])
    qkv = [np.concatenate([to_host(t, "bf16") for t in d.slots], axis=-1) for d in (q, k, v)]
    return cfg, p, (x, wq, wk, wv, wo), got_o, qkv


def test_attention_full_size(lib):
    """X [8192, 4096]; q/k/v/o [4096, 4096] over 4; o REDUCE_SCATTER to 4 x [2048, 4096].  Sampled rows."""
    cfg, p, (x, wq, wk, wv, wo), got_o, qkv = run_attention()
    rows = sample_rows(cfg["tokens"], seed=1)
    cols = chunk_bounds(cfg["hidden"], p)
    eo, eq, ek, ev = olin.attention_projections(w64(x[rows]), *[[w64(w[:, a:a + s]) for a, s in cols]
                                                                for w in (wq, wk, wv)],
                                                [w64(wo[a:a + s]) for a, s in cols], olin.ALL_REDUCE)
    check_fp32(got_o[rows], eo[0], "o sampled rows")
    for name, g, ref in zip("qkv", qkv, (eq, ek, ev)):
        check_bf16_pair(g[rows], np.concatenate(ref, axis=-1), f"{name} sampled rows")


def test_attention_full_size_every_element(lib):
    """The same launches, every element: q/k/v, o on the kernel's q, and o end to end."""
    cfg, p, (x, wq, wk, wv, wo), got_o, qkv = run_attention()
    cols = chunk_bounds(cfg["hidden"], p)
    wos = [w64(wo[a:a + s]) for a, s in cols]
    eo, eq, ek, ev = olin.attention_projections(w64(x), *[[w64(w[:, a:a + s]) for a, s in cols]
                                                          for w in (wq, wk, wv)], wos, olin.ALL_REDUCE)
    for name, g, ref in zip("qkv", qkv, (eq, ek, ev)):
        check_bf16_pair(g, np.concatenate(ref, axis=-1), f"{name}, every element")
    q = qkv[0]
    (on_q,) = olin.row_parallel([w64(q[:, a:a + s]) for a, s in cols], wos, None, olin.ALL_REDUCE)
    check_fp32(got_o, on_q, "o on the kernel's q, every element")
    assert rel_fro(got_o, eo[0]) <= REL_FRO_TOL, "o end to end"
