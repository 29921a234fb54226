"""GPU parity of the tensor-parallel linears against the fp64 oracle.

Tolerance (bf16 inputs, fp32 accumulation, unit-scale outputs), on the
fp32-output variant of every kernel: max |y - y_oracle| <= 2e-3 and
||y - y_oracle||_F / ||y_oracle||_F <= 1e-3.  The bf16-output variant of the
same launch is checked two ways: it equals the round-to-nearest-even bf16 of
the fp32 output bit for bit (one cast in the epilogue), and
|y_bf16 - y_oracle| <= 2e-3 + 2^-8 |y_oracle| (half a bf16 ulp on top).
"""
import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import bf16
from oracle import linear as olin
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import to_dev, to_host

pytestmark = pytest.mark.gpu

ABS_TOL = 2e-3
REL_FRO_TOL = 1e-3
ROW_MODES = [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER, tsl.PARTIAL]
OMODE = {tsl.ALL_REDUCE: olin.ALL_REDUCE, tsl.REDUCE_SCATTER: olin.REDUCE_SCATTER, tsl.PARTIAL: olin.PARTIAL}


def check_fp32(got: np.ndarray, expect: np.ndarray, what=""):
    got = got.astype(np.float64)
    err = np.abs(got - expect)
    assert np.isfinite(got).all(), what
    mx = float(err.max()) if err.size else 0.0
    fro = float(np.linalg.norm(got - expect) / max(np.linalg.norm(expect), 1e-30)) if err.size else 0.0
    assert mx <= ABS_TOL, f"{what}: max abs err {mx}"
    assert fro <= REL_FRO_TOL, f"{what}: rel Frobenius err {fro}"


def check_bf16_pair(got_bits: np.ndarray, ref_bits: np.ndarray, what=""):
    """A bf16 intermediate against the oracle's own bf16 rounding of the exact
    value: both are within half a bf16 ulp of values that agree to the fp32
    tolerance, so |g - r| <= 2e-3 + 2^-7 |r|."""
    g = bf16.widen64(got_bits)
    r = bf16.widen64(ref_bits)
    bad = np.abs(g - r) > ABS_TOL + 2.0 ** -7 * np.abs(r)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements, worst |g-r| = {float(np.abs(g - r).max())}"


def check_bf16(got_bits: np.ndarray, fp32_out: np.ndarray, expect: np.ndarray, what=""):
    np.testing.assert_array_equal(got_bits, bf16.round_rne(fp32_out), err_msg=f"{what}: bf16 != RNE(fp32)")
    g = bf16.widen64(got_bits)
    assert (np.abs(g - expect) <= ABS_TOL + 2.0 ** -8 * np.abs(expect)).all(), what


def mesh1(p):
    return tsl.DeviceMesh((p,), ("tp",))


def kmajor(a, dtype="bf16"):
    """[K, N] as a transposed view of [N, K] storage (the [out, in] layout)."""
    return to_dev(np.ascontiguousarray(a.T), dtype).t()


def col_dtensor(w_bits, p, dtype="bf16", views=False, k_major=False):
    """[K, N] weight, Shard(1) over p: separate slots, or column views of one parent."""
    K, N = w_bits.shape
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    if k_major:
        slots = [kmajor(w_bits[:, o:o + s], dtype) for o, s in chunk_bounds(N, p)]
    elif views:
        parent = to_dev(w_bits, dtype)
        slots = [parent[:, o:o + s] for o, s in chunk_bounds(N, p)]
    else:
        slots = [to_dev(np.ascontiguousarray(w_bits[:, o:o + s]), dtype) for o, s in chunk_bounds(N, p)]
    return tsl.DTensor(slots, mesh1(p), [tsl.Shard(1)], (K, N), td)


def row_dtensor(w_bits, p, dtype="bf16", k_major=False):
    K, N = w_bits.shape
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    if k_major:
        slots = [kmajor(w_bits[o:o + s], dtype) for o, s in chunk_bounds(K, p)]
    else:
        slots = [to_dev(np.ascontiguousarray(w_bits[o:o + s]), dtype) for o, s in chunk_bounds(K, p)]
    return tsl.DTensor(slots, mesh1(p), [tsl.Shard(0)], (K, N), td)


def x_rep(x_bits, p, dtype="bf16"):
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    return tsl.DTensor([to_dev(x_bits, dtype)], mesh1(p), [tsl.Replicate()], x_bits.shape, td)


def x_shard(x_bits, p, dtype="bf16"):
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    K = x_bits.shape[-1]
    slots = [to_dev(np.ascontiguousarray(x_bits[..., o:o + s]), dtype) for o, s in chunk_bounds(K, p)]
    return tsl.DTensor(slots, mesh1(p), [tsl.Shard(x_bits.ndim - 1)], x_bits.shape, td)


def w64(bits):
    return bf16.widen64(bits)


# ---------------------------------------------------------------- worked example

def test_worked_example_fp32(lib):
    """x[3, 8] @ W[8, 12], 4 parts, seed 0 ("Model parallelism", tensor-parallel
    linear layers): the column-parallel shards and the row-parallel sum against
    the pinned oracle (which equals dense x @ W), at the page's assert_close
    tolerance for fp32."""
    x, w = workloads.worked_example()
    p = 4
    cols, rows = chunk_bounds(12, p), chunk_bounds(8, p)
    x64, w64_ = x.astype(np.float64), w.astype(np.float64)
    y = tsl.column_parallel_linear(x_rep(x, p, "fp32"), col_dtensor(w, p, "fp32"))
    expect = olin.column_parallel(x64, [w64_[:, o:o + s] for o, s in cols])
    assert [t.shape for t in y.slots] == [(3, s) for _, s in cols]
    for t, e in zip(y.slots, expect):
        torch.testing.assert_close(torch.from_numpy(to_host(t, "fp32")), torch.from_numpy(e.astype(np.float32)))
    yr = tsl.row_parallel_linear(x_shard(x, p, "fp32"), row_dtensor(w, p, "fp32"), mode=tsl.ALL_REDUCE)
    (er,) = olin.row_parallel([x64[:, o:o + s] for o, s in rows], [w64_[o:o + s] for o, s in rows], None,
                              olin.ALL_REDUCE)
    assert yr.slots[0].shape == (3, 12)
    torch.testing.assert_close(torch.from_numpy(to_host(yr.slots[0], "fp32")), torch.from_numpy(er.astype(np.float32)))


# ---------------------------------------------------------------- column parallel

@pytest.mark.parametrize("M,K,N,p,views", [(300, 200, 1056, 4, False), (128, 64, 256, 1, False),
                                           (517, 328, 8 * 136, 8, True), (64, 1024, 4 * 264, 4, True)])
def test_column_parallel(lib, M, K, N, p, views):
    x = workloads.randn_bf16((M, K), 11)
    w = workloads.randn_bf16((K, N), 12, (1.0 / K) ** 0.5)
    b = workloads.randn_bf16((N,), 13, 0.5)
    xd = x_rep(x, p)
    wd = col_dtensor(w, p, views=views)
    bd = tsl.DTensor([to_dev(np.ascontiguousarray(b[o:o + s]), "bf16") for o, s in chunk_bounds(N, p)], mesh1(p),
                     [tsl.Shard(0)], (N,), torch.bfloat16)
    y32 = tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32)
    y16 = tsl.column_parallel_linear(xd, wd, bd)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)],
                                  [w64(b[o:o + s]) for o, s in chunk_bounds(N, p)])
    for i in range(p):
        f = to_host(y32.slots[i], "fp32")
        check_fp32(f, expect[i], f"shard {i}")
        check_bf16(to_host(y16.slots[i], "bf16"), f, expect[i], f"shard {i}")


def test_column_parallel_multi_qkv_small(lib):
    M, K, p = 384, 256, 4
    x = workloads.randn_bf16((M, K), 21)
    ws = [workloads.randn_bf16((K, K), 22 + j, (1.0 / K) ** 0.5) for j in range(3)]
    xd = x_rep(x, p)
    ys = tsl.column_parallel_linear_multi(xd, [col_dtensor(w, p) for w in ws], out_dtype=torch.float32)
    for j, w in enumerate(ws):
        expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(K, p)])
        for i in range(p):
            check_fp32(to_host(ys[j].slots[i], "fp32"), expect[i], f"w{j} shard {i}")


@pytest.mark.parametrize("k_major", [False, True])
def test_unaligned_shapes(lib, k_major):
    """Shard pitches TMA cannot describe (odd widths): without a workspace
    the launch runs on the CUDA-core kernel (counted), with the queried one
    the operands are copied to padded pitches and it runs on the tensor
    cores; both against the oracle."""
    M, K, N, p = 33, 50, 30, 4
    x = workloads.randn_bf16((M, K), 31 if not k_major else 81)
    w = workloads.randn_bf16((K, N), 32 if not k_major else 82, (1.0 / K) ** 0.5)
    xd, wd = x_rep(x, p), col_dtensor(w, p, k_major=k_major)
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
    for ws, cuda_cores in ((torch.empty(0, dtype=torch.uint8, device="cuda"), True), (None, False)):
        c0 = tsl.cuda_core_gemm_count()
        y = tsl.column_parallel_linear(xd, wd, out_dtype=torch.float32, workspace=ws)
        torch.cuda.synchronize()
        assert (tsl.cuda_core_gemm_count() > c0) == cuda_cores
        assert tsl.read_device_status() == 0
        for i in range(p):
            check_fp32(to_host(y.slots[i], "fp32"), expect[i], f"cuda_cores={cuda_cores} shard {i}")


# ---------------------------------------------------------------- row parallel

@pytest.mark.parametrize("mode", [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER, tsl.PARTIAL])
@pytest.mark.parametrize("M,K,N,p", [(300, 288, 320, 4), (256, 512, 512, 8), (130, 4 * 136, 200, 4)])
def test_row_parallel(lib, mode, M, K, N, p):
    x = workloads.randn_bf16((M, K), 41)
    w = workloads.randn_bf16((K, N), 42, (1.0 / K) ** 0.5)
    b = workloads.randn_bf16((N,), 43, 0.5)
    bd = tsl.DTensor([to_dev(b, "bf16")], mesh1(p), [tsl.Replicate()], (N,), torch.bfloat16)
    xd, wd = x_shard(x, p), row_dtensor(w, p)
    y32 = tsl.row_parallel_linear(xd, wd, bd, mode=mode, out_dtype=torch.float32)
    y16 = tsl.row_parallel_linear(xd, wd, bd, mode=mode)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    omode = OMODE[mode]
    expect = olin.row_parallel([w64(x[:, o:o + s]) for o, s in chunk_bounds(K, p)],
                               [w64(w[o:o + s]) for o, s in chunk_bounds(K, p)], w64(b), omode, parts=p)
    assert len(expect) == len(y32.slots)
    for i, e in enumerate(expect):
        f = to_host(y32.slots[i], "fp32")
        check_fp32(f, e, f"{mode} out {i}")
        check_bf16(to_host(y16.slots[i], "bf16"), f, e, f"{mode} out {i}")


def test_row_parallel_3d_reduce_scatter_on_batch(lib):
    """x [B, S, K] Shard(-1): REDUCE_SCATTER splits dim 0 (batch) into row blocks of S rows."""
    B, S_, K, N, p = 4, 96, 256, 192, 4
    x = workloads.randn_bf16((B, S_, K), 51)
    w = workloads.randn_bf16((K, N), 52, (1.0 / K) ** 0.5)
    y = tsl.row_parallel_linear(x_shard(x, p), row_dtensor(w, p), mode=tsl.REDUCE_SCATTER, out_dtype=torch.float32)
    dense = olin.row_sum([w64(x[..., o:o + s]) for o, s in chunk_bounds(K, p)],
                         [w64(w[o:o + s]) for o, s in chunk_bounds(K, p)])
    for i, (o, s) in enumerate(chunk_bounds(B, p)):
        check_fp32(to_host(y.slots[i], "fp32"), dense[o:o + s], f"block {i}")


# ---------------------------------------------------------------- MLP / attention

@pytest.mark.parametrize("M,K,F,N,p,mode", [(256, 256, 8 * 136, 384, 8, tsl.ALL_REDUCE),
                                            (200, 192, 4 * 96, 320, 4, tsl.REDUCE_SCATTER),
                                            (192, 256, 4 * 136, 264, 4, tsl.PARTIAL)])
def test_tp_mlp_small(lib, M, K, F, N, p, mode):
    x, wg, wu, wd = workloads.mlp_inputs(M, K, F, seed_base=600)
    wd = workloads.randn_bf16((F, N), 604, (1.0 / F) ** 0.5)
    xd = x_rep(x, p)
    wgd, wud, wdd = col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    y = tsl.tp_mlp_output(xd, wdd, mode=mode, out_dtype=torch.float32)
    ws = torch.empty(tsl.tp_mlp_workspace_bytes(xd, wgd, wud, wdd, y, mode=mode), dtype=torch.uint8, device="cuda")
    y = tsl.tp_mlp(xd, wgd, wud, wdd, mode=mode, out=y, workspace=ws)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    omode = OMODE[mode]
    cols = chunk_bounds(F, p)
    expect, hs = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols],
                             [w64(wd[o:o + s]) for o, s in cols], omode)
    # H: bf16 of SiLU(g) * u, allowed one bf16 ulp where fp32 and fp64 round apart
    check_bf16_pair(to_host(tsl.api.mlp_hidden_view(xd, col_dtensor(wg, p), ws), "bf16"),
                    np.concatenate(hs, axis=-1), "H")
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"mlp out {i}")


def test_attention_projections_small(lib):
    T, H, p = 512, 256, 4
    x, wq, wk, wv, wo = workloads.attention_inputs(T, H, seed_base=650)
    xd = x_rep(x, p)
    o, q, k, v = tsl.tp_attention_projections(xd, col_dtensor(wq, p), col_dtensor(wk, p), col_dtensor(wv, p),
                                              row_dtensor(wo, p), mode=tsl.REDUCE_SCATTER, out_dtype=torch.float32)
    cols = chunk_bounds(H, p)
    eo, eq, ek, ev = olin.attention_projections(w64(x), *[[w64(w[:, a:a + s]) for a, s in cols] for w in (wq, wk, wv)],
                                                [w64(wo[a:a + s]) for a, s in cols], olin.REDUCE_SCATTER)
    for i in range(p):
        for name, got, ref in (("q", q, eq), ("k", k, ek), ("v", v, ev)):
            check_bf16_pair(to_host(got.slots[i], "bf16"), ref[i], f"{name} shard {i}")
        check_fp32(to_host(o.slots[i], "fp32"), eo[i], f"o block {i}")


# ---------------------------------------------------------------- [out, in] weights (K-major B)

@pytest.mark.parametrize("M,K,N,p", [(300, 200, 1056, 4), (517, 328, 8 * 136, 8)])
def test_column_parallel_kmajor_weights(lib, M, K, N, p):
    x = workloads.randn_bf16((M, K), 61)
    w = workloads.randn_bf16((K, N), 62, (1.0 / K) ** 0.5)
    y = tsl.column_parallel_linear(x_rep(x, p), col_dtensor(w, p, k_major=True), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
    for i in range(p):
        check_fp32(to_host(y.slots[i], "fp32"), expect[i], f"shard {i}")


@pytest.mark.parametrize("mode", [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER])
def test_row_parallel_kmajor_weights(lib, mode):
    M, K, N, p = 300, 288, 320, 4
    x = workloads.randn_bf16((M, K), 71)
    w = workloads.randn_bf16((K, N), 72, (1.0 / K) ** 0.5)
    y = tsl.row_parallel_linear(x_shard(x, p), row_dtensor(w, p, k_major=True), mode=mode, out_dtype=torch.float32)
    omode = olin.ALL_REDUCE if mode == tsl.ALL_REDUCE else olin.REDUCE_SCATTER
    expect = olin.row_parallel([w64(x[:, o:o + s]) for o, s in chunk_bounds(K, p)],
                               [w64(w[o:o + s]) for o, s in chunk_bounds(K, p)], None, omode, parts=p)
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"{mode} out {i}")


def test_tp_mlp_kmajor_weights(lib):
    M, K, F, N, p = 256, 256, 8 * 136, 384, 8
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=680)
    wd = workloads.randn_bf16((F, N), 684, (1.0 / F) ** 0.5)
    xd = x_rep(x, p)
    y = tsl.tp_mlp(xd, col_dtensor(wg, p, k_major=True), col_dtensor(wu, p, k_major=True),
                   row_dtensor(wd, p, k_major=True), out_dtype=torch.float32)
    cols = chunk_bounds(F, p)
    (expect,), _ = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols],
                               [w64(wd[o:o + s]) for o, s in cols])
    check_fp32(to_host(y.slots[0], "fp32"), expect, "mlp")


# ---------------------------------------------------------------- uneven shards

def test_uneven_shards_run_on_tensor_cores_with_workspace(lib):
    """[512, 1024] x [1024, 8190] over 4: the last column shard is 2046 wide,
    a 4092-byte pitch TMA cannot read.  With the queried workspace the shard
    is copied to a padded pitch and the launch runs on the tensor cores; with
    none it runs on the CUDA-core kernel (counted).  Both match the oracle.
    The row-parallel layer on the same split (x shards [512, 2046]) likewise."""
    M, K, N, p = 512, 1024, 8190, 4
    x = workloads.randn_bf16((M, K), 961)
    w = workloads.randn_bf16((K, N), 962, (1.0 / K) ** 0.5)
    xd, wd = x_rep(x, p), col_dtensor(w, p)
    y = tsl.api._col_out(xd, wd, 0, torch.float32)
    need = tsl.column_parallel_linear_workspace_bytes(xd, [wd], [y])
    assert need >= 1024 * 2048 * 2  # at least the padded 2046-column shard
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in chunk_bounds(N, p)])
    c0 = tsl.cuda_core_gemm_count()
    tsl.column_parallel_linear(xd, wd, out=y, workspace=torch.empty(need, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert tsl.cuda_core_gemm_count() == c0
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"padded, shard {i}")
    tsl.column_parallel_linear(xd, wd, out=y, workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert tsl.cuda_core_gemm_count() > c0
    assert tsl.read_device_status() == 0
    for i, e in enumerate(expect):
        check_fp32(to_host(y.slots[i], "fp32"), e, f"CUDA-core, shard {i}")
    # row parallel: K = 8190 over 4, x shards [512, 2046]
    xr = workloads.randn_bf16((M, N), 963)
    wr = workloads.randn_bf16((N, 768), 964, (1.0 / N) ** 0.5)
    xrd, wrd = x_shard(xr, p), row_dtensor(wr, p)
    yr = tsl.api._row_out(xrd, wrd, 0, tsl.ALL_REDUCE, torch.float32)
    c1 = tsl.cuda_core_gemm_count()
    tsl.row_parallel_linear(xrd, wrd, out=yr)  # the Python API passes the queried workspace
    torch.cuda.synchronize()
    assert tsl.cuda_core_gemm_count() == c1
    assert tsl.read_device_status() == 0
    (er,) = olin.row_parallel([w64(xr[:, o:o + s]) for o, s in chunk_bounds(N, p)],
                              [w64(wr[o:o + s]) for o, s in chunk_bounds(N, p)], None, olin.ALL_REDUCE)
    check_fp32(to_host(yr.slots[0], "fp32"), er, "row, padded x shards")


# ---------------------------------------------------------------- degenerate sizes


def test_zero_tokens(lib):
    """x with no rows: every layer returns OK, launches nothing and gives empty outputs."""
    K, N, F, p = 256, 192, 4 * 96, 4
    x = workloads.randn_bf16((0, K), 61)
    w = workloads.randn_bf16((K, N), 62, (1.0 / K) ** 0.5)
    wg = workloads.randn_bf16((K, F), 63, (1.0 / K) ** 0.5)
    wu = workloads.randn_bf16((K, F), 64, (1.0 / K) ** 0.5)
    wd = workloads.randn_bf16((F, N), 65, (1.0 / F) ** 0.5)
    torch.cuda.synchronize()
    tsl.read_device_status(clear=True)
    n0 = lib.dt_launch_count()
    y = tsl.column_parallel_linear(x_rep(x, p), col_dtensor(w, p))
    assert [tuple(t.shape) for t in y.slots] == [(0, s) for _, s in chunk_bounds(N, p)]
    for mode in ROW_MODES:
        yr = tsl.row_parallel_linear(x_shard(x, p), row_dtensor(w, p), mode=mode, out_dtype=torch.float32)
        assert yr.slots and all(t.numel() == 0 for t in yr.slots)
    for mode in (tsl.ALL_REDUCE, tsl.REDUCE_SCATTER):
        xd = x_rep(x, p)
        ym = tsl.tp_mlp(xd, col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p), mode=mode)
        assert ym.slots and all(t.numel() == 0 for t in ym.slots)
    torch.cuda.synchronize()
    assert lib.dt_launch_count() == n0
    assert tsl.read_device_status() == 0


def test_zero_inner_dim_column(lib):
    """K = 0: X W is the zero matrix, so the column layer writes its bias."""
    M, N, p = 130, 200, 4
    x = workloads.randn_bf16((M, 0), 71)
    w = workloads.randn_bf16((0, N), 72)
    b = workloads.randn_bf16((N,), 73, 0.5)
    cols = chunk_bounds(N, p)
    bd = tsl.DTensor([to_dev(np.ascontiguousarray(b[o:o + s]), "bf16") for o, s in cols], mesh1(p), [tsl.Shard(0)],
                     (N,), torch.bfloat16)
    xd, wd = x_rep(x, p), col_dtensor(w, p)
    y32 = tsl.column_parallel_linear(xd, wd, bd, out_dtype=torch.float32)
    y16 = tsl.column_parallel_linear(xd, wd, bd)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    expect = olin.column_parallel(w64(x), [w64(w[:, o:o + s]) for o, s in cols], [w64(b[o:o + s]) for o, s in cols])
    for i, e in enumerate(expect):
        f = to_host(y32.slots[i], "fp32")
        np.testing.assert_array_equal(f, e, err_msg=f"shard {i}")  # the bias itself, exactly
        check_bf16(to_host(y16.slots[i], "bf16"), f, e, f"shard {i}")


@pytest.mark.parametrize("mode", ROW_MODES)
def test_zero_inner_dim_row(lib, mode):
    """K = 0 over p empty shards: the output is the bias, added once (PARTIAL: on part 0)."""
    M, N, p = 130, 200, 4
    x = workloads.randn_bf16((M, 0), 74)
    w = workloads.randn_bf16((0, N), 75)
    b = workloads.randn_bf16((N,), 76, 0.5)
    bd = tsl.DTensor([to_dev(b, "bf16")], mesh1(p), [tsl.Replicate()], (N,), torch.bfloat16)
    y = tsl.row_parallel_linear(x_shard(x, p), row_dtensor(w, p), bd, mode=mode, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    expect = olin.row_parallel([w64(x[:, o:o + s]) for o, s in chunk_bounds(0, p)],
                               [w64(w[o:o + s]) for o, s in chunk_bounds(0, p)], w64(b), OMODE[mode], parts=p)
    assert len(expect) == len(y.slots)
    for i, e in enumerate(expect):
        np.testing.assert_array_equal(to_host(y.slots[i], "fp32"), e, err_msg=f"{mode} out {i}")


@pytest.mark.parametrize("mode", [tsl.ALL_REDUCE, tsl.REDUCE_SCATTER])
def test_zero_ffn_width(lib, mode):
    """An MLP with no ffn columns: H is empty and Y = 0 (SiLU and the product never run)."""
    M, K, N, p = 130, 256, 200, 4
    x = workloads.randn_bf16((M, K), 77)
    wg, wu = workloads.randn_bf16((K, 0), 78), workloads.randn_bf16((K, 0), 79)
    wd = workloads.randn_bf16((0, N), 80)
    xd = x_rep(x, p)
    y = tsl.tp_mlp_output(xd, row_dtensor(wd, p), mode=mode, out_dtype=torch.float32)
    for t in y.slots:
        t.fill_(7.0)
    tsl.tp_mlp(xd, col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p), mode=mode, out=y)
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    cols = chunk_bounds(0, p)
    expect, _ = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols],
                            [w64(wd[o:o + s]) for o, s in cols], OMODE[mode])
    for i, e in enumerate(expect):
        assert not e.any()
        np.testing.assert_array_equal(to_host(y.slots[i], "fp32"), e, err_msg=f"{mode} out {i}")
