"""dt_tp_mlp_static_workspace: the TP MLP for callers that cannot allocate.

Some callers cannot allocate device memory when they run the MLP (a serving
loop that must not allocate once started, host code that does not own the
device allocator), so they cannot hand dt_tp_mlp a workspace for H.  This
entry point keeps H in an array built into the library instead.  The tests
call it through the C ABI:
  * twice in a row, on different inputs, against dt_tp_mlp with a caller
    workspace holding exactly H (the same whole-tile schedule, so the same
    bits) and within the linear tolerance the other tests use (max |err| <=
    2e-3, relative Frobenius <= 1e-3) against dt_tp_mlp with its full
    workspace and against the fp64 oracle;
  * on a shape whose down projection splits its last wave under dt_tp_mlp
    (the static entry runs it whole), on a stream it has not used, checking
    that the device's free memory does not change;
  * with H exactly the array's 32 MiB (accepted) and one row more (refused
    with DT_ERR_CAPACITY before anything launches).
The file name makes pytest collect it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle import linear as olin
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import _lib as L
from tensor_sharded_linear_gb300 import workloads

from helpers import to_host
from test_gpu_linear import REL_FRO_TOL, check_fp32, col_dtensor, row_dtensor, w64, x_rep

pytestmark = pytest.mark.gpu


def static_mlp(lib, x, wg, wu, wd, y, mode=L.TP_ALL_REDUCE):
    return lib.dt_tp_mlp_static_workspace(C.byref(x._desc()), C.byref(wg._desc()), C.byref(wu._desc()),
                                          C.byref(wd._desc()), C.byref(y._desc()), mode, 0, None,
                                          torch.cuda.current_stream().cuda_stream)


def h_bytes(m, f):
    return (m * f * 2 + 255) // 256 * 256


def oracle_mlp(x, wg, wu, wd, p):
    cols = chunk_bounds(wg.shape[1], p)
    (y,), _ = olin.tp_mlp(w64(x), [w64(wg[:, o:o + s]) for o, s in cols], [w64(wu[:, o:o + s]) for o, s in cols],
                          [w64(wd[o:o + s]) for o, s in cols])
    return y


def test_static_workspace_matches_caller_workspace_twice(lib):
    M, K, F, N, p = 256, 256, 8 * 136, 384, 8
    _, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=800)
    wd = workloads.randn_bf16((F, N), 804, (1.0 / F) ** 0.5)
    wgd, wud, wdd = col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    h_only = torch.empty(h_bytes(M, F), dtype=torch.uint8, device="cuda")
    tsl.read_device_status(clear=True)
    for call, seed in enumerate((810, 820)):
        x = workloads.randn_bf16((M, K), seed)
        xd = x_rep(x, p)
        same_schedule = tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, out_dtype=torch.float32, workspace=h_only)
        full = tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, out_dtype=torch.float32)
        y = tsl.DTensor.empty(xd.mesh, [tsl.Replicate()], (M, N), torch.float32)
        assert static_mlp(lib, xd, wgd, wud, wdd, y) == L.OK, lib.dt_last_error()
        torch.cuda.synchronize()
        assert tsl.read_device_status() == 0
        got = to_host(y.slots[0], "fp32")
        np.testing.assert_array_equal(got, to_host(same_schedule.slots[0], "fp32"), err_msg=f"call {call}")
        check_fp32(got, to_host(full.slots[0], "fp32").astype(np.float64), f"call {call} vs dt_tp_mlp")
        check_fp32(got, oracle_mlp(x, wg, wu, wd, p), f"call {call} vs the oracle")


def test_static_workspace_where_dt_tp_mlp_splits(lib):
    """Down projection of 20 tiles x 128 K iterations: dt_tp_mlp with its full
    workspace splits the last wave, the static entry runs it whole."""
    M, K, F, N, p = 512, 256, 8 * 1024, 2560, 8
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=830)
    wd = workloads.randn_bf16((F, N), 834, (1.0 / F) ** 0.5)
    xd, wgd, wud, wdd = x_rep(x, p), col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    ref = tsl.tp_mlp_output(xd, wdd, out_dtype=torch.float32)
    full_bytes = tsl.tp_mlp_workspace_bytes(xd, wgd, wud, wdd, ref)
    assert full_bytes > h_bytes(M, F)  # dt_tp_mlp would split
    tsl.tp_mlp(xd, wgd, wud, wdd, out=ref, workspace=torch.empty(full_bytes, dtype=torch.uint8, device="cuda"))
    y = tsl.DTensor.empty(xd.mesh, [tsl.Replicate()], (M, N), torch.float32)
    assert static_mlp(lib, xd, wgd, wud, wdd, y) == L.OK, lib.dt_last_error()  # the array is set up by now
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):
            assert static_mlp(lib, xd, wgd, wud, wdd, y) == L.OK, lib.dt_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert tsl.read_device_status() == 0
    got = to_host(y.slots[0], "fp32")
    check_fp32(got, to_host(ref.slots[0], "fp32").astype(np.float64), "vs dt_tp_mlp (split)")
    expect = oracle_mlp(x, wg, wu, wd, p)
    assert np.linalg.norm(got - expect) / np.linalg.norm(expect) <= REL_FRO_TOL


def test_static_workspace_at_capacity(lib):
    """H of 2048 x 8192 bf16 fills the 32 MiB array exactly; 2049 rows do not fit."""
    M, K, F, N, p = 2048, 128, 8192, 256, 8
    assert h_bytes(M, F) == L.TP_MLP_STATIC_WORKSPACE_BYTES
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=850)
    wd = workloads.randn_bf16((F, N), 854, (1.0 / F) ** 0.5)
    xd, wgd, wud, wdd = x_rep(x, p), col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    h_only = torch.empty(h_bytes(M, F), dtype=torch.uint8, device="cuda")
    ref = tsl.tp_mlp(xd, wgd, wud, wdd, out_dtype=torch.float32, workspace=h_only)
    y = tsl.DTensor.empty(xd.mesh, [tsl.Replicate()], (M, N), torch.float32)
    assert static_mlp(lib, xd, wgd, wud, wdd, y) == L.OK, lib.dt_last_error()
    torch.cuda.synchronize()
    assert tsl.read_device_status() == 0
    got = to_host(y.slots[0], "fp32")
    np.testing.assert_array_equal(got, to_host(ref.slots[0], "fp32"))
    expect = oracle_mlp(x, wg, wu, wd, p)
    assert np.linalg.norm(got - expect) / np.linalg.norm(expect) <= REL_FRO_TOL
    # one row more: refused on the host, nothing launched
    x1 = tsl.DTensor.empty(xd.mesh, [tsl.Replicate()], (M + 1, K), torch.bfloat16)
    y1 = tsl.DTensor.empty(xd.mesh, [tsl.Replicate()], (M + 1, N), torch.float32)
    launches = lib.dt_launch_count()
    assert static_mlp(lib, x1, wgd, wud, wdd, y1) == L.ERR_CAPACITY
    assert b"static workspace" in lib.dt_last_error()
    assert lib.dt_launch_count() == launches
