"""dt_tp_mlp_static_workspace: the TP MLP for callers that cannot allocate.

Some callers cannot allocate device memory when they run the MLP (a serving
loop that must not allocate once started, host code that does not own the
device allocator), so they cannot hand dt_tp_mlp a workspace for H.  This
entry point keeps H in an array built into the library instead.  The test
calls it through the C ABI twice in a row, on different inputs, and checks
each result against dt_tp_mlp with a caller-owned workspace, within the
linear tolerance the other tests use (max |err| <= 2e-3, relative Frobenius
<= 1e-3); it also checks that an H larger than the array is refused.
The file name makes pytest collect it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from tensor_sharded_linear_gb300 import _lib as L
from tensor_sharded_linear_gb300 import workloads

from helpers import to_host
from test_gpu_linear import check_fp32, col_dtensor, row_dtensor, x_rep

pytestmark = pytest.mark.gpu


def static_mlp(lib, x, wg, wu, wd, y, mode=L.TP_ALL_REDUCE):
    st = lib.dt_tp_mlp_static_workspace(C.byref(x._desc()), C.byref(wg._desc()), C.byref(wu._desc()),
                                        C.byref(wd._desc()), C.byref(y._desc()), mode, 0, None,
                                        torch.cuda.current_stream().cuda_stream)
    return st


def test_static_workspace_matches_caller_workspace_twice(lib):
    M, K, F, N, p = 256, 256, 8 * 136, 384, 8
    _, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=800)
    wd = workloads.randn_bf16((F, N), 804, (1.0 / F) ** 0.5)
    wgd, wud, wdd = col_dtensor(wg, p), col_dtensor(wu, p), row_dtensor(wd, p)
    tsl.read_device_status(clear=True)
    for call, seed in enumerate((810, 820)):
        x = workloads.randn_bf16((M, K), seed)
        xd = x_rep(x, p)
        ref = tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, out_dtype=torch.float32)
        y = tsl.DTensor.empty(xd.mesh, [tsl.Replicate()], (M, N), torch.float32)
        assert static_mlp(lib, xd, wgd, wud, wdd, y) == L.OK, lib.dt_last_error()
        torch.cuda.synchronize()
        assert tsl.read_device_status() == 0
        check_fp32(to_host(y.slots[0], "fp32"), to_host(ref.slots[0], "fp32").astype(np.float64), f"call {call}")


def test_static_workspace_refuses_oversized_h(lib):
    # H of 4096 x 8192 bf16 = 64 MiB exceeds the 32 MiB array; nothing is launched
    M, K, F, N, p = 4096, 64, 8192, 64, 8
    xd = tsl.DTensor.empty(tsl.DeviceMesh((p,), ("tp",)), [tsl.Replicate()], (M, K), torch.bfloat16)
    mesh = xd.mesh
    wg = tsl.DTensor.empty(mesh, [tsl.Shard(1)], (K, F), torch.bfloat16)
    wu = tsl.DTensor.empty(mesh, [tsl.Shard(1)], (K, F), torch.bfloat16)
    wd = tsl.DTensor.empty(mesh, [tsl.Shard(0)], (F, N), torch.bfloat16)
    y = tsl.DTensor.empty(mesh, [tsl.Replicate()], (M, N), torch.bfloat16)
    assert static_mlp(lib, xd, wg, wu, wd, y) == L.ERR_CAPACITY
    assert b"static workspace" in lib.dt_last_error()
