"""Failure detection without a GPU fault: every mbarrier wait in the GEMM
kernel is bounded.  With DT_GEMM_STARVE=1 the TMA producers issue no loads
(a flag that nothing sets: the MMA's "stage full" waits can never complete),
so the waits run out after DT_GEMM_WAIT_LIMIT_MS, the kernel records
DT_DEV_ERR_TIMEOUT in the status word, frees its tensor memory and returns.
The test then checks the CUDA context is still usable by running a
redistribute and comparing it with the oracle.  Each case runs in a child
process because the hooks are read once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import tensor_sharded_linear_gb300 as tsl
from tensor_sharded_linear_gb300 import _lib as L, workloads
from oracle import placement as opl, redistribute as ord_
from helpers import to_dev, dtensor_from_locals, locals_of
mesh = tsl.DeviceMesh((4,), ("tp",))
x = tsl.DTensor([to_dev(workloads.randn_bf16((256, 256), 1), "bf16")], mesh, [tsl.Replicate()], (256, 256), torch.bfloat16)
w = tsl.DTensor.distribute_tensor(to_dev(workloads.randn_bf16((256, 512), 2), "bf16"), mesh, [tsl.Shard(1)])
tsl.read_device_status(clear=True)
y = tsl.column_parallel_linear(x, w)
status = tsl.read_device_status(clear=True)
assert status & L.DEV_ERR_TIMEOUT, status
# the context still works: a redistribute, checked bit for bit
src = opl.Layout((4,), [opl.Shard(0)], (64, 96)); dst = opl.Layout((4,), [opl.Shard(1)], (64, 96))
loc = ord_.distribute(workloads.randn_bf16((64, 96), 3), src, "bf16")
out = dtensor_from_locals(loc, src, "bf16").redistribute([tsl.Shard(1)])
for g, e in zip(locals_of(out, "bf16"), ord_.redistribute(loc, src, dst, "bf16")):
    assert np.array_equal(g, e)
print("OK", status)
"""


def test_gemm_wait_runs_out_and_reports(lib):
    env = dict(os.environ, DT_GEMM_STARVE="1", DT_GEMM_WAIT_LIMIT_MS="50")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "OK" in r.stdout


CHILD_RD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import tensor_sharded_linear_gb300 as tsl
from tensor_sharded_linear_gb300 import _lib as L, workloads
from oracle import placement as opl, redistribute as ord_
from helpers import dtensor_from_locals, locals_of
tsl.read_device_status(clear=True)
# aligned rows: the bulk copy kernel, which issues no loads here
src = opl.Layout((4,), [opl.Shard(0)], (256, 2048)); dst = opl.Layout((4,), [opl.Shard(1)], (256, 2048))
loc = ord_.distribute(workloads.randn_bf16((256, 2048), 5), src, "bf16")
dtensor_from_locals(loc, src, "bf16").redistribute([tsl.Shard(1)])
status = tsl.read_device_status(clear=True)
assert status & L.DEV_ERR_TIMEOUT, status
# the context still works: an unaligned move (the warp kernel), checked bit for bit
src = opl.Layout((4,), [opl.Shard(0)], (64, 97)); dst = opl.Layout((4,), [opl.Shard(1)], (64, 97))
loc = ord_.distribute(workloads.randn_bf16((64, 97), 6), src, "bf16")
out = dtensor_from_locals(loc, src, "bf16").redistribute([tsl.Shard(1)])
for g, e in zip(locals_of(out, "bf16"), ord_.redistribute(loc, src, dst, "bf16")):
    assert np.array_equal(g, e)
assert tsl.read_device_status(clear=True) == 0
print("OK", status)
"""


def test_bulk_copy_wait_runs_out_and_reports(lib):
    """The bulk copy kernel's stage waits are bounded too: DT_RD_STARVE=1 makes
    it issue no loads, DT_RD_WAIT_LIMIT_MS=50 shortens the limit, and the
    redistribute reports DT_DEV_ERR_TIMEOUT in its status word."""
    env = dict(os.environ, DT_RD_STARVE="1", DT_RD_WAIT_LIMIT_MS="50")
    code = CHILD_RD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "OK" in r.stdout
