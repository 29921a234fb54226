"""Host logic of bench.py that needs no GPU: the multi-rank aggregation used
when N GPUs run independent replicas (world size 2 over gloo on the CPU), the
peak loader, and the reference arm's JSON line shape."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    r, w = bench.dist_init("gloo")
    # rank r did 1 + r roofline-seconds of work in 2 + r seconds
    roof, step = bench.aggregate(1.0 + r, 2.0 + r, w)
    bench.barrier(w)
    q.put((r, roof, step))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, roof, step in out:
        assert roof == pytest.approx(3.0)   # summed over ranks
        assert step == pytest.approx(3.0)   # slowest rank


def test_peaks_loader_reads_measured_file():
    p = bench.load_peaks()
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 100
    assert p["source"] in ("measured", "fallback")


def test_transitions_cover_the_sweep():
    names = [t[0] for t in bench.transitions()]
    assert names == ["S0->S1", "S1->S0", "S0->R", "S1->R", "R->S0", "R->S1", "P->R", "P->S0"]


def test_reference_arm_rank1_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    # rank 1 of the reference arm must return before any process-group setup or work
    code = ("import sys; sys.argv=['bench.py','--impl','reference','--steps','1','--warmup','3'];"
            "import bench; bench.dist_init=lambda b: (1, 2); bench.main(); print('quiet')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "quiet"
