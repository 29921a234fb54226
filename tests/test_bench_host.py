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


class _FakeNvml:
    """Scripted NVML: (SM MHz, watts, reason bits) per query, then the last one again."""

    def __init__(self, script):
        self.script = list(script)
        self.closed = False

    def sample(self):
        return self.script.pop(0) if len(self.script) > 1 else self.script[0]

    def max_sm(self):
        return 2070.0

    def close(self):
        self.closed = True


def test_clock_sampler_counts_only_the_timed_window(monkeypatch):
    """The sampler keeps the samples whose host time falls inside the timed
    region and decodes NVML's clock-event bits (0x4 power cap, 0x8 hw
    slowdown, 0x20 sw thermal, 0x40 hw thermal)."""
    import time

    fake = _FakeNvml([(1500.0, 100.0, 0x0)] * 3 + [(2070.0, 900.0, 0x4)] * 3 + [(1980.0, 1200.0, 0x4 | 0x20)] * 3 +
                     [(600.0, 50.0, 0x1)])
    monkeypatch.setattr(bench, "_Nvml", lambda uuid: fake)
    monkeypatch.setattr(bench.ClockSampler, "PERIOD_S", 0.0)
    s = bench.ClockSampler(0)
    s.start()
    deadline = time.time() + 5
    while len(s.samples) < 12 and time.time() < deadline:
        time.sleep(0.01)
    assert len(s.samples) >= 12
    times = [x[0] for x in s.samples]
    # start() queried once to check NVML, so the loop's samples begin at the
    # script's second entry: samples 2..7 are the 2070 MHz (power cap) and
    # 1980 MHz (power cap + sw thermal) queries, the timed region
    clk = s.stop((times[2], times[7]))
    assert fake.closed
    assert clk["samples"] == 6
    assert clk["sm_mhz"] == (2070.0 + 1980.0) / 2 and clk["sm_mhz_min"] == 1980.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["power_w_max"] == 1200.0
    assert clk["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]


def test_clock_sampler_without_nvml_or_nvidia_smi(monkeypatch):
    def no_nvml(uuid):
        raise OSError("libnvidia-ml.so.1: cannot open shared object file")

    def no_smi(*a, **k):
        raise FileNotFoundError("nvidia-smi")

    monkeypatch.setattr(bench, "_Nvml", no_nvml)
    monkeypatch.setattr(bench.subprocess, "Popen", no_smi)
    s = bench.ClockSampler(0)
    s.start()
    clk = s.stop((0.0, 1.0))
    assert clk["samples"] == 0 and clk["reasons"] == ["nvidia-smi unavailable"]
