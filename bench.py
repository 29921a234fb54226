#!/usr/bin/env python3
"""Benchmark of the DTensor tensor-parallel hot path on GB300.

One STEP is one pass of the whole path over one batch of synthetic input:
  1. EmbeddingWithReplicateOutput: table [128256, 4096] bf16 Shard(1) over 8,
     ids [4, 4096] -> Replicate [4, 4096, 4096]
  2. the redistribute sweep on a (dp=2, tp=4) mesh, dp kept Shard(0), for a
     bf16 [8192, 8192] tensor and an uneven [8191, 8190] one:
     S0->S1, S1->S0, S0->R, S1->R, R->S0, R->S1, P->R, P->S0 on tp, all 16
     moves in one dt_redistribute_batch call (one copy launch, one reduction
     launch); each move alone is also timed, outside the step
  3. the TP MLP: X [4096, 4096], gate/up [4096, 11008] Shard(1) over 8,
     SiLU*mul, down [11008, 4096] Shard(0), ALL_REDUCE
  4. the TP attention projections: X [8192, 4096], q/k/v [4096, 4096]
     Shard(1) over 4 (one launch), o Shard(0), REDUCE_SCATTER
Inputs are resident in HBM when the timed region starts.

value = 100 * (sum over GPUs of the step's roofline time) / (time per step):
the roofline time of a kernel is its algorithmic FLOPs / measured dense-bf16
peak, or its algorithmic bytes / measured HBM bandwidth.  Per-GPU work is
fixed as GPUs are added ("weak" scaling); every GPU runs an independent
replica (the logical mesh lives inside one GPU).

`--impl reference` times the CPU oracle (the plain fp64 / in-order fp32
model in oracle/) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TP-linear bf16 TFLOP/s and redistribute GB/s, as % of GB300 roofline"
UNIT = "% of one GB300 roofline, summed over GPUs"
WORKLOAD = ("tp_block: embedding [128256,4096]x ids[4,4096] P=8 + redistribute sweep 8 transitions x "
            "{[8192,8192],[8191,8190]} mesh(dp=2,tp=4) + TP MLP X[4096,4096] gate/up[4096,11008] "
            "down[11008,4096] P=8 ALL_REDUCE + TP attention X[8192,4096] qkv/o[4096,4096] P=4 REDUCE_SCATTER")
G_EVEN = 8192 * 8192 * 2
G_ODD = 8191 * 8190 * 2
EMB_BYTES = 4 * 4096 * 4096 * 2 * 2 + 4 * 4096 * 4
MLP_FLOPS = 3 * 2 * 4096 * 4096 * 11008
ATTN_FLOPS = 4 * 2 * 8192 * 4096 * 4096
GEMM_SOURCES = ["ptx_sm103.cuh", "gemm_sm103.cuh", "gemm_pair_kernel.cu", "gemm_host.cu"]
ALL_COMPONENTS = "embedding,redistribute,mlp,attention"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def transitions():
    return [("S0->S1", "S0S0", "S0S1"), ("S1->S0", "S0S1", "S0S0"), ("S0->R", "S0S0", "S0R"),
            ("S1->R", "S0S1", "S0R"), ("R->S0", "S0R", "S0S0"), ("R->S1", "S0R", "S0S1"),
            ("P->R", "S0P", "S0R"), ("P->S0", "S0P", "S0S0")]


# ---------------------------------------------------------------- distributed control plane

def dist_init(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(roofline_s: float, step_s: float, world: int, device="cpu"):
    """(sum over ranks of roofline seconds, max over ranks of step seconds)."""
    if world == 1:
        return roofline_s, step_s
    import torch.distributed as dist
    t = torch.tensor([roofline_s], dtype=torch.float64, device=device)
    m = torch.tensor([step_s], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(t.item()), float(m.item())


# ---------------------------------------------------------------- clocks

# NVML clock-event reason bits the timing rules name
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes):
    the SM clock, its maximum, board power and the active clock-event
    reasons of one GPU."""

    CLOCK_SM = 1

    def __init__(self, uuid: str):
        import ctypes
        self.C = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + uuid)
        try:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        C = self.C
        sm, mw, r = C.c_uint(), C.c_uint(), C.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, C.byref(sm)) != 0
                or self.lib.nvmlDeviceGetPowerUsage(self.h, C.byref(mw)) != 0
                or self.reasons_fn(self.h, C.byref(r)) != 0):
            raise RuntimeError("NVML query failed")
        return float(sm.value), mw.value / 1000.0, int(r.value)

    def max_sm(self):
        v = self.C.c_uint()
        return float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.C.byref(v)) == 0 else None

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock, power and throttle reasons while the timed region runs.

    NVML is read from a thread every 2 ms (ctypes releases the interpreter
    lock during each query), and only samples whose host timestamps fall
    inside the timed region count; a timed region of a few tens of ms still
    gets a dozen samples or more.  Where NVML cannot be loaded, nvidia-smi
    runs every 200 ms around the region instead."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, index: int):
        self.index = str(index)
        try:
            self.index = "GPU-" + str(torch.cuda.get_device_properties(index).uuid)
        except Exception:
            pass
        self.proc = None
        self.path = None
        self.nvml = None
        self.thread = None
        self.samples = []

    def start(self):
        try:
            self.nvml = _Nvml(self.index)
            self.nvml.sample()
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            import threading
            self.stop_flag = threading.Event()

            def loop():
                while not self.stop_flag.is_set():
                    t = time.perf_counter()
                    try:
                        self.samples.append((t, *self.nvml.sample()))
                    except Exception:
                        return
                    time.sleep(self.PERIOD_S)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.index, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self, window=None):
        """window: (t0, t1) host perf_counter bounds of the timed region."""
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
            inside = [x for x in self.samples if window is None or window[0] <= x[0] <= window[1]]
            mx = self.nvml.max_sm()
            self.nvml.close()
            reasons = sorted({name for _, _, _, r in inside for bit, name in NVML_REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(x[1] for x in inside) if inside else None, "sm_max_mhz": mx,
                    "sm_mhz_min": min(x[1] for x in inside) if inside else None,
                    "power_w_max": max(x[2] for x in inside) if inside else None, "reasons": reasons,
                    "samples": len(inside), "source": "NVML every 2 ms, samples inside the timed region"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm),
                "source": "nvidia-smi every 200 ms around the timed region"}


# ---------------------------------------------------------------- our arm

class Block:
    """Every tensor of one step, resident on one GPU, with prebuilt ABI descriptors."""

    def __init__(self, device, only=("embedding", "redistribute", "mlp", "attention"), weights_kmajor=False,
                 batch_sweep=True):
        import ctypes as C

        import tensor_sharded_linear_gb300 as tsl
        from tensor_sharded_linear_gb300 import _lib as L
        from tensor_sharded_linear_gb300 import workloads as W

        self.C, self.L, self.tsl = C, L, tsl
        self.lib = L.load()
        self.device = device
        bf = torch.bfloat16

        def dev(a):  # numpy bf16 bits / int32 -> device tensor
            if a.dtype == np.uint16:
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(bf).to(device)
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)

        def wdev(a):  # a [K, N] weight, stored [K, N] or (weights_kmajor) [N, K]
            return dev(np.ascontiguousarray(a.T)).t() if weights_kmajor else dev(a)

        self.wdev = wdev

        self.calls = []  # (name, kind, work, fn)
        self.call_io = []  # per call: (device inputs the host supplies, device outputs the host reads)
        self.sweep = []  # (name, bytes, src, dst) of every redistribute transition
        self.rd_fine = []  # the sweep as one batch call per shape: (name, kind, work, call, io)
        self.batch_sweep = batch_sweep
        stream = torch.cuda.current_stream(device).cuda_stream
        self.stream = stream

        from tensor_sharded_linear_gb300.api import DTensor
        S0, S1, R, Pp = tsl.Shard(0), tsl.Shard(1), tsl.Replicate(), tsl.Partial()
        if "embedding" in only:
            self._build_embedding(W, dev, DTensor, bf, device)
        if "redistribute" in only:
            self._build_redistribute(W, dev, DTensor, bf, device, S0, S1, R, Pp)
        if "mlp" in only:
            self._build_mlp(W, dev, DTensor, bf, device, S0, S1, R)
        if "attention" in only:
            self._build_attention(W, dev, DTensor, bf, device, S0, S1, R)
        torch.cuda.synchronize(device)

    def _build_embedding(self, W, dev, DTensor, bf, device):
        tsl = self.tsl
        P = W.EMBEDDING["parts"]
        tp = tsl.DeviceMesh((P,), ("tp",), device=device)
        table, ids = W.embedding_inputs()
        D = W.EMBEDDING["dim"]
        chunks = [(i * (D // P), D // P) for i in range(P)]
        tdt = DTensor([dev(table[:, o:o + s]) for o, s in chunks], tp, [tsl.Shard(1)], table.shape, bf)
        del table
        idt = DTensor([dev(ids)], tp, [tsl.Replicate()], ids.shape, torch.int32)
        odt = DTensor.empty(tp, [tsl.Replicate()], ids.shape + (D,), bf, device=device)
        self._add("embedding", "bytes", EMB_BYTES, "dt_tp_embedding", idt, tdt, odt, 0,
                  io=(list(idt.slots), list(odt.slots)))

    def _build_redistribute(self, W, dev, DTensor, bf, device, S0, S1, R, Pp):
        tsl = self.tsl
        mesh = tsl.DeviceMesh(W.REDISTRIBUTE["mesh"], ("dp", "tp"), device=device)
        pls = {"S0S0": [S0, S0], "S0S1": [S0, S1], "S0R": [S0, R], "S0P": [S0, Pp]}
        rd_in, rd_out = [], []
        for gshape, G in ((W.REDISTRIBUTE["shape"], G_EVEN), (W.REDISTRIBUTE["uneven"], G_ODD)):
            g = dev(W.redistribute_global(gshape))
            src = {k: DTensor.distribute_tensor(g, mesh, pls[k]) for k in ("S0S0", "S0S1", "S0R")}
            del g
            lay = DTensor.empty(mesh, pls["S0P"], gshape, bf, device=device)
            partial_slots = []
            for s, t in enumerate(lay.slots):
                partial_slots.append(dev(W.redistribute_partials(tuple(t.shape), 1, seed=310 + s)[0]))
            src["S0P"] = DTensor(partial_slots, mesh, pls["S0P"], gshape, bf)
            out = {k: DTensor.empty(mesh, pls[k], gshape, bf, device=device) for k in ("S0S0", "S0S1", "S0R")}
            shape_in = [t for k in src for t in src[k].slots]
            shape_out = [t for k in out for t in out[k].slots]
            rd_in += shape_in
            rd_out += shape_out
            tag = "x".join(str(s) for s in gshape)
            pairs, work_sum = [], 0
            for name, a, b in transitions():
                work = 5 * G if a == "S0P" else 2 * G
                self.sweep.append((f"redistribute {name} {tag}", work, src[a], out[b]))
                pairs.append((src[a], out[b]))
                work_sum += work
            self._add(f"redistribute sweep {tag}", "bytes", work_sum, "dt_redistribute_batch", pairs,
                      io=(shape_in, shape_out), target=self.rd_fine)
        if self.batch_sweep:
            # every transition in one dt_redistribute_batch call: one copy
            # launch and one reduction launch
            self._add(f"redistribute sweep ({len(self.sweep)} transitions, one batch)", "bytes",
                      sum(w for _, w, _, _ in self.sweep), "dt_redistribute_batch",
                      [(a, b) for _, _, a, b in self.sweep], io=(rd_in, rd_out))
        else:
            for i, (name, work, a, b) in enumerate(self.sweep):
                # the inputs and outputs ride on the first and last transition
                io = (rd_in if i == 0 else [], rd_out if i == len(self.sweep) - 1 else [])
                self._add(name, "bytes", work, "dt_redistribute", a, b, io=io)

    def _build_mlp(self, W, dev, DTensor, bf, device, S0, S1, R):
        tsl, L = self.tsl, self.L
        cfg = W.MLP
        P = cfg["parts"]
        tp8 = tsl.DeviceMesh((P,), ("tp",), device=device)
        x, wg, wu, wd = W.mlp_inputs()
        F = cfg["ffn"]
        fc = [(i * (F // P), F // P) for i in range(P)]
        xd = DTensor([dev(x)], tp8, [R], x.shape, bf)
        wdev = self.wdev
        wgd = DTensor([wdev(wg[:, o:o + s]) for o, s in fc], tp8, [S1], wg.shape, bf)
        wud = DTensor([wdev(wu[:, o:o + s]) for o, s in fc], tp8, [S1], wu.shape, bf)
        wdd = DTensor([wdev(wd[o:o + s]) for o, s in fc], tp8, [S0], wd.shape, bf)
        yd = DTensor.empty(tp8, [R], (cfg["tokens"], cfg["hidden"]), bf, device=device)
        nbytes = tsl.tp_mlp_workspace_bytes(xd, wgd, wud, wdd, yd)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self._add("tp_mlp", "flops", MLP_FLOPS, "dt_tp_mlp", xd, wgd, wud, wdd, yd,
                  io=(list(xd.slots), list(yd.slots)))

    def _build_attention(self, W, dev, DTensor, bf, device, S0, S1, R):
        tsl, L = self.tsl, self.L
        cfg = W.ATTENTION
        P = cfg["parts"]
        tp4 = tsl.DeviceMesh((P,), ("tp",), device=device)
        x, wq, wk, wv, wo = W.attention_inputs()
        H = cfg["hidden"]
        hc = [(i * (H // P), H // P) for i in range(P)]
        xa = DTensor([dev(x)], tp4, [R], x.shape, bf)
        wdev = self.wdev
        wcols = [DTensor([wdev(w[:, o:o + s]) for o, s in hc], tp4, [S1], w.shape, bf) for w in (wq, wk, wv)]
        wod = DTensor([wdev(wo[o:o + s]) for o, s in hc], tp4, [S0], wo.shape, bf)
        qkv = [DTensor.empty(tp4, [S1], (cfg["tokens"], H), bf, device=device) for _ in range(3)]
        od = DTensor.empty(tp4, [S0], (cfg["tokens"], H), bf, device=device)
        # caller-owned workspaces for the split tail (empty where a launch
        # would not split)
        self.ws_qkv = torch.empty(max(1, tsl.column_parallel_linear_workspace_bytes(xa, wcols, qkv)),
                                  dtype=torch.uint8, device=device)
        self.ws_o = torch.empty(max(1, tsl.row_parallel_linear_workspace_bytes(qkv[0], wod, od, tsl.REDUCE_SCATTER)),
                                dtype=torch.uint8, device=device)
        self._add("attention qkv", "flops", 3 * 2 * cfg["tokens"] * H * H, "qkv", xa, wcols, qkv,
                  io=(list(xa.slots), [t for d in qkv for t in d.slots]))
        self._add("attention o", "flops", 2 * cfg["tokens"] * H * H, "dt_row_parallel_linear", qkv[0], wod, od,
                  L.TP_REDUCE_SCATTER, io=([], list(od.slots)))

    def _add(self, name, kind, work, fn_name, *args, io=((), ()), target=None):
        C, L, lib, stream = self.C, self.L, self.lib, self.stream
        keep = list(args)  # the DTensors own the device memory the descriptors point at

        def desc(d):
            r = d._desc()
            keep.append(r)
            return C.byref(r)

        if fn_name == "dt_tp_embedding":
            ids, table, out, tp = args
            a = (desc(ids), desc(table), desc(out), tp)
            fn = lambda: lib.dt_tp_embedding(*a, None, stream)  # noqa: E731
        elif fn_name == "dt_redistribute":
            src, dst = args
            a = (desc(src), desc(dst))
            fn = lambda: lib.dt_redistribute(*a, None, stream)  # noqa: E731
        elif fn_name == "dt_redistribute_batch":
            (pairs,) = args
            sdescs = [a._desc() for a, _ in pairs]
            ddescs = [b._desc() for _, b in pairs]
            sa = (L.DTensorDesc * len(pairs))(*sdescs)
            da = (L.DTensorDesc * len(pairs))(*ddescs)
            keep.extend(sdescs + ddescs + [sa, da])
            npairs = len(pairs)
            fn = lambda: lib.dt_redistribute_batch(npairs, sa, da, None, stream)  # noqa: E731
        elif fn_name == "dt_tp_mlp":
            x, wg, wu, wd, y = args
            a = (desc(x), desc(wg), desc(wu), desc(wd), desc(y), L.TP_ALL_REDUCE, 0, self.ws.data_ptr(),
                 self.ws.numel())
            fn = lambda: lib.dt_tp_mlp(*a, None, stream)  # noqa: E731
        elif fn_name == "qkv":
            x, ws, ys = args
            wdescs = [w._desc() for w in ws]
            ydescs = [y._desc() for y in ys]
            keep.extend(wdescs + ydescs)
            wa = (L.DTensorDesc * 3)(*wdescs)
            ya = (L.DTensorDesc * 3)(*ydescs)
            keep.extend([wa, ya])
            xdesc = desc(x)
            wsa = (self.ws_qkv.data_ptr(), self.ws_qkv.numel())
            fn = lambda: lib.dt_column_parallel_linear_multi(xdesc, 3, wa, None, ya, 0, *wsa, None, stream)  # noqa: E731
        elif fn_name == "dt_row_parallel_linear":
            x, w, y, mode = args
            a = (desc(x), desc(w), None, desc(y), mode, 0, self.ws_o.data_ptr(), self.ws_o.numel())
            fn = lambda: lib.dt_row_parallel_linear(*a, None, stream)  # noqa: E731
        else:
            raise ValueError(fn_name)

        def call():
            st = fn()
            if st != L.OK:
                raise RuntimeError(f"{name}: {lib.dt_status_string(st).decode()}: {lib.dt_last_error().decode()}")

        call._keep = keep
        if target is not None:
            target.append((name, kind, work, call, (list(io[0]), list(io[1]))))
            return
        self.calls.append((name, kind, work, call))
        self.call_io.append((list(io[0]), list(io[1])))

    def pipeline_calls(self):
        """The step's calls with their inputs and outputs, the redistribute
        sweep split into one batch call per shape: the same work, in pieces
        small enough that copying one piece's next inputs overlaps the other
        piece's kernels."""
        out = []
        for (name, kind, work, call), io in zip(self.calls, self.call_io):
            if name.startswith("redistribute sweep") and self.rd_fine:
                out += self.rd_fine
            else:
                out.append((name, kind, work, call, io))
        return out

    @property
    def h2d(self):
        return [t for ins, _ in self.call_io for t in ins]

    @property
    def d2h(self):
        return [t for _, outs in self.call_io for t in outs]

    def step(self, events=None):
        for i, (_, _, _, call) in enumerate(self.calls):
            if events is not None:
                events[i][0].record()
            call()
            if events is not None:
                events[i][1].record()

    def measure_transitions(self, steps, peaks):
        """Each sweep transition alone, one dt_redistribute call per
        transition (outside the timed step): where the batch's time goes."""
        lib, stream, C = self.lib, self.stream, self.C
        rows = []
        for name, work, a, b in self.sweep:
            da, db = a._desc(), b._desc()
            rows.append((name, work, da, db))
        out = {}
        for name, work, da, db in rows:
            for _ in range(3):
                lib.dt_redistribute(C.byref(da), C.byref(db), None, stream)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            gc.disable()
            for e0, e1 in evs:
                e0.record()
                st = lib.dt_redistribute(C.byref(da), C.byref(db), None, stream)
                e1.record()
                if st != self.L.OK:
                    gc.enable()
                    raise RuntimeError(f"{name}: {lib.dt_last_error().decode()}")
            gc.enable()
            torch.cuda.synchronize()
            ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
            ach = work / (ms / 1e3) / 1e9
            out[name] = {"us": round(ms * 1e3, 2), "achieved": round(ach, 1), "unit": "GB/s",
                         "frac": round(ach / peaks["hbm_gbs"], 4)}
        return out

    def roofline_seconds(self, peaks):
        s = 0.0
        for _, kind, work, _ in self.calls:
            s += work / (peaks["bf16_tflops"] * 1e12) if kind == "flops" else work / (peaks["hbm_gbs"] * 1e9)
        return s


class Extras:
    """Rows built beyond the hot path, timed separately (not part of `value`):
    the sequence-parallel q/k/v entry (x token-sharded, read in place), the
    fused Replicate-output column linear, q/k/v with [out, in] weights (K-major
    B), the Ulysses Shard(2) -> Shard(1) move of [2, 32, 8192, 128], and the
    secondary rows of the step's own operations: S0/S1 -> Replicate with a
    materialised copy per rank, and the TP MLP and q/k/v with fp32 outputs."""

    def __init__(self, device, blk=None):
        import tensor_sharded_linear_gb300 as tsl
        from tensor_sharded_linear_gb300 import workloads as W
        from tensor_sharded_linear_gb300.api import DTensor
        self.tsl = tsl
        bf = torch.bfloat16
        self.items = []

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(bf).to(device)

        cfg = W.ATTENTION
        P, H, T = cfg["parts"], cfg["hidden"], cfg["tokens"]
        mesh = tsl.DeviceMesh((P,), ("tp",), device=device)
        x, wq, wk, wv, _ = W.attention_inputs()
        hc = [(i * (H // P), H // P) for i in range(P)]
        tc = [(i * (T // P), T // P) for i in range(P)]
        x_tok = DTensor([dev(x[o:o + s]) for o, s in tc], mesh, [tsl.Shard(0)], x.shape, bf)
        x_rep = DTensor([dev(x)], mesh, [tsl.Replicate()], x.shape, bf)
        ws = [DTensor([dev(w[:, o:o + s]) for o, s in hc], mesh, [tsl.Shard(1)], w.shape, bf) for w in (wq, wk, wv)]
        ws_k = [DTensor([dev(np.ascontiguousarray(w[:, o:o + s].T)).t() for o, s in hc], mesh, [tsl.Shard(1)],
                        w.shape, bf) for w in (wq, wk, wv)]
        outs = [DTensor.empty(mesh, [tsl.Shard(1)], (T, H), bf, device=device) for _ in range(3)]
        rep_out = DTensor.empty(mesh, [tsl.Replicate()], (T, H), bf, device=device)
        qkv_flops = 3 * 2 * T * H * H
        self._keep = (x_tok, x_rep, ws, ws_k, outs, rep_out)
        self.items.append(("sequence-parallel q/k/v entry", "flops", qkv_flops,
                           lambda: tsl.column_parallel_linear_multi(x_tok, ws, outs=outs)))
        self.items.append(("column linear, Replicate output", "flops", 2 * T * H * H,
                           lambda: tsl.column_parallel_linear(x_rep, ws[0], out=rep_out, output="replicate")))
        self.items.append(("q/k/v with [out, in] weights", "flops", qkv_flops,
                           lambda: tsl.column_parallel_linear_multi(x_rep, ws_k, outs=outs)))
        shape = (2, 32, 8192, 128)
        g = dev(W.randn_bf16(shape, 990))
        cp = tsl.DeviceMesh((4,), ("cp",), device=device)
        useq = DTensor.distribute_tensor(g, cp, [tsl.Shard(2)])
        uhead = DTensor.empty(cp, [tsl.Shard(1)], shape, bf, device=device)
        self._keep2 = (useq, uhead)
        self.items.append(("Ulysses S(2)->S(1) [2,32,8192,128]", "bytes", 2 * 2 * int(np.prod(shape)),
                           lambda: tsl.redistribute(useq, uhead)))
        # secondary rows: Replicate outputs materialised per rank (read G,
        # write 4G) and fp32-output variants of the GEMMs
        rmesh = tsl.DeviceMesh(W.REDISTRIBUTE["mesh"], ("dp", "tp"), device=device)
        rshape = W.REDISTRIBUTE["shape"]
        rg = dev(W.redistribute_global(rshape))
        S0, S1, R = tsl.Shard(0), tsl.Shard(1), tsl.Replicate()
        rsrc = {k: DTensor.distribute_tensor(rg, rmesh, pl) for k, pl in (("S0", [S0, S0]), ("S1", [S0, S1]))}
        rdst = DTensor.empty(rmesh, [S0, R], rshape, bf, materialize_replicas=True, device=device)
        del rg
        self._keep3 = (rsrc, rdst)
        G = 2 * int(np.prod(rshape))
        for k in ("S0", "S1"):
            self.items.append((f"redistribute {k}->R materialised [8192,8192]", "bytes", 5 * G,
                               lambda k=k: tsl.redistribute(rsrc[k], rdst)))
        mlp = [c for c in blk.calls if c[0] == "tp_mlp"] if blk is not None else []
        if mlp:
            # the step's own MLP tensors, an fp32 output, descriptors built once
            import ctypes as C
            from tensor_sharded_linear_gb300 import _lib as L
            xm, wgm, wum, wdm, ym16 = mlp[0][3]._keep[:5]
            ym = DTensor.empty(xm.mesh, [R], ym16.gshape, torch.float32, device=device)
            descs = [d._desc() for d in (xm, wgm, wum, wdm, ym)]
            lib, stream = L.load(), torch.cuda.current_stream(device).cuda_stream
            self._keep4 = (ym, descs)

            def mlp32():
                st = lib.dt_tp_mlp(*[C.byref(d) for d in descs], L.TP_ALL_REDUCE, 0, blk.ws.data_ptr(),
                                   blk.ws.numel(), None, stream)
                if st != L.OK:
                    raise RuntimeError(lib.dt_last_error().decode())
            self.items.append(("TP MLP, fp32 output", "flops", MLP_FLOPS, mlp32))
        outs32 = [DTensor.empty(mesh, [tsl.Shard(1)], (T, H), torch.float32, device=device) for _ in range(3)]
        self._keep5 = outs32
        self.items.append(("q/k/v, fp32 outputs", "flops", qkv_flops,
                           lambda: tsl.column_parallel_linear_multi(x_rep, ws, outs=outs32)))
        # an unevenly split weight: [4096, 8190] over 4 leaves a 2046-column
        # shard whose 4092-byte pitch TMA cannot read.  With the queried
        # workspace it is copied to a padded pitch (tensor cores); with none
        # the launch runs on the CUDA-core kernel
        Nu = 8190
        wu_bits = W.randn_bf16((H, Nu), 995, 1.0 / 64)
        step = -(-Nu // P)
        ucols = [(o, min(step, Nu - o)) for o in range(0, Nu, step)]
        wun = DTensor([dev(np.ascontiguousarray(wu_bits[:, o:o + s])) for o, s in ucols], mesh, [tsl.Shard(1)],
                      (H, Nu), bf)
        yun = DTensor.empty(mesh, [tsl.Shard(1)], (T, Nu), bf, device=device)
        wsu = torch.empty(tsl.column_parallel_linear_workspace_bytes(x_rep, [wun], [yun]), dtype=torch.uint8,
                          device=device)
        no_ws = torch.empty(0, dtype=torch.uint8, device=device)
        self._keep6 = (wun, yun, wsu, no_ws)
        self.items.append(("column linear, uneven shards [8192,4096]x[4096,8190]/4, padded in the workspace", "flops",
                           2 * T * H * Nu,
                           lambda: tsl.column_parallel_linear(x_rep, wun, out=yun, workspace=wsu)))
        self.items.append(("column linear, uneven shards, no workspace (CUDA-core kernel)", "flops", 2 * T * H * Nu,
                           lambda: tsl.column_parallel_linear(x_rep, wun, out=yun, workspace=no_ws)))

    def measure(self, steps, peaks):
        for _, _, _, fn in self.items:  # warm up every item (descriptor caches, first launches)
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        out = {}
        for name, kind, work, fn in self.items:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            gc.disable()
            for a, b in evs:
                a.record()
                fn()
                b.record()
            gc.enable()
            torch.cuda.synchronize()
            # median: these calls go through the Python API, and a host hiccup
            # in one iteration leaves the GPU waiting for that launch
            ms = statistics.median(a.elapsed_time(b) for a, b in evs)
            if kind == "flops":
                ach = work / (ms / 1e3) / 1e12
                out[name] = {"us": round(ms * 1e3, 2), "achieved": round(ach, 1), "unit": "TFLOP/s",
                             "frac": round(ach / peaks["bf16_tflops"], 4)}
            else:
                ach = work / (ms / 1e3) / 1e9
                out[name] = {"us": round(ms * 1e3, 2), "achieved": round(ach, 1), "unit": "GB/s",
                             "frac": round(ach / peaks["hbm_gbs"], 4)}
        return out


def gemm_source_hash():
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "tensor_sharded_linear_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def gemm_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "tcgen05_gemm_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_sha256_16") == gemm_source_hash():
            return d.get("bytes_per_launch_scaled"), d
    except Exception:
        pass
    return None, None


def run_ours(args):
    from tensor_sharded_linear_gb300 import build as B
    B.build()
    rank, world = dist_init("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peaks = load_peaks()
    blk = Block(device, only=tuple(args.only.split(",")))
    lib = blk.lib
    for _ in range(args.warmup):
        blk.step()
    # GEMM kernel launches per step, counted by the library on one more warm-up step
    blk.gemm_launches_per_step = 0
    for name, kind, _, call in blk.calls:
        c0 = lib.dt_launch_count()
        call()
        if kind == "flops":
            blk.gemm_launches_per_step += int(lib.dt_launch_count() - c0)
    torch.cuda.synchronize(device)
    n = len(blk.calls)
    events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
              for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(device)
    gc.disable()  # no collector pauses while the timed launches are issued
    launches0 = lib.dt_launch_count()
    wall0 = time.perf_counter()
    t0.record()
    for k in range(args.steps):
        blk.step(events[k])
    t1.record()
    torch.cuda.synchronize(device)
    wall1 = time.perf_counter()
    launches = lib.dt_launch_count() - launches0
    gc.enable()
    barrier(world)
    clk = clocks.stop((wall0, wall1))
    status = blk.tsl.read_device_status()
    total_ms = t0.elapsed_time(t1)
    step_s = total_ms / 1e3 / args.steps
    roof_s = blk.roofline_seconds(peaks)
    roof_sum, step_max = aggregate(roof_s, step_s, world, device)

    comps = {}
    gemm_flops = gemm_ms = red_bytes = red_ms = 0.0
    for i, (name, kind, work, _) in enumerate(blk.calls):
        ms = statistics.fmean(events[k][i][0].elapsed_time(events[k][i][1]) for k in range(args.steps))
        if kind == "flops":
            ach = work / (ms / 1e3) / 1e12
            comps[name] = {"us": round(ms * 1e3, 2), "achieved": round(ach, 1), "unit": "TFLOP/s",
                           "frac": round(ach / peaks["bf16_tflops"], 4)}
            gemm_flops += work
            gemm_ms += ms
        else:
            ach = work / (ms / 1e3) / 1e9
            comps[name] = {"us": round(ms * 1e3, 2), "achieved": round(ach, 1), "unit": "GB/s",
                           "frac": round(ach / peaks["hbm_gbs"], 4)}
            if name.startswith("redistribute"):
                red_bytes += work
                red_ms += ms
    gemm_tflops = gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms else 0.0
    ngemm = blk.gemm_launches_per_step
    traffic, _ = gemm_traffic()
    roofline = {"kernel": f"tcgen05_gemm_pair_kernel (TP MLP + attention projections, {ngemm} launches per step)",
                "bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(gemm_tflops / peaks["bf16_tflops"], 4),
                "peak_kind": f"dense bf16 burst, {peaks['source']}", "traffic": traffic,
                "algorithmic_flops_per_launch": round(gemm_flops / max(1, ngemm)),
                "launches_per_step": ngemm}
    red_gbs = red_bytes / (red_ms / 1e3) / 1e9 if red_ms else 0.0

    e2e = None if args.no_e2e else run_e2e(blk, args, peaks, world, device)
    extras = None
    if not args.no_extras and args.only == ALL_COMPONENTS:
        nx = max(3, min(args.steps, 10))
        transitions_alone = blk.measure_transitions(nx, peaks)
        ex = Extras(device, blk)
        extras = ex.measure(nx, peaks)
        extras["redistribute transitions, one call each"] = transitions_alone
        del ex

    line = {
        "metric": METRIC, "value": round(100.0 * roof_sum / step_max, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_max * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch CPU RNG, the workload shapes and distributions stated in config)",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}; logical TP mesh inside each GPU",
                   "l2": "no flush: every tensor is re-read only after >2.5 GB of other traffic per step "
                         "(L2 129 MB); each kernel's inputs are >=134 MB",
                   "peaks": peaks},
        "roofline": roofline,
        "tp_linear_tflops": round(gemm_tflops, 1),
        "redistribute_gbs": round(red_gbs, 1),
        "redistribute_frac": round(red_gbs / peaks["hbm_gbs"], 4),
        "components": comps,
        "extras": extras,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "device_status": status,
        "wall_s_timed": round(wall1 - wall0, 4),
    }
    if args.only != ALL_COMPONENTS:
        line["config"]["only"] = args.only
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(peaks, fraction=1.0 / 16)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(blk, args, peaks, world, device):
    """Same metric through the public API with host buffers: every step
    copies its activations in from pinned host memory and reads its results
    back.  The copies are pipelined with the compute on three streams, per
    call (the redistribute sweep as one batch per shape): a call's inputs for the next step go in once the call has finished
    this step, the call runs once its inputs are in and its previous results
    have been read back, and its results go out as soon as it finishes, so
    the link carries both directions while the kernels run.  The timed
    region ends when the last step's results are on the host."""
    comp = torch.cuda.current_stream(device)
    hs, ds = torch.cuda.Stream(device), torch.cuda.Stream(device)
    calls = blk.pipeline_calls()
    io = []
    for _, _, _, _, (ins, outs) in calls:
        hin = [(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for t in ins]
        hout = [(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for t in outs]
        for dev_t, host in hin:
            host.copy_(dev_t)
        io.append((hin, hout))
    bi = sum(t.numel() * t.element_size() for _, _, _, _, (ins, _) in calls for t in ins)
    bo = sum(t.numel() * t.element_size() for _, _, _, _, (_, outs) in calls for t in outs)
    n = len(calls)
    ev_in = [torch.cuda.Event() for _ in range(n)]     # call's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(n)]   # call finished (its inputs may be overwritten)
    ev_out = [torch.cuda.Event() for _ in range(n)]    # call's results are on the host
    for e in ev_done + ev_out:
        e.record(comp)
    steps = max(2, args.steps)  # the pipeline fills on the first step and drains after the last

    def one():
        for i, (_, _, _, call, _) in enumerate(calls):
            hin, hout = io[i]
            hs.wait_event(ev_done[i])
            with torch.cuda.stream(hs):
                for dev_t, host in hin:
                    dev_t.copy_(host, non_blocking=True)
            ev_in[i].record(hs)
            comp.wait_event(ev_in[i])
            comp.wait_event(ev_out[i])
            call()
            ev_done[i].record(comp)
            ds.wait_event(ev_done[i])
            with torch.cuda.stream(ds):
                for dev_t, host in hout:
                    host.copy_(dev_t, non_blocking=True)
            ev_out[i].record(ds)

    def timed(k):
        torch.cuda.synchronize(device)
        barrier(world)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        hs.wait_event(t0)  # no copy starts before the clock does
        ds.wait_event(t0)
        gc.disable()
        for _ in range(k):
            one()
        for e in ev_out:
            comp.wait_event(e)
        t1.record(comp)
        torch.cuda.synchronize(device)
        gc.enable()
        return t0.elapsed_time(t1) / 1e3 / k

    timed(1)  # warm-up: streams, events, pinned buffers
    step_s = timed(steps)
    roof_sum, step_max = aggregate(blk.roofline_seconds(peaks), step_s, world, device)
    return {"value": round(100.0 * roof_sum / step_max, 3), "unit": UNIT, "h2d_bytes_per_step": int(bi),
            "d2h_bytes_per_step": int(bo), "ms_per_step": round(step_max * 1e3, 3), "steps": steps,
            "copies": "pinned host buffers, copy streams overlapped with compute (per-call events)"}


# ---------------------------------------------------------------- the oracle on the host

def oracle_inputs():
    """The step's inputs on the host (generated once; not part of the timing)."""
    from tensor_sharded_linear_gb300 import workloads as W
    from oracle import placement as opl
    table, ids = W.embedding_inputs()
    inp = {"emb_shards": [np.ascontiguousarray(table[:, o:o + s]) for o, s in opl.chunk_bounds(4096, 8)],
           "ids": ids.reshape(-1)}
    del table
    inp["red"] = [(W.REDISTRIBUTE["shape"], G_EVEN, W.redistribute_global(W.REDISTRIBUTE["shape"])),
                  (W.REDISTRIBUTE["uneven"], G_ODD, W.redistribute_global(W.REDISTRIBUTE["uneven"]))]
    inp["mlp"] = W.mlp_inputs()
    inp["attn"] = W.attention_inputs()
    return inp


def oracle_sample(inp, fraction: float):
    """Run the oracle on `fraction` of every component of one step.

    Returns (seconds spent in the oracle, algorithmic work of the sample,
    per component {"seconds", "work", "kind"})."""
    from oracle import bf16 as ob
    from oracle import linear as olin
    from oracle import placement as opl
    from oracle import redistribute as ord_
    from oracle.embedding import tp_embedding as oemb
    from tensor_sharded_linear_gb300 import workloads as W

    work = {"flops": 0.0, "bytes": 0.0}
    t_total = 0.0
    per = {}

    def note(name, kind, secs, amount):
        c = per.setdefault(name, {"seconds": 0.0, "work": 0.0, "kind": kind})
        c["seconds"] += secs
        c["work"] += amount

    # embedding: the first tokens
    ntok = max(1, int(16384 * fraction))
    t = time.perf_counter()
    oemb(inp["ids"][:ntok], inp["emb_shards"], 4096)
    dt_ = time.perf_counter() - t
    t_total += dt_
    work["bytes"] += EMB_BYTES * ntok / 16384
    note("embedding", "bytes", dt_, EMB_BYTES * ntok / 16384)
    # redistribute: the same transitions on the first rows of each tensor
    for gshape, G, g_full in inp["red"]:
        rows = max(8, int(gshape[0] * fraction))
        sub = (rows, gshape[1])
        g = g_full[:rows]
        pls = {"S0S0": [opl.Shard(0), opl.Shard(0)], "S0S1": [opl.Shard(0), opl.Shard(1)],
               "S0R": [opl.Shard(0), opl.Replicate()], "S0P": [opl.Shard(0), opl.Partial()]}
        lays = {k: opl.Layout((2, 4), v, sub) for k, v in pls.items()}
        srcs = {k: ord_.distribute(g, lays[k], "bf16") for k in ("S0S0", "S0S1", "S0R")}
        srcs["S0P"] = [W.randn_bf16(lays["S0P"].local_shape(s), 310 + s) for s in range(8)]
        for _, a, b in transitions():
            t = time.perf_counter()
            ord_.redistribute(srcs[a], lays[a], lays[b], "bf16")
            dt_ = time.perf_counter() - t
            t_total += dt_
            work["bytes"] += (5 if a == "S0P" else 2) * G * rows / gshape[0]
            note("redistribute sweep", "bytes", dt_, (5 if a == "S0P" else 2) * G * rows / gshape[0])
    # MLP rows
    x, wg, wu, wd = inp["mlp"]
    rows = max(1, int(4096 * fraction))
    cols = opl.chunk_bounds(11008, 8)
    t = time.perf_counter()
    olin.tp_mlp(ob.widen64(x[:rows]), [ob.widen64(wg[:, o:o + s]) for o, s in cols],
                [ob.widen64(wu[:, o:o + s]) for o, s in cols], [ob.widen64(wd[o:o + s]) for o, s in cols])
    dt_ = time.perf_counter() - t
    t_total += dt_
    work["flops"] += MLP_FLOPS * rows / 4096
    note("tp_mlp", "flops", dt_, MLP_FLOPS * rows / 4096)
    # attention rows
    x, wq, wk, wv, wo = inp["attn"]
    rows = max(1, int(8192 * fraction))
    cols = opl.chunk_bounds(4096, 4)
    t = time.perf_counter()
    olin.attention_projections(ob.widen64(x[:rows]), *[[ob.widen64(w[:, o:o + s]) for o, s in cols]
                                                        for w in (wq, wk, wv)],
                               [ob.widen64(wo[o:o + s]) for o, s in cols], olin.ALL_REDUCE)
    dt_ = time.perf_counter() - t
    t_total += dt_
    work["flops"] += ATTN_FLOPS * rows / 8192
    note("attention", "flops", dt_, ATTN_FLOPS * rows / 8192)
    return t_total, work, per


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(peaks, fraction):
    secs, work, per = oracle_sample(oracle_inputs(), fraction)
    roof = work["flops"] / (peaks["bf16_tflops"] * 1e12) + work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    comps = {}
    for name, c in per.items():  # each component's own rate, in the GPU rows' units
        rate = c["work"] / max(c["seconds"], 1e-9)
        comps[name] = ({"seconds": round(c["seconds"], 3), "achieved": round(rate / 1e12, 4), "unit": "TFLOP/s"}
                       if c["kind"] == "flops" else
                       {"seconds": round(c["seconds"], 3), "achieved": round(rate / 1e9, 3), "unit": "GB/s"})
    return {"value": round(100.0 * roof / secs, 6), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "seconds": round(secs, 3), "components": comps,
            "sample": f"{fraction:.4g} of every component of one step: the first {fraction:.4g} of the tokens / "
                      f"rows of the embedding, the 16 redistribute transitions, the MLP and the attention "
                      f"projections (numpy fp64 matmul, in-order fp32 partial sums)"}


def run_reference(args):
    rank, world = dist_init("gloo")
    if rank != 0:
        return
    peaks = load_peaks()
    fraction = 1.0 / 256
    inp = oracle_inputs()
    for _ in range(args.warmup):
        oracle_sample(inp, fraction)
    secs_total = 0.0
    roof = 0.0
    for _ in range(args.steps):
        secs, work, _ = oracle_sample(inp, fraction)
        secs_total += secs
        roof += work["flops"] / (peaks["bf16_tflops"] * 1e12) + work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    value = round(100.0 * roof / secs_total, 6)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs_total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{fraction:.4g} of every component per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": cpu_cores(),
                         "sample": f"{fraction:.4g} of every component of one step per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_cublas_shapes(args):
    """Library context, not a bench line: cuBLAS (torch.matmul, bf16 in and
    out) on the step's dense GEMM shapes, each call after an L2 flush, CUDA
    events, median of --steps after --warmup.  The TP MLP has no fused
    counterpart there: gate and up run as one [T,H]x[H,2F] GEMM, SiLU(g)*u
    as torch elementwise ops, then the down GEMM.  The embedding gather is
    timed back to back three ways that move the same bytes: torch's
    index_select (the gather F.embedding runs) on the unsharded
    [128256, 4096] table (8 KiB rows); torch's index_select on each of the 8
    Shard(1) slots (1 KiB rows, 8 launches, outputs left unassembled); and
    this library's one-launch gather from the 8 slots into the Replicate
    output."""
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peaks = load_peaks()
    gen = torch.Generator(device=device).manual_seed(7)
    bf = torch.bfloat16

    def randn(*shape, std=1.0):
        return (torch.randn(*shape, device=device, generator=gen) * std).to(bf)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize(device)
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    from tensor_sharded_linear_gb300 import workloads as W
    T, H, F = W.MLP["tokens"], W.MLP["hidden"], W.MLP["ffn"]
    x, wgu, wd = randn(T, H), randn(H, 2 * F, std=H ** -0.5), randn(F, H, std=F ** -0.5)
    gu, h, y = torch.empty(T, 2 * F, device=device, dtype=bf), torch.empty(T, F, device=device, dtype=bf), \
        torch.empty(T, H, device=device, dtype=bf)
    rows = {}
    rows["MLP gate/up as one GEMM"] = (timed(lambda: torch.matmul(x, wgu, out=gu)), 2 * T * H * 2 * F)
    g, u = gu[:, :F], gu[:, F:]
    rows["MLP SiLU(g)*u, torch elementwise"] = (timed(lambda: torch.mul(torch.nn.functional.silu(g), u, out=h)), 0)
    rows["MLP down"] = (timed(lambda: torch.matmul(h, wd, out=y)), 2 * T * F * H)
    TA, HA = W.ATTENTION["tokens"], W.ATTENTION["hidden"]
    xa, wqkv, wo = randn(TA, HA), randn(HA, 3 * HA, std=HA ** -0.5), randn(HA, HA, std=HA ** -0.5)
    qkv, o = torch.empty(TA, 3 * HA, device=device, dtype=bf), torch.empty(TA, HA, device=device, dtype=bf)
    rows["attention q/k/v as one GEMM"] = (timed(lambda: torch.matmul(xa, wqkv, out=qkv)), 2 * TA * HA * 3 * HA)
    q = randn(TA, HA)  # contiguous, as the step's q/k/v output slots are
    rows["attention o"] = (timed(lambda: torch.matmul(q, wo, out=o)), 2 * TA * HA * HA)
    del x, wgu, wd, gu, h, y, xa, wqkv, wo, qkv, o, q
    import tensor_sharded_linear_gb300 as tsl
    from tensor_sharded_linear_gb300 import build as B
    B.build()
    E = W.EMBEDDING
    V, D, P = E["vocab"], E["dim"], E["parts"]
    ids = torch.randint(0, V, E["ids"], device=device, generator=gen, dtype=torch.int32)
    table = randn(V, D, std=E["std"])
    emb = torch.empty(*E["ids"], D, device=device, dtype=bf)
    ids64 = ids.long()

    def back_to_back(fn):
        """HBM-bound rows: --steps calls back to back between two events, as
        the bench times the step (a flush by writes would leave up to 129 MB
        of dirty lines for the timed call to write back)."""
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3 / args.steps

    # int64 ids: 64 KiB more than the int32 ids the library reads
    gathered = torch.empty_like(emb)
    brows = {"embedding, torch index_select (F.embedding's gather), unsharded table": (back_to_back(
        lambda: torch.index_select(table, 0, ids64.view(-1), out=gathered.view(-1, D))), EMB_BYTES + 4 * ids.numel())}
    tp = tsl.DeviceMesh((P,), ("tp",))
    shards = [t.contiguous() for t in table.chunk(P, dim=1)]
    del table
    tdt = tsl.DTensor(shards, tp, [tsl.Shard(1)], (V, D), bf)
    idt = tsl.DTensor([ids], tp, [tsl.Replicate()], tuple(E["ids"]), torch.int32)
    odt = tsl.DTensor([emb], tp, [tsl.Replicate()], tuple(E["ids"]) + (D,), bf)
    parts = [torch.empty(ids.numel(), t.shape[1], device=device, dtype=bf) for t in shards]

    def per_shard():
        for t, o in zip(shards, parts):
            torch.index_select(t, 0, ids64.view(-1), out=o)

    brows["embedding, torch index_select per Shard(1) slot (8 launches)"] = (back_to_back(per_shard),
                                                                              EMB_BYTES + (8 * P - 4) * ids.numel())
    brows["embedding, this library (8 Shard(1) slots -> Replicate)"] = (back_to_back(
        lambda: tsl.tp_embedding(idt, tdt, out=odt)), EMB_BYTES)
    out = {}
    for name, (us, flops) in rows.items():
        out[name] = {"us": round(us, 2)}
        if flops:
            tf = flops / (us / 1e6) / 1e12
            out[name].update(tflops=round(tf, 1), frac=round(tf / peaks["bf16_tflops"], 4))
    for name, (us, nbytes) in brows.items():
        gbs = nbytes / (us / 1e6) / 1e9
        out[name] = {"us": round(us, 2), "bytes": int(nbytes), "gbs": round(gbs, 1),
                     "frac": round(gbs / peaks["hbm_gbs"], 4)}
    mlp_us = sum(rows[k][0] for k in ("MLP gate/up as one GEMM", "MLP SiLU(g)*u, torch elementwise", "MLP down"))
    print(json.dumps({"impl": "cublas-shapes", "note": "library context on the step's dense shapes, not a bench line",
                      "rows": out, "tp_mlp_us_unfused": round(mlp_us, 2),
                      "peak_bf16_tflops": peaks["bf16_tflops"], "steps": args.steps, "warmup": args.warmup,
                      "l2": "GEMM rows: 256 MB written before every call; embedding rows: back to back"}),
          flush=True)


def run_profile_case(args):
    """One kernel of the step on its own, `--steps` calls after `--warmup`,
    each timed with CUDA events after a 512 MB write that flushes L2 (for ncu
    captures and A/B timing; prints one small JSON line, not a bench line).  Cases: `mlp_down` (the TP
    MLP's down projection: H [4096, 11008] Shard(-1) over 8, Wd Shard(0),
    ALL_REDUCE, split tail in its workspace), `qkv`, `o`, `sp_qkv` (q/k/v
    from the same x as 4 token shards, the sequence-parallel entry), and
    `rd:<transition>:<shape>` (one redistribute of the sweep, e.g.
    `rd:S1->S0:8191x8190`).  GEMM inputs are random device tensors of the
    step's shapes; redistribute inputs are the step's own."""
    import tensor_sharded_linear_gb300 as tsl
    from tensor_sharded_linear_gb300 import build as B
    B.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    bf = torch.bfloat16
    g = torch.Generator(device=dev).manual_seed(1)

    def rnd(*shape, std=1.0):
        return (torch.randn(*shape, device=dev, generator=g) * std).to(bf)

    S0, S1, R = tsl.Shard(0), tsl.Shard(1), tsl.Replicate()
    case = args.profile_case
    if case == "mlp_down":
        m8 = tsl.DeviceMesh((8,), ("tp",))
        h = tsl.DTensor([rnd(4096, 1376) for _ in range(8)], m8, [S1], (4096, 11008), bf)
        wd = tsl.DTensor([rnd(1376, 4096, std=0.0095) for _ in range(8)], m8, [S0], (11008, 4096), bf)
        y = tsl.DTensor.empty(m8, [R], (4096, 4096), bf)
        ws = torch.empty(max(1, tsl.row_parallel_linear_workspace_bytes(h, wd, y)), dtype=torch.uint8, device=dev)
        fn = lambda: tsl.row_parallel_linear(h, wd, out=y, workspace=ws)  # noqa: E731
    elif case in ("qkv", "o", "sp_qkv"):
        m4 = tsl.DeviceMesh((4,), ("tp",))
        xt = rnd(8192, 4096)
        x = tsl.DTensor([xt], m4, [R], (8192, 4096), bf)
        # the same tokens as 4 token shards (the sequence-parallel entry)
        x_tok = tsl.DTensor([xt[i * 2048:(i + 1) * 2048].contiguous() for i in range(4)], m4, [S0], (8192, 4096), bf)
        wq = [tsl.DTensor([rnd(4096, 1024, std=1 / 64) for _ in range(4)], m4, [S1], (4096, 4096), bf)
              for _ in range(3)]
        qkv = [tsl.DTensor.empty(m4, [S1], (8192, 4096), bf) for _ in range(3)]
        wo = tsl.DTensor([rnd(1024, 4096, std=1 / 64) for _ in range(4)], m4, [S0], (4096, 4096), bf)
        od = tsl.DTensor.empty(m4, [S0], (8192, 4096), bf)
        wsq = torch.empty(max(1, tsl.column_parallel_linear_workspace_bytes(x, wq, qkv)), dtype=torch.uint8,
                          device=dev)
        wso = torch.empty(max(1, tsl.row_parallel_linear_workspace_bytes(qkv[0], wo, od, tsl.REDUCE_SCATTER)),
                          dtype=torch.uint8, device=dev)
        tsl.column_parallel_linear_multi(x, wq, outs=qkv, workspace=wsq)
        if case == "qkv":
            fn = lambda: tsl.column_parallel_linear_multi(x, wq, outs=qkv, workspace=wsq)  # noqa: E731
        elif case == "sp_qkv":
            fn = lambda: tsl.column_parallel_linear_multi(x_tok, wq, outs=qkv)  # noqa: E731
        else:
            fn = lambda: tsl.row_parallel_linear(qkv[0], wo, mode=tsl.REDUCE_SCATTER, out=od, workspace=wso)  # noqa
    elif case.startswith("rd:"):
        _, name, shape = case.split(":")
        blk = Block(dev, only=("redistribute",))
        tag = f"redistribute {name} {shape}"
        hits = [(a, b) for n, _, a, b in blk.sweep if n == tag]
        if not hits:
            raise SystemExit(f"no sweep transition {tag!r}")
        a, b = hits[0]
        fn = lambda: tsl.redistribute(a, b)  # noqa: E731
    else:
        raise SystemExit(f"unknown --profile-case {case!r}")
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > L2: every call starts L2-cold
    times = []
    for _ in range(args.steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    if tsl.read_device_status() != 0:
        raise SystemExit("device status set")
    print(json.dumps({"profile_case": case, "warmup": args.warmup, "steps": args.steps,
                      "us_median": round(statistics.median(times), 2),
                      "bands": os.environ.get("DT_GEMM_BANDS", "default")}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the rows timed outside the step")
    ap.add_argument("--cublas-shapes", action="store_true",
                    help="time cuBLAS on the step's dense GEMM shapes and torch's embedding gather (library context) and exit")
    ap.add_argument("--only", default=ALL_COMPONENTS,
                    help="comma-separated subset of embedding,redistribute,mlp,attention (profiling)")
    ap.add_argument("--profile-case", default=None,
                    help="run one kernel of the step alone for a profiler and exit (see run_profile_case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile_case:
        run_profile_case(args)
    elif args.cublas_shapes:
        run_cublas_shapes(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
