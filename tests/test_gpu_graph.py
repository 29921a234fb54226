"""The hot path inside a CUDA graph.

One small step (embedding gather, a batched redistribute with copies and
Partial reductions, a TP MLP whose down projection splits its tail, fused
q/k/v and the o projection, an aligned move on the bulk-copy kernel and an
unevenly split column layer whose shard is copied to a padded pitch in its
workspace) runs eagerly, then the same calls are captured
into one CUDA graph.  Replays must reproduce the eager results bit for bit
(same kernels, same launch plans), and, after new inputs are written into
the same buffers, match an eager run on those inputs.  This exercises every
piece of the runtime that capture constrains: the reduction stream forked
from the caller's and joined back, the cached launch plans, and the GEMM's
split tail in the caller's workspace (its counters zeroed by a memset that
the graph captures with the launches).
"""
import numpy as np
import pytest
import torch

import tensor_sharded_linear_gb300 as tsl
from oracle.placement import chunk_bounds
from tensor_sharded_linear_gb300 import workloads

from helpers import to_dev

pytestmark = pytest.mark.gpu


def build_step():
    dev = torch.device("cuda")
    bf = torch.bfloat16
    S0, S1, R, P = tsl.Shard(0), tsl.Shard(1), tsl.Replicate(), tsl.Partial()
    inputs, outputs, calls = [], [], []

    # embedding: table Shard(1) over 4, ids Replicate
    tp4 = tsl.DeviceMesh((4,), ("tp",))
    table, ids = workloads.embedding_inputs(vocab=1000, dim=512, ids_shape=(2, 64), seed_base=70)
    tdt = tsl.DTensor([to_dev(np.ascontiguousarray(table[:, o:o + s]), "bf16") for o, s in chunk_bounds(512, 4)],
                      tp4, [S1], table.shape, bf)
    idt = tsl.DTensor([torch.from_numpy(ids).to(dev)], tp4, [R], ids.shape, torch.int32)
    emb = tsl.DTensor.empty(tp4, [R], ids.shape + (512,), bf, device=dev)
    inputs += idt.slots
    outputs += emb.slots
    calls.append(lambda: tsl.tp_embedding(idt, tdt, out=emb))

    # redistribute batch on a (2, 4) mesh: S0 -> S1 copies and P -> R reductions
    mesh = tsl.DeviceMesh((2, 4), ("dp", "tp"))
    g = (520, 384)
    src = tsl.DTensor.distribute_tensor(to_dev(workloads.randn_bf16(g, 71), "bf16"), mesh, [S0, S0])
    part = tsl.DTensor([to_dev(workloads.randn_bf16((260, 384), 72 + i), "bf16") for i in range(8)], mesh, [S0, P],
                       g, bf)
    o1 = tsl.DTensor.empty(mesh, [S0, S1], g, bf, device=dev)
    o2 = tsl.DTensor.empty(mesh, [S0, R], g, bf, device=dev)
    inputs += src.slots + part.slots
    outputs += o1.slots + o2.slots
    calls.append(lambda: tsl.redistribute_batch([(src, o1), (part, o2)]))

    # TP MLP over 8 (down projection: 20 tiles of 128 K steps, a split tail)
    M, K, F, N, p = 512, 256, 8 * 1024, 2560, 8
    x, wg, wu, _ = workloads.mlp_inputs(M, K, F, seed_base=80)
    wd = workloads.randn_bf16((F, N), 84, (1.0 / F) ** 0.5)
    tp8 = tsl.DeviceMesh((p,), ("tp",))
    cols = chunk_bounds(F, p)
    xd = tsl.DTensor([to_dev(x, "bf16")], tp8, [R], x.shape, bf)
    wgd = tsl.DTensor([to_dev(np.ascontiguousarray(wg[:, o:o + s]), "bf16") for o, s in cols], tp8, [S1], wg.shape, bf)
    wud = tsl.DTensor([to_dev(np.ascontiguousarray(wu[:, o:o + s]), "bf16") for o, s in cols], tp8, [S1], wu.shape, bf)
    wdd = tsl.DTensor([to_dev(np.ascontiguousarray(wd[o:o + s]), "bf16") for o, s in cols], tp8, [S0], wd.shape, bf)
    ym = tsl.DTensor.empty(tp8, [R], (M, N), torch.float32, device=dev)
    ws = torch.empty(tsl.tp_mlp_workspace_bytes(xd, wgd, wud, wdd, ym), dtype=torch.uint8, device=dev)
    inputs += xd.slots
    outputs += ym.slots
    calls.append(lambda: tsl.tp_mlp(xd, wgd, wud, wdd, mode=tsl.ALL_REDUCE, out=ym, workspace=ws))

    # attention projections over 4: fused q/k/v, o REDUCE_SCATTER on q
    T, H = 512, 512
    xa_bits, wq, wk, wv, wo = workloads.attention_inputs(T, H, seed_base=90)
    hc = chunk_bounds(H, 4)
    xa = tsl.DTensor([to_dev(xa_bits, "bf16")], tp4, [R], xa_bits.shape, bf)
    wqkv = [tsl.DTensor([to_dev(np.ascontiguousarray(w[:, o:o + s]), "bf16") for o, s in hc], tp4, [S1], w.shape, bf)
            for w in (wq, wk, wv)]
    wod = tsl.DTensor([to_dev(np.ascontiguousarray(wo[o:o + s]), "bf16") for o, s in hc], tp4, [S0], wo.shape, bf)
    qkv = [tsl.DTensor.empty(tp4, [S1], (T, H), bf, device=dev) for _ in range(3)]
    od = tsl.DTensor.empty(tp4, [S0], (T, H), torch.float32, device=dev)
    inputs += xa.slots
    for t in qkv:
        outputs += t.slots
    outputs += od.slots
    calls.append(lambda: tsl.column_parallel_linear_multi(xa, wqkv, outs=qkv))
    calls.append(lambda: tsl.row_parallel_linear(qkv[0], wod, mode=tsl.REDUCE_SCATTER, out=od))

    # an aligned move on its own (the bulk-copy kernel) and an unevenly split
    # column layer with its workspace (operand copy to a padded pitch, and
    # output rows at every alignment)
    g2 = (256, 2048)
    src2 = tsl.DTensor.distribute_tensor(to_dev(workloads.randn_bf16(g2, 95), "bf16"), tp4, [S0])
    o3 = tsl.DTensor.empty(tp4, [S1], g2, bf, device=dev)
    inputs += src2.slots
    outputs += o3.slots
    calls.append(lambda: tsl.redistribute(src2, o3))
    Nu = 1022  # over 4: 256, 256, 256, 254 columns
    wun = workloads.randn_bf16((H, Nu), 96, 1.0 / 23)
    wud_u = tsl.DTensor([to_dev(np.ascontiguousarray(wun[:, o:o + s]), "bf16") for o, s in chunk_bounds(Nu, 4)],
                        tp4, [S1], (H, Nu), bf)
    yu = tsl.DTensor.empty(tp4, [S1], (T, Nu), bf, device=dev)
    wsu = torch.empty(tsl.column_parallel_linear_workspace_bytes(xa, [wud_u], [yu]), dtype=torch.uint8, device=dev)
    assert wsu.numel() > 0
    outputs += yu.slots
    calls.append(lambda: tsl.column_parallel_linear(xa, wud_u, out=yu, workspace=wsu))
    keep = (tdt, idt, emb, src, part, o1, o2, xd, wgd, wud, wdd, ym, ws, xa, wqkv, wod, qkv, od, src2, o3, wud_u, yu,
            wsu)
    return calls, inputs, outputs, keep


def run(calls):
    for c in calls:
        c()


def snapshot(outputs):
    return [t.clone() for t in outputs]


def scribble(outputs):
    for t in outputs:
        t.view(torch.uint8).fill_(0x7F)


def same(a, b):
    return all(torch.equal(x.view(torch.uint8), y.view(torch.uint8)) for x, y in zip(a, b))


def test_step_in_a_cuda_graph(lib):
    calls, inputs, outputs, keep = build_step()
    # one stream for the eager runs and the capture: the linears' cached
    # plans are keyed by stream and workspace, so the captured calls replay
    # exactly the eager launches
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        run(calls)  # eager: plans made
    torch.cuda.synchronize()
    eager = snapshot(outputs)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run(calls)
    torch.cuda.synchronize()

    for _ in range(2):
        scribble(outputs)
        graph.replay()
        torch.cuda.synchronize()
        assert same(outputs, eager), "graph replay differs from the eager step"
    assert tsl.read_device_status() == 0

    # new inputs in the same buffers: the graph computes on them
    gen = torch.Generator(device="cuda").manual_seed(5)
    for t in inputs:
        if t.dtype == torch.int32:
            t.copy_(torch.randint(0, 1000, t.shape, device="cuda", generator=gen, dtype=torch.int32))
        else:
            t.copy_(torch.randn(t.shape, device="cuda", generator=gen).to(t.dtype))
    scribble(outputs)
    graph.replay()
    torch.cuda.synchronize()
    replayed = snapshot(outputs)
    assert not same(replayed, eager)
    scribble(outputs)
    with torch.cuda.stream(stream):
        run(calls)
    torch.cuda.synchronize()
    assert same(outputs, replayed), "graph replay on new inputs differs from the eager step"
    assert tsl.read_device_status() == 0
    del keep
