"""CUDA-graph capture of the device entry points.

An optimizer calls Newton-Schulz on the same buffers every step, so the whole
call can be captured once and replayed: no host work per launch (parameter
blocks, tensor maps) and no launch gaps. These tests capture
ns_orthogonalize_batched and the wave pipeline (its three streams join the
capture through events), replay them, and require the results of an eager
call bit for bit; a replay after the inputs change must follow them.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")


def test_graph_replays_orthogonalize_batched():
    dev = torch.device("cuda:0")
    shapes = [(128, 256)] * 4 + [(300, 700), (700, 300), (256, 64, 3, 3)]
    ts = workloads.gen_tensors(workloads.Workload("graph", shapes, 0.02, 101))
    ins = [t.to(dev) for t in ts]
    eager = [torch.empty_like(x) for x in ins]
    graphed = [torch.empty_like(x) for x in ins]
    plan = nsg.ns_plan_create(shapes, S=1)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    nsg.ns_orthogonalize_batched(plan, ins, eager, ws)   # first call: per-device set-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nsg.ns_orthogonalize_batched(plan, ins, graphed, ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for a, b in zip(eager, graphed):
        assert torch.equal(a, b)
    # new inputs in the same buffers: the replay computes on them
    for x in ins:
        x.copy_(torch.flip(x, dims=[0]))
    g.replay()
    nsg.ns_orthogonalize_batched(plan, ins, eager, ws)
    torch.cuda.synchronize()
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for a, b in zip(eager, graphed):
        assert torch.equal(a, b)


def test_graph_replays_wave_pipeline():
    dev = torch.device("cuda:0")
    w = workloads.gpt_24l_d2048()
    shapes = w.shapes[:4] + [(640, 384), (384, 640)]
    S = 8
    ts = workloads.gen_tensors(workloads.Workload("graphp", shapes, 0.02, 102))
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=0)
    _, hs, _ = plan.home_layout()
    rank_in = [torch.cat([t.reshape(S, -1)[r] for t in ts]).to(dev) for r in range(S)]
    home_in = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    home_out = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    eager = [torch.zeros_like(x) for x in rank_in]
    graphed = [torch.zeros_like(x) for x in rank_in]
    pipe = nsg.ns_pipeline_create(plan, 2)
    ws = torch.empty(pipe.workspace_bytes, dtype=torch.uint8, device=dev)
    nsg.ns_pipeline_run(pipe, rank_in, home_in, home_out, eager, ws)  # creates the pipeline's streams
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nsg.ns_pipeline_run(pipe, rank_in, home_in, home_out, graphed, ws)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for a, b in zip(eager, graphed):
        assert torch.equal(a, b)
