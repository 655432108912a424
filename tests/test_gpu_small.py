"""The one-CTA-per-matrix path for small matrices (m <= 128, n <= 512: the
whole iteration on one SM, X, A and B in shared memory, products in TMEM)
against the float64 oracle, and against the GEMM path it replaces.

* the 16 x 128x256 N(0, 1) workload: every matrix within 3e-2 of the oracle,
  in exactly one launch;
* ragged, transposed and 3-D shapes up to 128 x 512 and 512 x 128, step
  counts 0, 1, 3;
* the GEMM path (ns_set_small_path(False)) on the same inputs agrees;
* a plan mixing small and GEMM buckets in one call;
* the wave pipeline with small tensors read from and written to the rank
  buffers equals the serial calls bit for bit; with only small tensors it is
  one launch on the caller's stream.
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import BF16_TOL, oracle_ns, rel_err

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")


def _run(shapes, ts, steps=workloads.STEPS, small=True):
    dev = torch.device("cuda:0")
    ins = [t.to(dev) for t in ts]
    outs = [torch.full_like(x, float("nan")) for x in ins]
    plan = nsg.ns_plan_create(shapes, steps=steps, eps=workloads.EPS, S=1)
    ws = torch.empty(max(1, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
    nsg.ns_set_small_path(small)
    try:
        nsg.ns_profile_read(reset=True)
        nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
        rc = nsg.ns_check_status(plan)
        launches, _ = nsg.ns_profile_read(reset=True)
    finally:
        nsg.ns_set_small_path(True)
    assert rc == nsg.NS_OK, nsg.ns_status_string(rc)
    return outs, launches


def test_small_workload_one_launch():
    w = workloads.small_16x128x256()
    ts = workloads.gen_tensors(w)
    outs, launches = _run(w.shapes, ts)
    assert launches["small"] == 1 and sum(launches.values()) == 1, launches
    for t, o in zip(ts, outs):
        err = rel_err(o, oracle_ns(t))
        assert err <= BF16_TOL, err


RAGGED = [(5, 3), (1, 9), (9, 1), (128, 512), (512, 128), (64, 40), (100, 300), (300, 100), (8, 4, 16),
          (128, 64), (2, 2), (127, 129), (96, 448)]


@pytest.mark.parametrize("steps", [0, 1, 3, 5])
def test_small_ragged_shapes(steps):
    ts = workloads.gen_tensors(workloads.Workload("small", RAGGED, 1.0, 95))
    outs, launches = _run(RAGGED, ts, steps=steps)
    assert launches["small"] == 1 and launches["gram"] == 0
    for s, t, o in zip(RAGGED, ts, outs):
        assert o.shape == t.shape
        err = rel_err(o, oracle_ns(t, steps))
        assert err <= BF16_TOL, (s, steps, err)


def test_small_path_agrees_with_gemm_path():
    ts = workloads.gen_tensors(workloads.Workload("small2", RAGGED, 0.02, 96))
    a, la = _run(RAGGED, ts, small=True)
    b, lb = _run(RAGGED, ts, small=False)
    assert la["small"] == 1 and lb["small"] == 0 and lb["gram"] > 0
    for s, x, y in zip(RAGGED, a, b):
        assert rel_err(x, y.float().cpu().numpy()) <= BF16_TOL, s


def test_mixed_small_and_gemm_buckets():
    shapes = [(128, 256)] * 3 + [(300, 700), (64, 40), (700, 300)]
    ts = workloads.gen_tensors(workloads.Workload("mixed", shapes, 0.02, 97))
    outs, launches = _run(shapes, ts)
    assert launches["small"] == 1 and launches["gram"] == workloads.STEPS
    for s, t, o in zip(shapes, ts, outs):
        assert rel_err(o, oracle_ns(t)) <= BF16_TOL, s


@pytest.mark.parametrize("n_waves", [1, 2])
def test_pipeline_with_small_tensors_in_rank_buffers(n_waves):
    w = workloads.gpt_24l_d2048()
    w.shapes = w.shapes[:4] + [(128, 256), (256, 64), (64, 512), (8, 8, 8)]
    S, shapes = w.S, w.shapes
    dev = torch.device("cuda:0")
    ts = workloads.gen_tensors(w)
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=0)
    homes = plan.homes()
    ho, hs, _ = plan.home_layout()
    rank_in = [torch.cat([t.reshape(S, -1)[r] for t in ts]).to(dev) for r in range(S)]

    def bufs():
        return ([torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs],
                [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs],
                [torch.zeros_like(x) for x in rank_in])

    hi1, ho1, ro1 = bufs()
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ins = [hi1[homes[i]].data_ptr() + 2 * ho[i] for i in range(len(shapes))]
    outs = [ho1[homes[i]].data_ptr() + 2 * ho[i] for i in range(len(shapes))]
    nsg.ns_pack_to_home(plan, rank_in, hi1)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    nsg.ns_unpack_from_home(plan, ho1, ro1)
    hi2, ho2, ro2 = bufs()
    pipe = nsg.ns_pipeline_create(plan, n_waves)
    pws = torch.empty(pipe.workspace_bytes, dtype=torch.uint8, device=dev)
    nsg.ns_pipeline_run(pipe, rank_in, hi2, ho2, ro2, pws)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for a in hi2 + ho2:
        assert not a.any()          # rank buffers in, rank buffers out
    for a, b in zip(ro1, ro2):
        assert torch.equal(a, b)
    offs = np.concatenate([[0], np.cumsum([t.numel() // S for t in ts])])
    for i in range(4, len(shapes)):
        y = torch.cat([ro2[r][offs[i]:offs[i + 1]] for r in range(S)]).reshape(ts[i].shape)
        assert rel_err(y, oracle_ns(ts[i])) <= BF16_TOL, shapes[i]


def test_pipeline_all_small_one_launch_on_caller_stream():
    # every bucket small: the pipeline call is the single small-kernel launch,
    # ordered on the stream it is given (here a side stream), and equals the
    # serial pack -> NS -> unpack bit for bit
    w = workloads.small_16x128x256()
    w.shapes = w.shapes + [(256, 64), (64, 512), (8, 8, 8), (128, 128)]
    S, shapes = w.S, w.shapes
    dev = torch.device("cuda:0")
    ts = workloads.gen_tensors(w)
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=0)
    homes = plan.homes()
    ho, hs, _ = plan.home_layout()
    rank_in = [torch.cat([t.reshape(S, -1)[r] for t in ts]).to(dev) for r in range(S)]
    hi1 = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    ho1 = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    ro1 = [torch.zeros_like(x) for x in rank_in]
    ws = torch.empty(max(1, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
    nsg.ns_pack_to_home(plan, rank_in, hi1)
    nsg.ns_orthogonalize_batched(plan, [hi1[homes[i]].data_ptr() + 2 * ho[i] for i in range(len(shapes))],
                                 [ho1[homes[i]].data_ptr() + 2 * ho[i] for i in range(len(shapes))], ws)
    nsg.ns_unpack_from_home(plan, ho1, ro1)
    torch.cuda.synchronize()
    pipe = nsg.ns_pipeline_create(plan, 2)
    assert pipe.n_waves == 1
    pws = torch.empty(max(1, pipe.workspace_bytes), dtype=torch.uint8, device=dev)
    hi2 = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    ho2 = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    ro2 = [torch.zeros_like(x) for x in rank_in]
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    nsg.ns_profile_read(reset=True)
    with torch.cuda.stream(side):
        nsg.ns_pipeline_run(pipe, rank_in, hi2, ho2, ro2, pws, stream=side)
    side.synchronize()
    launches, _ = nsg.ns_profile_read(reset=True)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    assert launches["small"] == 1 and sum(launches.values()) == 1, launches
    for a in hi2 + ho2:
        assert not a.any()
    for a, b in zip(ro1, ro2):
        assert torch.equal(a, b)
