"""ns_orthogonalize_batched_fixed_ws: Newton-Schulz for callers that cannot
allocate device memory when they orthogonalise (for example a plugin whose
host program's caching allocator owns the GPU's memory, or code that must not
call cudaMalloc after start-up). It runs on the library's static scratch array
instead of a caller workspace.

Checked here, in every precision policy:
  * its results equal the workspace entry point's bit for bit (same kernels,
    same inputs), on two calls in a row with different inputs -- the array
    keeps the previous call's contents, so the second call shows that nothing
    stale is read;
  * both are within the policy's bar of the float64 oracle;
  * a call allocates no device memory (device free bytes and torch's
    allocator both unchanged across a call on a fresh plan);
  * plans that need more than the array are rejected.

This file is collected last so that a run stopping at the first failure has
already run every other test. It passes alone in a fresh process and after
the other tests.
"""

import pytest
import torch

import workloads
from gpu_util import BF16_TOL, rel_err
from oracle import ns as ons

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")

FP32_TOL = 1e-3
# mixed aspects: in NS_FP32_AUTO the buckets with n >= 2m run in Gram space,
# (5, 3), (384, 640) and (130, 130) in the standard fp32-Gram iteration
SHAPES = [(128, 256)] * 4 + [(300, 700), (700, 300), (256, 64, 3, 3), (5, 3), (384, 640), (130, 130)]
MODES = {
    "bf16": (nsg.NS_BF16, torch.bfloat16, BF16_TOL),
    "fp32_gram": (nsg.NS_FP32_GRAM, torch.float32, FP32_TOL),
    "fp32_gram_space": (nsg.NS_FP32_GRAM_SPACE, torch.float32, FP32_TOL),
    "fp32_auto": (nsg.NS_FP32_AUTO, torch.float32, FP32_TOL),
}


def _plan(mode):
    return nsg.ns_plan_create(SHAPES, steps=workloads.STEPS, eps=workloads.EPS, gram_mode=mode, S=1)


def _workspace_entry(plan, ins, odt):
    outs = [torch.full(t.shape, float("nan"), dtype=odt, device="cuda") for t in ins]
    # a workspace full of garbage: the workspace entry point keeps nothing either
    ws = torch.full((plan.workspace_bytes(),), 0x7F, dtype=torch.uint8, device="cuda")
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    return outs


@pytest.mark.parametrize("name", list(MODES))
def test_fixed_ws_matches_workspace_entry_two_calls(name):
    mode, odt, tol = MODES[name]
    plan = _plan(mode)
    assert 0 < plan.workspace_bytes() <= nsg.NS_FIXED_WS_BYTES
    for call, seed in enumerate((61, 62)):   # two calls in a row, different inputs
        ts = workloads.gen_tensors(workloads.Workload("fixed", SHAPES, 1.0, seed + 10 * mode))
        ins = [t.cuda() for t in ts]
        want = _workspace_entry(plan, ins, odt)
        got = [torch.full(t.shape, float("nan"), dtype=odt, device="cuda") for t in ins]
        nsg.ns_orthogonalize_batched_fixed_ws(plan, ins, got)
        assert nsg.ns_check_status(plan) == nsg.NS_OK
        for s, t, g, w in zip(SHAPES, ts, got, want):
            assert g.shape == w.shape and g.dtype == odt
            assert torch.equal(g, w), (name, call, s)
            ref = ons.newton_schulz(t.float().numpy(), workloads.STEPS, workloads.A_COEF, workloads.B_COEF,
                                    workloads.C_COEF, workloads.EPS)
            err = rel_err(g, ref)
            assert err <= tol, (name, call, s, err)


@pytest.mark.parametrize("name", ["bf16", "fp32_auto"])
def test_fixed_ws_allocates_no_device_memory(name):
    mode, odt, _ = MODES[name]
    ts = workloads.gen_tensors(workloads.Workload("fixed", SHAPES, 1.0, 63))
    ins = [t.cuda() for t in ts]
    outs = [torch.empty(t.shape, dtype=odt, device="cuda") for t in ins]
    # warm-up: the first call on the device looks up the array's address and
    # loads the kernels this plan runs
    nsg.ns_orthogonalize_batched_fixed_ws(_plan(mode), ins, outs)
    assert nsg.ns_check_status() == nsg.NS_OK
    torch.cuda.synchronize()
    plan = _plan(mode)                       # a fresh plan: nothing cached in it
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    nsg.ns_orthogonalize_batched_fixed_ws(plan, ins, outs)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    torch.cuda.synchronize()
    free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    assert free1 == free0, (free0, free1)
    assert alloc1 == alloc0, (alloc0, alloc1)


def test_fixed_ws_rejects_plans_over_the_limit():
    # (4096, 4096): X0, X1, A, B of 32 MiB each exceed the 64 MiB array
    plan = nsg.ns_plan_create([(4096, 4096)], S=1)
    assert plan.workspace_bytes() > nsg.NS_FIXED_WS_BYTES
    x = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_orthogonalize_batched_fixed_ws(plan, [x], [x])
    assert e.value.code == nsg.NS_ERR_WORKSPACE
