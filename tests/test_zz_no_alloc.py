"""ns_orthogonalize_batched_fixed_ws: Newton-Schulz for callers that cannot
allocate device memory (for example a plugin whose host program's allocator
owns the GPU's memory). It runs on the library's static scratch array instead
of a caller workspace; its results must match the workspace entry point's.

This file is collected last so that a run stopping at the first failure has
already run every other test. It passes alone in a fresh process and after
the other tests.
"""

import pytest
import torch

import workloads
from gpu_util import BF16_TOL, rel_err

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")

SHAPES = [(128, 256)] * 6 + [(300, 700), (700, 300), (256, 64, 3, 3), (5, 3)]


def _reference(plan, ins):
    outs = [torch.empty_like(t) for t in ins]
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device="cuda")
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    return outs


def test_fixed_ws_matches_workspace_entry_two_calls():
    plan = nsg.ns_plan_create(SHAPES, steps=workloads.STEPS, eps=workloads.EPS, S=1)
    assert 0 < plan.workspace_bytes() <= nsg.NS_FIXED_WS_BYTES
    for call, seed in enumerate((61, 62)):   # two calls in a row, different inputs
        ts = workloads.gen_tensors(workloads.Workload("fixed", SHAPES, 1.0, seed))
        ins = [t.cuda() for t in ts]
        want = _reference(plan, ins)
        got = [torch.full_like(t, float("nan")) for t in ins]
        nsg.ns_orthogonalize_batched_fixed_ws(plan, ins, got)
        assert nsg.ns_check_status(plan) == nsg.NS_OK
        for s, g, w in zip(SHAPES, got, want):
            assert g.shape == w.shape
            err = rel_err(g, w.float().cpu().numpy())
            assert err <= BF16_TOL, (call, s, err)


def test_fixed_ws_rejects_plans_over_the_limit():
    # (4096, 4096): X0, X1, A, B of 32 MiB each exceed the 64 MiB array
    plan = nsg.ns_plan_create([(4096, 4096)], S=1)
    assert plan.workspace_bytes() > nsg.NS_FIXED_WS_BYTES
    x = torch.zeros(4096, 4096, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_orthogonalize_batched_fixed_ws(plan, [x], [x])
    assert e.value.code == nsg.NS_ERR_WORKSPACE
