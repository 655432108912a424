"""Device-side error paths, driven without faulting or hanging the GPU.

* A bounded wait that runs out: ns_test_stall_next_gemm arms the next GEMM
  launch so that its TMA producer issues nothing; the MMA issuer's first wait
  for operands then runs out after a few milliseconds, the kernel records a
  timeout and unwinds with nothing in flight. ns_check_status must report
  NS_ERR_TIMEOUT once, and the next call on the same device must be correct.
  Both GEMM forms: the 1-SM kernel (one 128-row tile) and the 2-SM kernel
  (a 256-row pair).
* A refused index: a routing entry given an out-of-range home (host-side
  injection) makes the pack kernel skip that tensor and report
  NS_ERR_DEVICE_CHECK; the tensor's home slots keep their previous contents,
  the other tensors are moved, and restoring the home restores the result.
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import BF16_TOL, bits, oracle_ns, rel_err
from oracle import routing as orr

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")


@pytest.mark.parametrize("shape", [(128, 256), (256, 512)])
def test_gemm_wait_runs_out_and_the_device_stays_usable(shape):
    dev = torch.device("cuda:0")
    shapes = [shape]
    ts = workloads.gen_tensors(workloads.Workload("stall", shapes, 1.0, 93))
    ins = [t.to(dev) for t in ts]
    outs = [torch.empty_like(x) for x in ins]
    plan = nsg.ns_plan_create(shapes, steps=workloads.STEPS, eps=workloads.EPS, S=1)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    # a 128-row matrix would otherwise run as one CTA with no GEMM launch
    nsg.ns_set_small_path(False)
    try:
        nsg.ns_test_stall_next_gemm(3_000_000)          # 3 ms
        nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
        assert nsg.ns_check_status(plan) == nsg.NS_ERR_TIMEOUT
        assert nsg.ns_check_status(plan) == nsg.NS_OK   # read and cleared
        # the next call on the same device runs normally and is right
        outs = [torch.full_like(x, float("nan")) for x in ins]
        nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
        assert nsg.ns_check_status(plan) == nsg.NS_OK
    finally:
        nsg.ns_set_small_path(True)
    assert rel_err(outs[0], oracle_ns(ts[0])) <= BF16_TOL


def test_out_of_range_home_is_refused():
    dev = torch.device("cuda:0")
    shapes = [(8, 6), (4, 10), (12, 2), (6, 6)]
    S = 2
    ts = workloads.gen_tensors(workloads.Workload("badhome", shapes, 1.0, 94))
    np_ts = [bits(t).reshape(t.shape) for t in ts]
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=0)
    homes = plan.homes()
    ho, hs, _ = plan.home_layout()
    ranks_np = orr.make_rank_buffers(np_ts, S, 0)
    want = orr.route_to_ns_home(ranks_np, shapes, dict(enumerate(homes)), S, 0)
    rank_t = [torch.from_numpy(r.view(np.int16).copy()).view(torch.bfloat16).to(dev) for r in ranks_np]

    def pack():
        home_t = [torch.full((max(1, n),), -7.0, dtype=torch.bfloat16, device=dev) for n in hs]
        nsg.ns_pack_to_home(plan, rank_t, home_t)
        return home_t, nsg.ns_check_status(plan)

    home_t, rc = pack()                               # uploads the routing table
    assert rc == nsg.NS_OK
    bad = 1
    nsg.ns_test_set_route_home(plan, bad, S + 3)
    home_t, rc = pack()
    assert rc == nsg.NS_ERR_DEVICE_CHECK
    sentinel = bits(torch.full((1,), -7.0, dtype=torch.bfloat16))[0]
    for i, s in enumerate(shapes):
        n_el = int(np.prod(s))
        got = bits(home_t[homes[i]])[ho[i]:ho[i] + n_el]
        if i == bad:
            assert (got == sentinel).all()             # not moved
        else:
            assert np.array_equal(got, want[homes[i]][ho[i]:ho[i] + n_el])
    nsg.ns_test_set_route_home(plan, bad, homes[bad])  # restore
    home_t, rc = pack()
    assert rc == nsg.NS_OK
    for h in range(S):
        assert np.array_equal(bits(home_t[h])[:hs[h]], want[h])
