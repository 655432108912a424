"""Split-QKV: pack the fused QKV projections whole, orthogonalise the Q, K
and V row blocks separately, unpack whole (Megatron-LM issue #6720 lists
split-QKV support among the layer-sharded Muon features).

The routing plan covers complete tensors; an NS plan over the row blocks gets
pointers offset into the home buffers (a row block of a row-major tensor is
contiguous). Oracle: NS of each block on its own.
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import BF16_TOL, bits, oracle_ns, rel_err

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")


@pytest.mark.parametrize("layers,d", [(1, 4096), (2, 2048)])
def test_split_qkv_pack_ns_unpack(layers, d):
    w = workloads.llama8b_32l() if d == 4096 else workloads.gpt_24l_d2048()
    w.shapes = w.shapes[:layers * (5 if d == 4096 else 4)]
    S, shapes = w.S, w.shapes
    dev = torch.device("cuda:0")
    ts = workloads.gen_tensors(w)
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=0)
    homes = plan.homes()
    ho, hs, rs = plan.home_layout()
    rank_in = [torch.cat([t.reshape(S, -1)[r] for t in ts]).to(dev) for r in range(S)]
    home_in = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    home_out = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    rank_out = [torch.empty_like(x) for x in rank_in]
    blocks, parents = workloads.split_rows(shapes)
    assert len(blocks) > len(shapes)
    cols = [int(np.prod(s)) // s[0] for s in shapes]
    ins = [home_in[homes[i]].data_ptr() + 2 * (ho[i] + r0 * cols[i]) for i, r0 in parents]
    outs = [home_out[homes[i]].data_ptr() + 2 * (ho[i] + r0 * cols[i]) for i, r0 in parents]
    ns_plan = nsg.ns_plan_create(blocks, S=1)
    ws = torch.empty(ns_plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    nsg.ns_pack_to_home(plan, rank_in, home_in)
    nsg.ns_orthogonalize_batched(ns_plan, ins, outs, ws)
    nsg.ns_unpack_from_home(plan, home_out, rank_out)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    # every block against the oracle of that block alone
    for (i, r0), blk in zip(parents, blocks):
        t = ts[i].reshape(shapes[i][0], -1)[r0:r0 + blk[0]]
        y = home_out[homes[i]][ho[i] + r0 * cols[i]: ho[i] + (r0 + blk[0]) * cols[i]].reshape(blk)
        assert rel_err(y, oracle_ns(t.reshape(blk))) <= BF16_TOL, (i, r0, blk)
    # unpack hands every rank its shard of every whole result
    for r in range(S):
        want = torch.cat([home_out[homes[i]][ho[i]:ho[i] + ts[i].numel()].reshape(S, -1)[r].cpu()
                          for i in range(len(shapes))])
        assert np.array_equal(bits(rank_out[r]), bits(want))
