"""Pins for the routing oracle (CPU only).

* OwnerGatherPlan worked example (owner_planning page), value for value.
* Row-shard pack equals torch.cat of the shards along shard_dim (a library
  routine), unpack inverts pack bit for bit, S = 1 is the identity
  (layer_sharded_a2a: a trivial group performs no communication).
* Flat-buffer gather/scatter metadata seen from every rank is consistent:
  every owner reconstructs every owned tensor exactly.
"""

import json
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import planning as op
from oracle import routing as orr

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def example():
    with open(os.path.join(GOLD, "owner_gather_example.json")) as f:
        return json.load(f)


def example_flat():
    # param_0 = 0..23 (6x4), param_1 = 100..115 (4x4), at offsets 0 and 24
    flat = np.zeros(40, np.int64)
    flat[0:24] = np.arange(24)
    flat[24:40] = 100 + np.arange(16)
    return flat


@pytest.mark.parametrize("rho", [0, 1])
def test_owner_gather_example(rho):
    ex = example()
    numels = [s[0] * s[1] for s in ex["shapes"]]
    owners = {int(k): v for k, v in ex["explicit_owners"].items()}
    plan = orr.owner_gather_plan(ex["tensor_to_offset"], numels, ex["size"], 2, owners, rho)
    view = ex["views"][str(rho)]
    assert plan["send_sizes"] == {int(k): v for k, v in view["send_sizes"].items()}
    assert plan["recv_sizes"] == {int(k): v for k, v in view["recv_sizes"].items()}
    assert {i: hi - lo for i, (lo, hi) in plan["own_shards"].items()} == \
        {int(k): v for k, v in view["own_shards_numel"].items()}
    assert plan["recv_offsets"] == {(i, s): o for i, s, o in view["recv_offsets"]}
    # local shard sizes of every param on this rank
    for i, (off, n) in enumerate(zip(ex["tensor_to_offset"], numels)):
        p = orr.piece(off, n, rho, ex["size"], 2)
        assert (0 if p is None else p[1] - p[0]) == ex["local_shard_numel"][str(rho)][i]
    if "send_contents" in view:
        flat = example_flat()
        bufs = orr.gather_send_buffers(plan, flat)
        for o, items in view["send_contents"].items():
            want = np.concatenate([flat[ex["tensor_to_offset"][i] + s: ex["tensor_to_offset"][i] + s + c]
                                   for i, s, c in items])
            assert np.array_equal(bufs[int(o)], want)


def test_owner_gather_example_reconstruct():
    ex = example()
    numels = [s[0] * s[1] for s in ex["shapes"]]
    owners = {int(k): v for k, v in ex["explicit_owners"].items()}
    flat = example_flat()
    p0 = orr.owner_gather_plan(ex["tensor_to_offset"], numels, 40, 2, owners, 0)
    p1 = orr.owner_gather_plan(ex["tensor_to_offset"], numels, 40, 2, owners, 1)
    recv = {0: orr.gather_send_buffers(p0, flat)[1]}
    assert recv[0].size == ex["reconstruct"]["0"]["received_from_rank0"]
    full0 = orr.reconstruct_full(p1, 0, ex["tensor_to_offset"], numels, 40, 2, 1, recv, flat[20:40])
    full1 = orr.reconstruct_full(p1, 1, ex["tensor_to_offset"], numels, 40, 2, 1, recv, flat[20:40])
    assert full0.size == ex["reconstruct"]["0"]["total"] and np.array_equal(full0, np.arange(24))
    assert full1.size == ex["reconstruct"]["1"]["total"] and np.array_equal(full1, 100 + np.arange(16))


def test_owner_scatter_example():
    # Scatter mirror of the example's owners {0: 1, 1: 1}: rank 1 returns the
    # 20 elements of param_0 that rank 0 holds; rank 0 unpacks {0: 20}.
    ex = example()
    numels = [s[0] * s[1] for s in ex["shapes"]]
    owners = {int(k): v for k, v in ex["explicit_owners"].items()}
    s1 = orr.owner_scatter_plan(ex["tensor_to_offset"], numels, 40, 2, owners, 1)
    s0 = orr.owner_scatter_plan(ex["tensor_to_offset"], numels, 40, 2, owners, 0)
    assert s1["send_sizes"] == {0: 20} and s1["recv_sizes"] == {}
    assert s0["send_sizes"] == {} and s0["recv_sizes"] == {1: 20}
    assert s0["recv_offsets"] == {(0, 1): 0}
    result = -example_flat()
    out = orr.scatter_unpack(s0, ex["tensor_to_offset"], numels, 40, 2, owners, 0,
                             {1: orr.gather_send_buffers(s1, result)[0]})
    assert list(out) == [0] and np.array_equal(out[0], result[0:20])


def test_default_owner_gather_metadata():
    # With the balancer's owners {0: 0, 1: 1}: rank 1 sends param_0's last 4
    # elements to rank 0, which receives them at offset 0.
    ex = example()
    numels = [24, 16]
    owners = op.lpt_owners_flat(ex["shapes"], ex["tensor_to_offset"], 40, 2)
    p0 = orr.owner_gather_plan(ex["tensor_to_offset"], numels, 40, 2, owners, 0)
    p1 = orr.owner_gather_plan(ex["tensor_to_offset"], numels, 40, 2, owners, 1)
    assert p1["send_sizes"] == {0: 4} and p0["recv_sizes"] == {1: 4}
    assert p0["recv_offsets"] == {(0, 1): 0}


def _random_flat_layout(seed, S):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 12))
    shapes = [(int(g.integers(1, 9)), int(g.integers(1, 7))) for _ in range(n)]
    numels = [a * b for a, b in shapes]
    offsets, pos = [], 0
    for k in numels:
        pos += int(g.integers(0, 3))      # padding / ineligible gaps
        offsets.append(pos)
        pos += k
    size = ((pos + S - 1) // S) * S
    return shapes, offsets, numels, size


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("S", [1, 2, 3, 5])
def test_flat_gather_scatter_roundtrip(seed, S):
    shapes, offsets, numels, size = _random_flat_layout(seed, S)
    owners = op.lpt_owners_flat(shapes, offsets, size, S)
    flat = np.arange(size, dtype=np.int64) * 7 + 3
    plans = [orr.owner_gather_plan(offsets, numels, size, S, owners, r) for r in range(S)]
    sends = [orr.gather_send_buffers(p, flat) for p in plans]
    for rho in range(S):
        per = size // S
        recv = {src: sends[src][rho] for src in range(S) if rho in sends[src]}
        assert {k: v.size for k, v in recv.items()} == plans[rho]["recv_sizes"]
        for i, o in owners.items():
            if o != rho:
                continue
            full = orr.reconstruct_full(plans[rho], i, offsets, numels, size, S, rho, recv,
                                        flat[rho * per:(rho + 1) * per])
            assert np.array_equal(full, flat[offsets[i]:offsets[i] + numels[i]])
    homes = orr.flat_pack_to_owner([flat[r * (size // S):(r + 1) * (size // S)] for r in range(S)],
                                   offsets, numels, size, S, owners)
    before = [np.full(size // S, -1, np.int64) for _ in range(S)]
    back = np.concatenate(orr.flat_unpack_from_owner(homes, before, offsets, numels, size, S, owners))
    for i in owners:
        assert np.array_equal(back[offsets[i]:offsets[i] + numels[i]], flat[offsets[i]:offsets[i] + numels[i]])
    covered = np.zeros(size, bool)
    for i in owners:
        covered[offsets[i]:offsets[i] + numels[i]] = True
    assert np.all(back[~covered] == -1)
    # scatter metadata is the mirror image of the gather metadata
    sp = [orr.owner_scatter_plan(offsets, numels, size, S, owners, r) for r in range(S)]
    for r in range(S):
        for q in range(S):
            assert sp[r]["send_sizes"].get(q, 0) == plans[q]["send_sizes"].get(r, 0)


def test_owner_must_hold_elements():
    with pytest.raises(ValueError):
        orr.owner_gather_plan([0, 24], [24, 16], 40, 2, {1: 0}, 0)


@pytest.mark.parametrize("S,shard_dim", [(1, 0), (2, 0), (4, 0), (3, 1), (2, 2)])
def test_row_shard_pack_is_torch_cat(S, shard_dim):
    shapes = [(12, 6, 4), (24, 12, 6), (24, 3, 6), (12, 6, 6)]
    tensors = [torch.arange(int(np.prod(s)), dtype=torch.int32).reshape(s) * 3 + i
               for i, s in enumerate(shapes)]
    home_of = {0: S - 1, 1: 0, 2: S - 1, 3: 0}
    ranks = orr.make_rank_buffers([t.numpy() for t in tensors], S, shard_dim)
    # each rank buffer is torch.chunk's shard of every tensor, in index order
    for r in range(S):
        want = torch.cat([torch.chunk(t, S, dim=shard_dim)[r].reshape(-1) for t in tensors])
        assert np.array_equal(ranks[r], want.numpy())
    homes = orr.route_to_ns_home(ranks, shapes, home_of, S, shard_dim)
    for h in range(S):
        mine = [i for i in range(len(shapes)) if home_of[i] == h]
        want = (torch.cat([torch.cat([torch.chunk(tensors[i], S, dim=shard_dim)[r] for r in range(S)],
                                     dim=shard_dim).reshape(-1) for i in mine])
                if mine else torch.zeros(0, dtype=torch.int32))
        assert np.array_equal(homes[h], want.numpy())
    back = orr.route_from_ns_home(homes, shapes, home_of, S, shard_dim)
    for r in range(S):
        assert np.array_equal(back[r], ranks[r])


def test_row_shard_trivial_group_is_identity():
    shapes = [(4, 5), (2, 3)]
    ts = [np.arange(20).reshape(4, 5), np.arange(6).reshape(2, 3) + 50]
    ranks = orr.make_rank_buffers(ts, 1, 0)
    homes = orr.route_to_ns_home(ranks, shapes, {0: 0, 1: 0}, 1, 0)
    assert np.array_equal(homes[0], ranks[0])


def test_row_shard_bf16_bits_roundtrip():
    w = workloads.Workload("t", [(16, 8), (8, 24), (24, 8)], 1.0, 77, S=8)
    ts = [t.view(torch.int16).numpy().view(np.uint16) for t in workloads.gen_tensors(w)]
    home_of = op.lpt_homes_row_shard(w.shapes, 8)
    ranks = orr.make_rank_buffers(ts, 8, 0)
    homes = orr.route_to_ns_home(ranks, w.shapes, home_of, 8, 0)
    assert np.array_equal(np.concatenate(orr.route_from_ns_home(homes, w.shapes, home_of, 8, 0)),
                          np.concatenate(ranks))
    off = orr.home_offsets(w.shapes, home_of, 8)
    for i, t in enumerate(ts):
        h = home_of[i]
        assert np.array_equal(homes[h][off[i]:off[i] + t.size], t.reshape(-1))


def test_row_shard_not_divisible():
    with pytest.raises(ValueError):
        orr.make_rank_buffers([np.zeros((5, 2))], 2, 0)


# ------------------------------------------------------- two-stage exchange

def _ts_tensors(shapes, seed=0):
    g = np.random.default_rng(seed)
    return [g.integers(0, 60000, size=s).astype(np.uint16) for s in shapes]


def test_two_stage_with_one_tp_rank_is_the_row_shard_route():
    shapes = [(12, 6), (24, 4), (6, 6, 2)]
    ts = _ts_tensors(shapes)
    home_of = {0: 2, 1: 0, 2: 1}
    R = 3
    two = orr.route_two_stage(orr.make_rank_buffers_two_stage(ts, R, 1, [1, 1, 2]), shapes, [1, 1, 2],
                              home_of, R, 1)
    one = orr.route_to_ns_home(orr.make_rank_buffers(ts, R, 0), shapes, home_of, R, 0)
    for a, b in zip(two, one):
        assert np.array_equal(a, b)


def test_two_stage_with_one_remat_rank_is_a_partition_dim_route():
    shapes = [(4, 12), (6, 6), (2, 6, 4)]
    ts = _ts_tensors(shapes, 1)
    home_of = {0: 1, 1: 1, 2: 0}
    T = 2
    pd = [1, 1, 1]
    two = orr.route_two_stage(orr.make_rank_buffers_two_stage(ts, 1, T, pd), shapes, pd, home_of, 1, T)
    one = orr.route_to_ns_home(orr.make_rank_buffers(ts, T, 1), shapes, home_of, T, 1)
    for a, b in zip(two, one):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("R,T", [(2, 2), (2, 4), (3, 2)])
def test_two_stage_homes_hold_complete_tensors_and_back(R, T):
    shapes = [(24, 8), (12, 16, 4), (48, 4), (24, 4, 4)]
    pd = [1, 2, 0, 1]
    ts = _ts_tensors(shapes, 2)
    S = R * T
    home_of = {i: (3 * i + 1) % S for i in range(len(shapes))}
    ranks = orr.make_rank_buffers_two_stage(ts, R, T, pd)
    homes = orr.route_two_stage(ranks, shapes, pd, home_of, R, T)
    for h in range(S):
        mine = [i for i in range(len(shapes)) if home_of[i] == h]
        want = np.concatenate([ts[i].reshape(-1) for i in mine]) if mine else np.zeros(0, np.uint16)
        assert np.array_equal(homes[h], want)
    back = orr.route_two_stage_back(homes, shapes, pd, home_of, R, T)
    for a, b in zip(back, ranks):
        assert np.array_equal(a, b)
