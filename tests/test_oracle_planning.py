"""Pins for the planning oracle (CPU only): hand-derived costs and LPT cases,
the OwnerGatherPlan worked example's owners, and invariants.

Sources: Megatron-Core API pages owner_planning (ns_cost_fn,
assign_owner_work, OwnerGatherPlan example) and layer_sharded_a2a
(params_by_home).
"""

import json
import os

import pytest

from oracle import planning as op

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_ns_cost_hand_values():
    for case in load("planning_hand_cases.json")["ns_cost"]:
        assert op.ns_cost(case["shape"], case["steps"]) == case["cost"], case


@pytest.mark.parametrize("case", load("planning_hand_cases.json")["lpt"], ids=lambda c: c["name"])
def test_lpt_hand_cases(case):
    works = [op.OwnerWork(i, c, cand) for i, (c, cand) in enumerate(zip(case["costs"], case["candidates"]))]
    got = op.assign_owner_work(works)
    assert [got[i] for i in range(len(case["costs"]))] == case["owners"]


def test_example_default_owners():
    ex = load("owner_gather_example.json")
    want = {int(k): v for k, v in load("planning_hand_cases.json")["example_default_owners"]["owners"].items()}
    got = op.lpt_owners_flat(ex["shapes"], ex["tensor_to_offset"], ex["size"], ex["world_size"])
    assert got == want


def test_example_candidates_and_ranges():
    ex = load("owner_gather_example.json")
    assert [list(op.rank_range(r, ex["size"], 2)) for r in range(2)] == ex["rank_ranges"]
    numels = [s[0] * s[1] for s in ex["shapes"]]
    assert op.flat_candidates(ex["tensor_to_offset"], numels, ex["size"], 2) == [[0, 1], [1]]


def test_round_robin_invariant_equal_costs():
    for S in (1, 2, 3, 8):
        homes = op.lpt_homes_row_shard([(1408, 2048)] * 50, S)
        assert [homes[i] for i in range(50)] == [i % S for i in range(50)]


def test_single_candidates_never_move():
    works = [op.OwnerWork(0, 100, [0, 1]), op.OwnerWork(1, 1, [1]), op.OwnerWork(2, 5, [0])]
    got = op.assign_owner_work(works)
    assert got[1] == 1 and got[2] == 0


def test_params_by_home():
    assert op.params_by_home(5, {0: 2, 1: 0, 2: 2, 3: 0, 4: 1}, 4) == [[1, 3], [4], [0, 2], []]
    with pytest.raises(KeyError):
        op.params_by_home(3, {0: 0, 2: 1}, 2)
    with pytest.raises(ValueError):
        op.params_by_home(1, {0: 3}, 2)


def test_view_and_eligibility():
    assert op.view_2d((256, 64, 3, 3)) == (256, 576)
    assert op.select_ge_2d((3, 4)) and not op.select_ge_2d((7,))
    with pytest.raises(ValueError):
        op.ns_cost((7,))
