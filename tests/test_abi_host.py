"""C-ABI host logic against the oracle, CPU only (no CUDA call is made).

* libnsgb300.so loads and exports every function include/nsgb300.h declares.
* ns_cost, ns_assign_owner_work, row-shard homes and home offsets, flat
  owners and the OwnerGatherPlan / OwnerScatterPlan metadata agree with the
  oracle exactly, including the owner_planning page's worked example.
* Invalid inputs return the documented status codes.
"""

import ctypes
import json
import os

import numpy as np
import pytest

import workloads
from oracle import planning as op
from oracle import routing as orr

nsg = pytest.importorskip("newton_schulz_shape_gb300")

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_library_exports_every_header_symbol():
    syms = nsg.header_symbols()
    assert len(syms) >= 16
    for s in syms:
        assert hasattr(nsg.lib, s), s
    from newton_schulz_shape_gb300._lib import _SIGS
    assert sorted(_SIGS) == syms


def test_header_constants_match_the_binding():
    # every enumerator of the header has the same value in the binding
    import re
    from newton_schulz_shape_gb300 import _lib
    with open(os.path.join(os.path.dirname(GOLD), "..", "include", "nsgb300.h")) as f:
        hdr = f.read()
    consts = dict((k, int(v)) for k, v in re.findall(r"\b(NS_[A-Z0-9_]+)\s*=\s*(-?\d+)", hdr))
    assert len(consts) >= 17
    for k, v in consts.items():
        assert getattr(_lib, k) == v, k
    # sizes the header defines as (value << shift)
    defs = re.findall(r"#define\s+(NS_[A-Z0-9_]+)\s+\((\d+)ull\s*<<\s*(\d+)\)", hdr)
    assert [k for k, _, _ in defs] == ["NS_FIXED_WS_BYTES"]
    for k, v, sh in defs:
        assert getattr(nsg, k) == int(v) << int(sh), k


def test_ns_cost_hand_values_and_oracle():
    with open(os.path.join(GOLD, "planning_hand_cases.json")) as f:
        cases = json.load(f)["ns_cost"]
    for c in cases:
        assert nsg.ns_cost(c["shape"], c["steps"]) == c["cost"]
    for s in workloads.gen_random_shapes(200, 5, max_dim=5000):
        for k in (0, 1, 5):
            assert nsg.ns_cost(s, k) == op.ns_cost(s, k)


def test_ns_cost_errors():
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_cost([7], 5)
    assert e.value.code == nsg.NS_ERR_SHAPE
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_cost([2**40, 2**40], 5)
    assert e.value.code == nsg.NS_ERR_ARG


def test_lpt_hand_cases():
    with open(os.path.join(GOLD, "planning_hand_cases.json")) as f:
        cases = json.load(f)["lpt"]
    for c in cases:
        n_ranks = 1 + max(max(x) for x in c["candidates"])
        assert nsg.ns_assign_owner_work(c["costs"], c["candidates"], n_ranks) == c["owners"]


@pytest.mark.parametrize("seed", range(40))
def test_lpt_random_vs_oracle(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 60))
    R = int(g.integers(1, 9))
    costs = [int(g.integers(1, 6)) * int(g.choice([1, 1000, 10**9])) for _ in range(n)]
    cands = []
    for _ in range(n):
        k = int(g.integers(1, R + 1))
        cands.append(sorted(g.choice(R, size=k, replace=False).tolist()))
    want = op.assign_owner_work([op.OwnerWork(i, costs[i], cands[i]) for i in range(n)])
    assert nsg.ns_assign_owner_work(costs, cands, R) == [want[i] for i in range(n)]


def test_lpt_errors():
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_assign_owner_work([5], [[]], 2)
    assert e.value.code == nsg.NS_ERR_HOME
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_assign_owner_work([5], [[3]], 2)
    assert e.value.code == nsg.NS_ERR_HOME


@pytest.mark.parametrize("S", [1, 2, 3, 8])
@pytest.mark.parametrize("seed", range(6))
def test_row_shard_plan_vs_oracle(S, seed):
    shapes = workloads.gen_random_shapes(int(np.random.default_rng(seed).integers(1, 40)), seed, 400, S)
    plan = nsg.ns_plan_create(shapes, S=S)
    want = op.lpt_homes_row_shard(shapes, S)
    assert plan.homes() == [want[i] for i in range(len(shapes))]
    ho, hs, rs = plan.home_layout()
    assert ho == orr.home_offsets(shapes, want, S)
    for h in range(S):
        assert hs[h] == sum(int(np.prod(shapes[i])) for i in range(len(shapes)) if want[i] == h)
    assert rs == [sum(int(np.prod(s)) // S for s in shapes)] * S


def test_row_shard_explicit_homes_and_workloads():
    for w in (workloads.gpt_24l_d2048(), workloads.moe_16l_64e()):
        plan = nsg.ns_plan_create(w.shapes, S=w.S)
        want = op.lpt_homes_row_shard(w.shapes, w.S)
        assert plan.homes() == [want[i] for i in range(len(w.shapes))]
    # equal costs, all candidates: round robin
    plan = nsg.ns_plan_create([(1408, 2048)] * 20, S=8)
    assert plan.homes() == [i % 8 for i in range(20)]
    plan = nsg.ns_plan_create([(4, 6), (8, 2)], S=2, home_of=[1, 1])
    assert plan.homes() == [1, 1]
    assert plan.home_layout()[1] == [0, 40]


def test_row_shard_errors():
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create([(5, 4)], S=2)
    assert e.value.code == nsg.NS_ERR_NOT_DIVISIBLE
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create([(4,)], S=2)
    assert e.value.code == nsg.NS_ERR_SHAPE
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create([(4, 4)], S=2, home_of=[2])
    assert e.value.code == nsg.NS_ERR_HOME
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create([(4, 4)], S=0)
    assert e.value.code == nsg.NS_ERR_ARG
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create([(4, 4)], S=1, ridge=1e-3)   # ridge belongs to the fp32-Gram mode
    assert e.value.code == nsg.NS_ERR_ARG


def _example():
    with open(os.path.join(GOLD, "owner_gather_example.json")) as f:
        return json.load(f)


def test_flat_worked_example():
    ex = _example()
    owners = [ex["explicit_owners"][str(i)] for i in range(2)]
    plan = nsg.ns_plan_create_flat(ex["shapes"], ex["tensor_to_offset"], ex["size"], S=2, owner_of=owners)
    for rho in (0, 1):
        view = ex["views"][str(rho)]
        send, recv, roff, own = plan.owner_gather_meta(rho)
        assert {o: v for o, v in enumerate(send) if v} == {int(k): v for k, v in view["send_sizes"].items()}
        assert {s: v for s, v in enumerate(recv) if v} == {int(k): v for k, v in view["recv_sizes"].items()}
        assert {i: v for i, v in enumerate(own) if v >= 0} == \
            {int(k): v for k, v in view["own_shards_numel"].items()}
        got = {(i, s): roff[i][s] for i in range(2) for s in range(2) if roff[i][s] >= 0}
        assert got == {(i, s): o for i, s, o in view["recv_offsets"]}
    # default balancer on the example: {0: 0, 1: 1}
    plan = nsg.ns_plan_create_flat(ex["shapes"], ex["tensor_to_offset"], ex["size"], S=2)
    assert plan.homes() == [0, 1]


def _random_flat(seed, S):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 14))
    shapes, offsets, pos = [], [], 0
    part = []
    for _ in range(n):
        if g.random() < 0.2:
            shp = (int(g.integers(1, 9)),)          # 1-D: not eligible
        else:
            shp = (int(g.integers(1, 9)), int(g.integers(1, 7)))
        pos += int(g.integers(0, 3))
        offsets.append(pos)
        shapes.append(shp)
        pos += int(np.prod(shp))
    size = ((pos + S - 1) // S) * S
    return shapes, offsets, size


@pytest.mark.parametrize("S", [1, 2, 3, 5])
@pytest.mark.parametrize("seed", range(10))
def test_flat_plan_vs_oracle(S, seed):
    shapes, offsets, size = _random_flat(seed, S)
    plan = nsg.ns_plan_create_flat(shapes, offsets, size, S=S)
    part = [i for i, s in enumerate(shapes) if len(s) >= 2]
    numels = [int(np.prod(s)) for s in shapes]
    want = op.lpt_owners_flat(shapes, offsets, size, S, tensor_indices=part)
    homes = plan.homes()
    assert homes == [want.get(i, -1) for i in range(len(shapes))]
    for rho in range(S):
        g = orr.owner_gather_plan(offsets, numels, size, S, want, rho)
        send, recv, roff, own = plan.owner_gather_meta(rho)
        assert {o: v for o, v in enumerate(send) if v} == g["send_sizes"]
        assert {s: v for s, v in enumerate(recv) if v} == g["recv_sizes"]
        assert {i: v for i, v in enumerate(own) if v >= 0} == {i: hi - lo for i, (lo, hi) in g["own_shards"].items()}
        assert {(i, s): roff[i][s] for i in range(len(shapes)) for s in range(S) if roff[i][s] >= 0} == \
            g["recv_offsets"]
        sc = orr.owner_scatter_plan(offsets, numels, size, S, want, rho)
        send, recv, roff = plan.owner_scatter_meta(rho)
        assert {o: v for o, v in enumerate(send) if v} == sc["send_sizes"]
        assert {s: v for s, v in enumerate(recv) if v} == sc["recv_sizes"]
        assert {(i, s): roff[i][s] for i in range(len(shapes)) for s in range(S) if roff[i][s] >= 0} == \
            sc["recv_offsets"]


def test_flat_errors():
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create_flat([(6, 4), (4, 4)], [0, 24], 41, S=2)
    assert e.value.code == nsg.NS_ERR_NOT_DIVISIBLE
    with pytest.raises(nsg.NsError) as e:   # rank 0 holds nothing of param_1
        nsg.ns_plan_create_flat([(6, 4), (4, 4)], [0, 24], 40, S=2, owner_of=[0, 0])
    assert e.value.code == nsg.NS_ERR_HOME
    with pytest.raises(nsg.NsError) as e:   # overlapping tensors
        nsg.ns_plan_create_flat([(6, 4), (4, 4)], [0, 20], 40, S=2)
    assert e.value.code == nsg.NS_ERR_ARG


def test_workspace_bytes_layout():
    plan = nsg.ns_plan_create([(128, 256)] * 3 + [(300, 70)], S=1)
    ws = plan.workspace_bytes()
    # (128,256) x3: X 128x256 x2 + A,B 128x128 x2 in bf16; (70, 300) -> padded (128, 320)
    lower = 3 * (2 * 128 * 256 + 2 * 128 * 128) * 2 + (2 * 128 * 320 + 2 * 128 * 128) * 2
    assert lower <= ws <= lower + 64 * 1024
    assert plan.n_buckets == 2
    assert nsg.ns_plan_create([], S=1).workspace_bytes() == 0


def test_fp32_auto_workspace_follows_each_bucket_mode():
    # a bucket with n >= 2m takes the Gram-space layout, others the standard
    # fp32 layout: single-bucket auto plans equal the plan of that mode
    for shape, mode in [((256, 1024), nsg.NS_FP32_GRAM_SPACE), ((1024, 256), nsg.NS_FP32_GRAM_SPACE),
                        ((300, 500), nsg.NS_FP32_GRAM), ((512, 512), nsg.NS_FP32_GRAM)]:
        auto = nsg.ns_plan_create([shape], gram_mode=nsg.NS_FP32_AUTO, S=1)
        pure = nsg.ns_plan_create([shape], gram_mode=mode, S=1)
        assert auto.workspace_bytes() == pure.workspace_bytes(), shape
        assert auto.gram_mode == nsg.NS_FP32_AUTO and auto.out_bytes == 4
    mixed = nsg.ns_plan_create([(256, 1024), (512, 512)], gram_mode=nsg.NS_FP32_AUTO, S=1)
    parts = [nsg.ns_plan_create([s], gram_mode=m, S=1).workspace_bytes()
             for s, m in [((256, 1024), nsg.NS_FP32_GRAM_SPACE), ((512, 512), nsg.NS_FP32_GRAM)]]
    assert mixed.workspace_bytes() == sum(parts)
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create([(4, 4)], gram_mode=4, S=1)
    assert e.value.code == nsg.NS_ERR_ARG


@pytest.mark.parametrize("R,T", [(1, 1), (2, 2), (4, 2), (2, 4)])
def test_two_stage_plan_vs_oracle(R, T):
    shapes = [(32, 16), (16, 32, 2), (64, 8), (8, 8, 8), (16, 24)]
    pd = [1, 1, 0, 2, 1]
    plan = nsg.ns_plan_create_two_stage(shapes, pd, R, T)
    S = R * T
    want = op.lpt_homes_row_shard(shapes, S)
    assert plan.homes() == [want[i] for i in range(len(shapes))]
    ho, hs, rs = plan.home_layout()
    assert ho == orr.home_offsets(shapes, want, S)
    assert rs == [sum(int(np.prod(s)) // S for s in shapes)] * S


def test_two_stage_errors():
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create_two_stage([(6, 8)], [0], 2, 2)   # 6 rows not divisible by R*T = 4
    assert e.value.code == nsg.NS_ERR_NOT_DIVISIBLE
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create_two_stage([(8, 6)], [1], 2, 4)   # 6 columns not divisible by T = 4
    assert e.value.code == nsg.NS_ERR_NOT_DIVISIBLE
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_plan_create_two_stage([(8, 8)], [2], 2, 2)   # no dim 2
    assert e.value.code == nsg.NS_ERR_ARG


def test_pipeline_wave_split_host():
    w = workloads.gpt_24l_d2048()
    plan = nsg.ns_plan_create(w.shapes, S=8)
    for n in (1, 2, 4, 7, 500):
        pipe = nsg.ns_pipeline_create(plan, n)
        assert 1 <= pipe.n_waves <= min(n, len(w.shapes))
        assert pipe.workspace_bytes > 0
        # two wave workspaces, each at most the whole plan's
        assert pipe.workspace_bytes <= 2 * plan.workspace_bytes() + 2048
    # every bucket small (one CTA per matrix): one wave, unless that path is off
    small = nsg.ns_plan_create([(128, 256)] * 16, S=8)
    assert nsg.ns_pipeline_create(small, 4).n_waves == 1
    nsg.ns_set_small_path(False)
    try:
        assert nsg.ns_pipeline_create(small, 4).n_waves == 4
    finally:
        nsg.ns_set_small_path(True)
    fp32 = nsg.ns_plan_create([(128, 256)], gram_mode=nsg.NS_FP32_GRAM, S=1)
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_pipeline_create(fp32, 2)
    assert e.value.code == nsg.NS_ERR_UNSUPPORTED


def test_symmetric_store_modes():
    # 0 (upper pair blocks, the default) and 1 (also the mirror); anything else is refused
    for bad in (-1, 2, 3):
        with pytest.raises(nsg.NsError) as e:
            nsg.ns_set_symmetric_store(bad)
        assert e.value.code == nsg.NS_ERR_ARG
    nsg.ns_set_symmetric_store(1)
    nsg.ns_set_symmetric_store(0)


def test_pipeline_with_nothing_participating():
    # a plan without participating tensors gives a pipeline of no waves
    for plan in (nsg.ns_plan_create([], S=2),
                 nsg.ns_plan_create_flat([(4, 4)], [0], 16, participating=[False], S=1)):
        pipe = nsg.ns_pipeline_create(plan, 3)
        assert pipe.n_waves == 0
        assert pipe.workspace_bytes == 0
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_pipeline_create(nsg.ns_plan_create([(8, 8)], S=1), 0)
    assert e.value.code == nsg.NS_ERR_ARG


@pytest.mark.parametrize("kind,S", [("row", 1), ("row", 3), ("row", 8), ("row_dim1", 4), ("two_stage", 4)])
def test_rank_splits_simulated_all_to_allv(kind, S):
    # every rank's view of the exchange, simulated with numpy: the pieces each
    # home receives are exactly the pieces the sources hold
    if kind == "row":
        shapes = workloads.gen_random_shapes(17, 300 + S, 120, S)
        plan = nsg.ns_plan_create(shapes, S=S, shard_dim=0)
    elif kind == "row_dim1":
        shapes = [(5, 12, 7), (3, 24, 4), (2, 36, 8), (6, 12, 4), (1, 4)]
        plan = nsg.ns_plan_create(shapes, S=S, shard_dim=1)
    else:
        shapes = [(48, 24), (24, 48, 4), (96, 16), (24, 8, 8), (48, 12)]
        plan = nsg.ns_plan_create_two_stage(shapes, [1, 1, 0, 2, 1], 2, 2)
    homes = plan.homes()
    _, _, rank_sizes = plan.home_layout()
    n = len(shapes)
    piece = [int(np.prod(s)) // S for s in shapes]
    roff = np.concatenate([[0], np.cumsum(piece)])
    # rank r's buffer: a distinct value per (rank, element)
    bufs = [np.arange(rank_sizes[r]) + 10**6 * (r + 1) for r in range(S)]
    views = [plan.rank_splits(r) for r in range(S)]
    sends = []
    for r, (sc, sd, rc, rd, sp, rp) in enumerate(views):
        assert sum(sc) == rank_sizes[r] and sd == list(np.concatenate([[0], np.cumsum(sc)[:-1]]))
        snd = np.full(sum(sc), -1)
        for i in range(n):
            snd[sp[i]:sp[i] + piece[i]] = bufs[r][roff[i]:roff[i + 1]]
        assert (snd >= 0).all()                      # the pieces tile the send buffer
        sends.append(snd)
    for r, (sc, sd, rc, rd, sp, rp) in enumerate(views):
        # all_to_allv: segment s of r's receive buffer is what s sends to r
        recv = np.concatenate([sends[s][views[s][1][r]:views[s][1][r] + views[s][0][r]] for s in range(S)])
        assert list(rc) == [views[s][0][r] for s in range(S)]
        for i in range(n):
            for s in range(S):
                if homes[i] == r:
                    got = recv[rp[i][s]:rp[i][s] + piece[i]]
                    assert np.array_equal(got, bufs[s][roff[i]:roff[i + 1]]), (kind, i, s, r)
                else:
                    assert rp[i][s] == -1


def test_rank_splits_rejects_flat_plans():
    plan = nsg.ns_plan_create_flat([(6, 4), (4, 4)], [0, 24], 40, S=2)
    with pytest.raises(nsg.NsError) as e:
        plan.rank_splits(0)
    assert e.value.code == nsg.NS_ERR_ARG


def test_test_hooks_reject_bad_arguments():
    for v in (0, 99_999, 10_000_000_001):
        with pytest.raises(nsg.NsError) as e:
            nsg.ns_test_stall_next_gemm(v)
        assert e.value.code == nsg.NS_ERR_ARG
    plan = nsg.ns_plan_create([(4, 4), (2, 6)], S=2)
    for t in (-1, 2):
        with pytest.raises(nsg.NsError) as e:
            nsg.ns_test_set_route_home(plan, t, 0)
        assert e.value.code == nsg.NS_ERR_ARG
    # host-only: no device table uploaded yet, so no CUDA call is made
    nsg.ns_test_set_route_home(plan, 1, 0)
