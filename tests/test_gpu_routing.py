"""GPU pack (shard -> home) and unpack (home -> shard) against the oracle,
bit for bit, for the row-shard and flat-buffer models."""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import bits
from oracle import planning as op
from oracle import routing as orr

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")


def _row_shard_case(shapes, S, shard_dim, seed, home_of=None):
    dev = torch.device("cuda:0")
    ts = workloads.gen_tensors(workloads.Workload("route", shapes, 1.0, seed))
    np_ts = [bits(t).reshape(t.shape) for t in ts]
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=shard_dim, home_of=home_of)
    homes = plan.homes()
    home_of_d = {i: h for i, h in enumerate(homes)}
    ranks_np = orr.make_rank_buffers(np_ts, S, shard_dim)
    want_homes = orr.route_to_ns_home(ranks_np, shapes, home_of_d, S, shard_dim)
    rank_t = [torch.from_numpy(r.view(np.int16).copy()).view(torch.bfloat16).to(dev) for r in ranks_np]
    _, hs, _ = plan.home_layout()
    home_t = [torch.full((max(1, n),), -1.0, dtype=torch.bfloat16, device=dev) for n in hs]
    nsg.ns_pack_to_home(plan, rank_t, home_t)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for h in range(S):
        assert np.array_equal(bits(home_t[h])[:hs[h]], want_homes[h])
    back = [torch.zeros_like(r) for r in rank_t]
    nsg.ns_unpack_from_home(plan, home_t, back)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for r in range(S):
        assert np.array_equal(bits(back[r]), ranks_np[r])


@pytest.mark.parametrize("S", [1, 2, 8])
def test_row_shard_dim0(S):
    shapes = workloads.gen_random_shapes(25, 100 + S, 300, S)
    _row_shard_case(shapes, S, 0, 21)


@pytest.mark.parametrize("S,shard_dim", [(2, 1), (3, 1), (4, 2)])
def test_row_shard_other_dims(S, shard_dim):
    shapes = [(5, 12, 7), (3, 24, 4), (2, 36, 8), (6, 12, 4)] if shard_dim == 1 else \
             [(3, 5, 8, 2), (2, 3, 12, 5), (4, 1, 4, 3)]
    _row_shard_case(shapes, S, shard_dim, 22)


def test_row_shard_empty_homes_and_odd_alignment():
    # every param homed on rank 2: ranks 0, 1, 3 own nothing; odd element counts
    shapes = [(4, 3), (8, 5), (4, 7), (12, 1)]
    _row_shard_case(shapes, 4, 0, 23, home_of=[2, 2, 2, 2])


def test_row_shard_large_moe_slice():
    shapes = [(1408, 2048), (1408, 2048), (2048, 1408)] * 8
    _row_shard_case(shapes, 8, 0, 24)


def _flat_case(shapes, offsets, size, S, seed, owner_of=None):
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(seed)
    flat = (torch.randn(size, generator=g)).to(torch.bfloat16)
    flat_np = bits(flat)
    per = size // S
    plan = nsg.ns_plan_create_flat(shapes, offsets, size, S=S, owner_of=owner_of)
    owners = {i: h for i, h in enumerate(plan.homes()) if h >= 0}
    numels = [int(np.prod(s)) for s in shapes]
    ranks_np = [flat_np[r * per:(r + 1) * per] for r in range(S)]
    want = orr.flat_pack_to_owner(ranks_np, offsets, numels, size, S, owners)
    rank_t = [flat[r * per:(r + 1) * per].clone().to(dev) for r in range(S)]
    _, hs, _ = plan.home_layout()
    home_t = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    nsg.ns_pack_to_home(plan, rank_t, home_t)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for h in range(S):
        assert np.array_equal(bits(home_t[h])[:hs[h]], want[h])
    # unpack into buffers pre-filled with a marker: non-participating slots keep it
    marker = [torch.full((per,), 7.0, dtype=torch.bfloat16, device=dev) for _ in range(S)]
    nsg.ns_unpack_from_home(plan, home_t, marker)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    before = [bits(torch.full((per,), 7.0, dtype=torch.bfloat16)) for _ in range(S)]
    want_back = orr.flat_unpack_from_owner([bits(h)[:n] for h, n in zip(home_t, hs)], before, offsets,
                                           numels, size, S, owners)
    for r in range(S):
        assert np.array_equal(bits(marker[r]), want_back[r])


def test_flat_worked_example_on_gpu():
    _flat_case([(6, 4), (4, 4)], [0, 24], 40, 2, 31, owner_of=[1, 1])
    _flat_case([(6, 4), (4, 4)], [0, 24], 40, 2, 32)


@pytest.mark.parametrize("S", [2, 3, 5])
def test_flat_random(S):
    g = np.random.default_rng(S)
    shapes, offsets, pos = [], [], 0
    for _ in range(30):
        shp = (int(g.integers(1, 40)),) if g.random() < 0.2 else (int(g.integers(1, 60)), int(g.integers(1, 90)))
        pos += int(g.integers(0, 5))
        offsets.append(pos)
        shapes.append(shp)
        pos += int(np.prod(shp))
    size = ((pos + S - 1) // S) * S
    _flat_case(shapes, offsets, size, S, 40 + S)


@pytest.mark.parametrize("R,T", [(2, 2), (2, 4), (4, 2), (1, 4), (3, 1)])
def test_two_stage_fused_gather_equals_two_stages(R, T):
    # one fused gather on the GPU == GTP_remat stage (dim 0) then TP stage
    # (partition_dim), done literally by the oracle
    shapes = [(48, 24), (24, 48, 4), (96, 16), (24, 8, 8), (48, 12)]
    pd = [1, 1, 0, 2, 1]
    dev = torch.device("cuda:0")
    ts = workloads.gen_tensors(workloads.Workload("two", shapes, 1.0, 91))
    np_ts = [bits(t).reshape(t.shape) for t in ts]
    plan = nsg.ns_plan_create_two_stage(shapes, pd, R, T)
    S = R * T
    home_of = dict(enumerate(plan.homes()))
    ranks = orr.make_rank_buffers_two_stage(np_ts, R, T, pd)
    want = orr.route_two_stage(ranks, shapes, pd, home_of, R, T)
    rank_t = [torch.from_numpy(r.view(np.int16).copy()).view(torch.bfloat16).to(dev) for r in ranks]
    _, hs, _ = plan.home_layout()
    home_t = [torch.full((max(1, n),), -3.0, dtype=torch.bfloat16, device=dev) for n in hs]
    nsg.ns_pack_to_home(plan, rank_t, home_t)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for h in range(S):
        assert np.array_equal(bits(home_t[h])[:hs[h]], want[h])
    back = [torch.zeros_like(r) for r in rank_t]
    nsg.ns_unpack_from_home(plan, home_t, back)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    back_want = orr.route_two_stage_back(want, shapes, pd, home_of, R, T)
    for r in range(S):
        assert np.array_equal(bits(back[r]), back_want[r])


@pytest.mark.parametrize("n_waves", [1, 2, 3, 7])
def test_wave_pipeline_equals_serial_step(n_waves):
    # issue #6720 wave dispatch: the pipelined pack -> NS -> unpack must give
    # the serial result bit for bit
    w = workloads.gpt_24l_d2048()
    w.shapes = w.shapes[:8] + [(640, 384), (384, 640), (256, 64, 3, 3)]
    S, shapes = w.S, w.shapes
    dev = torch.device("cuda:0")
    ts = workloads.gen_tensors(w)
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=0)
    homes = plan.homes()
    ho, hs, rs = plan.home_layout()
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
    for _ in range(2):   # run twice: the second run reuses streams, events and workspaces
        nsg.ns_pipeline_run(pipe, rank_in, hi2, ho2, ro2, pws)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    # row shards along dim 0: the pipeline reads the rank buffers and its last
    # B*X launches write them, so the home buffers stay untouched
    for a in hi2 + ho2:
        assert not a.any()
    for a, b in zip(ro1, ro2):
        assert torch.equal(a, b)
    # and the result itself is right (sampled): tensor i rebuilt from its row
    # shards in the output rank buffers
    from gpu_util import BF16_TOL, oracle_ns, rel_err
    offs = [0]
    for t in ts:
        offs.append(offs[-1] + t.numel() // S)
    for i in (0, 3, len(shapes) - 1):
        y = torch.cat([ro2[r][offs[i]:offs[i + 1]] for r in range(S)]).reshape(ts[i].shape)
        assert rel_err(y, oracle_ns(ts[i])) <= BF16_TOL
        assert torch.equal(y, ho1[homes[i]][ho[i]:ho[i] + ts[i].numel()].reshape(ts[i].shape))


def _e2e_check(plan, shapes, ts, rank_in, S, participating, pipe_waves=0):
    from gpu_util import BF16_TOL, oracle_ns, rel_err
    dev = torch.device("cuda:0")
    homes = plan.homes()
    ho, hs, rs = plan.home_layout()
    home_in = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    home_out = [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs]
    rank_out = [torch.full_like(x, 5.0) for x in rank_in]
    if pipe_waves:
        pipe = nsg.ns_pipeline_create(plan, pipe_waves)
        ws = torch.empty(pipe.workspace_bytes, dtype=torch.uint8, device=dev)
        nsg.ns_pipeline_run(pipe, rank_in, home_in, home_out, rank_out, ws)
    else:
        part = [i for i in range(len(shapes)) if participating[i]]
        ws = torch.empty(max(1, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
        ins = [home_in[homes[i]].data_ptr() + 2 * ho[i] for i in part]
        outs = [home_out[homes[i]].data_ptr() + 2 * ho[i] for i in part]
        nsg.ns_pack_to_home(plan, rank_in, home_in)
        nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
        nsg.ns_unpack_from_home(plan, home_out, rank_out)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for i, t in enumerate(ts):
        if not participating[i]:
            continue
        y = home_out[homes[i]][ho[i]:ho[i] + t.numel()].reshape(t.shape)
        assert rel_err(y, oracle_ns(t)) <= BF16_TOL, i
    return home_out, rank_out


@pytest.mark.parametrize("waves", [0, 3])
def test_flat_model_pack_ns_unpack(waves):
    # owner_planning data model end to end: a flat buffer with 1-D (ineligible)
    # and padded gaps, owners by the default balancer
    g = np.random.default_rng(5)
    shapes, offsets, pos = [], [], 0
    for k in range(14):
        shp = (int(g.integers(8, 60)),) if k % 5 == 4 else (int(g.integers(16, 300)), int(g.integers(16, 300)))
        pos += int(g.integers(0, 9))
        offsets.append(pos)
        shapes.append(shp)
        pos += int(np.prod(shp))
    S = 4
    size = ((pos + S - 1) // S) * S
    dev = torch.device("cuda:0")
    flat = torch.zeros(size, dtype=torch.bfloat16)
    ts = []
    for i, (s, off) in enumerate(zip(shapes, offsets)):
        t = workloads.gen_tensor(s, 1.0, 95, i)
        ts.append(t)
        flat[off:off + t.numel()] = t.reshape(-1)
    per = size // S
    rank_in = [flat[r * per:(r + 1) * per].clone().to(dev) for r in range(S)]
    plan = nsg.ns_plan_create_flat(shapes, offsets, size, S=S)
    part = [len(s) >= 2 for s in shapes]
    home_out, rank_out = _e2e_check(plan, shapes, ts, rank_in, S, part, waves)
    # the scatter puts every result back at its flat position; others keep 5.0
    back = torch.cat([x.cpu() for x in rank_out])
    for i, (t, off) in enumerate(zip(ts, offsets)):
        if part[i]:
            homes = plan.homes()
            ho, _, _ = plan.home_layout()
            want = home_out[homes[i]][ho[i]:ho[i] + t.numel()].cpu()
            assert torch.equal(back[off:off + t.numel()], want)
        else:
            assert torch.all(back[off:off + t.numel()] == 5.0)


@pytest.mark.parametrize("waves", [0, 2])
def test_two_stage_model_pack_ns_unpack(waves):
    shapes = [(512, 256), (256, 512, 2), (1024, 128), (256, 64, 4)]
    pd = [1, 1, 0, 2]
    R, T = 2, 2
    ts = workloads.gen_tensors(workloads.Workload("tsn", shapes, 1.0, 96))
    np_ts = [bits(t).reshape(t.shape) for t in ts]
    dev = torch.device("cuda:0")
    ranks = orr.make_rank_buffers_two_stage(np_ts, R, T, pd)
    rank_in = [torch.from_numpy(r.view(np.int16).copy()).view(torch.bfloat16).to(dev) for r in ranks]
    plan = nsg.ns_plan_create_two_stage(shapes, pd, R, T)
    home_out, rank_out = _e2e_check(plan, shapes, ts, rank_in, R * T, [True] * len(shapes), waves)
    # unpack: every rank gets its two-stage piece of every result
    homes = plan.homes()
    full = orr.route_two_stage_back([bits(h) for h in home_out], shapes, pd, dict(enumerate(homes)), R, T)
    for r in range(R * T):
        assert np.array_equal(bits(rank_out[r]), full[r][:rank_out[r].numel()])


def _pipeline_vs_serial(shapes, S, shard_dim, n_waves, seed):
    """Run pack -> NS -> unpack as three serial calls and through the wave
    pipeline; the rank outputs must agree bit for bit. Returns both results."""
    dev = torch.device("cuda:0")
    ts = workloads.gen_tensors(workloads.Workload("pipe", shapes, 0.02, seed))
    plan = nsg.ns_plan_create(shapes, S=S, shard_dim=shard_dim)
    homes = plan.homes()
    ho, hs, rs = plan.home_layout()
    shards = [[_rank_piece(t, S, shard_dim, r) for t in ts] for r in range(S)]
    rank_in = [torch.cat(sh).to(dev) if sh else torch.zeros(1, dtype=torch.bfloat16, device=dev) for sh in shards]

    def bufs():
        return ([torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs],
                [torch.zeros(max(1, n), dtype=torch.bfloat16, device=dev) for n in hs],
                [torch.full_like(x, 7.0) for x in rank_in])

    hi1, ho1, ro1 = bufs()
    ws = torch.empty(max(1, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
    ins = [hi1[homes[i]].data_ptr() + 2 * ho[i] for i in range(len(shapes))]
    outs = [ho1[homes[i]].data_ptr() + 2 * ho[i] for i in range(len(shapes))]
    nsg.ns_pack_to_home(plan, rank_in, hi1)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    nsg.ns_unpack_from_home(plan, ho1, ro1)
    hi2, ho2, ro2 = bufs()
    pipe = nsg.ns_pipeline_create(plan, n_waves)
    pws = torch.empty(max(1, pipe.workspace_bytes), dtype=torch.uint8, device=dev)
    nsg.ns_pipeline_run(pipe, rank_in, hi2, ho2, ro2, pws)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for a, b in zip(ro1, ro2):
        assert torch.equal(a, b)
    return ts, ho1, homes, ho


def _rank_piece(t, S, shard_dim, r):
    # rank r's (…, D/S, …) slice of t along shard_dim, flattened (torch.chunk)
    return torch.chunk(t, S, dim=shard_dim)[r].contiguous().reshape(-1)


@pytest.mark.parametrize("n_waves", [1, 3])
def test_pipeline_ragged_shapes_fused_paths(n_waves):
    # row shards along dim 0 take the fused paths (prologue reading the rank
    # buffers, last B*X writing them); odd column counts and shard offsets
    # exercise the unaligned fallbacks of both, tall shapes the transposed ones
    from gpu_util import BF16_TOL, oracle_ns, rel_err
    shapes = [(8, 5), (16, 3), (24, 40), (40, 24), (8, 7, 3), (200, 130), (136, 72), (64, 64)]
    ts, ho1, homes, ho = _pipeline_vs_serial(shapes, 8, 0, n_waves, 91)
    for i, t in enumerate(ts):
        y = ho1[homes[i]][ho[i]:ho[i] + t.numel()].reshape(t.shape)
        assert rel_err(y, oracle_ns(t)) <= BF16_TOL, shapes[i]


def test_pipeline_shard_dim1_keeps_pack_and_unpack():
    # shards along dim 1 are not contiguous rows: the pipeline packs and
    # unpacks through the home buffers, with the same result as the serial calls
    _pipeline_vs_serial([(64, 256), (256, 64), (128, 128), (96, 32)], 4, 1, 2, 92)


def test_pipeline_with_no_participating_tensor_is_a_no_op():
    # a flat plan in which nothing participates: no waves, the run only orders
    # the streams and leaves every buffer as it was
    dev = torch.device("cuda:0")
    plan = nsg.ns_plan_create_flat([(4, 4)], [0], 16, participating=[False], S=2)
    pipe = nsg.ns_pipeline_create(plan, 2)
    assert pipe.n_waves == 0
    bufs = [torch.full((8,), float(r + 1), dtype=torch.bfloat16, device=dev) for r in range(2)]
    homes = [torch.full((1,), -1.0, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    out = [torch.zeros(8, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws = torch.empty(max(1, pipe.workspace_bytes), dtype=torch.uint8, device=dev)
    nsg.ns_pipeline_run(pipe, bufs, homes, homes, out, ws)
    torch.cuda.synchronize()
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for r in range(2):
        assert torch.equal(out[r], torch.zeros_like(out[r]))
        assert torch.equal(bufs[r], torch.full_like(bufs[r], float(r + 1)))
