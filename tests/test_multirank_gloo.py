"""Multi-rank host logic on CPU (world size 2, gloo, 127.0.0.1).

* Every rank builds the plan independently through the C ABI and gets the
  same homes and home layout (a real exchange needs all ranks to agree).
* The plan's split sizes drive a real all_to_all of the row shards
  (layer_sharded_a2a, route_to_ns_home on a 2-rank group): each home's
  reconstructed buffer equals the oracle's, bit for bit; the reverse
  all_to_all (route_from_ns_home) gives every rank its shards back.
* The bench's max-over-ranks timing and whole-job value.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, port, errfile):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=WORLD)
        import bench
        import newton_schulz_shape_gb300 as nsg
        import workloads
        from oracle import routing as orr

        w = workloads.Workload("mr", [(8, 6), (4, 10), (12, 2), (6, 6), (2, 3, 4)], 1.0, 5)
        plan = nsg.ns_plan_create(w.shapes, S=WORLD, shard_dim=0)
        homes = plan.homes()
        ho, hs, rs = plan.home_layout()
        mine = torch.tensor(homes + ho + hs + rs, dtype=torch.int64)
        allp = [torch.zeros_like(mine) for _ in range(WORLD)]
        dist.all_gather(allp, mine)
        assert all(torch.equal(allp[0], x) for x in allp), "ranks disagree on the plan"

        # this rank's shards of every param (index order), as int16 bit patterns
        # gloo exchanges int32: carry the bf16 bit patterns widened to int32
        ts = [t.view(torch.int16).numpy().astype(np.int32) for t in workloads.gen_tensors(w)]
        ranks = orr.make_rank_buffers(ts, WORLD, 0)
        local = torch.from_numpy(ranks[rank].copy())
        # send split to home h: this rank's shards of the params homed on h
        shard = [int(np.prod(s)) // WORLD for s in w.shapes]
        send_idx = [[i for i in range(len(w.shapes)) if homes[i] == h] for h in range(WORLD)]
        off = np.concatenate([[0], np.cumsum(shard)])
        send = torch.cat([torch.cat([local[off[i]:off[i + 1]] for i in send_idx[h]]) if send_idx[h]
                          else torch.zeros(0, dtype=torch.int32) for h in range(WORLD)])
        in_splits = [sum(shard[i] for i in send_idx[rank])] * WORLD
        out_splits = [sum(shard[i] for i in send_idx[h]) for h in range(WORLD)]
        recv = torch.zeros(sum(in_splits), dtype=torch.int32)
        dist.all_to_all_single(recv, send, in_splits, out_splits)
        # reconstruct the complete params homed here: shards in rank order
        parts, pos = {i: [] for i in send_idx[rank]}, 0
        for src in range(WORLD):
            for i in send_idx[rank]:
                parts[i].append(recv[pos:pos + shard[i]].numpy())
                pos += shard[i]
        home = np.concatenate([np.concatenate([p.reshape(w.shapes[i][0] // WORLD, -1) for p in parts[i]],
                                              axis=0).reshape(-1) for i in send_idx[rank]]) \
            if send_idx[rank] else np.zeros(0, np.int32)
        want = orr.route_to_ns_home(ranks, w.shapes, dict(enumerate(homes)), WORLD, 0)[rank]
        assert np.array_equal(home, want)
        assert home.size == hs[rank]

        # reverse exchange: every rank gets its shard of every param back
        back_send = torch.cat([torch.from_numpy(home[ho[i]:ho[i] + int(np.prod(w.shapes[i]))].copy())
                               .reshape(WORLD, -1)[dst] for dst in range(WORLD) for i in send_idx[rank]]) \
            if send_idx[rank] else torch.zeros(0, dtype=torch.int32)
        back = torch.zeros(local.numel(), dtype=torch.int32)
        dist.all_to_all_single(back, back_send, out_splits, in_splits)
        got, pos = {}, 0
        for h in range(WORLD):
            for i in send_idx[h]:
                got[i] = back[pos:pos + shard[i]]
                pos += shard[i]
        assert torch.equal(torch.cat([got[i] for i in range(len(w.shapes))]), local)

        # bench aggregation: max over ranks, whole-job value
        t = bench.max_over_ranks(10.0 + rank, WORLD)
        assert t == 10.0 + WORLD - 1
        assert bench.job_value(96, WORLD, t) == 96 * WORLD * 1000.0 / t
        assert bench.replica_seed(2000, rank, WORLD) != bench.replica_seed(2000, 1 - rank, WORLD)
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover
        import traceback
        with open(errfile + f".{rank}", "w") as f:
            f.write(traceback.format_exc())
        raise


def test_two_rank_plan_agreement_exchange_and_timing(tmp_path):
    nsg = pytest.importorskip("newton_schulz_shape_gb300")  # noqa: F841
    err = str(tmp_path / "err")
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, err)) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    msgs = []
    for r in range(WORLD):
        if os.path.exists(err + f".{r}"):
            msgs.append(open(err + f".{r}").read())
    assert all(p.exitcode == 0 for p in procs), "\n".join(msgs)
