"""Multi-rank host logic on CPU (world size 2, gloo, 127.0.0.1).

* Every rank builds the plan independently through the C ABI and gets the
  same homes and home layout (a real exchange needs all ranks to agree).
* The plan's all_to_allv splits and piece positions (ns_plan_rank_splits)
  drive a real all_to_all of the row shards (layer_sharded_a2a,
  route_to_ns_home on a 2-rank group): each home's reconstructed buffer
  equals the oracle's, bit for bit; the reverse all_to_all
  (route_from_ns_home, the same splits with the sides swapped) gives every
  rank its shards back.
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
        # the all_to_allv splits and piece positions come from the plan
        send_counts, send_displs, recv_counts, recv_displs, send_pos, recv_pos = plan.rank_splits(rank)
        shard = [int(np.prod(s)) // WORLD for s in w.shapes]
        off = np.concatenate([[0], np.cumsum(shard)])
        send = torch.zeros(sum(send_counts), dtype=torch.int32)
        for i in range(len(w.shapes)):
            send[send_pos[i]:send_pos[i] + shard[i]] = local[off[i]:off[i + 1]]
        recv = torch.zeros(sum(recv_counts), dtype=torch.int32)
        dist.all_to_all_single(recv, send, recv_counts, send_counts)
        # reconstruct the complete params homed here: pieces in rank order
        mine = [i for i in range(len(w.shapes)) if homes[i] == rank]
        home = np.concatenate([np.concatenate([recv[recv_pos[i][src]:recv_pos[i][src] + shard[i]].numpy()
                                               .reshape(w.shapes[i][0] // WORLD, -1) for src in range(WORLD)],
                                              axis=0).reshape(-1) for i in mine]) \
            if mine else np.zeros(0, np.int32)
        want = orr.route_to_ns_home(ranks, w.shapes, dict(enumerate(homes)), WORLD, 0)[rank]
        assert np.array_equal(home, want)
        assert home.size == hs[rank]

        # reverse exchange (route_from_ns_home): the same splits with the
        # sides swapped; every rank gets its shard of every param back
        back_send = torch.zeros(sum(recv_counts), dtype=torch.int32)
        for i in mine:
            full = torch.from_numpy(home[ho[i]:ho[i] + int(np.prod(w.shapes[i]))].copy()).reshape(WORLD, -1)
            for dst in range(WORLD):
                back_send[recv_pos[i][dst]:recv_pos[i][dst] + shard[i]] = full[dst]
        back_recv = torch.zeros(sum(send_counts), dtype=torch.int32)
        dist.all_to_all_single(back_recv, back_send, send_counts, recv_counts)
        back = torch.cat([back_recv[send_pos[i]:send_pos[i] + shard[i]] for i in range(len(w.shapes))])
        assert torch.equal(back, local)

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
            with open(err + f".{r}") as f:
                msgs.append(f.read())
    assert all(p.exitcode == 0 for p in procs), "\n".join(msgs)
