"""Parity of the exact call bench.py times, at full size, on every matrix.

bench.py's step is ``ns_pipeline_run`` with 2 waves over a row-shard plan
(S = 8 simulated ranks, shard_dim 0, LPT homes): the rank buffers go in, the
prologue reads them directly, and the last B*X launches of each wave write the
results straight back into the output rank buffers. These tests make that
call with the bench's buffers and check its results:

  * GPT-style 24 layers (96 matrices, 2.42 GB): every matrix, rebuilt from its
    8 row shards in the output rank buffers, against the float64 oracle
    (relative Frobenius error <= 3e-2), with the oracle spread over the host
    cores; and the pipelined result equals the serial pack -> NS -> unpack
    calls bit for bit;
  * MoE 16 layers x 64 experts x 3 (3072 matrices, 17.7 GB): per layer one
    gate, one up and one down matrix (a different expert in every layer)
    against the oracle, and every matrix finite with ||Y||_F / sqrt(m) inside
    the band the 5-step map allows.
"""

import concurrent.futures as cf

import numpy as np
import pytest
import torch

import workloads
from gpu_util import BF16_TOL, bits
from oracle_pool import OraclePool

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")

WAVES = 2   # bench.py's default


def _inputs(w, keep):
    """Rank buffers of the workload on the GPU (rank r: its row shard of every
    tensor, in index order) and the bf16 bits of the tensors in `keep`."""
    dev = torch.device("cuda:0")
    S, shapes = w.S, w.shapes
    numels = [int(np.prod(s)) for s in shapes]
    L = sum(numels) // S
    rank_in = [torch.empty(L, dtype=torch.bfloat16, device=dev) for _ in range(S)]
    offs = np.concatenate([[0], np.cumsum([n // S for n in numels])]).astype(np.int64)
    kept = {}
    gen = lambda i: workloads.gen_tensor(shapes[i], w.sigma, w.seed, i)  # noqa: E731
    with cf.ThreadPoolExecutor(8) as ex:
        for i, t in enumerate(ex.map(gen, range(len(shapes)))):
            sh = t.reshape(S, -1).to(dev)
            for r in range(S):
                rank_in[r][offs[i]:offs[i + 1]].copy_(sh[r])
            if i in keep:
                kept[i] = bits(t).reshape(-1)
    return rank_in, offs, kept


def _bench_call(w, rank_in, waves=WAVES):
    """ns_pipeline_run exactly as bench.py makes it; returns the output rank buffers."""
    dev = torch.device("cuda:0")
    plan = nsg.ns_plan_create(w.shapes, steps=workloads.STEPS, eps=workloads.EPS, S=w.S, shard_dim=0)
    _, home_sizes, rank_sizes = plan.home_layout()
    assert rank_sizes[0] == rank_in[0].numel()
    home_in = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in home_sizes]
    home_out = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in home_sizes]
    rank_out = [torch.full_like(x, float("nan")) for x in rank_in]
    pipe = nsg.ns_pipeline_create(plan, waves)
    assert pipe.n_waves == waves
    ws = torch.empty(pipe.workspace_bytes, dtype=torch.uint8, device=dev)
    nsg.ns_pipeline_run(pipe, rank_in, home_in, home_out, rank_out, ws)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    del ws, home_in, home_out
    return plan, rank_out


def _result_bits(rank_out, offs, i, S):
    """Tensor i's result rebuilt from its row shards (bf16 bits, row-major)."""
    return np.concatenate([bits(rank_out[r][offs[i]:offs[i + 1]]) for r in range(S)])


def _job(w, i, in_bits, out_bits):
    return (i, tuple(w.shapes[i]), in_bits, out_bits, workloads.STEPS, workloads.A_COEF, workloads.B_COEF,
            workloads.C_COEF, workloads.EPS, 0.0)


def test_gpt_24l_bench_call_every_matrix():
    w = workloads.gpt_24l_d2048()
    S, n = w.S, len(w.shapes)
    rank_in, offs, kept = _inputs(w, keep=set(range(n)))
    plan, rank_out = _bench_call(w, rank_in)

    # the serial calls (pack, NS, unpack) give the same bits
    dev = torch.device("cuda:0")
    homes = plan.homes()
    ho, hs, _ = plan.home_layout()
    home_in = [torch.empty(max(1, k), dtype=torch.bfloat16, device=dev) for k in hs]
    home_out = [torch.empty(max(1, k), dtype=torch.bfloat16, device=dev) for k in hs]
    serial_out = [torch.empty_like(x) for x in rank_in]
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ins = [home_in[homes[i]].data_ptr() + 2 * ho[i] for i in range(n)]
    outs = [home_out[homes[i]].data_ptr() + 2 * ho[i] for i in range(n)]
    nsg.ns_pack_to_home(plan, rank_in, home_in)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    nsg.ns_unpack_from_home(plan, home_out, serial_out)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    for a, b in zip(rank_out, serial_out):
        assert torch.equal(a, b)
    del ws, home_in, home_out, serial_out

    jobs = [_job(w, i, kept[i], _result_bits(rank_out, offs, i, S)) for i in range(n)]
    del rank_in, rank_out
    with OraclePool() as pool:
        errs = pool.errors(jobs)
    assert len(errs) == n
    bad = {i: e for i, e in errs.items() if not e <= BF16_TOL}
    assert not bad, bad
    assert max(errs.values()) > 1e-3   # bf16 rounding is visible: the comparison is real


def _moe_sample(w):
    """Per layer: one gate, one up and one down matrix, of expert (5 * layer) % 64."""
    per_layer = 64 * 3
    out = []
    for layer in range(len(w.shapes) // per_layer):
        e = (5 * layer) % 64
        base = layer * per_layer + 3 * e
        out += [base, base + 1, base + 2]
    return out


def test_moe_16l_64e_bench_call():
    w = workloads.moe_16l_64e()
    S, n = w.S, len(w.shapes)
    sample = _moe_sample(w)
    assert len(sample) == 48 and {w.shapes[i] for i in sample} == {(1408, 2048), (2048, 1408)}
    rank_in, offs, kept = _inputs(w, keep=set(sample))
    plan, rank_out = _bench_call(w, rank_in)
    del rank_in

    # every matrix: finite, and ||Y||_F / sqrt(m) in the 5-step map's band;
    # every tensor has the same numel, so a rank buffer is a (n, numel / S) array
    shard = int(np.prod(w.shapes[0])) // S
    sq = torch.zeros(n, dtype=torch.float64, device="cuda")
    for r in range(S):
        v = rank_out[r].view(n, shard)
        assert torch.isfinite(v).all(), r
        sq += v.double().square().sum(dim=1)
    f = (sq / 1408.0).sqrt()
    assert bool(((f > 0.5) & (f < 1.2)).all()), (float(f.min()), float(f.max()))

    jobs = [_job(w, i, kept[i], _result_bits(rank_out, offs, i, S)) for i in sample]
    with OraclePool() as pool:
        errs = pool.errors(jobs)
    bad = {i: e for i, e in errs.items() if not e <= BF16_TOL}
    assert not bad, bad
