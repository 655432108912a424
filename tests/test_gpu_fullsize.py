"""Parity at full workload sizes, in the launch configuration bench.py times.

The whole workload runs as pack (S = 8 row shards -> LPT homes) -> shape-
batched Newton-Schulz -> unpack. The float64 oracle then checks sampled
matrices (one per (m, n) bucket, first and last tensor):
  * pack: the home buffer holds the complete tensor, bit for bit;
  * NS: per-matrix relative Frobenius error <= 3e-2;
  * unpack: every rank buffer holds its shard of the result, bit for bit.
Every matrix is also checked for properties that hold at any size: finite,
and ||Y||_F / sqrt(m) inside the band the 5-step map allows for these inputs.
At the sweep's largest size, where the oracle cannot run in seconds, a
structured input with orthogonal rows is checked against its closed form
(tied to the oracle on small sizes by test_closed_form_inputs.py).
"""

import math

import numpy as np
import pytest
import torch

import workloads
from closed_forms import hadamard_row_norms, row_gains
from gpu_util import BF16_TOL, bits, oracle_ns, rel_err

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")


def view_mn(s):
    c = int(np.prod(s[1:]))
    return min(s[0], c), max(s[0], c)


def run_pipeline(w, sample=None):
    dev = torch.device("cuda:0")
    S, shapes = w.S, w.shapes
    plan = nsg.ns_plan_create(shapes, steps=workloads.STEPS, eps=workloads.EPS, S=S, shard_dim=0)
    home_off, home_sizes, rank_sizes = plan.home_layout()
    homes = plan.homes()
    L = rank_sizes[0]
    if sample is None:
        seen, sample = set(), [0, len(shapes) - 1]
        for i, s in enumerate(shapes):
            if view_mn(s) not in seen:
                seen.add(view_mn(s))
                sample.append(i)
        sample = sorted(set(sample))
    rank_in = [torch.empty(L, dtype=torch.bfloat16, device=dev) for _ in range(S)]
    rank_off, kept, pos = [], {}, 0
    for i, s in enumerate(shapes):
        t = workloads.gen_tensor(s, w.sigma, w.seed, i)
        if i in sample:
            kept[i] = t
        n = t.numel() // S
        sh = t.reshape(S, n).to(dev)
        for r in range(S):
            rank_in[r][pos:pos + n].copy_(sh[r])
        rank_off.append(pos)
        pos += n
    home_in = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in home_sizes]
    home_out = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in home_sizes]
    rank_out = [torch.empty(L, dtype=torch.bfloat16, device=dev) for _ in range(S)]
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ins = [home_in[homes[i]].data_ptr() + 2 * home_off[i] for i in range(len(shapes))]
    outs = [home_out[homes[i]].data_ptr() + 2 * home_off[i] for i in range(len(shapes))]
    nsg.ns_pack_to_home(plan, rank_in, home_in)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    nsg.ns_unpack_from_home(plan, home_out, rank_out)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    del ws

    # properties of every matrix
    for i, s in enumerate(shapes):
        n_el = int(np.prod(s))
        y = home_out[homes[i]][home_off[i]:home_off[i] + n_el].float()
        assert torch.isfinite(y).all(), i
        m, _ = view_mn(s)
        f = float(torch.linalg.vector_norm(y)) / np.sqrt(m)
        assert 0.5 < f < 1.2, (i, s, f)

    # sampled matrices against the oracle
    for i in sample:
        s = shapes[i]
        t = kept[i]
        n_el = t.numel()
        h = homes[i]
        got_in = home_in[h][home_off[i]:home_off[i] + n_el]
        assert np.array_equal(bits(got_in), bits(t).reshape(-1)), ("pack", i)
        y = home_out[h][home_off[i]:home_off[i] + n_el]
        err = rel_err(y.reshape(s), oracle_ns(t))
        assert err <= BF16_TOL, ("ns", i, s, err)
        ysh = bits(y).reshape(S, -1)
        for r in range(S):
            got = bits(rank_out[r][rank_off[i]:rank_off[i] + n_el // S])
            assert np.array_equal(got, ysh[r]), ("unpack", i, r)
    return plan


def test_gpt_24l_d2048_full():
    run_pipeline(workloads.gpt_24l_d2048())


def test_llama8b_32l_full():
    run_pipeline(workloads.llama8b_32l())


def test_moe_full_size_matrices_two_layers():
    w = workloads.moe_16l_64e()
    w.shapes = w.shapes[:2 * 64 * 3]          # 384 matrices at the workload's full per-matrix size
    run_pipeline(w, sample=[0, 1, 2, 191, 383])


@pytest.mark.parametrize("m,aspect", [(1024, 1), (1024, 8), (2048, 2), (4096, 4)])
def test_sweep_points(m, aspect):
    w = workloads.sweep_shapes(m, aspect, 2)
    w.shapes = [w.shapes[0], (aspect * m, m)]   # one wide, one tall (exercises the transpose back)
    run_pipeline(w, sample=[0, 1])


def test_sweep_conv_3d():
    run_pipeline(workloads.conv_3d(), sample=[0, 31, 63])


def test_sweep_8192_square():
    w = workloads.sweep_shapes(8192, 1, 1)
    run_pipeline(w, sample=[0])


@pytest.mark.parametrize("mode", ["bf16", "fp32_auto"])
def test_max_sweep_size_closed_form(mode):
    # the sweep's largest matrix, 8192 x 65536 (1 GiB of bf16), wide and tall
    # in one batch, against the closed form NS_k(X)_i = g_i X_i of an input
    # with orthogonal rows. Checked per matrix (relative Frobenius error, the
    # policy's bar) and per 128 x 256 output tile, so that one wrong tile
    # anywhere in the 2^29 elements fails. fp32_auto runs these shapes in Gram
    # space (n = 8m).
    gram_mode, odt, tol, tile_tol = {"bf16": (nsg.NS_BF16, torch.bfloat16, BF16_TOL, 0.1),
                                     "fp32_auto": (nsg.NS_FP32_AUTO, torch.float32, 1e-3, 1e-2)}[mode]
    dev = torch.device("cuda:0")
    m, blocks = 8192, 8
    x, r, d = workloads.gen_hadamard_rows(m, blocks, seed=5807, device="cuda")
    shapes = [(m, m * blocks), (m * blocks, m)]
    ins = [x, x.t().contiguous()]
    outs = [torch.empty(t.shape, dtype=odt, device=dev) for t in ins]
    plan = nsg.ns_plan_create(shapes, steps=workloads.STEPS, eps=workloads.EPS, gram_mode=gram_mode, S=1)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    del ws
    g = torch.tensor(row_gains(hadamard_row_norms(m, r, d), workloads.STEPS, workloads.A_COEF,
                               workloads.B_COEF, workloads.C_COEF, workloads.EPS),
                     dtype=torch.float64, device=dev)
    for y, tall in zip(outs, (False, True)):
        yw = y.t() if tall else y
        num = den = 0.0
        worst_tile = 0.0
        for i0 in range(0, m, 1024):
            want = g[i0:i0 + 1024, None] * x[i0:i0 + 1024].double()
            diff = yw[i0:i0 + 1024].double() - want
            num += float(diff.square().sum())
            den += float(want.square().sum())
            dt = diff.square().reshape(8, 128, -1, 256).sum(dim=(1, 3))
            wt = want.square().reshape(8, 128, -1, 256).sum(dim=(1, 3))
            worst_tile = max(worst_tile, float((dt / wt).sqrt().max()))
            del want, diff
        err = math.sqrt(num / den)
        assert err <= tol, (mode, tall, err)
        assert worst_tile <= tile_tol, (mode, tall, worst_tile)
