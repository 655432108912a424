"""GPU parity of shape-batched Newton-Schulz against the float64 oracle.

Bar (per matrix): relative Frobenius error <= 3e-2 on the bf16 path. Inputs
are the seeded bf16 Gaussians of ``workloads``; the oracle sees the same bf16
values in float64. Sizes span several 128 x 256 tiles and ragged tails, plus
the degenerate cases (zero matrix, zero-size tensor, empty batch, in-place).
"""

import numpy as np
import pytest
import torch

import workloads
from gpu_util import BF16_TOL, oracle_ns, rel_err, run_ns

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")


def test_small_16x128x256_all_matrices():
    w = workloads.small_16x128x256()
    ts = workloads.gen_tensors(w)
    outs = run_ns(nsg, w.shapes, ts)
    for t, o in zip(ts, outs):
        assert o.shape == t.shape and o.dtype == torch.bfloat16
        assert rel_err(o, oracle_ns(t)) <= BF16_TOL


RAGGED = [(300, 700), (700, 300), (256, 64, 3, 3), (130, 130), (64, 1000), (5, 3), (1, 9), (9, 1),
          (200, 456), (456, 200), (128, 64), (384, 640)]


def test_ragged_mixed_buckets():
    shapes = RAGGED
    w = workloads.Workload("ragged", shapes, 1.0, 11)
    ts = workloads.gen_tensors(w)
    outs = run_ns(nsg, shapes, ts)
    for s, t, o in zip(shapes, ts, outs):
        assert o.shape == t.shape
        err = rel_err(o, oracle_ns(t))
        assert err <= BF16_TOL, (s, err)


@pytest.mark.parametrize("steps", [0, 1, 3])
def test_step_counts(steps):
    shapes = [(192, 320), (320, 192)]
    ts = workloads.gen_tensors(workloads.Workload("steps", shapes, 0.02, 12))
    outs = run_ns(nsg, shapes, ts, steps=steps)
    for t, o in zip(ts, outs):
        assert rel_err(o, oracle_ns(t, steps)) <= BF16_TOL


def test_many_matrices_one_bucket():
    shapes = [(256, 512)] * 40
    ts = workloads.gen_tensors(workloads.Workload("many", shapes, 0.02, 13))
    outs = run_ns(nsg, shapes, ts)
    for i in (0, 17, 39):
        assert rel_err(outs[i], oracle_ns(ts[i])) <= BF16_TOL


def test_in_place():
    shapes = [(128, 384), (384, 128)]
    ts = workloads.gen_tensors(workloads.Workload("inplace", shapes, 1.0, 14))
    outs = run_ns(nsg, shapes, [t.clone() for t in ts], inplace=True)
    for t, o in zip(ts, outs):
        assert rel_err(o, oracle_ns(t)) <= BF16_TOL


def test_degenerate():
    shapes = [(64, 96), (0, 5), (7, 0, 3), (16, 16)]
    ts = [torch.zeros(64, 96, dtype=torch.bfloat16), torch.zeros(0, 5, dtype=torch.bfloat16),
          torch.zeros(7, 0, 3, dtype=torch.bfloat16),
          workloads.gen_tensor((16, 16), 1.0, 15, 0)]
    outs = run_ns(nsg, shapes, ts)
    assert torch.all(outs[0] == 0)
    assert outs[1].numel() == 0 and outs[2].numel() == 0
    assert rel_err(outs[3], oracle_ns(ts[3])) <= BF16_TOL
    # empty batch
    plan = nsg.ns_plan_create([], S=1)
    nsg.ns_orthogonalize_batched(plan, [], [], None, 0)


def test_bad_workspace_rejected():
    plan = nsg.ns_plan_create([(128, 256)], S=1)
    x = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(nsg.NsError) as e:
        nsg.ns_orthogonalize_batched(plan, [x], [x], small)
    assert e.value.code == nsg.NS_ERR_WORKSPACE


def test_repeatable_bitwise():
    shapes = [(256, 768)] * 4
    ts = workloads.gen_tensors(workloads.Workload("rep", shapes, 0.02, 16))
    a = run_ns(nsg, shapes, ts)
    b = run_ns(nsg, shapes, ts)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("cl", [0, 1, 3])
def test_cluster_pairs_odd_tile_rows(cl):
    # m_pad = 384, 384, 640: odd tile-row counts leave a spare CTA in the last pair
    shapes = [(300, 700), (700, 300), (640, 960), (256, 256)]
    ts = workloads.gen_tensors(workloads.Workload("odd", shapes, 0.02, 17))
    nsg.ns_set_gemm_cluster(cl)
    try:
        outs = run_ns(nsg, shapes, ts)
    finally:
        nsg.ns_set_gemm_cluster(0)
    for s_, t, o in zip(shapes, ts, outs):
        assert rel_err(o, oracle_ns(t)) <= BF16_TOL, (cl, s_)


@pytest.mark.parametrize("cl", [0, 1, 3])
def test_symmetric_store_modes_agree(cl):
    # A and B stored as upper pair blocks (readers take the rest transposed)
    # or with their mirror (readers take rows): the same products in the same
    # K order, so bitwise-equal results; odd and even tile-row counts, one and
    # several pair rows, two buckets in one launch
    shapes = [(300, 700), (700, 300), (640, 960), (1024, 3072), (2048, 1024), (256, 256)]
    ts = workloads.gen_tensors(workloads.Workload("symstore", shapes, 0.02, 23))
    nsg.ns_set_gemm_cluster(cl)
    try:
        nsg.ns_set_symmetric_store(1)
        a = run_ns(nsg, shapes, ts)
        nsg.ns_set_symmetric_store(0)
        b = run_ns(nsg, shapes, ts)
    finally:
        nsg.ns_set_symmetric_store(0)
        nsg.ns_set_gemm_cluster(0)
    for s_, x, y in zip(shapes, a, b):
        assert torch.equal(x, y), (cl, s_)
    for s_, t, y in zip(shapes[:3], ts, b):
        assert rel_err(y, oracle_ns(t)) <= BF16_TOL, (cl, s_)


@pytest.mark.parametrize("cl", [3])
def test_cluster_and_single_cta_agree(cl):
    shapes = [(1024, 3072), (2048, 1024)]
    ts = workloads.gen_tensors(workloads.Workload("agree", shapes, 0.02, 18))
    nsg.ns_set_gemm_cluster(1)
    try:
        a = run_ns(nsg, shapes, ts)
        nsg.ns_set_gemm_cluster(cl)
        b = run_ns(nsg, shapes, ts)
    finally:
        nsg.ns_set_gemm_cluster(0)
    for x, y in zip(a, b):
        # the same products in the same K order: bitwise equal
        assert torch.equal(x, y)
