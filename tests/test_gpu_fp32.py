"""GPU parity of the fp32-Gram path (NS_FP32_GRAM) against the float64 oracle.

Bar (per matrix): relative Frobenius error <= 1e-3. Inputs are bf16 (the
momentum shards the pack moves); results are fp32. The trace ridge is
compared with the oracle's reading of it, A <- A + ridge * (tr A / m) * I
before B is formed (parity unpinned: the pages do not fix the form).
"""

import pytest
import torch

import workloads
from gpu_util import oracle_ns, rel_err
from oracle import ns as ons

pytestmark = pytest.mark.gpu
nsg = pytest.importorskip("newton_schulz_shape_gb300")

FP32_TOL = 1e-3


def run_f32(shapes, ts, steps=workloads.STEPS, ridge=0.0):
    dev = torch.device("cuda:0")
    ins = [t.to(dev) for t in ts]
    outs = [torch.full(t.shape, float("nan"), dtype=torch.float32, device=dev) for t in ins]
    plan = nsg.ns_plan_create(shapes, steps=steps, eps=workloads.EPS, gram_mode=nsg.NS_FP32_GRAM, ridge=ridge, S=1)
    assert plan.out_bytes == 4
    ws = torch.empty(max(1, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    rc = nsg.ns_check_status(plan)
    assert rc == nsg.NS_OK, nsg.ns_status_string(rc)
    return outs


def oracle(t, steps=workloads.STEPS, ridge=0.0):
    return ons.newton_schulz(t.float().numpy(), steps, workloads.A_COEF, workloads.B_COEF, workloads.C_COEF,
                             workloads.EPS, ridge=ridge)


SHAPES = [(128, 256), (128, 256), (300, 700), (700, 300), (256, 64, 3, 3), (130, 130), (5, 3), (200, 456)]


def test_fp32_gram_small_and_ragged():
    ts = workloads.gen_tensors(workloads.Workload("f32", SHAPES, 1.0, 71))
    outs = run_f32(SHAPES, ts)
    for s, t, o in zip(SHAPES, ts, outs):
        assert o.dtype == torch.float32 and o.shape == t.shape
        err = rel_err(o, oracle(t))
        assert err <= FP32_TOL, (s, err)


@pytest.mark.parametrize("steps", [0, 1, 3])
def test_fp32_gram_step_counts(steps):
    shapes = [(192, 320), (320, 192)]
    ts = workloads.gen_tensors(workloads.Workload("f32s", shapes, 0.02, 72))
    outs = run_f32(shapes, ts, steps=steps)
    for t, o in zip(ts, outs):
        assert rel_err(o, oracle(t, steps)) <= FP32_TOL


@pytest.mark.parametrize("ridge", [1e-5, 1e-3])
def test_fp32_gram_trace_ridge(ridge):
    shapes = [(256, 512), (512, 256), (100, 300)]
    ts = workloads.gen_tensors(workloads.Workload("ridge", shapes, 0.02, 73))
    outs = run_f32(shapes, ts, ridge=ridge)
    for t, o in zip(ts, outs):
        assert rel_err(o, oracle(t, ridge=ridge)) <= FP32_TOL
        # the ridge moves the result measurably at 1e-3
        if ridge >= 1e-3:
            assert rel_err(o, oracle(t)) > 5 * rel_err(o, oracle(t, ridge=ridge))


def test_fp32_gram_sweep_sizes():
    shapes = [(1024, 2048), (2048, 1024), (1024, 1024)]
    ts = workloads.gen_tensors(workloads.Workload("f32big", shapes, 0.02, 74))
    outs = run_f32(shapes, ts)
    for s, t, o in zip(shapes, ts, outs):
        assert rel_err(o, oracle(t)) <= FP32_TOL, s


def test_fp32_gram_beats_bf16_path():
    shapes = [(256, 768)]
    ts = workloads.gen_tensors(workloads.Workload("cmp", shapes, 0.02, 75))
    ref = oracle(ts[0])
    f32 = rel_err(run_f32(shapes, ts)[0], ref)
    dev = torch.device("cuda:0")
    x = ts[0].to(dev)
    y = torch.empty_like(x)
    plan = nsg.ns_plan_create(shapes, S=1)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    nsg.ns_orthogonalize_batched(plan, [x], [y], ws)
    bf16 = rel_err(y, ref)
    assert f32 < bf16 / 10, (f32, bf16)


def run_mode(shapes, ts, mode, steps=workloads.STEPS, ridge=0.0):
    dev = torch.device("cuda:0")
    ins = [t.to(dev) for t in ts]
    outs = [torch.full(t.shape, float("nan"), dtype=torch.float32, device=dev) for t in ins]
    plan = nsg.ns_plan_create(shapes, steps=steps, eps=workloads.EPS, gram_mode=mode, ridge=ridge, S=1)
    ws = torch.empty(max(1, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    rc = nsg.ns_check_status(plan)
    assert rc == nsg.NS_OK, nsg.ns_status_string(rc)
    return outs


# Gram-space NS (issue #6720's gram_once): the same iteration carried on m x m
# matrices; the result must match the oracle of the standard iteration.
GS_SHAPES = [(128, 512), (512, 128), (256, 64, 3, 3), (200, 900), (130, 130), (5, 3)]


def test_gram_space_matches_oracle():
    ts = workloads.gen_tensors(workloads.Workload("gs", GS_SHAPES, 1.0, 81))
    outs = run_mode(GS_SHAPES, ts, nsg.NS_FP32_GRAM_SPACE)
    for s, t, o in zip(GS_SHAPES, ts, outs):
        assert o.shape == t.shape
        err = rel_err(o, oracle(t))
        assert err <= FP32_TOL, (s, err)


@pytest.mark.parametrize("steps", [1, 2, 5])
def test_gram_space_step_counts(steps):
    shapes = [(256, 1024), (1024, 256)]
    ts = workloads.gen_tensors(workloads.Workload("gss", shapes, 0.02, 82))
    outs = run_mode(shapes, ts, nsg.NS_FP32_GRAM_SPACE, steps=steps)
    for t, o in zip(ts, outs):
        assert rel_err(o, oracle(t, steps)) <= FP32_TOL


@pytest.mark.parametrize("ridge", [1e-5, 1e-3])
def test_gram_space_trace_ridge(ridge):
    shapes = [(256, 1024), (300, 800)]
    ts = workloads.gen_tensors(workloads.Workload("gsr", shapes, 0.02, 83))
    outs = run_mode(shapes, ts, nsg.NS_FP32_GRAM_SPACE, ridge=ridge)
    for t, o in zip(ts, outs):
        assert rel_err(o, oracle(t, ridge=ridge)) <= FP32_TOL


def test_gram_space_agrees_with_fp32_gram_path():
    shapes = [(1024, 4096), (2048, 2048)]
    ts = workloads.gen_tensors(workloads.Workload("gsa", shapes, 0.02, 84))
    a = run_mode(shapes, ts, nsg.NS_FP32_GRAM_SPACE)
    b = run_mode(shapes, ts, nsg.NS_FP32_GRAM)
    for t, x, y in zip(ts, a, b):
        assert rel_err(x, y.cpu().numpy()) <= FP32_TOL
        assert rel_err(x, oracle(t)) <= FP32_TOL


# NS_FP32_AUTO: per shape bucket, Gram space when n >= 2m, else the standard
# fp32-Gram iteration. Each matrix must come out bit for bit as in the plan of
# the mode its bucket was given, and within the fp32 bar of the oracle.
AUTO_SHAPES = [(256, 1024), (1024, 256), (300, 300), (200, 350), (128, 2048), (130, 130)]


def test_fp32_auto_matches_the_mode_of_each_bucket():
    ts = workloads.gen_tensors(workloads.Workload("auto", AUTO_SHAPES, 0.02, 85))
    auto = run_mode(AUTO_SHAPES, ts, nsg.NS_FP32_AUTO)
    for s, t, o in zip(AUTO_SHAPES, ts, auto):
        r, c = s[0], s[1]
        m, n = min(r, c), max(r, c)
        mode = nsg.NS_FP32_GRAM_SPACE if n >= 2 * m else nsg.NS_FP32_GRAM
        alone = run_mode([s], [t], mode)[0]
        assert torch.equal(o.cpu(), alone.cpu()), s
        assert rel_err(o, oracle(t)) <= FP32_TOL, s


# Full sweep sizes (the size/aspect sweep's points, whole batches as the
# sweep runs them): every matrix finite with ||Y||_F / sqrt(m) in the 5-step
# band, the first of the batch against the oracle at the fp32 bar.
SWEEP_BATCH = {(m, a): bt for m, a, bt in workloads.sweep_points()}


@pytest.mark.parametrize("m,aspect,mode", [(4096, 1, nsg.NS_FP32_GRAM), (4096, 4, nsg.NS_FP32_AUTO),
                                           (8192, 1, nsg.NS_FP32_GRAM), (2048, 8, nsg.NS_FP32_AUTO)])
def test_fp32_sweep_points_full_size(m, aspect, mode):
    w = workloads.sweep_shapes(m, aspect, SWEEP_BATCH[(m, aspect)])
    ts = workloads.gen_tensors(w, indices=[0])
    dev = torch.device("cuda:0")
    # the batch's other matrices come from the same generator, on the GPU side only
    ins = [ts[0].to(dev)] + [workloads.gen_tensor(s, w.sigma, w.seed, i).to(dev)
                             for i, s in enumerate(w.shapes) if i > 0]
    outs = [torch.full(t.shape, float("nan"), dtype=torch.float32, device=dev) for t in ins]
    plan = nsg.ns_plan_create(w.shapes, steps=workloads.STEPS, eps=workloads.EPS, gram_mode=mode, S=1)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    assert nsg.ns_check_status(plan) == nsg.NS_OK
    del ws
    for i, o in enumerate(outs):
        assert torch.isfinite(o).all(), i
        f = float(torch.linalg.vector_norm(o.double())) / m ** 0.5
        assert 0.5 < f < 1.2, (i, f)
    err = rel_err(outs[0], oracle(ts[0]))
    assert err <= FP32_TOL, (m, aspect, err)


# The fp32 products run on CTA pairs (2-SM MMA) when every bucket of a launch
# has two or more 128-row tiles; ns_set_gemm_cluster(1) forces one CTA per
# tile. Same products in the same K order: identical bits. Odd tile-row
# counts (m_pad = 384, 640; n_pad = 640, 1152) leave a spare half pair.
@pytest.mark.parametrize("mode", [nsg.NS_FP32_GRAM, nsg.NS_FP32_GRAM_SPACE, nsg.NS_FP32_AUTO])
def test_fp32_pairs_equal_single_cta(mode):
    shapes = [(384, 640), (640, 384), (300, 1100), (512, 512), (256, 1152)]
    ts = workloads.gen_tensors(workloads.Workload("pairs", shapes, 0.02, 86))
    nsg.ns_set_gemm_cluster(1)
    try:
        single = run_mode(shapes, ts, mode)
    finally:
        nsg.ns_set_gemm_cluster(0)
    paired = run_mode(shapes, ts, mode)
    for s, t, a, b in zip(shapes, ts, single, paired):
        assert torch.equal(a, b), (mode, s)
        assert rel_err(b, oracle(t)) <= FP32_TOL, (mode, s)
