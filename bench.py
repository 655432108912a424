#!/usr/bin/env python
"""Throughput of the shape-batched Newton-Schulz hot path on GB300.

One step = pack (S = 8 simulated row-shard ranks -> LPT homes) -> quintic
Newton-Schulz on every matrix (5 steps, bf16 path) -> unpack (homes -> ranks),
all through the C ABI of libnsgb300.so. Default workload: GPT-style 24 layers,
d = 2048, ffn = 8192 (QKV 6144x2048, O 2048x2048, up 8192x2048,
down 2048x8192 per layer; 96 matrices, 2.42 GB of bf16 per step).

Prints one JSON line (rank 0). ``value`` is matrices/s with inputs resident in
HBM; ``e2e`` is the same metric with the host->device copy of the rank shards
and the device->host copy of the results inside the timed region.
``--impl reference`` times the float64 CPU oracle instead, on a bounded
sample of the same workload.

Multi-GPU (torchrun): every rank runs its own replica of the workload (weak
scaling, no data-path collective); the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NS matrices/s and achieved TFLOP/s vs GB300 dense bf16 peak (1 GPU)"
UNIT = "matrices/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["gpt", "small", "llama", "moe", "sweep"], default="gpt")
    ap.add_argument("--gram", choices=["bf16", "fp32", "fp32gs", "fp32auto"], default="bf16",
                    help="precision policy (sweep workload): bf16 path, fp32-Gram (split TF32) path, "
                         "its Gram-space form, or per bucket the faster of the two (Gram space when n >= 2m)")
    ap.add_argument("--ridge", type=float, default=0.0, help="trace ridge (fp32-Gram path only)")
    ap.add_argument("--points", type=str, default="",
                    help="sweep subset, e.g. '1024x1,4096x8' (m x aspect); default: all")
    ap.add_argument("--layers", type=int, default=0,
                    help="keep only the first N layers of the workload (small cases for ncu captures)")
    ap.add_argument("--gemm-cluster", type=int, default=0, choices=[0, 1, 3],
                    help="GEMM tiling: 0 automatic, 1 single CTA, 3 2-SM MMA")
    ap.add_argument("--sym-store", choices=["upper", "mirror"], default="upper",
                    help="bf16 A and B: upper 256x256 pair blocks only (readers load the rest "
                         "transposed) or also their mirror")
    ap.add_argument("--waves", type=int, default=2,
                    help="run the step through the wave pipeline with this many waves (0: serial calls)")
    ap.add_argument("--split-qkv", action="store_true",
                    help="orthogonalise Q, K and V blocks of fused QKV projections separately")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-budget", type=float, default=20.0,
                    help="seconds of oracle work per cpu_baseline / reference sample")
    ap.add_argument("--no-1thread", action="store_true",
                    help="skip the single-thread oracle run reported beside cpu_baseline")
    return ap.parse_args()


PER_LAYER = {"gpt": 4, "llama": 5, "moe": 3 * 64, "small": 1, "sweep": 1}


def sweep_workload():
    import workloads
    shapes = []
    for (m, a, bt) in workloads.sweep_points():
        shapes += [(m, a * m)] * bt
    shapes += [(256, 64, 3, 3)] * 64
    return workloads.Workload("size/aspect sweep", shapes, 0.02, 5000, S=1)


def get_workload(name: str, layers: int = 0):
    import workloads
    w = {"gpt": workloads.gpt_24l_d2048, "small": workloads.small_16x128x256,
         "llama": workloads.llama8b_32l, "moe": workloads.moe_16l_64e, "sweep": sweep_workload}[name]()
    if layers > 0:
        w.shapes = w.shapes[:layers * PER_LAYER[name]]
        w.name += f" (first {layers} layers)"
    return w


def view_mn(shape):
    rows = shape[0]
    cols = 1
    for d in shape[1:]:
        cols *= d
    return min(rows, cols), max(rows, cols)


def is_small(shape) -> bool:
    """The library runs bf16 matrices with m <= 128 and n <= 512 as one CTA
    per matrix (kind "small") unless its small path is switched off."""
    m, n = view_mn(shape)
    return m <= 128 and n <= 512


def flops_by_kind(shapes, k, small_path=True):
    """Algorithmic flops per call by kernel kind: Gram 2 m^2 n, A*A 2 m^3,
    B*X 2 m^2 n per matrix per step (useful total k (4 m^2 n + 2 m^3));
    all three of a small matrix's products count for kind "small"."""
    g = a2 = bx = sm = 0
    for s in shapes:
        m, n = view_mn(s)
        if small_path and is_small(s):
            sm += k * (4 * m * m * n + 2 * m * m * m)
            continue
        g += 2 * m * m * n * k
        a2 += 2 * m * m * m * k
        bx += 2 * m * m * n * k
    return {"gram": g, "a2b": a2, "bx": bx, "small": sm}


# NVIDIA's dense (no 2:4 sparsity) bf16 tensor-core figure for one GB300 GPU
NOMINAL_BF16_TFLOPS = 2250.0


def executed_flops_by_kind(shapes, k, cluster_mode: int = 0):
    """Tensor-core flops the kernels execute per call, by kind: whole tiles on
    the zero-padded operands, only the upper tiles of the symmetric products,
    spare half pairs of odd tile-row counts included. Useful flops
    (flops_by_kind) can exceed the tensor-pipe rate because SYRK skips work."""
    ex = {"gram": 0, "a2b": 0, "bx": 0, "small": 0}
    big = [s for s in shapes if not is_small(s)]
    for s in shapes:
        m, n = view_mn(s)
        m_pad, n_pad = -(-m // 128) * 128, -(-n // 64) * 64
        if is_small(s):
            # the whole padded products: 128 x 128 x n_pad, 128^3, 128 x n_pad x 128
            ex["small"] += k * (2 * 128 * 128 * n_pad * 2 + 2 * 128 ** 3)
            continue
        tm, tn_sym, tn_bx = m_pad // 128, -(-m_pad // 256), -(-n_pad // 256)
        for kind, kdim in (("gram", n_pad), ("a2b", m_pad), ("bx", m_pad)):
            mode = int(gemm_kernel_for(kind, cluster_mode, big)[0].startswith("ns_gemm2sm")) if tm >= 2 else 0
            if kind == "bx":
                tiles = (-(-tm // 2) * 2 if mode else tm) * tn_bx
            elif mode:
                tiles = 2 * sum(tn_sym - q for q in range(-(-tm // 2)))
            else:
                tiles = sum(tn_sym - (r * 128) // 256 for r in range(tm))
            ex[kind] += 2 * 128 * 256 * kdim * tiles * k
    return ex


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["bf16_tflops"], d["bf16_tflops_sustained"], d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def gemm_kernel_for(kind: str, cluster_mode: int, shapes=()):
    """(kernel name, source file) of the GEMM kind under a tiling mode: the
    library's default runs the 2-SM kernel for Gram, and for A*A and B*X when
    every bucket has an even number of 128-row tile rows (else the 1-SM one);
    small matrices run in ns_small_kernel."""
    if kind == "small":
        return "ns_small_kernel", "small.cu"
    even = all(((view_mn(s)[0] + 127) // 128) % 2 == 0 for s in shapes if not is_small(s))
    mode = cluster_mode if cluster_mode else (3 if kind in ("gram", "a2b") or even else 1)
    if mode == 3:
        return f"ns_gemm2sm_kernel<{kind}>", "gemm2sm.cu"
    return f"ns_gemm_kernel<{kind}>", "gemm.cu"


def traffic_for(kind: str, cluster_mode: int, shapes=()):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel (else None)."""
    name, fname = gemm_kernel_for(kind, cluster_mode, shapes)
    csrc = os.path.join(ROOT, "newton_schulz_shape_gb300", "csrc")
    summ = os.path.join(ROOT, "profiles", "gemm_traffic.md")
    try:
        # the kernel's own file and the epilogue it includes
        sha = hashlib.sha256(b"".join(open(os.path.join(csrc, f), "rb").read()
                                      for f in (fname, "epilogue.cuh"))).hexdigest()[:16]
        for line in open(summ):
            if line.startswith("traffic:"):
                kv = dict(x.strip().split("=", 1) for x in line[len("traffic:"):].split(";") if "=" in x)
                if kv.get("kernel") == name and kv.get("source") == fname and kv.get("sha256") == sha:
                    return int(kv["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


# ------------------------------------------------------------- multi-rank
def replica_seed(seed: int, rank: int, world: int) -> int:
    """Each rank runs its own replica of the workload (weak scaling)."""
    return seed + 7919 * rank if world > 1 else seed


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank time over all ranks (the only collective the bench uses)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(n_mats: int, world: int, ms_step: float) -> float:
    """Whole-job matrices/s: every rank processes n_mats per step."""
    return n_mats * world * 1000.0 / ms_step


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"nsgb300_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- CPU oracle
def cpu_oracle_sample(w, budget_s: float = 20.0):
    """Time the float64 oracle on one matrix per shape bucket (and the routing
    oracle on those tensors), smallest buckets first, until `budget_s` is
    spent; extrapolate to the whole workload by count, and by useful flops at
    the sampled rate for buckets not sampled."""
    import numpy as np  # noqa: F401
    import workloads
    from oracle import ns as ons
    from oracle import routing as orr
    buckets = {}
    for i, s in enumerate(w.shapes):
        buckets.setdefault(view_mn(s), []).append(i)
    order = sorted(buckets, key=lambda mn: mn[0] * mn[0] * mn[1])
    total_est, spent, sampled_flops = 0.0, 0.0, 0
    sample, unsampled = [], []
    for mn in order:
        idx = buckets[mn]
        i = idx[0]
        fl = sum(flops_by_kind([w.shapes[i]], workloads.STEPS).values())
        if spent > budget_s:
            unsampled.append((len(idx), fl))
            continue
        t = workloads.gen_tensor(w.shapes[i], w.sigma, w.seed, i)
        x = t.float().numpy()
        bits = t.view(__import__("torch").int16).numpy()
        t0 = time.perf_counter()
        ons.newton_schulz(x, workloads.STEPS, workloads.A_COEF, workloads.B_COEF, workloads.C_COEF, workloads.EPS)
        ranks = orr.make_rank_buffers([bits], w.S, 0)
        homes = orr.route_to_ns_home(ranks, [w.shapes[i]], {0: 0}, w.S, 0)
        orr.route_from_ns_home(homes, [w.shapes[i]], {0: 0}, w.S, 0)
        dt = time.perf_counter() - t0
        spent += dt
        sampled_flops += fl
        total_est += dt * len(idx)
        sample.append(f"{len(idx)}x{tuple(w.shapes[i])}: {dt:.2f}s")
    if unsampled:
        rate = sampled_flops / spent
        total_est += sum(c * fl / rate for c, fl in unsampled)
        sample.append(f"{sum(c for c, _ in unsampled)} matrices in {len(unsampled)} larger buckets "
                      f"extrapolated at the sampled {rate / 1e9:.0f} GFLOP/s")
    threads = blas_threads() or os.cpu_count()
    return len(w.shapes) / total_est, threads, "one matrix per (m, n) bucket, NS + pack/unpack oracle, " \
        "extrapolated by bucket count: " + "; ".join(sample)


def blas_threads():
    """Threads of the BLAS numpy's matmul runs on: threadpoolctl when it is
    installed, else the OpenBLAS library numpy loaded, asked directly."""
    try:
        import threadpoolctl
        return max(p.get("num_threads", 1) for p in threadpoolctl.threadpool_info())
    except Exception:
        pass
    try:
        import ctypes

        import numpy as np
        np.ones(2) @ np.ones(2)
        paths = {ln.split()[-1] for ln in open("/proc/self/maps") if "openblas" in ln.lower() and "/" in ln}
        for path in sorted(paths):
            lib = ctypes.CDLL(path)
            for sym in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                        "openblas_get_num_threads64_", "openblas_get_num_threads"):
                fn = getattr(lib, sym, None)
                if fn is not None:
                    return int(fn())
    except Exception:
        pass
    v = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(v) if v and v.isdigit() else None


def oracle_single_thread(args, budget_s: float = 8.0):
    """The same oracle sample with every BLAS/OpenMP pool limited to one
    thread (a child process: the limits must be set before numpy loads)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               RANK="0", WORLD_SIZE="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", args.workload,
           "--layers", str(args.layers), "--steps", "1", "--warmup", "0", "--no-1thread",
           "--oracle-budget", str(budget_s)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])["value"]
    except Exception:
        return None


def cpu_baseline_entry(w, args, v, threads, sample):
    d = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
         "host_cpus": os.cpu_count(), "blas_threads": blas_threads()}
    if not args.no_1thread:
        d["value_1thread"] = oracle_single_thread(args)
    return d


def oracle_step(w, idx):
    """The float64 oracle over tensors `idx` of the workload: NS plus the
    pack/unpack routing oracle. Returns the seconds it took (inputs are
    generated before the clock starts)."""
    import torch

    import workloads
    from oracle import ns as ons
    from oracle import routing as orr
    ts = [workloads.gen_tensor(w.shapes[i], w.sigma, w.seed, i) for i in idx]
    xs = [t.float().numpy() for t in ts]
    bits = [t.view(torch.int16).numpy() for t in ts]
    t0 = time.perf_counter()
    for i, x, b in zip(idx, xs, bits):
        ons.newton_schulz(x, workloads.STEPS, workloads.A_COEF, workloads.B_COEF, workloads.C_COEF, workloads.EPS)
        ranks = orr.make_rank_buffers([b], w.S, 0)
        homes = orr.route_to_ns_home(ranks, [w.shapes[i]], {0: 0}, w.S, 0)
        orr.route_from_ns_home(homes, [w.shapes[i]], {0: 0}, w.S, 0)
    return time.perf_counter() - t0


def split_by_flops(w, k):
    """Tensor indices in exactly min(k, n) non-empty groups of consecutive
    tensors with about equal oracle flops."""
    import workloads
    fl = [sum(flops_by_kind([s], workloads.STEPS).values()) for s in w.shapes]
    n = len(fl)
    k = max(1, min(k, n))
    total, groups, cur, acc = sum(fl), [], [], 0.0
    for i, f in enumerate(fl):
        cur.append(i)
        acc += f
        left = n - i - 1                   # tensors not yet placed
        need = k - (len(groups) + 1)       # groups still to fill once this one closes
        if need > 0 and left >= need and (acc >= total * (len(groups) + 1) / k or left == need):
            groups.append(cur)
            cur = []
    groups.append(cur)
    return groups


def run_reference(args):
    """The float64 oracle on the host cores, timed like our arm: W warm-up
    steps, then K timed steps. When the whole workload fits in about four
    minutes of oracle work (estimated from the warm-up's rate) the K steps
    split it, so that together they run every matrix exactly once and nothing
    is extrapolated; otherwise each step runs a bounded sample (one matrix per
    shape bucket) and the workload's rate is extrapolated from it."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import workloads
    w = get_workload(args.workload, args.layers)
    flops = [sum(flops_by_kind([s], workloads.STEPS).values()) for s in w.shapes]
    small = min(range(len(w.shapes)), key=lambda i: flops[i])
    warm_s = [oracle_step(w, [small]) for _ in range(max(1, args.warmup))]
    rate = flops[small] / max(1e-9, min(warm_s))          # oracle flop/s on this host
    full_est = sum(flops) / rate
    t0 = time.perf_counter()
    if full_est <= 240.0 and args.steps <= len(w.shapes):
        groups = split_by_flops(w, max(1, args.steps))
        step_s = [oracle_step(w, g) for g in groups]
        value = len(w.shapes) / sum(step_s)
        extrapolated = False
        sample = (f"the whole workload once: {len(w.shapes)} matrices split over {len(groups)} timed steps "
                  f"of about equal oracle flops, NS + pack/unpack oracle")
    else:
        budget = min(args.oracle_budget, max(2.0, 150.0 / max(1, args.steps)))
        step_s, vals = [], []
        for _ in range(args.steps):
            s0 = time.perf_counter()
            v, _, sample = cpu_oracle_sample(w, budget)
            step_s.append(time.perf_counter() - s0)
            vals.append(v)
        value = statistics.median(vals)
        extrapolated = True
    wall = time.perf_counter() - t0
    threads = blas_threads() or os.cpu_count()
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": len(step_s),
            "warmup": len(warm_s), "ms_per_step": 1000.0 * statistics.mean(step_s), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "extrapolated": extrapolated,
            "config": {"workload": w.name, "matrices": len(w.shapes), "S": w.S},
            "cpu_baseline": cpu_baseline_entry(w, args, value, threads, sample),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall, "oracle_full_workload_estimate_s": full_est}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our path
def run_ours(args):
    import torch
    import torch.distributed as dist

    import newton_schulz_shape_gb300 as nsg
    import workloads

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    w = get_workload(args.workload, args.layers)
    w.seed = replica_seed(w.seed, rank, world)
    nsg.ns_set_gemm_cluster(args.gemm_cluster)
    nsg.ns_set_symmetric_store(1 if args.sym_store == "mirror" else 0)
    S, shapes = w.S, w.shapes
    plan = nsg.ns_plan_create(shapes, steps=workloads.STEPS, eps=workloads.EPS, S=S, shard_dim=0)
    home_off, home_sizes, rank_sizes = plan.home_layout()
    homes = plan.homes()
    L = rank_sizes[0]

    # host inputs: rank r's shards of every tensor, in index order (pinned)
    rank_host = [torch.empty(L, dtype=torch.bfloat16, pin_memory=True) for _ in range(S)]
    pos = 0
    for i, s in enumerate(shapes):
        t = workloads.gen_tensor(s, w.sigma, w.seed, i).reshape(S, -1)
        n = t.shape[1]
        for r in range(S):
            rank_host[r][pos:pos + n].copy_(t[r])
        pos += n
    # pinned buffers are touched by the CPU once: untouched pinned pages make the
    # first device -> host copy into them run at a fraction of the link speed
    out_host = [torch.zeros(L, dtype=torch.bfloat16, pin_memory=True) for _ in range(S)]

    rank_in = [h.to(dev) for h in rank_host]
    home_in = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in home_sizes]
    home_out = [torch.empty(max(1, n), dtype=torch.bfloat16, device=dev) for n in home_sizes]
    rank_out = [torch.empty(L, dtype=torch.bfloat16, device=dev) for _ in range(S)]
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ins = [home_in[homes[i]].data_ptr() + 2 * home_off[i] for i in range(len(shapes))]
    outs = [home_out[homes[i]].data_ptr() + 2 * home_off[i] for i in range(len(shapes))]
    ns_shapes = shapes
    ns_plan = plan
    if args.split_qkv:
        # split-QKV: NS over the row blocks of each fused QKV tensor; a row block
        # of a row-major tensor is contiguous, so its pointer is an offset
        ns_shapes, parents = workloads.split_rows(shapes)
        ins = [ins[i] + 2 * r0 * (int(np.prod(shapes[i])) // shapes[i][0]) for i, r0 in parents]
        outs = [outs[i] + 2 * r0 * (int(np.prod(shapes[i])) // shapes[i][0]) for i, r0 in parents]
        ns_plan = nsg.ns_plan_create(ns_shapes, steps=workloads.STEPS, eps=workloads.EPS, S=1)
        ws = torch.empty(ns_plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    pipe = None
    if args.waves > 0 and not args.split_qkv:
        pipe = nsg.ns_pipeline_create(plan, args.waves)
        ws = torch.empty(pipe.workspace_bytes, dtype=torch.uint8, device=dev)

    def step(rin=None, rout=None):
        rin = rank_in if rin is None else rin
        rout = rank_out if rout is None else rout
        if pipe is not None:
            nsg.ns_pipeline_run(pipe, rin, home_in, home_out, rout, ws, stream=stream)
            return
        nsg.ns_pack_to_home(plan, rin, home_in, stream=stream)
        nsg.ns_orthogonalize_batched(ns_plan, ins, outs, ws, stream=stream)
        nsg.ns_unpack_from_home(plan, home_out, rout, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    rc = nsg.ns_check_status(plan, stream)
    if rc != nsg.NS_OK:
        raise RuntimeError(f"device status after warm-up: {nsg.ns_status_string(rc)}")

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    uuid = ""
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)

    # ---- device-resident timed region (per-phase events on the launch stream)
    nsg.ns_profile_read(reset=True)
    nsg.ns_profile_enable(True)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier()
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        if pipe is not None:
            # the pipeline overlaps the phases; only whole steps are timed
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
            continue
        ev[k][0].record(stream)
        nsg.ns_pack_to_home(plan, rank_in, home_in, stream=stream)
        ev[k][1].record(stream)
        nsg.ns_orthogonalize_batched(ns_plan, ins, outs, ws, stream=stream)
        ev[k][2].record(stream)
        nsg.ns_unpack_from_home(plan, home_out, rank_out, stream=stream)
        ev[k][3].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    nsg.ns_profile_enable(False)
    launches, kms = nsg.ns_profile_read(reset=True)
    rc = nsg.ns_check_status(plan, stream)
    if rc != nsg.NS_OK:
        raise RuntimeError(f"device status after timing: {nsg.ns_status_string(rc)}")
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ms_step = ms_total / args.steps
    pack_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    ns_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev) if pipe is None else None
    unpack_ms = statistics.median(e[2].elapsed_time(e[3]) for e in ev) if pipe is None else None
    n_mats = len(ns_shapes)
    value = job_value(n_mats, world, ms_step)

    # ---- raw copy bandwidth (context for e2e)
    copy_gbs = {}
    for name, fn in (("h2d", lambda: [rank_in[r].copy_(rank_host[r], non_blocking=True) for r in range(S)]),
                     ("d2h", lambda: [out_host[r].copy_(rank_out[r], non_blocking=True) for r in range(S)])):
        fn()
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        fn()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        copy_gbs[name] = 2 * S * L / (c0.elapsed_time(c1) * 1e-3) / 1e9

    # ---- end to end: every step copies its inputs host -> device (pinned),
    # runs pack -> NS -> unpack, and copies its results device -> host. The
    # copies run on their own streams while other steps compute, through a
    # ring of NB device buffer sets (inputs, outputs): step k's input copy may
    # start once step k - NB has read its set, so the copy streams can fall
    # behind for a while (the shared host link stalls single copies at times)
    # and catch up without holding the GPU. NB is 2-4, as device memory
    # allows. On the host side every step reads the same pinned input buffer
    # and writes the same pinned output buffer (the output copies run in step
    # order on one stream): rotating the output copies over several host
    # buffers made every one of them several times slower on this machine.
    e2e = None
    if not args.no_e2e:
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        set_dev = 2 * 2 * S * L                      # inputs + outputs, bf16
        free_dev = torch.cuda.mem_get_info(dev)[0]
        NB = max(2, min(4, 1 + int(0.5 * free_dev // set_dev)))
        rin = [rank_in] + [[torch.empty_like(x) for x in rank_in] for _ in range(NB - 1)]
        rout = [rank_out] + [[torch.empty_like(x) for x in rank_out] for _ in range(NB - 1)]
        hout = [out_host] * NB                       # one pinned host output buffer
        ev_in = [torch.cuda.Event() for _ in range(NB)]
        ev_cmp = [torch.cuda.Event() for _ in range(NB)]
        ev_out = [torch.cuda.Event() for _ in range(NB)]

        trace = []   # per step: events around the input copies, the compute and the output copies

        def e2e_steps(n):
            for k in range(n):
                b = k % NB
                tr = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
                with torch.cuda.stream(s_in):
                    if k >= NB:
                        s_in.wait_event(ev_cmp[b])     # rin[b] was read by step k - NB
                    tr[0].record(s_in)
                    for r in range(S):
                        rin[b][r].copy_(rank_host[r], non_blocking=True)
                    tr[1].record(s_in)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                if k >= NB:
                    stream.wait_event(ev_out[b])       # rout[b] was copied out by step k - NB
                tr[2].record(stream)
                step(rin[b], rout[b])
                tr[3].record(stream)
                ev_cmp[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[b])
                    tr[4].record(s_out)
                    for r in range(S):
                        hout[b][r].copy_(rout[b][r], non_blocking=True)
                    tr[5].record(s_out)
                    ev_out[b].record(s_out)
                trace.append(tr)

        e2e_steps(NB)                                   # warm-up of the pipeline
        barrier()
        for h in out_host:                              # so that the check below sees this region's copies
            h.zero_()
        e2e_clocks = ClockSampler(uuid)
        e2e_clocks.start()
        time.sleep(0.3)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        trace.clear()
        e2e_steps(args.steps)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)
        e1.record(stream)
        barrier()
        clk_e2e = e2e_clocks.stop()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
        # the results of the last step really came back
        ok = all(torch.equal(hout[(args.steps - 1) % NB][r], rank_out[r].cpu()) for r in range(S))
        nbytes = 2 * S * L
        # per-step timings (ms): each group is the step's S copies of one direction
        groups = {"h2d_ms": [t[0].elapsed_time(t[1]) for t in trace],
                  "compute_ms": [t[2].elapsed_time(t[3]) for t in trace],
                  "d2h_ms": [t[4].elapsed_time(t[5]) for t in trace]}
        timeline = {k: {"median": statistics.median(v), "max": max(v),
                        "over_2x_median": sum(x > 2 * statistics.median(v) for x in v)} for k, v in groups.items()}
        e2e = {"value": job_value(n_mats, world, ms_e2e), "unit": UNIT, "ms_per_step": ms_e2e,
               "timeline": timeline,
               "copy_gbs_in_region": {"h2d": nbytes / (timeline["h2d_ms"]["median"] * 1e-3) / 1e9,
                                      "d2h": nbytes / (timeline["d2h_ms"]["median"] * 1e-3) / 1e9},
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
               "pipelining": f"copies on their own streams overlap the compute of other steps; ring of {NB} "
                             "device buffer sets (in/out); one pinned host input and one pinned host output buffer",
               "results_returned": ok, "copy_gbs": copy_gbs, "clocks": clk_e2e}

    # ---- roofline of the dominant kernel
    burst, sustained, hbm, peak_src = peaks()
    fl = flops_by_kind(ns_shapes, workloads.STEPS)
    ex = executed_flops_by_kind(ns_shapes, workloads.STEPS, args.gemm_cluster)
    # the last step's B*X launches also store the results (kind bx_final):
    # split the B*X flops between the two kinds by launch count (every B*X
    # launch of a step covers the same matrices)
    n_bx = launches.get("bx", 0) + launches.get("bx_final", 0)
    for d in (fl, ex):
        tot = d["bx"]
        d["bx"] = tot * launches.get("bx", 0) / max(1, n_bx)
        d["bx_final"] = tot - d["bx"]
    gemm_kinds = ["gram", "a2b", "bx", "bx_final", "small"]
    # the roofline kernel: the pure GEMM launches (or the small-matrix
    # kernel) with the most time
    dom = max(["gram", "a2b", "bx", "small"], key=lambda k: kms.get(k, 0.0))
    per_launch_ms = kms[dom] / max(1, launches[dom])
    launches_per_step = launches[dom] / args.steps
    flops_per_launch = fl[dom] / launches_per_step
    achieved = flops_per_launch / (per_launch_ms * 1e-3) / 1e12
    useful = sum(fl.values())
    # the recorded traffic is for one launch over the whole 24-layer GPT-style
    # workload (one NS step of one phase); scale it by this launch's share of
    # that work (waves split a phase into several launches)
    traffic = traffic_for(dom, args.gemm_cluster, ns_shapes) if args.workload == "gpt" and not args.layers \
        and not args.split_qkv and dom != "small" and args.sym_store == "upper" else None
    if traffic is not None:
        traffic = int(traffic * flops_per_launch / (sum(fl[k] for k in gemm_kinds if k.startswith(dom))
                                                    / workloads.STEPS))
    roofline = {"bound": "tensor", "kernel": gemm_kernel_for(dom, args.gemm_cluster, ns_shapes)[0], "achieved": achieved,
                "peak": sustained, "unit": "TFLOP/s", "frac": achieved / sustained,
                "traffic": traffic,
                "peak_note": f"{peak_src} sustained bf16 (kernel timed inside a long step); burst {burst}",
                "nominal_peak": NOMINAL_BF16_TFLOPS, "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                "useful_tflops_step": useful / (ms_step * 1e-3) / 1e12,
                "flops_per_launch": flops_per_launch, "avg_launch_ms": per_launch_ms}
    if dom == "small":
        roofline["note"] = (f"latency-bound: one CTA per matrix, {n_mats} CTAs on "
                            f"{torch.cuda.get_device_properties(dev).multi_processor_count} SMs; "
                            "the fraction is of the whole GPU's peak")
    per_kernel = {k: {"launches_per_step": launches[k] / args.steps, "ms_per_step": kms[k] / args.steps}
                  for k in launches}
    for k in gemm_kinds:
        if kms.get(k, 0) > 0:
            per_kernel[k]["tflops"] = fl[k] / (kms[k] / args.steps * 1e-3) / 1e12
            per_kernel[k]["executed_tflops"] = ex[k] / (kms[k] / args.steps * 1e-3) / 1e12
    pack_bytes = 2 * 2 * S * L   # read + write, bf16
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0, sigma) bf16 per tensor (sigma 0.02)",
        "config": {"workload": f"{w.name}: {n_mats} matrices, S={S} row shards, LPT homes, "
                               f"pack -> NS (5 steps) -> unpack",
                   "matrices": n_mats, "S": S, "ns_steps": workloads.STEPS, "gemm_cluster": args.gemm_cluster,
                   "symmetric_store": args.sym_store, "split_qkv": bool(args.split_qkv), "waves": pipe.n_waves if pipe is not None else 0,
                   "l2": f"inputs larger than L2 ({2 * S * L / 1e9:.2f} GB of bf16 per step)"},
        "tflops_useful": useful / (ms_step * 1e-3) / 1e12 * world,
        "ns_only": ({"ms": ns_ms, "tflops_useful": useful / (ns_ms * 1e-3) / 1e12,
                     "frac_of_burst_peak": useful / (ns_ms * 1e-3) / 1e12 / burst} if pipe is None else None),
        "phases_ms": ({"pack": pack_ms, "ns": ns_ms, "unpack": unpack_ms} if pipe is None
                      else {"pipelined_step": pack_ms, "waves": pipe.n_waves}),
        "pack_gbs": pack_bytes / (pack_ms * 1e-3) / 1e9 if pipe is None else None,
        "unpack_gbs": pack_bytes / (unpack_ms * 1e-3) / 1e9 if pipe is None and unpack_ms > 0 else None,
        "per_kernel": per_kernel,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": int(sum(launches.values())),
        "roofline": roofline,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, threads, sample = cpu_oracle_sample(w, args.oracle_budget)
        line["cpu_baseline"] = cpu_baseline_entry(w, args, v, threads, sample)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ sweep
def run_sweep(args):
    """Size/aspect sweep: NS alone (no pack) on each point's batch, one plan
    per point, inputs resident in HBM; per-point useful TFLOP/s and the whole
    sweep's matrices/s."""
    import torch

    import newton_schulz_shape_gb300 as nsg
    import workloads

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    pts = [(m, a, bt) for (m, a, bt) in workloads.sweep_points()]
    if args.points:
        want = {tuple(int(x) for x in p.split("x")) for p in args.points.split(",")}
        pts = [p for p in pts if (p[0], p[1]) in want]
    mode = {"bf16": nsg.NS_BF16, "fp32": nsg.NS_FP32_GRAM, "fp32gs": nsg.NS_FP32_GRAM_SPACE,
            "fp32auto": nsg.NS_FP32_AUTO}[args.gram]
    stream = torch.cuda.current_stream(dev)
    results, tot_ms, tot_mats, tot_flops = [], 0.0, 0, 0
    runs = [(f"{m}x{a * m}", [(m, a * m)] * bt, 5000 + m + a) for (m, a, bt) in pts]
    if not args.points:
        runs.append(("256x64x3x3", [(256, 64, 3, 3)] * 64, 5999))
    clocks = ClockSampler("")
    clocks.start()
    for name, shapes, seed in runs:
        w = workloads.Workload(name, shapes, 0.02, seed)
        ins = [workloads.gen_tensor(s, w.sigma, w.seed, i).to(dev) for i, s in enumerate(shapes)]
        odt = torch.bfloat16 if mode == nsg.NS_BF16 else torch.float32
        outs = [torch.empty(s, dtype=odt, device=dev) for s in shapes]
        plan = nsg.ns_plan_create(shapes, steps=workloads.STEPS, eps=workloads.EPS, gram_mode=mode,
                                  ridge=args.ridge, S=1)
        ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
        for _ in range(max(3, args.warmup)):
            nsg.ns_orthogonalize_batched(plan, ins, outs, ws, stream=stream)
        rc = nsg.ns_check_status(plan, stream)
        if rc != nsg.NS_OK:
            raise RuntimeError(f"{name}: {nsg.ns_status_string(rc)}")
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            nsg.ns_orthogonalize_batched(plan, ins, outs, ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        fl = sum(sum(flops_by_kind([s], workloads.STEPS).values()) for s in shapes)
        results.append({"point": name, "matrices": len(shapes), "ms": ms,
                        "tflops_useful": fl / (ms * 1e-3) / 1e12})
        tot_ms += ms
        tot_mats += len(shapes)
        tot_flops += fl
        del ins, outs, ws, plan
        torch.cuda.empty_cache()
    clk = clocks.stop()
    burst, sustained, _, src = peaks()
    line = {"metric": METRIC, "value": tot_mats * 1000.0 / tot_ms, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": tot_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if mode == nsg.NS_BF16 else "f32 (split-TF32 products)",
            "data": "synthetic: seeded N(0, 0.02) bf16 per tensor",
            "config": {"workload": "size/aspect sweep: m in {1024..8192} x aspect {1,2,4,8} (+ 256x64x3x3), NS only",
                       "gram": args.gram, "ridge": args.ridge},
            "tflops_useful": tot_flops / (tot_ms * 1e-3) / 1e12,
            "peak_bf16_tflops": {"burst": burst, "sustained": sustained, "source": src},
            "points": results, "clocks": clk}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "sweep":
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
