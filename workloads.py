"""Seeded synthetic inputs for the Newton-Schulz hot path.

Shared by the tests, the bench and the oracle legs. It holds the workload
shape lists and a seeded Gaussian generator, and none of the method's
arithmetic (no views, norms, costs or routing).

Recipe: tensor ``i`` of a workload with seed ``s`` is drawn from its own CPU
generator seeded with ``s * 1_000_003 + i`` as float32 ``randn * sigma`` and
rounded to bf16 (round to nearest even). Per-tensor seeding lets a test
regenerate any one tensor of a large workload on its own. The same bf16 bytes
feed the GPU path and the oracle.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

A_COEF, B_COEF, C_COEF = 3.4445, -4.7750, 2.0315
EPS = 1e-7
STEPS = 5


@dataclass
class Workload:
    name: str
    shapes: list
    sigma: float
    seed: int
    S: int = 8
    shard_dim: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)


def small_16x128x256() -> Workload:
    """16 matrices 128x256, entries N(0, 1)."""
    return Workload("16x(128x256) N(0,1)", [(128, 256)] * 16, 1.0, 1000, S=8)


def gpt_24l_d2048() -> Workload:
    """GPT-style 24 layers, d=2048, ffn=8192: QKV 6144x2048, O 2048x2048,
    up 8192x2048, down 2048x8192 per layer; N(0, 0.02)."""
    shapes = []
    for _ in range(24):
        shapes += [(6144, 2048), (2048, 2048), (8192, 2048), (2048, 8192)]
    return Workload("gpt-24L-d2048-ffn8192", shapes, 0.02, 2000, S=8)


def llama8b_32l() -> Workload:
    """Llama-8B-shaped 32 layers, d=4096, ffn=14336: GQA QKV 6144x4096,
    O 4096x4096, gate/up 14336x4096, down 4096x14336; N(0, 0.02)."""
    shapes = []
    for _ in range(32):
        shapes += [(6144, 4096), (4096, 4096), (14336, 4096), (14336, 4096), (4096, 14336)]
    return Workload("llama8b-32L-d4096-ffn14336", shapes, 0.02, 3000, S=8)


def moe_16l_64e() -> Workload:
    """MoE: 16 layers x 64 experts x (gate 1408x2048, up 1408x2048,
    down 2048x1408); S = 8 row shards; N(0, 0.02)."""
    shapes = []
    for _ in range(16 * 64):
        shapes += [(1408, 2048), (1408, 2048), (2048, 1408)]
    return Workload("moe-16L-64E-1408x2048", shapes, 0.02, 4000, S=8)


def sweep_shapes(m: int, aspect: int, batch: int) -> Workload:
    """One point of the size/aspect sweep: `batch` matrices m x (aspect*m)."""
    return Workload(f"sweep-{m}x{aspect * m}", [(m, aspect * m)] * batch, 0.02,
                    5000 + m + aspect, S=8)


def sweep_points() -> list:
    """(m, aspect, batch) of the sweep: m in {1024..8192}, aspect 1..8."""
    pts = []
    for m in (1024, 2048, 4096, 8192):
        for rho in (1, 2, 4, 8):
            batch = 4 if (m == 8192 and rho >= 4) else 8
            pts.append((m, rho, batch))
    return pts


def conv_3d() -> Workload:
    """The (256, 64, 3, 3) tensor of the sweep, 64 of them."""
    return Workload("conv-256x64x3x3", [(256, 64, 3, 3)] * 64, 0.02, 5999, S=8)


def tensor_seed(seed: int, i: int) -> int:
    return seed * 1_000_003 + i


def gen_tensor(shape, sigma: float, seed: int, i: int) -> torch.Tensor:
    """Tensor i of a workload: bf16 on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(tensor_seed(seed, i))
    return (torch.randn(tuple(shape), generator=g, dtype=torch.float32) * sigma).to(torch.bfloat16)


def gen_tensors(w: Workload, indices=None) -> list:
    if indices is None:
        indices = range(len(w.shapes))
    return [gen_tensor(w.shapes[i], w.sigma, w.seed, i) for i in indices]


def gen_random_shapes(n: int, seed: int, max_dim: int = 300, S: int = 1,
                      max_ndim: int = 4) -> list:
    """Random tensor shapes (ndim 2..max_ndim) whose first dim is a multiple
    of S, for planner and routing tests."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shapes = []
    for _ in range(n):
        nd = int(torch.randint(2, max_ndim + 1, (1,), generator=g))
        first = S * int(torch.randint(1, max(2, max_dim // S), (1,), generator=g))
        rest = [int(torch.randint(1, 9 if nd > 2 else max_dim, (1,), generator=g))
                for _ in range(nd - 1)]
        shapes.append(tuple([first] + rest))
    return shapes


# Row splits of fused QKV projections (split-QKV): Q rows, then K, then V.
QKV_SPLITS = {
    (6144, 2048): (2048, 2048, 2048),   # GPT-style MHA, d = 2048
    (6144, 4096): (4096, 1024, 1024),   # Llama-8B GQA: 32 query heads, 8 KV heads, head dim 128
}


def split_rows(shapes, splits=None):
    """Expand each tensor whose shape has a row split into its row blocks.
    Returns (block_shapes, parents) with parents[j] = (tensor index, first row)."""
    splits = QKV_SPLITS if splits is None else splits
    out, parents = [], []
    for i, s in enumerate(shapes):
        sp = splits.get(tuple(s))
        if sp is None:
            out.append(tuple(s))
            parents.append((i, 0))
            continue
        r0 = 0
        for rows in sp:
            out.append((rows,) + tuple(s[1:]))
            parents.append((i, r0))
            r0 += rows
    return out, parents


def gen_hadamard_rows(m: int, blocks: int, seed: int, device: str = "cpu"):
    """Seeded structured input with orthogonal rows, for closed-form checks at
    sizes the float64 oracle cannot run in seconds.

    X (m x blocks*m, m a power of two) is `blocks` column blocks; block j is
    d_j * diag(r) * P * H_m * Q_j, where H_m is the Sylvester Hadamard matrix
    (entry (i, k) = (-1)^popcount(i & k)), P a seeded row permutation, Q_j a
    seeded signed column permutation, and r_i, d_j are drawn from
    {1, 1.125, ..., 1.875}. Every entry is +-(8 + u)(8 + v) / 64 with
    u, v < 8: at most 8 significant bits, so X is exact in bf16.
    Returns (X as bf16 on `device`, r, d) with r and d as lists of floats.
    The seeded draws come from numpy; the rest is integer and exact float
    arithmetic, so every device gives the same bits.
    """
    import numpy as np

    if m < 1 or m & (m - 1):
        raise ValueError("m must be a power of two")
    rng = np.random.default_rng(seed)
    r = (8 + rng.integers(0, 8, m)) / 8.0
    d = (8 + rng.integers(0, 8, blocks)) / 8.0
    rows = torch.from_numpy(rng.permutation(m).astype(np.int32)).to(device)
    r_t = torch.from_numpy(r.astype(np.float32)).to(device)
    out = torch.empty((m, blocks * m), dtype=torch.bfloat16, device=device)
    for j in range(blocks):
        cols = torch.from_numpy(rng.permutation(m).astype(np.int32)).to(device)
        sign = torch.from_numpy((1 - 2 * rng.integers(0, 2, m)).astype(np.float32)).to(device)
        v = rows[:, None] & cols[None, :]
        for sh in (16, 8, 4, 2, 1):
            v ^= v >> sh
        mag = r_t[:, None] * (sign * float(d[j]))[None, :]        # exact: <= 8 significant bits
        out[:, j * m:(j + 1) * m] = torch.where((v & 1).bool(), -mag, mag).to(torch.bfloat16)
    return out, [float(x) for x in r], [float(x) for x in d]
