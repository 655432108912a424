"""Oracle: owner / home planning on the CPU, in exact Python integers.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Sources
-------
* Megatron-Core API page ``core.distributed.fsdp.src.megatron_fsdp.
  experimental.owner_planning``: ``select_ge_2d_params``, ``ns_cost_fn``,
  ``_OwnerWork``, ``assign_owner_work``, and the OwnerGatherPlan example
  (a flat buffer split evenly across ranks).
* Megatron-Core API page ``core.optimizer.layer_sharded_a2a``:
  ``params_by_home`` and the (P/S, Q) row-shard model of ``route_to_ns_home``.

Readings where the pages are silent:

* costs are exact integers (``ns_cost_fn`` is documented to return an int);
* the buffer-order tie rule applies both to equal costs (stable order by
  tensor index, tensors being in buffer order) and to equally loaded holders
  (the earliest candidate in buffer order, i.e. the lowest rank);
* single-candidate tensors are taken in tensor-index order and their cost
  counts toward the load seen by later tensors.
"""

from __future__ import annotations

from dataclasses import dataclass


def view_2d(shape) -> tuple[int, int]:
    """(rows, cols) = (shape[0], prod(shape[1:])) -- owner_planning, ns_cost_fn."""
    if len(shape) < 2:
        raise ValueError("needs ndim >= 2")
    cols = 1
    for s in shape[1:]:
        cols *= int(s)
    return int(shape[0]), cols


def select_ge_2d(shape) -> bool:
    """Eligibility: the tensor has at least 2 dims -- owner_planning, select_ge_2d_params."""
    return len(shape) >= 2


def ns_cost(shape, num_ns_steps: int = 5) -> int:
    """numel * (min(rows, cols) * num_ns_steps + 1) -- owner_planning, ns_cost_fn."""
    rows, cols = view_2d(shape)
    return rows * cols * (min(rows, cols) * num_ns_steps + 1)


@dataclass
class OwnerWork:
    """A tensor's cost and eligible owners in buffer order -- owner_planning, _OwnerWork."""

    tensor_index: int
    cost: int
    candidates: list


def assign_owner_work(works: list[OwnerWork]) -> dict[int, int]:
    """Greedy LPT owner assignment -- owner_planning, assign_owner_work.

    Tensors with one candidate go first (in tensor-index order); then the
    rest in descending cost order (ties keep tensor-index order). Each goes
    to its least-loaded candidate; equal loads go to the candidate that comes
    first in buffer order. Returns {tensor_index: owner}.
    """
    works = sorted(works, key=lambda w: w.tensor_index)
    load: dict[int, int] = {}
    for w in works:
        if not w.candidates:
            raise ValueError(f"tensor {w.tensor_index} has no holder")
        for r in w.candidates:
            load.setdefault(r, 0)
    single = [w for w in works if len(w.candidates) == 1]
    multi = [w for w in works if len(w.candidates) > 1]
    # Python's sort is stable: equal costs keep tensor-index (buffer) order.
    multi.sort(key=lambda w: -w.cost)
    owner: dict[int, int] = {}
    for w in single + multi:
        best = w.candidates[0]
        for r in w.candidates[1:]:
            if load[r] < load[best]:
                best = r
        owner[w.tensor_index] = best
        load[best] += w.cost
    return owner


def params_by_home(num_params: int, home_of: dict, size: int) -> list[list[int]]:
    """result[r] = indices homed on r, increasing -- layer_sharded_a2a, params_by_home."""
    result: list[list[int]] = [[] for _ in range(size)]
    for i in range(num_params):
        if i not in home_of:
            raise KeyError(f"home_of does not cover param {i}")
        h = home_of[i]
        if not 0 <= h < size:
            raise ValueError(f"home {h} of param {i} outside group of size {size}")
        result[h].append(i)
    return result


# ---------------------------------------------------------------- candidates

def row_shard_candidates(num_params: int, S: int) -> list[list[int]]:
    """Row-shard model: every rank holds a (P/S, Q) shard of every param
    (layer_sharded_a2a, route_to_ns_home), so every rank is a candidate."""
    return [list(range(S)) for _ in range(num_params)]


def rank_range(r: int, size: int, S: int) -> tuple[int, int]:
    """[lo, hi) of rank r when a flat buffer of `size` is split evenly
    (owner_planning, OwnerGatherPlan example: rank 0 holds [0, 20), rank 1
    holds [20, 40) of a 40-element buffer)."""
    if size % S:
        raise ValueError("buffer size must be divisible by the number of ranks")
    per = size // S
    return r * per, (r + 1) * per


def flat_candidates(offsets, numels, size: int, S: int) -> list[list[int]]:
    """Flat-buffer model: the ranks whose range intersects a tensor's
    [offset, offset + numel), in buffer (rank) order."""
    cands = []
    for off, n in zip(offsets, numels):
        c = []
        for r in range(S):
            lo, hi = rank_range(r, size, S)
            if max(lo, off) < min(hi, off + n):
                c.append(r)
        cands.append(c)
    return cands


def lpt_homes_row_shard(shapes, S: int, steps: int = 5) -> dict[int, int]:
    """Default homes for the row-shard model: LPT with all S candidates."""
    cands = row_shard_candidates(len(shapes), S)
    works = [OwnerWork(i, ns_cost(s, steps), cands[i]) for i, s in enumerate(shapes)]
    return assign_owner_work(works)


def lpt_owners_flat(shapes, offsets, size: int, S: int, tensor_indices=None,
                    steps: int = 5) -> dict[int, int]:
    """Default owners for the flat-buffer model (assign_owner_work over the
    participating tensors, default cost = NS with `steps` iterations)."""
    numels = []
    for s in shapes:
        n = 1
        for d in s:
            n *= int(d)
        numels.append(n)
    cands = flat_candidates(offsets, numels, size, S)
    if tensor_indices is None:
        tensor_indices = range(len(shapes))
    works = [OwnerWork(i, ns_cost(shapes[i], steps), cands[i]) for i in tensor_indices]
    return assign_owner_work(works)
