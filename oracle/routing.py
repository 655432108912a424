"""Oracle: shard -> home pack and home -> shard unpack, on the CPU.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Two data models, one per page:

Row-shard model -- Megatron-Core API page ``core.optimizer.layer_sharded_a2a``
    (``route_to_ns_home`` / ``route_from_ns_home``). Every rank r holds a
    (P/S, Q) shard of every param: the slice r of S equal slices along
    ``shard_dim``. The home assembles the complete (P, Q) tensor; the
    backward exchange hands every rank its shard of every result. On one GPU
    "rank r" is a flat buffer holding rank r's shards of all params in index
    order, and "home h" is a flat buffer holding the complete params homed on
    h, in increasing index order (the order ``params_by_home`` fixes).

Flat-buffer model -- Megatron-Core API page ``core.distributed.fsdp.src.
    megatron_fsdp.experimental.owner_planning`` (``OwnerGatherPlan``,
    ``OwnerScatterPlan``). One flat buffer of ``size`` elements is split into
    S equal rank ranges; tensor i occupies [offset_i, offset_i + numel_i).
    The metadata of both plans is computed here from one rank's point of view,
    as the page's worked example does.

Everything here is data movement written with numpy slicing and
concatenation; values are never interpreted, so bit patterns (e.g. uint16
views of bf16) pass through unchanged.
"""

from __future__ import annotations

import numpy as np

from .planning import params_by_home, rank_range


# ------------------------------------------------------------ row-shard model

def _split_dims(shape, shard_dim: int) -> tuple[int, int, int]:
    pre = 1
    for d in shape[:shard_dim]:
        pre *= int(d)
    post = 1
    for d in shape[shard_dim + 1:]:
        post *= int(d)
    return pre, int(shape[shard_dim]), post


def _numel(shape) -> int:
    n = 1
    for d in shape:
        n *= int(d)
    return n


def shard_of(t: np.ndarray, r: int, S: int, shard_dim: int) -> np.ndarray:
    """Rank r's (P/S, Q) shard of t: slice r of S equal slices along
    shard_dim (layer_sharded_a2a, route_to_ns_home)."""
    D = t.shape[shard_dim]
    if D % S:
        raise ValueError("shard_dim size is not divisible by S")
    w = D // S
    idx = [slice(None)] * t.ndim
    idx[shard_dim] = slice(r * w, (r + 1) * w)
    return t[tuple(idx)]


def make_rank_buffers(tensors, S: int, shard_dim: int) -> list[np.ndarray]:
    """Rank r's flat buffer: its shard of every param, in param index order."""
    out = []
    for r in range(S):
        parts = [np.ascontiguousarray(shard_of(t, r, S, shard_dim)).reshape(-1)
                 for t in tensors]
        out.append(np.concatenate(parts) if parts else np.zeros(0, np.uint16))
    return out


def route_to_ns_home(rank_buffers, shapes, home_of: dict, S: int,
                     shard_dim: int) -> list[np.ndarray]:
    """Pack (layer_sharded_a2a, route_to_ns_home): S rank buffers -> S home
    buffers. Home h holds the complete tensors of params_by_home(...)[h],
    each assembled by concatenating the S shards along shard_dim, in
    increasing param index order."""
    n = len(shapes)
    dtype = rank_buffers[0].dtype if S else np.uint16
    # cut every rank buffer into its per-param shards (index order)
    shards = [[None] * S for _ in range(n)]
    for r in range(S):
        pos = 0
        for i, shp in enumerate(shapes):
            pre, D, post = _split_dims(shp, shard_dim)
            cnt = pre * (D // S) * post
            shards[i][r] = rank_buffers[r][pos:pos + cnt].reshape(pre, D // S, post)
            pos += cnt
        if pos != rank_buffers[r].size:
            raise ValueError("rank buffer size does not match the shapes")
    homes = params_by_home(n, home_of, S)
    out = []
    for h in range(S):
        parts = [np.concatenate(shards[i], axis=1).reshape(-1) for i in homes[h]]
        out.append(np.concatenate(parts) if parts else np.zeros(0, dtype))
    return out


def route_from_ns_home(home_buffers, shapes, home_of: dict, S: int,
                       shard_dim: int) -> list[np.ndarray]:
    """Unpack (layer_sharded_a2a, route_from_ns_home): S home buffers of
    complete results -> S rank buffers, rank r getting its (P/S, Q) shard of
    every result in param index order."""
    n = len(shapes)
    homes = params_by_home(n, home_of, S)
    full = [None] * n
    for h in range(S):
        pos = 0
        for i in homes[h]:
            cnt = _numel(shapes[i])
            full[i] = home_buffers[h][pos:pos + cnt].reshape(shapes[i])
            pos += cnt
        if pos != home_buffers[h].size:
            raise ValueError("home buffer size does not match the shapes")
    return make_rank_buffers(full, S, shard_dim)


def home_offsets(shapes, home_of: dict, S: int) -> list[int]:
    """Element offset of each param inside its home buffer."""
    homes = params_by_home(len(shapes), home_of, S)
    off = [0] * len(shapes)
    for h in range(S):
        pos = 0
        for i in homes[h]:
            off[i] = pos
            pos += _numel(shapes[i])
    return off


# --------------------------------------------------------- flat-buffer model

def piece(off: int, numel: int, r: int, size: int, S: int):
    """Global [lo, hi) of tensor [off, off+numel) held by rank r, or None."""
    lo_r, hi_r = rank_range(r, size, S)
    lo, hi = max(off, lo_r), min(off + numel, hi_r)
    return (lo, hi) if lo < hi else None


def _check_owners(offsets, numels, size, S, owner_of):
    for i, o in owner_of.items():
        if piece(offsets[i], numels[i], o, size, S) is None:
            raise ValueError(f"owner {o} of tensor {i} holds none of it")


def owner_gather_plan(offsets, numels, size: int, S: int, owner_of: dict, rho: int) -> dict:
    """OwnerGatherPlan metadata seen from rank rho (owner_planning page).

    Returns a dict with
      send:         {owner: [(i, lo, hi), ...]}  pieces in tensor-index order;
                    only owners != rho with a non-zero total appear;
      send_sizes:   {owner: total}
      recv_sizes:   {src: total} for src != rho, non-zero only;
      own_shards:   {i: (lo, hi)} rho's own piece of each tensor it owns;
      recv_offsets: {(i, src): offset} of i's piece inside src's buffer to
                    rho, only where src holds elements of i.
    Ranges are global [lo, hi) positions in the flat buffer.
    """
    _check_owners(offsets, numels, size, S, owner_of)
    order = sorted(owner_of)
    send: dict[int, list] = {}
    for i in order:
        o = owner_of[i]
        if o == rho:
            continue
        p = piece(offsets[i], numels[i], rho, size, S)
        if p is not None:
            send.setdefault(o, []).append((i, p[0], p[1]))
    send_sizes = {o: sum(hi - lo for _, lo, hi in v) for o, v in send.items()}
    recv_sizes: dict[int, int] = {}
    recv_offsets: dict[tuple, int] = {}
    own: dict[int, tuple] = {}
    for src in range(S):
        if src == rho:
            continue
        pos = 0
        for i in order:
            if owner_of[i] != rho:
                continue
            p = piece(offsets[i], numels[i], src, size, S)
            if p is None:
                continue
            recv_offsets[(i, src)] = pos
            pos += p[1] - p[0]
        if pos:
            recv_sizes[src] = pos
    for i in order:
        if owner_of[i] == rho:
            own[i] = piece(offsets[i], numels[i], rho, size, S)
    return {"send": send, "send_sizes": send_sizes, "recv_sizes": recv_sizes,
            "own_shards": own, "recv_offsets": recv_offsets}


def gather_send_buffers(plan: dict, flat: np.ndarray) -> dict:
    """Materialise rho's send buffers from the global flat buffer's contents
    (OwnerGatherPlan.pack: this rank's shards for each owner, index order)."""
    return {o: np.concatenate([flat[lo:hi] for _, lo, hi in v])
            for o, v in plan["send"].items()}


def reconstruct_full(plan: dict, i: int, offsets, numels, size: int, S: int,
                     rho: int, recv_buffers: dict, flat_local: np.ndarray) -> np.ndarray:
    """OwnerGatherPlan.reconstruct_full: concatenate the per-rank pieces of
    owned tensor i in buffer order; rho's own piece comes from its local
    range ``flat_local`` (the contents of [lo_rho, hi_rho))."""
    lo_rho, _ = rank_range(rho, size, S)
    parts = []
    for r in range(S):
        p = piece(offsets[i], numels[i], r, size, S)
        if p is None:
            continue
        n = p[1] - p[0]
        if r == rho:
            parts.append(flat_local[p[0] - lo_rho:p[1] - lo_rho])
        else:
            off = plan["recv_offsets"][(i, r)]
            parts.append(recv_buffers[r][off:off + n])
    return np.concatenate(parts)


def owner_scatter_plan(offsets, numels, size: int, S: int, owner_of: dict, rho: int) -> dict:
    """OwnerScatterPlan metadata seen from rank rho (owner_planning page).

    send:         {dest: [(i, lo, hi), ...]} pieces of results rho owns that
                  dest holds (dest != rho), tensor-index order, non-zero only;
    send_sizes:   {dest: total};
    recv_sizes:   {owner: total} rho receives from each owner != rho;
    recv_offsets: {(i, owner): offset} of i's piece inside owner's buffer to
                  rho, only where rho holds elements of i.
    """
    _check_owners(offsets, numels, size, S, owner_of)
    order = sorted(owner_of)
    send: dict[int, list] = {}
    for dest in range(S):
        if dest == rho:
            continue
        for i in order:
            if owner_of[i] != rho:
                continue
            p = piece(offsets[i], numels[i], dest, size, S)
            if p is not None:
                send.setdefault(dest, []).append((i, p[0], p[1]))
    send_sizes = {d: sum(hi - lo for _, lo, hi in v) for d, v in send.items()}
    recv_sizes: dict[int, int] = {}
    recv_offsets: dict[tuple, int] = {}
    for o in range(S):
        if o == rho:
            continue
        pos = 0
        for i in order:
            if owner_of[i] != o:
                continue
            p = piece(offsets[i], numels[i], rho, size, S)
            if p is None:
                continue
            recv_offsets[(i, o)] = pos
            pos += p[1] - p[0]
        if pos:
            recv_sizes[o] = pos
    return {"send": send, "send_sizes": send_sizes, "recv_sizes": recv_sizes,
            "recv_offsets": recv_offsets}


def scatter_unpack(plan: dict, offsets, numels, size: int, S: int, owner_of: dict,
                   rho: int, recv_buffers: dict) -> dict:
    """OwnerScatterPlan.unpack: {i: rho's flat result piece} for tensors rho
    holds elements of but does not own."""
    out = {}
    for (i, o), off in plan["recv_offsets"].items():
        p = piece(offsets[i], numels[i], rho, size, S)
        out[i] = recv_buffers[o][off:off + (p[1] - p[0])]
    return out


def flat_pack_to_owner(rank_buffers, offsets, numels, size: int, S: int,
                       owner_of: dict) -> list[np.ndarray]:
    """Single-GPU end result of the owner gather: owner h's buffer holds the
    complete flat tensors it owns, in tensor-index order (what
    reconstruct_full returns for each owned tensor)."""
    flat = np.concatenate(rank_buffers)
    if flat.size != size:
        raise ValueError("rank buffers do not add up to the buffer size")
    out = []
    for h in range(S):
        parts = [flat[offsets[i]:offsets[i] + numels[i]]
                 for i in sorted(owner_of) if owner_of[i] == h]
        out.append(np.concatenate(parts) if parts else np.zeros(0, flat.dtype))
    return out


def flat_unpack_from_owner(home_buffers, rank_buffers_before, offsets, numels,
                           size: int, S: int, owner_of: dict) -> list[np.ndarray]:
    """Single-GPU end result of the owner scatter: every rank's range of the
    flat buffer receives the results of the participating tensors; elements
    outside participating tensors keep their previous contents."""
    flat = np.concatenate([np.array(b, copy=True) for b in rank_buffers_before])
    if flat.size != size:
        raise ValueError("rank buffers do not add up to the buffer size")
    for h in range(S):
        pos = 0
        for i in sorted(owner_of):
            if owner_of[i] != h:
                continue
            flat[offsets[i]:offsets[i] + numels[i]] = home_buffers[h][pos:pos + numels[i]]
            pos += numels[i]
    per = size // S
    return [flat[r * per:(r + 1) * per] for r in range(S)]


# --------------------------------------------------- two-stage (GTP_remat x TP)
#
# Megatron-Core API page core.optimizer.layer_sharded_a2a: the exchange runs
# in two stages, first over the GTP_remat group along dim 0, then over the TP
# group along the param's partition_dim; the Megatron-LM issue #6720 reports
# fusing the two into one exchange. Model: R remat ranks x T TP ranks, rank
# rho = r * T + t. TP shard t of a param is slice t of T along partition_dim;
# rank (r, t) holds slice r of R along dim 0 of that TP shard. The home of a
# param is one of the R * T ranks.

def two_stage_piece(x: np.ndarray, r: int, t: int, R: int, T: int, pdim: int) -> np.ndarray:
    """Rank (r, t)'s piece: TP slice t along pdim, then remat slice r along dim 0."""
    tp = shard_of(x, t, T, pdim)
    return shard_of(tp, r, R, 0)


def make_rank_buffers_two_stage(tensors, R: int, T: int, pdims) -> list[np.ndarray]:
    out = []
    for r in range(R):
        for t in range(T):
            parts = [np.ascontiguousarray(two_stage_piece(x, r, t, R, T, pd)).reshape(-1)
                     for x, pd in zip(tensors, pdims)]
            out.append(np.concatenate(parts) if parts else np.zeros(0, np.uint16))
    return out


def route_two_stage(rank_buffers, shapes, pdims, home_of: dict, R: int, T: int) -> list[np.ndarray]:
    """The two exchanges done literally: stage 1 gathers, inside each TP rank's
    remat group, the dim-0 slices of every param onto the remat coordinate of
    its home (concatenation along dim 0 rebuilds the TP shard); stage 2
    gathers, inside the home's TP group, the TP shards onto the home
    (concatenation along partition_dim). Returns the R*T home buffers."""
    n = len(shapes)
    S = R * T
    # cut every rank buffer into pieces
    pieces = {}
    for r in range(R):
        for t in range(T):
            buf = rank_buffers[r * T + t]
            pos = 0
            for i, shp in enumerate(shapes):
                shp_t = list(shp)
                shp_t[pdims[i]] //= T
                shp_p = list(shp_t)
                shp_p[0] //= R
                cnt = _numel(shp_p)
                pieces[(i, r, t)] = buf[pos:pos + cnt].reshape(shp_p)
                pos += cnt
    # stage 1: remat group of TP rank t gathers along dim 0
    tp_shards = {}
    for i in range(n):
        for t in range(T):
            tp_shards[(i, t)] = np.concatenate([pieces[(i, r, t)] for r in range(R)], axis=0)
    # stage 2: the home's TP group gathers along partition_dim
    full = [np.concatenate([tp_shards[(i, t)] for t in range(T)], axis=pdims[i]) for i in range(n)]
    homes = params_by_home(n, home_of, S)
    return [np.concatenate([full[i].reshape(-1) for i in homes[h]]) if homes[h]
            else np.zeros(0, rank_buffers[0].dtype) for h in range(S)]


def route_two_stage_back(home_buffers, shapes, pdims, home_of: dict, R: int, T: int) -> list[np.ndarray]:
    """Inverse of route_two_stage: every rank gets its piece of every result."""
    n = len(shapes)
    homes = params_by_home(n, home_of, R * T)
    full = [None] * n
    for h in range(R * T):
        pos = 0
        for i in homes[h]:
            cnt = _numel(shapes[i])
            full[i] = home_buffers[h][pos:pos + cnt].reshape(shapes[i])
            pos += cnt
    return make_rank_buffers_two_stage(full, R, T, pdims)
