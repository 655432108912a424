"""Shape-batched quintic Newton-Schulz for GB300 (sm_103a), with the
shard -> home pack and home -> shard unpack of layer-sharded Muon.

Thin Python binding of ``libnsgb300.so`` (C ABI in ``include/nsgb300.h``):
the functions below keep the C names and only marshal arguments. Every step
of the hot path runs in the library's CUDA kernels; if the library is missing
the import fails.

Buffers are torch CUDA tensors (or raw device addresses as ints); streams
default to torch's current stream.
"""

from __future__ import annotations

import ctypes

from ._lib import (NS_BF16, NS_ERR_ARG, NS_ERR_CUDA, NS_ERR_DEVICE_CHECK, NS_ERR_HOME,  # noqa: F401
                   NS_ERR_NOT_DIVISIBLE, NS_ERR_SHAPE, NS_ERR_TIMEOUT, NS_ERR_UNSUPPORTED,
                   NS_ERR_WORKSPACE, NS_FP32_GRAM, NS_FP32_GRAM_SPACE, NS_FP32_AUTO, NS_LAYOUT_FLAT, NS_LAYOUT_ROW_SHARD, NS_LAYOUT_TWO_STAGE, NS_OK,
                   LIB_PATH, NsError, check, header_symbols, i32_array, i64_array, lib, ptr_array)

A_COEF, B_COEF, C_COEF = 3.4445, -4.7750, 2.0315


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "is_contiguous") and not x.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def ns_status_string(code: int) -> str:
    return lib.ns_status_string(code).decode()


def ns_cost(shape, steps: int = 5) -> int:
    """owner_planning, ns_cost_fn: numel * (min(rows, cols) * steps + 1)."""
    out = ctypes.c_int64()
    check(lib.ns_cost(i64_array(shape), len(shape), steps, ctypes.byref(out)), "ns_cost")
    return out.value


def ns_assign_owner_work(costs, candidates, n_ranks: int) -> list:
    """owner_planning, assign_owner_work (greedy LPT). candidates[i] lists the
    ranks holding tensor i, in buffer order."""
    n = len(costs)
    ptr, idx = [0], []
    for c in candidates:
        idx += list(c)
        ptr.append(len(idx))
    out = (ctypes.c_int32 * max(1, n))()
    check(lib.ns_assign_owner_work(n, i64_array(costs), i32_array(ptr), i32_array(idx), n_ranks, out),
          "ns_assign_owner_work")
    return list(out[:n])


class NsPlan:
    """Owns an ns_plan_t*; destroyed with the object."""

    def __init__(self, handle: ctypes.c_void_p, n_tensors: int, S: int):
        self._h = handle
        self.n_tensors = n_tensors
        self.S = S
        info = self.info()
        self.n_participating = int(info[1])
        self.layout = int(info[3])
        self.gram_mode = int(info[4])
        self.steps = int(info[5])
        self.n_buckets = int(info[6])
        self.rank_len = int(info[7])
        self.in_bytes = int(info[8])
        self.out_bytes = int(info[9])

    @property
    def handle(self):
        return self._h

    def info(self) -> list:
        buf = (ctypes.c_int64 * 10)()
        check(lib.ns_plan_info(self._h, buf), "ns_plan_info")
        return list(buf)

    def homes(self) -> list:
        buf = (ctypes.c_int32 * max(1, self.n_tensors))()
        check(lib.ns_plan_homes(self._h, buf), "ns_plan_homes")
        return list(buf[:self.n_tensors])

    def home_layout(self):
        ho = (ctypes.c_int64 * max(1, self.n_tensors))()
        hs = (ctypes.c_int64 * self.S)()
        rs = (ctypes.c_int64 * self.S)()
        check(lib.ns_plan_home_layout(self._h, ho, hs, rs), "ns_plan_home_layout")
        return list(ho[:self.n_tensors]), list(hs), list(rs)

    def workspace_bytes(self) -> int:
        out = ctypes.c_uint64()
        check(lib.ns_plan_workspace_bytes(self._h, ctypes.byref(out)), "ns_plan_workspace_bytes")
        return out.value

    def owner_gather_meta(self, rho: int):
        n, S = self.n_tensors, self.S
        send, recv = (ctypes.c_int64 * S)(), (ctypes.c_int64 * S)()
        roff, own = (ctypes.c_int64 * max(1, n * S))(), (ctypes.c_int64 * max(1, n))()
        check(lib.ns_owner_gather_meta(self._h, rho, send, recv, roff, own), "ns_owner_gather_meta")
        return list(send), list(recv), [list(roff[i * S:(i + 1) * S]) for i in range(n)], list(own[:n])

    def owner_scatter_meta(self, rho: int):
        n, S = self.n_tensors, self.S
        send, recv = (ctypes.c_int64 * S)(), (ctypes.c_int64 * S)()
        roff = (ctypes.c_int64 * max(1, n * S))()
        check(lib.ns_owner_scatter_meta(self._h, rho, send, recv, roff), "ns_owner_scatter_meta")
        return list(send), list(recv), [list(roff[i * S:(i + 1) * S]) for i in range(n)]

    def rank_splits(self, rho: int):
        """route_to_ns_home as one all_to_allv seen from rank rho:
        (send_counts, send_displs, recv_counts, recv_displs, send_pos, recv_pos)
        with recv_pos[i][s] the offset of rank s's piece of tensor i."""
        n, S = self.n_tensors, self.S
        sc, sd, rc, rd = [(ctypes.c_int64 * S)() for _ in range(4)]
        sp, rp = (ctypes.c_int64 * max(1, n))(), (ctypes.c_int64 * max(1, n * S))()
        check(lib.ns_plan_rank_splits(self._h, rho, sc, sd, rc, rd, sp, rp), "ns_plan_rank_splits")
        return (list(sc), list(sd), list(rc), list(rd), list(sp[:n]),
                [list(rp[i * S:(i + 1) * S]) for i in range(n)])

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.ns_plan_destroy(h)
            self._h = None


def _shape_args(shapes):
    ndims = [len(s) for s in shapes]
    flat = [int(d) for s in shapes for d in s]
    return i32_array(ndims), i64_array(flat)


def ns_plan_create(shapes, steps: int = 5, a: float = A_COEF, b: float = B_COEF, c: float = C_COEF,
                   eps: float = 1e-7, gram_mode: int = NS_BF16, ridge: float = 0.0, S: int = 1,
                   shard_dim: int = 0, home_of=None) -> NsPlan:
    """Row-shard plan (layer_sharded_a2a): homes from home_of, or LPT if None."""
    nd, sh = _shape_args(shapes)
    h = ctypes.c_void_p()
    homes = i32_array(home_of) if home_of is not None else None
    check(lib.ns_plan_create(len(shapes), nd, sh, steps, a, b, c, eps, gram_mode, ridge, S, shard_dim,
                             homes, ctypes.byref(h)), "ns_plan_create")
    plan = NsPlan(h, len(shapes), S)
    plan.shard_dim = shard_dim
    return plan


def ns_plan_create_two_stage(shapes, partition_dims, R: int, T: int, steps: int = 5, a: float = A_COEF,
                             b: float = B_COEF, c: float = C_COEF, eps: float = 1e-7, gram_mode: int = NS_BF16,
                             ridge: float = 0.0, home_of=None) -> NsPlan:
    """Two-stage (GTP_remat x TP) plan (layer_sharded_a2a), fused into one gather."""
    nd, sh = _shape_args(shapes)
    h = ctypes.c_void_p()
    homes = i32_array(home_of) if home_of is not None else None
    check(lib.ns_plan_create_two_stage(len(shapes), nd, sh, i32_array(partition_dims), R, T, steps, a, b, c, eps,
                                       gram_mode, ridge, homes, ctypes.byref(h)), "ns_plan_create_two_stage")
    plan = NsPlan(h, len(shapes), R * T)
    plan.shard_dim = 0
    return plan


def ns_plan_create_flat(shapes, offsets, buffer_size: int, participating=None, steps: int = 5,
                        a: float = A_COEF, b: float = B_COEF, c: float = C_COEF, eps: float = 1e-7,
                        gram_mode: int = NS_BF16, ridge: float = 0.0, S: int = 1, owner_of=None) -> NsPlan:
    """Flat-buffer plan (owner_planning): owners from owner_of, or LPT if None."""
    nd, sh = _shape_args(shapes)
    h = ctypes.c_void_p()
    part = (ctypes.c_uint8 * max(1, len(shapes)))(*[1 if p else 0 for p in participating]) \
        if participating is not None else None
    owners = i32_array([(-1 if o is None else o) for o in owner_of]) if owner_of is not None else None
    check(lib.ns_plan_create_flat(len(shapes), nd, sh, i64_array(offsets), buffer_size, part, steps, a, b, c,
                                  eps, gram_mode, ridge, S, owners, ctypes.byref(h)), "ns_plan_create_flat")
    plan = NsPlan(h, len(shapes), S)
    plan.shard_dim = 0
    return plan


def ns_orthogonalize_batched(plan: NsPlan, ins, outs, workspace, workspace_bytes=None, stream=None) -> None:
    """Newton-Schulz on the plan's participating tensors (index order)."""
    n = len(ins)
    if len(outs) != n:
        raise ValueError("ins and outs differ in length")
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.ns_orthogonalize_batched(plan.handle, ptr_array([_addr(t) for t in ins]),
                                       ptr_array([_addr(t) for t in outs]), n, _addr(workspace),
                                       int(workspace_bytes), _stream(stream)), "ns_orthogonalize_batched")


NS_FIXED_WS_BYTES = 64 << 20


def ns_orthogonalize_batched_fixed_ws(plan: NsPlan, ins, outs, stream=None) -> None:
    """Same as ns_orthogonalize_batched, for callers that cannot allocate a
    workspace: the library's static scratch array of NS_FIXED_WS_BYTES is used
    instead. Plans needing more raise NS_ERR_WORKSPACE; calls that overlap on
    the GPU share that array and race."""
    n = len(ins)
    if len(outs) != n:
        raise ValueError("ins and outs differ in length")
    check(lib.ns_orthogonalize_batched_fixed_ws(plan.handle, ptr_array([_addr(t) for t in ins]),
                                                ptr_array([_addr(t) for t in outs]), n, _stream(stream)),
          "ns_orthogonalize_batched_fixed_ws")


def ns_pack_to_home(plan: NsPlan, rank_bufs, home_bufs, shard_dim=None, stream=None) -> None:
    """route_to_ns_home / OwnerGatherPlan: S rank buffers -> S home buffers."""
    sd = 0 if plan.layout != NS_LAYOUT_ROW_SHARD else (shard_dim if shard_dim is not None else _plan_shard_dim(plan))
    check(lib.ns_pack_to_home(plan.handle, ptr_array([_addr(t) for t in rank_bufs]), len(rank_bufs), sd,
                              ptr_array([_addr(t) for t in home_bufs]), _stream(stream)), "ns_pack_to_home")


def ns_unpack_from_home(plan: NsPlan, home_bufs, rank_bufs, shard_dim=None, stream=None) -> None:
    """route_from_ns_home / OwnerScatterPlan: S home buffers -> S rank buffers."""
    sd = 0 if plan.layout != NS_LAYOUT_ROW_SHARD else (shard_dim if shard_dim is not None else _plan_shard_dim(plan))
    check(lib.ns_unpack_from_home(plan.handle, ptr_array([_addr(t) for t in home_bufs]), len(home_bufs), sd,
                                  ptr_array([_addr(t) for t in rank_bufs]), _stream(stream)), "ns_unpack_from_home")


def _plan_shard_dim(plan: NsPlan) -> int:
    return getattr(plan, "shard_dim", 0)


def ns_check_status(plan: NsPlan = None, stream=None) -> int:
    """Synchronise the stream and return the device status (NS_OK or an error code)."""
    return lib.ns_check_status(plan.handle if plan is not None else None, _stream(stream))


KERNEL_KINDS = ("gram", "a2b", "bx", "prologue_store", "pack_unpack", "bx_final", "small")


def ns_profile_enable(enable: bool = True) -> None:
    """Per-launch CUDA-event timing inside the library (measurement only)."""
    check(lib.ns_profile_enable(1 if enable else 0), "ns_profile_enable")


def ns_profile_read(reset: bool = False):
    """Return ({kind: launches}, {kind: summed gpu ms}) since the last reset."""
    n = (ctypes.c_int64 * len(KERNEL_KINDS))()
    ms = (ctypes.c_double * len(KERNEL_KINDS))()
    check(lib.ns_profile_read(1 if reset else 0, n, ms), "ns_profile_read")
    return dict(zip(KERNEL_KINDS, list(n))), dict(zip(KERNEL_KINDS, list(ms)))


def ns_set_gemm_cluster(cl: int) -> None:
    """GEMM tiling: 0 automatic (2-SM MMA for the Gram and A*A, and for B*X when
    every bucket has an even number of 128-row tile rows), 1 single CTA,
    3 2-SM MMA."""
    check(lib.ns_set_gemm_cluster(cl), "ns_set_gemm_cluster")


def ns_set_small_path(enable: bool) -> None:
    """bf16 buckets with m <= 128 and n <= 512: one CTA per matrix for the whole
    iteration (True, the default) or the GEMM launches (False)."""
    check(lib.ns_set_small_path(1 if enable else 0), "ns_set_small_path")


def ns_set_symmetric_store(mode: int) -> None:
    """bf16 A and B: 0 stores only the upper 256 x 256 pair blocks (readers
    take the rest transposed; the default), 1 also stores the mirror."""
    check(lib.ns_set_symmetric_store(mode), "ns_set_symmetric_store")


class NsPipeline:
    """Owns an ns_pipeline_t* (wave-dispatched pack -> NS -> unpack)."""

    def __init__(self, plan: NsPlan, n_waves: int):
        self.plan = plan          # keeps the plan alive
        self._h = ctypes.c_void_p()
        check(lib.ns_pipeline_create(plan.handle, n_waves, ctypes.byref(self._h)), "ns_pipeline_create")
        w = ctypes.c_int()
        b = ctypes.c_uint64()
        check(lib.ns_pipeline_info(self._h, ctypes.byref(w), ctypes.byref(b)), "ns_pipeline_info")
        self.n_waves = w.value
        self.workspace_bytes = b.value

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.ns_pipeline_destroy(h)
            self._h = None


def ns_pipeline_create(plan: NsPlan, n_waves: int) -> NsPipeline:
    return NsPipeline(plan, n_waves)


def ns_pipeline_run(pipe: NsPipeline, rank_in, home_in, home_out, rank_out, workspace, stream=None) -> None:
    """Wave-dispatched pack -> Newton-Schulz -> unpack over the whole plan."""
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.ns_pipeline_run(pipe._h, ptr_array([_addr(t) for t in rank_in]),
                              ptr_array([_addr(t) for t in home_in]), ptr_array([_addr(t) for t in home_out]),
                              ptr_array([_addr(t) for t in rank_out]), _addr(workspace), nbytes, _stream(stream)),
          "ns_pipeline_run")


def ns_test_stall_next_gemm(wait_limit_ns: int) -> None:
    """Test support: the next bf16 GEMM launch stalls and its bounded waits run
    out after wait_limit_ns; ns_check_status then reports NS_ERR_TIMEOUT."""
    check(lib.ns_test_stall_next_gemm(int(wait_limit_ns)), "ns_test_stall_next_gemm")


def ns_test_set_route_home(plan: NsPlan, tensor: int, home: int) -> None:
    """Test support: overwrite a tensor's home in the plan's routing table
    (out-of-range values make pack/unpack refuse it: NS_ERR_DEVICE_CHECK)."""
    check(lib.ns_test_set_route_home(plan.handle, tensor, home), "ns_test_set_route_home")
