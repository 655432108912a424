"""Helpers shared by the GPU parity tests (data plumbing only)."""

import numpy as np
import torch

import workloads
from oracle import ns as ons

BF16_TOL = 3e-2          # per-matrix relative Frobenius error, bf16 path


def oracle_ns(t: torch.Tensor, steps=workloads.STEPS) -> np.ndarray:
    return ons.newton_schulz(t.float().numpy(), steps, workloads.A_COEF, workloads.B_COEF,
                             workloads.C_COEF, workloads.EPS)


def rel_err(gpu_out: torch.Tensor, ref: np.ndarray) -> float:
    return ons.rel_fro_error(gpu_out.float().cpu().numpy(), ref)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a tensor (for bit-exact comparisons)."""
    t = t.contiguous().cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


def run_ns(nsg, shapes, tensors, steps=workloads.STEPS, inplace=False):
    dev = torch.device("cuda:0")
    ins = [t.to(dev) for t in tensors]
    outs = ins if inplace else [torch.empty_like(t) for t in ins]
    plan = nsg.ns_plan_create(shapes, steps=steps, eps=workloads.EPS, S=1)
    ws = torch.empty(max(1, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
    nsg.ns_orthogonalize_batched(plan, ins, outs, ws)
    rc = nsg.ns_check_status(plan)
    assert rc == nsg.NS_OK, nsg.ns_status_string(rc)
    return outs
