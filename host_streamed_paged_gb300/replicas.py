"""Host-side helpers for running the path as independent replicas, one per GPU.

The attention path has no exchange between GPUs (one sequence's history lives
on one device), so N processes each run their own replica; the only
cross-process steps are the timing barrier, the max over ranks of the step
time and the aggregate throughput.  These helpers work with any
``torch.distributed`` backend (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations

import hashlib
import struct


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (the value itself without a process group)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rows_per_s(rows_per_step: int, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every replica processes `rows_per_step` rows per step,
    and the slowest replica's step time bounds the job."""
    if ms_per_step <= 0:
        raise ValueError("step time must be positive")
    return world * rows_per_step / (ms_per_step * 1e-3)


def plan_signature(trace) -> str:
    """A digest of a plan-only trace (the ordered operations a context would
    enqueue): replicas given the same configuration and calls must agree."""
    h = hashlib.sha256()
    for t in trace:
        h.update(struct.pack("<8q", *(int(t[k]) for k in ("op", "stream", "layer", "event", "a", "b", "c", "d"))))
    return h.hexdigest()
