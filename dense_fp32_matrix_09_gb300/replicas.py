"""Replica bookkeeping for a run on several GPUs of one node.

The GEMM does not shard: one call is one problem on one GPU, and the method
has no exchange step.  Several GPUs therefore run independent replicas (one
process per GPU, each with its own copy of the inputs), and the only thing the
ranks share is the timing: every rank times its own steps, the job's time is
the slowest rank's (a MAX reduction over the process group, after a barrier),
and the job's rate is the work of all ranks divided by that time.  No
collective touches the data path.
"""
from __future__ import annotations


def slowest(ms: float, dist=None, device: str = "cpu") -> float:
    """The largest `ms` over the ranks of the default process group (`dist` =
    torch.distributed, initialised), or `ms` itself when dist is None.
    `device`: where the reduction tensor lives ("cuda" for NCCL, "cpu" for gloo)."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job rate in TFLOP/s: every rank did flop_per_rank_step per step,
    and a step of the job takes the slowest rank's ms_per_step."""
    if ms_per_step <= 0:
        raise ValueError("ms_per_step must be positive")
    return flop_per_rank_step * world / (ms_per_step * 1e-3) / 1e12
