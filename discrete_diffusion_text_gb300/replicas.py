"""Host logic of data-parallel replicas (one process per GPU, independent canvases).

Canvases are independent requests, so the denoising core shards as replicas with no data
exchange: each rank draws its own canvases (distinct Philox seeds), runs the same workload,
and only the timing is combined: the job's time is the slowest rank's, and throughput counts
every rank's canvases.
"""

from __future__ import annotations


def replica_seed(base_seed: int, rank: int, step: int) -> int:
    """A 64-bit Philox seed unique to (workload seed, rank, benchmark step)."""
    return ((int(base_seed) << 32) + 1_000_003 * int(rank) + int(step)) & 0xFFFFFFFFFFFFFFFF


def max_over_ranks(value: float, group=None) -> float:
    """Maximum of a per-rank float over the process group (identity without one)."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized():
        return float(value)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def job_throughput(world: int, L: int, B: int, denoise_steps: float, seconds_per_step: float) -> float:
    """Canvas tokens x denoising steps per second for the whole job (all ranks)."""
    return world * L * B * denoise_steps / seconds_per_step
