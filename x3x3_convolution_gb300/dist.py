"""Rank-level helpers for running the library as independent replicas on several GPUs.

The path shards into independent units (images of a batch, passes of a video, frames of a pass), so
several GPUs run replicas with no collective on the data path. What the ranks do share is host-side
bookkeeping, which these helpers implement over torch.distributed (NCCL on GPUs, gloo on CPUs):
  * agreement on whether every rank could build and load the kernels before any of them uses them
    (FastVideo wan22_vae_decode commit message: the ranks of the parallel decode agree on whether
    every one of them could build the kernel, and fall back together otherwise);
  * the maximum over ranks of a measured time (a job is as slow as its slowest rank);
  * a contiguous, balanced assignment of independent units to ranks.
"""
from __future__ import annotations


def _dist():
    import torch.distributed as dist
    return dist


def _device():
    import torch
    dist = _dist()
    backend = dist.get_backend()
    return torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")


def agree_all(ok: bool) -> bool:
    """True on every rank iff `ok` is true on every rank (all-reduce MIN of a flag)."""
    import torch
    dist = _dist()
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return bool(ok)
    t = torch.tensor([1 if ok else 0], dtype=torch.int32, device=_device())
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def max_over_ranks(value: float) -> float:
    """The largest `value` of all ranks, on every rank."""
    import torch
    dist = _dist()
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard(n_units: int, rank: int, world: int) -> range:
    """Contiguous block of [0, n_units) owned by `rank`; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or n_units < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n_units, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))
