"""Independent replicas, one process per GPU.

A paged MoE layer step keeps one residency state (slot table, LRU clock,
counters) per handle, and the method runs each layer whole on one device, so
several GPUs run as unrelated replicas: each holds its own K-slot tables and
pinned host store and serves its own request stream, with no collective on the
data path.  The only cross-process traffic is host-side bookkeeping around a
timed run: barriers at its edges and one max-reduction of the elapsed time, so
that job throughput = (units all replicas processed) / (slowest replica's
time).  Everything here works on any ``torch.distributed`` backend (NCCL on
GPUs, gloo on the CPU).
"""

from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class Replica:
    rank: int
    world: int
    local_rank: int

    @property
    def is_root(self) -> bool:
        return self.rank == 0


def from_env(env=None) -> Replica:
    """Rank, world size and local rank as set by ``torch.distributed.run``
    (defaults: a single replica)."""
    env = os.environ if env is None else env
    rank, world = int(env.get("RANK", "0")), int(env.get("WORLD_SIZE", "1"))
    local = int(env.get("LOCAL_RANK", str(rank)))
    if world < 1 or not 0 <= rank < world or local < 0:
        raise ValueError(f"bad replica layout: rank {rank}, world {world}, local rank {local}")
    return Replica(rank, world, local)


def init(rep: Replica, backend: str, device=None, timeout_s: float | None = None) -> None:
    """Join the process group of a multi-replica run (no-op for one replica).
    ``timeout_s`` bounds every later barrier and reduction, so a replica that
    died between steps ends the others' next collective with an error instead
    of a hang."""
    if rep.world == 1:
        return
    import datetime

    import torch.distributed as dist

    kw = {"device_id": device} if device is not None and backend == "nccl" else {}
    if timeout_s is not None:
        kw["timeout"] = datetime.timedelta(seconds=timeout_s)
    dist.init_process_group(backend, rank=rep.rank, world_size=rep.world, **kw)


def finish(rep: Replica) -> None:
    if rep.world > 1:
        import torch.distributed as dist

        if dist.is_initialized():
            dist.destroy_process_group()


def barrier(rep: Replica) -> None:
    if rep.world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_replicas(rep: Replica, value: float, device="cpu") -> float:
    """The largest ``value`` over all replicas (every rank gets it)."""
    if rep.world == 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_replica: float, world: int, slowest_ms: float) -> float:
    """Whole-job throughput: every replica processed ``units_per_replica``
    units; the job took as long as its slowest replica."""
    if slowest_ms <= 0:
        raise ValueError("elapsed time must be positive")
    return world * units_per_replica / (slowest_ms * 1e-3)


def input_seed(base: int, rep: Replica) -> int:
    """Seed of a replica's own request stream.  Replica 0 keeps ``base``, so a
    one-replica run sees exactly the single-GPU inputs."""
    return base + 7919 * rep.rank
