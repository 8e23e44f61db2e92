"""Target-sharded all-pairs forces over several GPUs, one process per GPU.

The force grid of N targets x N sources splits into independent row blocks
(GPU Gems 3 ch.31 study page, section 2: each thread block owns a set of
targets and runs over every source).  Rank r owns a contiguous range of
targets -- its bodies and their velocities -- and every step:

1. all-gathers the positions of every rank into one N-body array in global
   order (the only exchange: 16 N bytes in total);
2. evaluates its own targets against all N sources with nbody_forces_ts;
3. applies the Euler step to its own bodies.

No reduction is needed and Euler stays local.  All compute runs in the
library's kernels; this module only moves tensors between ranks
(torch.distributed: NCCL on GPUs, gloo in the CPU tests).  Each rank's
results equal those of nbody_forces_ts on one GPU for the same target range.
"""
from __future__ import annotations


def shard_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """Targets [lo, hi) of `rank`: contiguous, in rank order, sizes differing
    by at most one (the first n % world ranks take one more)."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"bad shard: n={n}, rank={rank}, world={world}")
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def shard_counts(n: int, world: int) -> list[int]:
    return [hi - lo for lo, hi in (shard_range(n, r, world) for r in range(world))]


def gather_bodies(local, n: int, group=None, out=None):
    """The [n, 4] array of every rank's `local` rows in rank order.

    Each rank passes its own [count_r, 4] rows (count_r from shard_range).
    The ranks' blocks are padded to the largest count for one all_gather and
    compacted into `out` (allocated if None)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    counts = shard_counts(n, world)
    if local.shape != (counts[rank], 4):
        raise ValueError(f"rank {rank} holds {tuple(local.shape)} rows, expected ({counts[rank]}, 4)")
    width = max(counts)
    pad = torch.zeros((width, 4), dtype=local.dtype, device=local.device)
    pad[:counts[rank]].copy_(local)
    blocks = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(blocks, pad, group=group)
    if out is None:
        out = torch.empty((n, 4), dtype=local.dtype, device=local.device)
    lo = 0
    for r, c in enumerate(counts):
        out[lo:lo + c].copy_(blocks[r][:c])
        lo += c
    return out


def forces_sharded(local_pm, n: int, eps2: float, acc_pot=None, sources=None, group=None,
                   workspace=None):
    """(a, p) of this rank's targets from all n bodies: gather, then
    nbody_forces_ts(local targets, all sources).  `sources` may be a
    preallocated [n, 4] buffer for the gathered positions; `workspace` a
    caller-owned workspace tensor (then the library allocates nothing).
    Everything runs on the current torch stream of the bodies' device."""
    from . import _binding as B
    full = gather_bodies(local_pm, n, group=group, out=sources)
    if workspace is None:
        return B.nbody_forces_ts(local_pm, full, eps2, acc_pot)
    return B.nbody_forces_ts_ws(local_pm, full, eps2, acc_pot, workspace=workspace)


def simulate_sharded(local_pm, local_vel, local_acc, n: int, eps2: float, dt: float, steps: int,
                     group=None, workspace=None):
    """`steps` sharded steps in place on this rank's bodies: gather, forces
    of the local targets, local Euler step (positions first)."""
    import torch
    from . import _binding as B
    full = torch.empty((n, 4), dtype=local_pm.dtype, device=local_pm.device)
    for _ in range(int(steps)):
        forces_sharded(local_pm, n, eps2, local_acc, sources=full, group=group,
                       workspace=workspace)
        B.nbody_euler_step(local_pm, local_vel, local_acc, dt)
