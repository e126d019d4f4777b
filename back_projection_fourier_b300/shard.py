"""Data parallelism over poses: one process per GPU, each with its own shard of the batch.

Items (poses) are independent (torch-projectors summaries, Method section: batches over
images and poses), so rank r of w projects its own poses with no collective.  The volume
gradient is a sum over poses: each rank computes the share of its poses and one all-reduce
(sum) of the volume-sized buffer gives every rank the gradient of the whole batch.  The
rotation and shift gradients of a pose depend on that pose alone and stay on its rank.

The same three pieces serve the benchmark's multi-GPU run and the CPU test of this module:
``workload_shard`` draws a rank's shard of a seeded workload (and nothing else),
``shard_step`` runs one forward + backward step on it with whatever projection operators
it is given, and ``volume_allreduce`` is the one collective.
"""
from __future__ import annotations


def pose_range(n_pose: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [start, stop) of poses owned by `rank` (sizes differ by <= 1)."""
    if world < 1 or not 0 <= rank < world or n_pose < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, n_pose >= 0")
    base, extra = divmod(n_pose, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def workload_shard(name: str, per_rank: int | None, rank: int, world: int, **kw):
    """Rank `rank`'s shard of the workload `name` run on `world` ranks with `per_rank`
    projections each (weak scaling: the whole batch is per_rank * world projections, drawn
    from the workload's seed; None takes the workload's own batch per rank).  Every rank
    holds the same reconstruction(s) and the poses pose_range(n_pose, rank, world) of each.
    Only the shard's per-pose arrays are drawn.  Returns a synth.Workload."""
    from . import synth

    entry = synth.WORKLOADS[name]   # (number, ndim, op, interp, D, B, rc, amp, falloff[, n_rec])
    if entry[1] != 3:
        raise ValueError("pose sharding applies to the 3D workloads")
    n_rec = entry[9] if len(entry) > 9 else 1
    per_rank = entry[5] if per_rank is None else per_rank
    total = per_rank * world
    wl = synth.make_workload(name, B=total, poses=pose_range(total // n_rec, rank, world), **kw)
    wl.extra.update(rank=rank, world=world)
    return wl


def volume_allreduce(t, group=None) -> None:
    """Sum the volume-sized tensor `t` (complex or real) over the ranks of `group`, in place:
    the one exchange step of the data-parallel backward.  No-op without a process group."""
    import torch
    import torch.distributed as dist

    if t is None or not dist.is_available() or not dist.is_initialized():
        return
    if dist.get_world_size(group) == 1:
        return
    dist.all_reduce(torch.view_as_real(t) if t.is_complex() else t, group=group)


def shard_step(project, backward, vol, rot, shift, grad, group=None):
    """One data-parallel step on this rank's shard: y = project(vol, rot, shift) and
    (g_vol, g_rot, g_shift) = backward(vol, rot, shift, grad), then g_vol summed over the
    ranks.  `project` and `backward` are the projection operators (the CUDA library's calls
    in the benchmark); returns (y, g_vol, g_rot, g_shift), g_vol the whole batch's."""
    y = project(vol, rot, shift)
    g_vol, g_rot, g_sh = backward(vol, rot, shift, grad)
    volume_allreduce(g_vol, group)
    return y, g_vol, g_rot, g_sh
