"""Host-side sharding of a batch of poses over ranks (data parallelism).

Items (poses) are independent: rank r of w projects poses [start, stop) of the batch with
no collective; the volume gradient (and the back-projected volumes) are sums over poses,
so the per-rank partial sums are added with one all-reduce.
"""
from __future__ import annotations


def pose_range(n_pose: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [start, stop) of poses owned by `rank` (sizes differ by <= 1)."""
    if world < 1 or not 0 <= rank < world or n_pose < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, n_pose >= 0")
    base, extra = divmod(n_pose, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)
