"""Multi-rank path on CPU: the package's data-parallel step (back_projection_fourier_b300.shard)
on two gloo ranks, with the fp64 oracle standing in for the CUDA operators.  Each rank draws
only its shard of the batch (workload_shard), runs shard_step on it and the one volume
all-reduce; the forward and pose gradients of its shard must equal the unsharded ones exactly
and the all-reduced volume gradient (and insertion) the unsharded sums.  No GPU."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from back_projection_fourier_b300 import shard, synth
from back_projection_fourier_b300.shard import pose_range


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a))


def _worker(rank, world, port, res, name, per_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle

        wl = shard.workload_shard(name, per_rank, rank, world)
        kw = dict(interp=wl.interp, layout=wl.layout, cutoff=wl.rc, nthreads=1)

        def project(V, R, S):
            return _t(oracle.project(3, V.numpy(), R.numpy(), S.numpy(), **kw))

        def backward(V, R, S, G):
            return tuple(_t(x) for x in oracle.project_backward(3, V.numpy(), R.numpy(),
                                                                 G.numpy(), S.numpy(), **kw))

        y, g_vol, g_rot, g_sh = shard.shard_step(project, backward, _t(wl.rec), _t(wl.rot),
                                                 _t(wl.shift), _t(wl.grad))
        vol, wvol = (_t(x) for x in oracle.backproject(3, wl.grad, wl.rot, shift=wl.shift, **kw))
        shard.volume_allreduce(vol)
        shard.volume_allreduce(wvol)
        # the unsharded batch, drawn whole, computed on one rank's worth of arithmetic
        full = synth.make_workload(name, B=per_rank * world)
        a, b = wl.extra["poses"]
        f_y = oracle.project(3, full.rec, full.rot, full.shift, **kw)
        f_rec, f_rot, f_sh = oracle.project_backward(3, full.rec, full.rot, full.grad, full.shift, **kw)
        f_vol, f_w = oracle.backproject(3, full.grad, full.rot, shift=full.shift, **kw)

        def rel(x, ref):
            return float(np.abs(x.numpy() - ref).max() / np.abs(ref).max())

        res[f"rec{rank}"] = rel(g_vol, f_rec)
        res[f"vol{rank}"] = rel(vol, f_vol)
        res[f"wvol{rank}"] = rel(wvol, f_w)
        res[f"fwd{rank}"] = float(np.abs(y.numpy() - f_y[:, a:b]).max())
        res[f"rot{rank}"] = float(np.abs(g_rot.numpy() - f_rot[:, a:b]).max())
        res[f"sh{rank}"] = float(np.abs(g_sh.numpy() - f_sh[:, a:b]).max())
        res[f"B{rank}"] = wl.B
    finally:
        dist.destroy_process_group()


def test_pose_range_partitions():
    for n in (0, 1, 7, 23, 4096):
        for w in (1, 2, 3, 8):
            spans = [pose_range(n, r, w) for r in range(w)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[i][1] == spans[i + 1][0] for i in range(w - 1))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
    with pytest.raises(ValueError):
        pose_range(5, 2, 2)


@pytest.mark.parametrize("name,per_rank,world", [("fwdbwd3d_d64_cubic_b4096", 5, 3),
                                                 ("fwdbwd3d_d128_cubic_r8_b16384", 16, 2)])
def test_workload_shards_tile_the_whole_batch(name, per_rank, world):
    """Shards drawn alone concatenate, pose range by pose range, to the batch drawn whole."""
    full = synth.make_workload(name, B=per_rank * world)
    parts = [shard.workload_shard(name, per_rank, r, world) for r in range(world)]
    for key in ("rot", "shift", "grad"):
        cat = np.concatenate([getattr(p, key) for p in parts], axis=1)
        assert np.array_equal(cat, getattr(full, key)), key
    assert all(np.array_equal(p.rec, full.rec) for p in parts)
    assert sum(p.B for p in parts) == full.B


@pytest.mark.parametrize("name,per_rank", [("fwdbwd3d_d64_cubic_b4096", 12),
                                           ("fwdbwd3d_d128_cubic_r8_b16384", 16)])
def test_two_rank_gloo_step_matches_unsharded(name, per_rank):
    """With several reconstructions each rank all-reduces all of their gradient volumes at
    once (one collective of the whole [n_rec] stack)."""
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        res = m.dict()
        port = 29500 + (os.getpid() + per_rank) % 1000
        mp.start_processes(_worker, args=(2, port, res, name, per_rank), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(res)
    for r in range(2):
        assert res[f"rec{r}"] < 1e-13 and res[f"vol{r}"] < 1e-13 and res[f"wvol{r}"] < 1e-13, res
        assert res[f"fwd{r}"] == 0.0 and res[f"rot{r}"] == 0.0 and res[f"sh{r}"] == 0.0, res
        assert res[f"B{r}"] == per_rank, res
