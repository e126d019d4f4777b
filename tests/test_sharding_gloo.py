"""Multi-rank path on CPU: two gloo ranks each take a shard of the poses; the forward
outputs concatenate to the unsharded result and the all-reduced (summed) volume gradient
and back-projection equal the unsharded ones.  Computed with the oracle; no GPU."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from back_projection_fourier_b300.shard import pose_range


def _worker(rank, world, port, res, name, B):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from back_projection_fourier_b300 import synth

        wl = synth.make_workload(name, B=B)
        kw = dict(interp=wl.interp, layout=wl.layout, cutoff=wl.rc, nthreads=1)
        a, b = pose_range(wl.n_pose, rank, world)
        sl = lambda x: None if x is None else np.ascontiguousarray(x[:, a:b])  # noqa: E731
        y = oracle.project(3, wl.rec, sl(wl.rot), sl(wl.shift), **kw)
        g_rec, g_rot, g_sh = oracle.project_backward(3, wl.rec, sl(wl.rot), sl(wl.grad), sl(wl.shift), **kw)
        vol, wvol = oracle.backproject(3, sl(wl.grad), sl(wl.rot), shift=sl(wl.shift), **kw)
        t = torch.from_numpy(np.concatenate([g_rec.view(np.float64).ravel(),
                                             vol.view(np.float64).ravel(), wvol.ravel()]))
        dist.all_reduce(t)
        if rank == 0:
            full_y = oracle.project(3, wl.rec, wl.rot, wl.shift, **kw)
            f_rec, f_rot, f_sh = oracle.project_backward(3, wl.rec, wl.rot, wl.grad, wl.shift, **kw)
            f_vol, f_w = oracle.backproject(3, wl.grad, wl.rot, shift=wl.shift, **kw)
            n1, n2 = f_rec.size * 2, f_vol.size * 2
            red = t.numpy()
            res["rec"] = float(np.abs(red[:n1] - f_rec.view(np.float64).ravel()).max() / np.abs(f_rec).max())
            res["vol"] = float(np.abs(red[n1:n1 + n2] - f_vol.view(np.float64).ravel()).max() / np.abs(f_vol).max())
            res["wvol"] = float(np.abs(red[n1 + n2:] - f_w.ravel()).max() / np.abs(f_w).max())
            res["fwd_shard0"] = float(np.abs(y - full_y[:, a:b]).max())
            res["rot_shard0"] = float(np.abs(g_rot - f_rot[:, a:b]).max())
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


@pytest.mark.parametrize("name,B", [("fwdbwd3d_d64_cubic_b4096", 23),
                                    ("fwdbwd3d_d128_cubic_r8_b16384", 24)])
def test_two_rank_gloo_sharding_matches_unsharded(name, B):
    """Shards of every reconstruction's poses; with several reconstructions each rank
    all-reduces all of their gradient volumes at once."""
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        res = m.dict()
        port = 29500 + (os.getpid() + B) % 1000
        mp.start_processes(_worker, args=(2, port, res, name, B), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(res)
    assert res["rec"] < 1e-13 and res["vol"] < 1e-13 and res["wvol"] < 1e-13, res
    assert res["fwd_shard0"] == 0.0 and res["rot_shard0"] == 0.0, res
