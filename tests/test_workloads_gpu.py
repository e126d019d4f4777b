"""GPU parity on the benchmark workloads, at full size, in the launch configuration the
benchmark times.

Where the oracle finishes in seconds the whole output is compared; elsewhere the oracle
computes sampled outputs one by one (forward pixels; rotation / shift gradients of
sampled poses, which depend on that pose alone; whole images of the 2D workload, which
depend on that image alone), and the volume-sized results are checked through the
adjoint identity Re <P V, Y> = Re <V, P^T Y> against the (pinned) forward projection.
"""
import numpy as np
import pytest
import torch

from parity_util import TOL_BWD, TOL_FWD, crandn32, dev, host, max_rel, opts, oracle
from back_projection_fourier_b300 import synth, tp

pytestmark = pytest.mark.gpu


def wl_opts(wl):
    return opts(wl.interp, wl.layout, 1.0, wl.rc)


def oracle_kw(wl):
    return dict(interp=wl.interp, layout=wl.layout, cutoff=wl.rc)


def sub(a, idx, axis=1):
    return None if a is None else np.ascontiguousarray(np.take(a, idx, axis=axis))


def adjoint_gap(PV, Y, V, PtY):
    """|Re<PV, Y> - Re<V, PtY>| / (|PV| |Y|), in fp64 on the device."""
    a = torch.vdot(PV.reshape(-1).to(torch.complex128), Y.reshape(-1).to(torch.complex128)).real
    b = torch.vdot(V.reshape(-1).to(torch.complex128), PtY.reshape(-1).to(torch.complex128)).real
    nrm = torch.linalg.vector_norm(PV.to(torch.complex128)) * torch.linalg.vector_norm(Y.to(torch.complex128))
    return float(abs(a - b) / nrm)


def test_fwd3d_d32_linear_full():
    wl = synth.make_workload("fwd3d_d32_linear_b64")
    y = tp.project(dev(wl.rec), dev(wl.rot), dev(wl.shift), opts=wl_opts(wl))
    ref = oracle.project(3, wl.rec, wl.rot, wl.shift, **oracle_kw(wl))
    assert max_rel(host(y), ref) <= TOL_FWD


def test_fwdbwd3d_d64_cubic_full():
    wl = synth.make_workload("fwdbwd3d_d64_cubic_b4096")
    V, R, S, G = dev(wl.rec), dev(wl.rot), dev(wl.shift), dev(wl.grad)
    y = tp.project(V, R, S, opts=wl_opts(wl))
    g_rec, g_rot, g_sh = tp.project_backward(V, R, G, S, opts=wl_opts(wl))
    ref = oracle.project(3, wl.rec, wl.rot, wl.shift, **oracle_kw(wl))
    assert max_rel(host(y), ref) <= TOL_FWD
    r_rec, r_rot, r_sh = oracle.project_backward(3, wl.rec, wl.rot, wl.grad, wl.shift, **oracle_kw(wl))
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    assert max_rel(host(g_sh), r_sh) <= TOL_BWD


@pytest.mark.parametrize("interp", [0, 1])
def test_insert3d_d128(interp):
    wl = synth.make_workload("insert3d_d128_b16384", interp=interp)
    P, R, W = dev(wl.grad), dev(wl.rot), dev(np.ascontiguousarray(wl.weights))
    op = wl_opts(wl)
    # sub-batch of 512 slices: whole-volume parity with the oracle
    idx = np.arange(512)
    vol_s, w_s = tp.backproject(P[:, :512].contiguous(), R[:, :512].contiguous(), None,
                                W[:, :512].contiguous(), opts=op)
    r_vol, r_w = oracle.backproject(3, sub(wl.grad, idx), sub(wl.rot, idx),
                                    weights=sub(np.ascontiguousarray(wl.weights), idx), **oracle_kw(wl))
    assert max_rel(host(vol_s), r_vol) <= TOL_BWD
    assert max_rel(host(w_s), r_w) <= TOL_BWD
    # full batch: adjoint identity against the forward projection, and the weights volume
    # equals the back-projection of the weights as real data (no shift in this workload)
    vol, wvol = tp.backproject(P, R, None, W, opts=op)
    rng = np.random.default_rng(5)
    Vr = dev(crandn32(rng, vol.shape))
    PV = tp.project(Vr, R, None, opts=op)
    assert adjoint_gap(PV, P, Vr, vol) <= 1e-5
    vol_w, _ = tp.backproject(W.to(torch.complex64), R, None, None, want_weights=False, opts=op)
    assert max_rel(host(vol_w).real, host(wvol)) <= TOL_BWD
    assert float(vol_w.imag.abs().max()) <= 1e-5 * float(vol_w.real.abs().max())


def test_rot2d_d256_cubic_full_sampled_images():
    wl = synth.make_workload("rot2d_d256_cubic_b8192")
    V, R, S, G = dev(wl.rec), dev(wl.rot), dev(wl.shift), dev(wl.grad)
    op = wl_opts(wl)
    y = tp.project(V, R, S, opts=op)
    g_rec, g_rot, g_sh = tp.project_backward(V, R, G, S, opts=op)
    idx = np.random.default_rng(3).choice(wl.B, 24, replace=False)
    ti = torch.from_numpy(idx).cuda()
    kw = oracle_kw(wl)
    rec_s, rot_s, sh_s, g_s = (np.ascontiguousarray(a[idx]) for a in (wl.rec, wl.rot, wl.shift, wl.grad))
    ref = oracle.project(2, rec_s, rot_s, sh_s, **kw)
    assert max_rel(host(y[ti]), ref) <= TOL_FWD
    r_rec, r_rot, r_sh = oracle.project_backward(2, rec_s, rot_s, g_s, sh_s, **kw)
    assert max_rel(host(g_rec[ti]), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot[ti]), r_rot) <= TOL_BWD
    assert max_rel(host(g_sh[ti]), r_sh) <= TOL_BWD


def test_rot2d_d256_cubic_insertion_with_weights_sampled_images():
    """The 2D insertion with weights (the half-warp tile scatter) over the whole 2D workload:
    every image has its own output image, so sampled images compare exactly with the oracle."""
    wl = synth.make_workload("rot2d_d256_cubic_b8192")
    R, S, G = dev(wl.rot), dev(wl.shift), dev(wl.grad)
    rng = np.random.default_rng(5)
    w = rng.uniform(0.1, 2.0, wl.grad.shape).astype(np.float32)
    op = wl_opts(wl)
    img, wimg = tp.backproject(G, R, S, dev(w), Dv=wl.D, opts=op, ndim=2)
    idx = rng.choice(wl.B, 24, replace=False)
    ti = torch.from_numpy(idx).cuda()
    kw = oracle_kw(wl)
    g_s, rot_s, sh_s, w_s = (np.ascontiguousarray(a[idx]) for a in (wl.grad, wl.rot, wl.shift, w))
    r_img, r_w = oracle.backproject(2, g_s, rot_s, weights=w_s, shift=sh_s, Dv=wl.D, **kw)
    assert max_rel(host(img[ti]), r_img) <= TOL_BWD
    assert max_rel(host(wimg[ti]), r_w) <= TOL_BWD


def _fwdbwd3d_sampled(name, n_pix=6000, n_poses=48, n_sub=None):
    """n_sub: None compares the whole volume gradient of the full batch with the oracle;
    an integer compares the whole volume gradient of the first n_sub poses of every
    reconstruction (the same kernel and launch shape on a batch the oracle finishes in
    seconds)."""
    wl = synth.make_workload(name)
    V, R, S, G = dev(wl.rec), dev(wl.rot), dev(wl.shift), dev(wl.grad)
    op = wl_opts(wl)
    kw = oracle_kw(wl)
    # the benchmark's calls: the gathers read the grouped copy in a workspace
    ws = tp.workspace_for(V, op)
    y = torch.empty_like(G)
    tp.tp_project_3d_to_2d_ws(V, R, S, y, ws, op)
    assert torch.equal(y, tp.project(V, R, S, opts=op))
    g_rec, g_rot = torch.empty_like(V), torch.empty_like(R)
    g_sh = torch.empty((S.shape[0], wl.n_pose, 2), device="cuda")
    tp.tp_project_backward_ws(3, V, R, S, G, None, g_rot, g_sh, ws, op)
    tp.tp_project_backward(3, V, R, S, G, g_rec, None, None, op)
    rng = np.random.default_rng(11)
    n_items = wl.n_rec * wl.n_pose
    items = rng.integers(0, n_items, n_pix)
    pix = rng.integers(0, wl.D * wl.H, n_pix)
    got = y.reshape(n_items, -1)[torch.from_numpy(items).cuda(), torch.from_numpy(pix).cuda()]
    ref = oracle.project_samples(3, wl.rec, wl.rot, items, pix, wl.shift, **kw)
    # relative to the largest output value of the whole projection stack
    scale = float(y.abs().max())
    assert float(np.abs(host(got) - ref).max()) <= TOL_FWD * scale
    # rotation / shift gradients of sampled poses depend on those poses alone
    poses = np.sort(rng.choice(wl.n_pose, n_poses // wl.n_rec, replace=False))
    _, r_rot, r_sh = oracle.project_backward(3, wl.rec, sub(wl.rot, poses), sub(wl.grad, poses),
                                             sub(wl.shift, poses), want_rec=False, **kw)
    tpo = torch.from_numpy(poses).cuda()
    assert max_rel(host(g_rot[:, tpo]), r_rot) <= TOL_BWD
    assert max_rel(host(g_sh[:, tpo]), r_sh) <= TOL_BWD
    # the volume gradient voxel by voxel against the oracle, over every voxel of the box
    if n_sub is None:
        r_rec, _, _ = oracle.project_backward(3, wl.rec, wl.rot, wl.grad, wl.shift,
                                              want_rot=False, want_shift=False, **kw)
        assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    else:
        idx = np.arange(n_sub)
        g_sub = torch.empty_like(V)
        sl = lambda t: t[:, :n_sub].contiguous()  # noqa: E731
        tp.tp_project_backward(3, V, sl(R), sl(S), sl(G), g_sub, None, None, op)
        r_rec, _, _ = oracle.project_backward(3, wl.rec, sub(wl.rot, idx), sub(wl.grad, idx),
                                              sub(wl.shift, idx), want_rot=False,
                                              want_shift=False, **kw)
        assert max_rel(host(g_sub), r_rec) <= TOL_BWD
    # and the full batch's volume gradient through the adjoint identity
    Vr = dev(crandn32(rng, wl.rec.shape))
    PV = tp.project(Vr, R, S, opts=op)
    assert adjoint_gap(PV, G, Vr, g_rec) <= 1e-5


def test_fwdbwd3d_d128_cubic_full_sampled():
    _fwdbwd3d_sampled("fwdbwd3d_d128_cubic_b16384")


def test_fwdbwd3d_d128_cubic_r8_full_sampled():
    """Eight reconstructions, each with 2048 poses of its own (per-reconstruction rotations
    and shifts): items index (reconstruction, pose), gradients land in their own volume."""
    _fwdbwd3d_sampled("fwdbwd3d_d128_cubic_r8_b16384")


def test_fwdbwd3d_d256_cubic_full_sampled():
    _fwdbwd3d_sampled("fwdbwd3d_d256_cubic_b50000", n_pix=4000, n_poses=24, n_sub=256)


def test_fwdbwd3d_d128_cubic_fused_backward():
    """tp_project_backward_fused (one kernel pass) on the headline workload: the whole batch
    against the two-kernel call, the pose gradients of sampled poses and the volume gradient of
    a 512-pose sub-batch (every voxel) against the oracle."""
    wl = synth.make_workload("fwdbwd3d_d128_cubic_b16384")
    V, R, S, G = dev(wl.rec), dev(wl.rot), dev(wl.shift), dev(wl.grad)
    op = wl_opts(wl)
    kw = oracle_kw(wl)
    fused = tp.project_backward(V, R, G, S, opts=op, fused=True)
    two = tp.project_backward(V, R, G, S, opts=op)
    for a, b in zip(fused, two):
        assert max_rel(host(a), host(b)) <= TOL_BWD
    rng = np.random.default_rng(12)
    poses = np.sort(rng.choice(wl.n_pose, 48, replace=False))
    _, r_rot, r_sh = oracle.project_backward(3, wl.rec, sub(wl.rot, poses), sub(wl.grad, poses),
                                             sub(wl.shift, poses), want_rec=False, **kw)
    tpo = torch.from_numpy(poses).cuda()
    assert max_rel(host(fused[1][:, tpo]), r_rot) <= TOL_BWD
    assert max_rel(host(fused[2][:, tpo]), r_sh) <= TOL_BWD
    n_sub = 512
    sl = lambda t: t[:, :n_sub].contiguous()  # noqa: E731
    g_sub, _, _ = tp.project_backward(V, sl(R), sl(G), sl(S), opts=op, fused=True)
    idx = np.arange(n_sub)
    r_rec, _, _ = oracle.project_backward(3, wl.rec, sub(wl.rot, idx), sub(wl.grad, idx),
                                          sub(wl.shift, idx), want_rot=False, want_shift=False, **kw)
    assert max_rel(host(g_sub), r_rec) <= TOL_BWD


def test_chunked_volume_gradient_equals_the_backward():
    """The pipelined end-to-end step sums each pose chunk's volume gradient with the insertion
    call (accumulate = 1): the same transpose as the backward's volume gradient."""
    wl = synth.make_workload("fwdbwd3d_d128_cubic_b16384", B=1000)
    V, R, S, G = dev(wl.rec), dev(wl.rot), dev(wl.shift), dev(wl.grad)
    op = wl_opts(wl)
    g_rec, _, _ = tp.project_backward(V, R, G, S, want_rot=False, want_shift=False, opts=op)
    acc = torch.empty_like(V)
    for c, (a, b) in enumerate([(0, 300), (300, 301), (301, 1000)]):
        tp.tp_backproject_2d_to_3d(G[:, a:b], None, R[:, a:b], S[:, a:b], acc, None, wl.D, c > 0, op)
    assert max_rel(host(acc), host(g_rec)) <= TOL_BWD
