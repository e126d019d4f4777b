"""GPU: degenerate inputs.  Rotations that are NaN, infinite, huge or zero and huge shifts must
neither fault nor disturb the other poses of the batch: the kernels clamp every sample
coordinate to +-2^23, where all taps fall outside the stored band and touch no memory.  The
valid poses are compared with the oracle on those poses alone."""
import numpy as np
import pytest
import torch

from parity_util import TOL_BWD, TOL_FWD, crandn32, dev, host, max_rel, opts, oracle, rotations
from back_projection_fourier_b300 import tp

pytestmark = pytest.mark.gpu


def batch(rng, k):
    good = rotations(rng, 3, k)
    bad = np.stack([np.full((k, k), np.nan), np.full((k, k), np.inf), 1e30 * good[0],
                    np.zeros((k, k))]).astype(np.float32)
    rot = np.concatenate([good[:1], bad, good[1:]])[None]            # valid poses 0, 5, 6
    shift = rng.uniform(-4, 4, (1, rot.shape[1], 2)).astype(np.float32)
    shift[0, 1] = (1e30, -1e30)        # huge shift on an excluded pose
    shift[0, 6] = (1e5, -3e4)          # large shift on a valid pose (fp64 still resolves it)
    return rot, shift


@pytest.mark.parametrize("interp", [0, 1])
def test_degenerate_poses_3d(interp):
    rng = np.random.default_rng(31 + interp)
    D = 24
    op = opts(interp)
    kw = dict(interp=interp, layout=1)
    rot, shift = batch(rng, 3)
    vol = crandn32(rng, (1, D, D, D // 2 + 1))
    grad = crandn32(rng, (1, rot.shape[1], D, D // 2 + 1))
    w = rng.uniform(0.1, 1, grad.shape).astype(np.float32)
    # a huge but finite rotation (pose 3) still maps the pixel (0, 0) to c = 0, a valid sample:
    # zero its data so that its (correct) contribution to the volume needs no oracle term
    grad[:, 3] = 0
    w[:, 3] = 0
    V, R, S, G = dev(vol), dev(rot), dev(shift), dev(grad)
    ok = np.array([0, 4, 5, 6])                       # finite poses (4: the zero matrix)
    sub = lambda a: np.ascontiguousarray(a[:, ok])    # noqa: E731
    y = tp.project(V, R, S, opts=op)
    ws = tp.workspace_for(V, op)
    y_ws = torch.empty_like(y)
    tp.tp_project_3d_to_2d_ws(V, R, S, y_ws, ws, op)
    g_rot = torch.empty_like(R)
    g_sh = torch.empty((1, rot.shape[1], 2), device="cuda")
    g_rec = torch.empty_like(V)
    tp.tp_project_backward_ws(3, V, R, S, G, g_rec, g_rot, g_sh, ws, op)
    vol_bp, w_bp = tp.backproject(G, R, S, dev(w), opts=op)
    torch.cuda.synchronize()
    ref = oracle.project(3, vol, sub(rot), sub(shift), **kw)
    assert max_rel(host(y)[:, ok], ref) <= TOL_FWD
    assert torch.equal(y[:, ok], y_ws[:, ok])
    r_rec, r_rot, r_sh = oracle.project_backward(3, vol, sub(rot), sub(grad), sub(shift), **kw)
    # pose 6 (large shift, finite rotation) lands and counts in the volume gradient
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot)[:, ok[:3]], r_rot[:, :3]) <= TOL_BWD
    r_vol, r_w = oracle.backproject(3, sub(grad), sub(rot), weights=sub(w), shift=sub(shift), **kw)
    assert max_rel(host(vol_bp), r_vol) <= TOL_BWD
    assert max_rel(host(w_bp), r_w) <= TOL_BWD


def test_degenerate_poses_2d():
    rng = np.random.default_rng(41)
    D = 32
    op = opts(1)
    rot, shift = batch(rng, 2)
    n = rot.shape[1]
    img = crandn32(rng, (n, D, D // 2 + 1))
    rot = np.ascontiguousarray(rot.transpose(1, 0, 2, 3))           # one image per pose
    shift = np.ascontiguousarray(shift.transpose(1, 0, 2))
    grad = crandn32(rng, (n, 1, D, D // 2 + 1))
    y = tp.project(dev(img), dev(rot), dev(shift), opts=op)
    g_rec, g_rot, g_sh = tp.project_backward(dev(img), dev(rot), dev(grad), dev(shift), opts=op)
    torch.cuda.synchronize()
    ok = np.array([0, 4, 5, 6])
    r = oracle.project(2, img[ok], rot[ok], shift[ok], interp=1, layout=1)
    assert max_rel(host(y)[ok], r) <= TOL_FWD
    rr, rg, _ = oracle.project_backward(2, img[ok], rot[ok], grad[ok], shift[ok], interp=1, layout=1)
    assert max_rel(host(g_rec)[ok], rr) <= TOL_BWD
    assert max_rel(host(g_rot)[ok], rg) <= TOL_BWD


@pytest.mark.parametrize("interp", [0, 1])
def test_huge_finite_rotation_with_data(interp):
    """A finite rotation scaled by 1e7 sends every pixel but (0, 0) far outside the band, where
    the kernels clamp the coordinate to +-2^23: tiles of the scatter then span extents near 2^24
    and take the per-tap path.  With non-zero upstream data on that pose the volume gradient
    and the insertion still match the oracle (fp64, no clamp needed at 1e7), which counts only
    pixel (0, 0) of it."""
    rng = np.random.default_rng(41 + interp)
    D = 24
    op = opts(interp)
    kw = dict(interp=interp, layout=1)
    rot = rotations(rng, 4, 3).astype(np.float32)
    rot[1] *= 1e7
    rot = rot[None]
    shift = rng.uniform(-4, 4, (1, 4, 2)).astype(np.float32)
    vol = crandn32(rng, (1, D, D, D // 2 + 1))
    grad = crandn32(rng, (1, 4, D, D // 2 + 1))
    w = rng.uniform(0.1, 1, grad.shape).astype(np.float32)
    V, R, S, G = dev(vol), dev(rot), dev(shift), dev(grad)
    g_rec = torch.empty_like(V)
    tp.tp_project_backward(3, V, R, S, G, g_rec, None, None, op)
    vol_bp, w_bp = tp.backproject(G, R, S, dev(w), opts=op)
    r_rec, _, _ = oracle.project_backward(3, vol, rot, grad, shift, want_rot=False,
                                          want_shift=False, **kw)
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    r_vol, r_w = oracle.backproject(3, grad, rot, weights=w, shift=shift, **kw)
    assert max_rel(host(vol_bp), r_vol) <= TOL_BWD
    assert max_rel(host(w_bp), r_w) <= TOL_BWD
