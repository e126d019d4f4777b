"""GPU: the differentiable PyTorch operators (back_projection_fourier_b300.autograd) against the
fp64 oracle -- forward values and the gradients autograd returns for every input."""
import numpy as np
import pytest
import torch

from parity_util import TOL_BWD, TOL_FWD, crandn32, dev, host, max_rel, oracle, rotations
from back_projection_fourier_b300 import autograd as tpa

pytestmark = pytest.mark.gpu


def leaf(a):
    return dev(a).requires_grad_(True)


@pytest.mark.parametrize("ndim,interp,layout", [(3, 1, 1), (3, 0, 0), (2, 1, 1)])
def test_project_autograd(ndim, interp, layout):
    rng = np.random.default_rng(90 + ndim + interp)
    D, n_pose = 24, 7
    shape = (2, D, D, D // 2 + 1) if ndim == 3 else (2, D, D // 2 + 1)
    rec = crandn32(rng, shape)
    rot = rotations(rng, 2 * n_pose, ndim).reshape(2, n_pose, ndim, ndim)
    shift = rng.uniform(-4, 4, (2, n_pose, 2)).astype(np.float32)
    G = crandn32(rng, (2, n_pose, D, D // 2 + 1))
    r, R, s = leaf(rec), leaf(rot), leaf(shift)
    out = tpa.project(r, R, s, interp=interp, layout=layout)
    out.backward(dev(G))
    kw = dict(interp=interp, layout=layout)
    assert max_rel(host(out), oracle.project(ndim, rec, rot, shift, **kw)) <= TOL_FWD
    g_rec, g_rot, g_sh = oracle.project_backward(ndim, rec, rot, G, shift, **kw)
    assert max_rel(host(r.grad), g_rec) <= TOL_BWD
    assert max_rel(host(R.grad), g_rot) <= TOL_BWD
    assert max_rel(host(s.grad), g_sh) <= TOL_BWD


@pytest.mark.parametrize("ndim,with_weights", [(3, True), (3, False), (2, True)])
def test_backproject_autograd(ndim, with_weights):
    rng = np.random.default_rng(95 + ndim)
    D, n_pose = 20, 6
    proj = crandn32(rng, (1, n_pose, D, D // 2 + 1))
    w = rng.uniform(0.1, 2.0, proj.shape).astype(np.float32) if with_weights else None
    rot = rotations(rng, n_pose, ndim)[None]
    shift = rng.uniform(-3, 3, (1, n_pose, 2)).astype(np.float32)
    vshape = (1, D, D, D // 2 + 1) if ndim == 3 else (1, D, D // 2 + 1)
    Gv = crandn32(rng, vshape)
    GW = rng.standard_normal(vshape).astype(np.float32)
    p, R, s = leaf(proj), leaf(rot), leaf(shift)
    W = leaf(w) if with_weights else None
    res = tpa.backproject(p, R, s, W, ndim=ndim)
    r_vol, r_w = oracle.backproject(ndim, proj, rot, weights=w, shift=shift)
    if with_weights:
        vol, wvol = res
        torch.autograd.backward([vol, wvol], [dev(Gv), dev(GW)])
        assert max_rel(host(wvol), r_w) <= TOL_BWD
    else:
        vol = res
        vol.backward(dev(Gv))
    assert max_rel(host(vol), r_vol) <= TOL_BWD
    gP, gW, gR, gs = oracle.backproject_backward(ndim, proj, rot, Gv, GW if with_weights else None,
                                                 w, shift)
    assert max_rel(host(p.grad), gP) <= TOL_FWD
    assert max_rel(host(R.grad), gR) <= TOL_BWD
    assert max_rel(host(s.grad), gs) <= TOL_BWD
    if with_weights:
        assert max_rel(host(W.grad), gW) <= TOL_FWD


@pytest.mark.parametrize("ndim,factor,interp", [(3, 1, 1), (3, 2, 0), (3, 3, 0), (2, 2, 0), (2, 1, 1)])
def test_pipeline_autograd(ndim, factor, interp):
    """Real-space volume -> pad -> FFT -> projection, and the volume / pose gradients."""
    rng = np.random.default_rng(100 + ndim * 10 + factor)
    D, n_pose = 16, 5
    vol = rng.standard_normal((1,) + (D,) * ndim).astype(np.float32)
    rot = rotations(rng, n_pose, ndim)[None]
    shift = rng.uniform(-3, 3, (1, n_pose, 2)).astype(np.float32)
    G = crandn32(rng, (1, n_pose, D, D // 2 + 1))
    v, R, s = leaf(vol), leaf(rot), leaf(shift)
    out = tpa.project_real(v, R, s, factor=factor, interp=interp, ndim=ndim)
    out.backward(dev(G))
    ref = oracle.project_real(ndim, vol, rot, shift, factor=factor, interp=interp)
    assert max_rel(host(out), ref) <= TOL_FWD
    g_v, g_R, g_s = oracle.project_real_backward(ndim, vol, rot, G, shift, factor=factor,
                                                 interp=interp)
    assert max_rel(host(v.grad), g_v) <= TOL_BWD
    assert max_rel(host(R.grad), g_R) <= TOL_BWD
    assert max_rel(host(s.grad), g_s) <= TOL_BWD
