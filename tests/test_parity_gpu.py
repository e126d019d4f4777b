"""GPU parity: every C-ABI entry point against the fp64 oracle on the same seeded inputs.

Small cases span several CTAs and ragged pixel tails, both interpolations and layouts,
2D and 3D, oversampling, custom cutoffs, shifts on/off, several reconstructions with
shared or per-reconstruction poses.  Metric: max |gpu - oracle| / max |oracle| per output
tensor; bar: 1e-5 for forward projection, 1e-4 for back-projection and gradients.
"""
import numpy as np
import pytest
import torch

from parity_util import TOL_BWD, TOL_FWD, crandn32, dev, host, max_rel, opts, oracle, rotations
from back_projection_fourier_b300 import tp

pytestmark = pytest.mark.gpu

# ndim, interp, layout, o, Dv, Do, cutoff, shifted, n_rec, n_rot, n_pose
CASES = [
    (3, 1, 1, 1.0, 32, 32, -1.0, True, 1, 1, 37),
    (3, 0, 1, 1.0, 32, 32, -1.0, True, 1, 1, 37),
    (3, 1, 0, 1.0, 24, 24, 9.5, True, 2, 2, 13),
    (3, 0, 0, 1.5, 24, 16, -1.0, False, 2, 1, 11),
    (3, 1, 1, 2.0, 32, 16, 100.0, True, 1, 1, 9),
    (3, 1, 1, 1.0, 2, 2, -1.0, True, 1, 1, 5),
    (3, 1, 0, 1.0, 30, 30, -1.0, True, 2, 2, 7),
    (3, 0, 1, 1.25, 40, 32, 12.0, True, 3, 1, 6),
    # linear at o = 2: many 8 x 4 tiles of the linear scatter exceed its box (wider than 16
    # voxels) and take the per-tap path with global atomics
    (3, 0, 1, 2.0, 48, 24, -1.0, True, 2, 1, 5),
    (2, 1, 1, 1.0, 48, 48, -1.0, True, 5, 5, 3),
    (2, 0, 0, 1.0, 30, 30, -1.0, True, 3, 1, 4),
    (2, 1, 0, 1.5, 36, 24, 10.0, False, 4, 4, 2),
    (2, 0, 1, 1.0, 64, 64, 0.0, True, 2, 2, 3),
    # image boxes larger than the volume (Do > Dv): the outer samples fall outside the stored
    # range and read zero
    (3, 1, 1, 1.0, 16, 24, -1.0, True, 1, 1, 7),
    (3, 0, 0, 1.0, 16, 20, -1.0, True, 2, 2, 5),
    (2, 1, 1, 1.0, 16, 24, -1.0, True, 3, 3, 2),
    (2, 0, 0, 1.0, 12, 30, -1.0, True, 2, 1, 3),
]


CASES2 = [c for c in CASES if c[0] == 2]
PARTIAL = [c for c in CASES if c[0] == 3][:3] + CASES2[:2]   # three 3D and two 2D cases


def make_case(case, seed=0):
    ndim, interp, layout, o, Dv, Do, rc, shifted, n_rec, n_rot, n_pose = case
    rng = np.random.default_rng(seed + hash(case) % 10000)
    Hv, Ho = Dv // 2 + 1, Do // 2 + 1
    shape = (n_rec, Dv, Dv, Hv) if ndim == 3 else (n_rec, Dv, Hv)
    rec = crandn32(rng, shape)
    rot = rotations(rng, n_rot * n_pose, ndim).reshape(n_rot, n_pose, ndim, ndim)
    shift = rng.uniform(-6, 6, (n_rot, n_pose, 2)).astype(np.float32) if shifted else None
    grad = crandn32(rng, (n_rec, n_pose, Do, Ho))
    w = rng.uniform(0.0, 2.0, (n_rec, n_pose, Do, Ho)).astype(np.float32)
    kw = dict(interp=interp, layout=layout, oversampling=o, cutoff=rc)
    return rec, rot, shift, grad, w, kw, opts(interp, layout, o, rc)


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_forward(case):
    ndim, Do = case[0], case[5]
    rec, rot, shift, _, _, kw, op = make_case(case)
    y = tp.project(dev(rec), dev(rot), dev(shift), Do=Do, opts=op)
    ref = oracle.project(ndim, rec, rot, shift, Do=Do, **kw)
    assert max_rel(host(y), ref) <= TOL_FWD


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_backward(case):
    ndim = case[0]
    rec, rot, shift, grad, _, kw, op = make_case(case, seed=1)
    g_rec, g_rot, g_sh = tp.project_backward(dev(rec), dev(rot), dev(grad), dev(shift),
                                             want_shift=shift is not None, opts=op)
    r_rec, r_rot, r_sh = oracle.project_backward(ndim, rec, rot, grad, shift, **kw)
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    if ndim == 3:
        assert np.all(host(g_rot)[..., 2] == 0)
    if shift is not None:
        assert max_rel(host(g_sh), r_sh) <= TOL_BWD


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_backward_fused(case):
    """tp_project_backward_fused: in 3D cubic one kernel pass emits the volume, rotation and
    shift gradients (including the cases whose taps reach the x <= 0 planes, the rim, or
    tiles too large for a box at o = 2); elsewhere it is the two-kernel call.  Either way the
    oracle's gradients."""
    ndim = case[0]
    rec, rot, shift, grad, _, kw, op = make_case(case, seed=1)
    r_rec, r_rot, r_sh = oracle.project_backward(ndim, rec, rot, grad, shift, **kw)
    g_rec, g_rot, g_sh = tp.project_backward(dev(rec), dev(rot), dev(grad), dev(shift),
                                             want_shift=shift is not None, opts=op, fused=True)
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    if ndim == 3:
        assert np.all(host(g_rot)[..., 2] == 0)
    if shift is not None:
        assert max_rel(host(g_sh), r_sh) <= TOL_BWD
        # the shift gradient alone beside the volume gradient (still one pass)
        g_rec2, g_none, g_sh2 = tp.project_backward(dev(rec), dev(rot), dev(grad), dev(shift),
                                                    want_rot=False, opts=op, fused=True)
        assert g_none is None
        assert max_rel(host(g_rec2), r_rec) <= TOL_BWD
        assert max_rel(host(g_sh2), r_sh) <= TOL_BWD


@pytest.mark.parametrize("case", [c for c in CASES if c[0] == 3 and c[1] == 1][:4],
                         ids=[str(c) for c in CASES if c[0] == 3 and c[1] == 1][:4])
def test_backward_gradient_at_odd_8_byte_offset(case):
    """The volume gradient may start at any 8-byte boundary (the C ABI asks for 8): a buffer at
    an odd multiple of 8 bytes gives the oracle's result like an aligned one."""
    ndim = case[0]
    rec, rot, shift, grad, _, kw, op = make_case(case, seed=6)
    r_rec, _, _ = oracle.project_backward(ndim, rec, rot, grad, shift, want_rot=False,
                                          want_shift=False, **kw)
    V = dev(rec)
    buf = torch.empty(V.numel() + 1, dtype=V.dtype, device="cuda")
    g_rec = buf[1:].view(V.shape)
    assert g_rec.data_ptr() % 16 == 8
    tp.tp_project_backward(ndim, V, dev(rot), dev(shift), dev(grad), g_rec, None, None, op)
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD


@pytest.mark.parametrize("case", PARTIAL, ids=[str(c) for c in PARTIAL])
def test_backward_partial_outputs(case):
    """Each gradient output may be skipped (NULL); the others are unchanged."""
    ndim = case[0]
    rec, rot, shift, grad, _, kw, op = make_case(case, seed=2)
    r_rec, r_rot, r_sh = oracle.project_backward(ndim, rec, rot, grad, shift, **kw)
    g_rec, _, _ = tp.project_backward(dev(rec), dev(rot), dev(grad), dev(shift), want_rot=False,
                                      want_shift=False, opts=op)
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    _, g_rot, g_sh = tp.project_backward(dev(rec), dev(rot), dev(grad), dev(shift), want_rec=False,
                                         want_shift=shift is not None, opts=op)
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    if shift is not None:
        assert max_rel(host(g_sh), r_sh) <= TOL_BWD
    # without a shift the shift gradient is defined as zero
    _, _, g0 = tp.project_backward(dev(rec), dev(rot), dev(grad), None, want_rec=False, opts=op)
    assert np.all(host(g0) == 0)


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
@pytest.mark.parametrize("with_weights", [True, False])
def test_backproject(case, with_weights):
    ndim, Dv = case[0], case[4]
    _, rot, shift, proj, w, kw, op = make_case(case, seed=3)
    weights = w if with_weights else None
    vol, wvol = tp.backproject(dev(proj), dev(rot), dev(shift), dev(weights), Dv=Dv, opts=op,
                               ndim=ndim)
    r_vol, r_w = oracle.backproject(ndim, proj, rot, weights=weights, shift=shift, Dv=Dv, **kw)
    assert max_rel(host(vol), r_vol) <= TOL_BWD
    assert max_rel(host(wvol), r_w) <= TOL_BWD


@pytest.mark.parametrize("ndim", [2, 3])
def test_backproject_accumulate_and_skips(ndim):
    case = (ndim, 1, 1, 1.0, 24, 24, -1.0, True, 2, 2, 5)
    _, rot, shift, proj, w, kw, op = make_case(case, seed=4)
    r_vol, r_w = oracle.backproject(ndim, proj, rot, weights=w, shift=shift, Dv=24, **kw)
    vol, wvol = tp.backproject(dev(proj), dev(rot), dev(shift), dev(w), Dv=24, opts=op, ndim=ndim)
    fn = tp.tp_backproject_2d_to_3d if ndim == 3 else tp.tp_backproject_2d_to_2d
    fn(dev(proj), dev(w), dev(rot), dev(shift), vol, wvol, 24, True, op)       # accumulate
    assert max_rel(host(vol), 2 * r_vol) <= TOL_BWD
    assert max_rel(host(wvol), 2 * r_w) <= TOL_BWD
    # weights only (no data output), then data only, each overwriting (accumulate = 0)
    fn(dev(proj), dev(w), dev(rot), dev(shift), None, wvol, 24, False, op)
    assert max_rel(host(wvol), r_w) <= TOL_BWD
    fn(dev(proj), None, dev(rot), dev(shift), vol, None, 24, False, op)
    assert max_rel(host(vol), r_vol) <= TOL_BWD


CASES3 = [c for c in CASES if c[0] == 3]


@pytest.mark.parametrize("case", CASES3, ids=[str(c) for c in CASES3])
def test_workspace_path(case):
    """The gathers reading the grouped copy in a workspace give the plain call's forward bit
    for bit (same taps, weights and order) and the oracle's gradients."""
    ndim, Do = case[0], case[5]
    rec, rot, shift, grad, _, kw, op = make_case(case, seed=7)
    V, R, S, G = dev(rec), dev(rot), dev(shift), dev(grad)
    ws = tp.workspace_for(V, op)
    assert ws is not None and ws.numel() == tp.tp_workspace_size(3, rec.shape[0], rec.shape[1], op)
    y0 = tp.project(V, R, S, Do=Do, opts=op)
    y1 = torch.empty_like(y0)
    tp.tp_project_3d_to_2d_ws(V, R, S, y1, ws, op)
    assert torch.equal(y0, y1)
    g_rot = torch.empty_like(R)
    g_sh = torch.empty((1 if S is None else S.shape[0], R.shape[1], 2), device="cuda")
    g_rec = torch.empty_like(V)
    tp.tp_project_backward_ws(3, V, R, S, G, g_rec, g_rot, g_sh, ws, op)
    r_rec, r_rot, r_sh = oracle.project_backward(ndim, rec, rot, grad, shift, **kw)
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    if shift is not None:
        assert max_rel(host(g_sh), r_sh) <= TOL_BWD
    # a NULL workspace is the plain path
    y2 = torch.empty_like(y0)
    tp.tp_project_3d_to_2d_ws(V, R, S, y2, None, op)
    assert torch.equal(y0, y2)


def test_workspace_ignored_in_2d():
    """ndim = 2 has no grouped copy: a workspace passed to the backward is ignored."""
    case = CASES2[0]
    rec, rot, shift, grad, _, kw, op = make_case(case, seed=8)
    V, R, S, G = dev(rec), dev(rot), dev(shift), dev(grad)
    assert tp.tp_workspace_size(2, rec.shape[0], rec.shape[1], op) == 0
    ws = torch.empty(1 << 12, dtype=torch.uint8, device="cuda")
    g0 = tp.project_backward(V, R, G, S, opts=op)
    g1 = (torch.empty_like(V), torch.empty_like(R), torch.empty_like(g0[2]))
    tp.tp_project_backward_ws(2, V, R, S, G, g1[0], g1[1], g1[2], ws, op)
    for a, b in zip(g0, g1):
        assert max_rel(host(b), host(a)) <= TOL_BWD


# rotations per reconstruction with one shared set of shifts, and the reverse
MIXED = [(ndim, n_rot, n_sh) for ndim in (3, 2) for n_rot, n_sh in ((3, 1), (1, 3))]


@pytest.mark.parametrize("ndim,n_rot,n_sh", MIXED)
def test_mixed_pose_broadcast(ndim, n_rot, n_sh):
    """Rotations and shifts broadcast over the reconstructions independently (n_rot and n_sh
    each 1 or n_rec): every entry point, the gradient of the shared array summed over the
    reconstructions, on the plain, the workspace and the one-pass calls."""
    rng = np.random.default_rng(40 + 10 * ndim + n_rot)
    n_rec, n_pose, D = 3, 9, 26
    H = D // 2 + 1
    rec = crandn32(rng, (n_rec, D, D, H) if ndim == 3 else (n_rec, D, H))
    rot = rotations(rng, n_rot * n_pose, ndim).reshape(n_rot, n_pose, ndim, ndim)
    shift = rng.uniform(-6, 6, (n_sh, n_pose, 2)).astype(np.float32)
    grad = crandn32(rng, (n_rec, n_pose, D, H))
    w = rng.uniform(0.0, 2.0, (n_rec, n_pose, D, H)).astype(np.float32)
    kw = dict(interp=1, layout=1, oversampling=1.0, cutoff=-1.0)
    op = opts(1, 1, 1.0, -1.0)
    V, R, S, G = dev(rec), dev(rot), dev(shift), dev(grad)

    y = tp.project(V, R, S, Do=D, opts=op)
    assert max_rel(host(y), oracle.project(ndim, rec, rot, shift, Do=D, **kw)) <= TOL_FWD
    r_rec, r_rot, r_sh = oracle.project_backward(ndim, rec, rot, grad, shift, **kw)
    g_rec, g_rot, g_sh = tp.project_backward(V, R, G, S, want_shift=True, opts=op)
    assert g_rot.shape == R.shape and g_sh.shape == S.shape
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    assert max_rel(host(g_sh), r_sh) <= TOL_BWD
    vol, wvol = tp.backproject(G, R, S, dev(w), Dv=D, opts=op, ndim=ndim)
    r_vol, r_w = oracle.backproject(ndim, grad, rot, weights=w, shift=shift, Dv=D, **kw)
    assert max_rel(host(vol), r_vol) <= TOL_BWD
    assert max_rel(host(wvol), r_w) <= TOL_BWD
    if ndim == 3:
        ws = tp.workspace_for(V, op)
        y1 = torch.empty_like(y)
        tp.tp_project_3d_to_2d_ws(V, R, S, y1, ws, op)
        assert torch.equal(y, y1)
        g1 = (torch.empty_like(V), torch.empty_like(R), torch.empty_like(S))
        tp.tp_project_backward_ws(3, V, R, S, G, g1[0], g1[1], g1[2], ws, op)
        assert max_rel(host(g1[0]), r_rec) <= TOL_BWD
        assert max_rel(host(g1[1]), r_rot) <= TOL_BWD
        assert max_rel(host(g1[2]), r_sh) <= TOL_BWD
        # the one-pass backward: a shared pose's gradient gathers every reconstruction's terms
        g2 = tp.project_backward(V, R, G, S, want_shift=True, opts=op, fused=True)
        assert max_rel(host(g2[0]), r_rec) <= TOL_BWD
        assert max_rel(host(g2[1]), r_rot) <= TOL_BWD
        assert max_rel(host(g2[2]), r_sh) <= TOL_BWD


def _bp_grads(case, with_weights, seed):
    ndim = case[0]
    Gv, rot, shift, proj, w, kw, op = make_case(case, seed=seed)
    rng = np.random.default_rng(seed + 100)
    GW = rng.standard_normal(Gv.shape).astype(np.float32)
    weights = w if with_weights else None
    return ndim, Gv, GW, rot, shift, proj, weights, kw, op


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
@pytest.mark.parametrize("with_weights", [True, False])
def test_backproject_backward(case, with_weights):
    """Gradients of the insertion for upstream gradients of both the data and weight volumes."""
    ndim, Gv, GW, rot, shift, proj, weights, kw, op = _bp_grads(case, with_weights, 5)
    gP, gW, gR, gs = tp.backproject_backward(dev(proj), dev(rot), dev(Gv), dev(GW), dev(shift),
                                             dev(weights), want_shift=shift is not None, opts=op,
                                             ndim=ndim)
    rP, rW, rR, rs = oracle.backproject_backward(ndim, proj, rot, Gv, GW, weights, shift, **kw)
    assert max_rel(host(gP), rP) <= TOL_FWD
    if with_weights:
        assert max_rel(host(gW), rW) <= TOL_FWD
    assert max_rel(host(gR), rR) <= TOL_BWD
    if ndim == 3:
        assert np.all(host(gR)[..., 2] == 0)
    if shift is not None:
        assert max_rel(host(gs), rs) <= TOL_BWD


@pytest.mark.parametrize("case", [CASES[0], CASES[3], CASES2[0]], ids=str)
def test_backproject_backward_partial(case):
    """Either upstream gradient may be absent (= 0) and any output skipped."""
    ndim, Gv, GW, rot, shift, proj, weights, kw, op = _bp_grads(case, True, 6)
    # data volume only
    rP, _, rR, rs = oracle.backproject_backward(ndim, proj, rot, Gv, None, weights, shift, **kw)
    gP, gW, gR, gs = tp.backproject_backward(dev(proj), dev(rot), dev(Gv), None, dev(shift),
                                             dev(weights), opts=op, ndim=ndim)
    assert max_rel(host(gP), rP) <= TOL_FWD
    assert np.all(host(gW) == 0)
    assert max_rel(host(gR), rR) <= TOL_BWD
    if shift is not None:
        assert max_rel(host(gs), rs) <= TOL_BWD
    else:
        assert np.all(host(gs) == 0)
    # weight volume only: no proj needed; the data gradients are zero
    _, rW, rR, _ = oracle.backproject_backward(ndim, proj, rot, None, GW, weights, shift, **kw)
    gP, gW, gR, gs = tp.backproject_backward(dev(proj), dev(rot), None, dev(GW), dev(shift),
                                             dev(weights), opts=op, ndim=ndim)
    assert np.all(host(gP) == 0) and np.all(host(gs) == 0)
    assert max_rel(host(gW), rW) <= TOL_FWD
    assert max_rel(host(gR), rR) <= TOL_BWD
    # pose gradients only, then the image gradients only (proj not needed)
    _, rW, rR, rs = oracle.backproject_backward(ndim, proj, rot, Gv, GW, weights, shift, **kw)
    _, _, gR, gs = tp.backproject_backward(dev(proj), dev(rot), dev(Gv), dev(GW), dev(shift),
                                           dev(weights), want_proj=False, want_weights=False,
                                           opts=op, ndim=ndim)
    assert max_rel(host(gR), rR) <= TOL_BWD
    gP = torch.empty(proj.shape, dtype=torch.complex64, device="cuda")
    gW = torch.empty(proj.shape, dtype=torch.float32, device="cuda")
    tp.tp_backproject_backward(ndim, None, None, dev(rot), dev(shift), dev(Gv), dev(GW), gP, gW,
                               None, None, op)
    rP = oracle.project(ndim, Gv, rot, shift, Do=proj.shape[2], **kw)
    assert max_rel(host(gP), rP) <= TOL_FWD
    assert max_rel(host(gW), rW) <= TOL_FWD


def test_empty_batches():
    vol = torch.ones((1, 8, 8, 5), dtype=torch.complex64, device="cuda")
    rot = torch.zeros((1, 0, 3, 3), device="cuda")
    out = torch.empty((1, 0, 8, 5), dtype=torch.complex64, device="cuda")
    tp.tp_project_3d_to_2d(vol, rot, None, out)
    w = torch.ones((1, 8, 8, 5), device="cuda")
    tp.tp_backproject_2d_to_3d(out, None, rot, None, vol, w, 8, False)   # zeroes the outputs
    torch.cuda.synchronize()
    assert torch.all(vol == 0) and torch.all(w == 0)
    g_rot = torch.full((1, 0, 3, 3), 7.0, device="cuda")
    tp.tp_project_backward(3, vol, rot, None, out, vol, g_rot, None)
    gw = torch.empty((1, 0, 8, 5), device="cuda")
    tp.tp_backproject_backward(3, out, gw, rot, None, vol, w, out, gw, g_rot, None)
    torch.cuda.synchronize()


def test_many_items_grid_stride():
    """More work units than one grid holds: the kernels stride over items."""
    rng = np.random.default_rng(7)
    n_pose = 90000
    rec = crandn32(rng, (1, 4, 4, 3))
    rot = rotations(rng, n_pose, 3)[None]
    shift = rng.uniform(-1, 1, (1, n_pose, 2)).astype(np.float32)
    y = tp.project(dev(rec), dev(rot), dev(shift), opts=opts(1))
    items = rng.integers(0, n_pose, 3000)
    pix = rng.integers(0, 4 * 3, 3000)
    ref = oracle.project_samples(3, rec, rot, items, pix, shift, interp=1)
    got = host(y).reshape(n_pose, -1)[items, pix]
    assert max_rel(got, ref) <= TOL_FWD
    grec, grot, gsh = tp.project_backward(dev(rec), dev(rot), dev(crandn32(rng, (1, n_pose, 4, 3))),
                                          dev(shift), opts=opts(1))
    torch.cuda.synchronize()
    assert torch.isfinite(grot).all()


def test_large_box_sampled():
    """D = 512 volume (32-bit in-volume offsets near their largest use) on a few poses."""
    rng = np.random.default_rng(8)
    D = 512
    rec = crandn32(rng, (1, D, D, D // 2 + 1))
    rot = rotations(rng, 3, 3)[None]
    shift = rng.uniform(-20, 20, (1, 3, 2)).astype(np.float32)
    y = host(tp.project(dev(rec), dev(rot), dev(shift), opts=opts(1)))
    items = rng.integers(0, 3, 4000)
    pix = rng.integers(0, D * (D // 2 + 1), 4000)
    ref = oracle.project_samples(3, rec, rot, items, pix, shift, interp=1)
    assert max_rel(y.reshape(3, -1)[items, pix], ref) <= TOL_FWD


def test_large_2d_box_fallback_kernels():
    """2D boxes beyond the shared-memory tables: at D = 4100 the gathers take the per-pixel
    kernels (image boxes above 4096) and the insertion and image gradient the direct-atomic
    kernel (boxes above 1024).  Forward on sampled pixels, full backward and insertion with
    weights against the oracle."""
    rng = np.random.default_rng(21)
    D = 4100
    H = D // 2 + 1
    rec = crandn32(rng, (2, D, H))
    rot = rotations(rng, 2, 2).reshape(2, 1, 2, 2)
    shift = rng.uniform(-40, 40, (2, 1, 2)).astype(np.float32)
    grad = crandn32(rng, (2, 1, D, H))
    w = rng.uniform(0.0, 2.0, (2, 1, D, H)).astype(np.float32)
    op, kw = opts(1), dict(interp=1, layout=1)
    y = host(tp.project(dev(rec), dev(rot), dev(shift), opts=op))
    items, pix = rng.integers(0, 2, 4000), rng.integers(0, D * H, 4000)
    ref = oracle.project_samples(2, rec, rot, items, pix, shift, **kw)
    assert max_rel(y.reshape(2, -1)[items, pix], ref) <= TOL_FWD
    g_rec, g_rot, g_sh = tp.project_backward(dev(rec), dev(rot), dev(grad), dev(shift), opts=op)
    r_rec, r_rot, r_sh = oracle.project_backward(2, rec, rot, grad, shift, **kw)
    assert max_rel(host(g_rec), r_rec) <= TOL_BWD
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    assert max_rel(host(g_sh), r_sh) <= TOL_BWD
    vol, wvol = tp.backproject(dev(grad), dev(rot), dev(shift), dev(w), Dv=D, opts=op, ndim=2)
    r_vol, r_w = oracle.backproject(2, grad, rot, weights=w, shift=shift, Dv=D, **kw)
    assert max_rel(host(vol), r_vol) <= TOL_BWD
    assert max_rel(host(wvol), r_w) <= TOL_BWD


def test_largest_3d_box():
    """D = 1024, the largest 3D box (a 4.3 GB volume): in-volume offsets at their largest and
    no grouped copy (its offsets would not fit 32 bits).  Forward on sampled pixels and the
    pose gradients against the oracle; the volume gradient by the transpose identity
    Re<g, P V> = Re<P^T g, V>, summed in complex128 from the library's own outputs."""
    rng = np.random.default_rng(22)
    D, n_pose = 1024, 3
    H = D // 2 + 1
    rec = rng.standard_normal((1, D, D, H, 2), dtype=np.float32).view(np.complex64)
    rec = rec.reshape(1, D, D, H)
    rot = rotations(rng, n_pose, 3)[None]
    shift = rng.uniform(-20, 20, (1, n_pose, 2)).astype(np.float32)
    grad = crandn32(rng, (1, n_pose, D, H))
    op, kw = opts(1), dict(interp=1, layout=1)
    assert tp.tp_workspace_size(3, 1, D, op) == 0
    V, R, S, G = dev(rec), dev(rot), dev(shift), dev(grad)
    y = tp.project(V, R, S, opts=op)
    items, pix = rng.integers(0, n_pose, 4000), rng.integers(0, D * H, 4000)
    ref = oracle.project_samples(3, rec, rot, items, pix, shift, **kw)
    assert max_rel(host(y).reshape(n_pose, -1)[items, pix], ref) <= TOL_FWD
    g_rec, g_rot, g_sh = tp.project_backward(V, R, G, S, opts=op)
    _, r_rot, r_sh = oracle.project_backward(3, rec, rot, grad, shift, want_rec=False, **kw)
    assert max_rel(host(g_rot), r_rot) <= TOL_BWD
    assert max_rel(host(g_sh), r_sh) <= TOL_BWD
    t_l = (G.to(torch.complex128).conj() * y.to(torch.complex128))
    lhs, scale_l = float(t_l.real.sum()), float(t_l.abs().sum())
    rhs = scale_r = 0.0
    for z0 in range(0, D, 128):                      # complex128 in slabs: bounded memory
        t_r = g_rec[:, z0:z0 + 128].to(torch.complex128).conj() * V[:, z0:z0 + 128].to(torch.complex128)
        rhs += float(t_r.real.sum())
        scale_r += float(t_r.abs().sum())
    assert abs(lhs - rhs) <= 1e-5 * max(scale_l, scale_r)
