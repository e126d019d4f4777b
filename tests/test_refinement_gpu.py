"""GPU, end to end through the differentiable operators: refine poses and shifts by gradient
descent.  Projections of a synthetic volume at true rotations and shifts are the targets; from
rotations perturbed by a few degrees and shifts off by a pixel, Adam on the squared error
(gradients from tp_project_backward through torch.autograd) must bring both back.  This is the
use the method is made for: projections inside an optimisation loop, with gradients for the
rotation matrices and the shifts."""
import numpy as np
import pytest
import torch

from back_projection_fourier_b300 import autograd as tpa
from back_projection_fourier_b300 import synth, tp

pytestmark = pytest.mark.gpu


def small_rotation(rng, n, deg):
    axis = rng.standard_normal((n, 3))
    axis /= np.linalg.norm(axis, axis=1, keepdims=True)
    ang = np.deg2rad(deg) * np.ones(n)
    K = np.zeros((n, 3, 3))
    K[:, 0, 1], K[:, 0, 2], K[:, 1, 2] = -axis[:, 2], axis[:, 1], -axis[:, 0]
    K = K - K.transpose(0, 2, 1)
    I = np.eye(3)[None]
    return I + np.sin(ang)[:, None, None] * K + (1 - np.cos(ang))[:, None, None] * (K @ K)


@pytest.mark.parametrize("interp", [tp.TP_CUBIC, tp.TP_LINEAR])
def test_pose_and_shift_refinement(interp):
    rng = np.random.default_rng(123)
    D, n = 64, 8
    vol = torch.from_numpy(synth.volume_spectrum(rng, D, falloff=True)[None]).cuda()
    R_true = synth.rotations_3d(rng, n).astype(np.float64)
    s_true = rng.uniform(-3, 3, (1, n, 2))
    with torch.no_grad():
        target = tpa.project(vol, torch.from_numpy(R_true[None].astype(np.float32)).cuda(),
                             torch.from_numpy(s_true.astype(np.float32)).cuda(), interp=interp,
                             cutoff=D / 4)
    R0 = np.einsum("nab,nbc->nac", small_rotation(rng, n, 4.0), R_true)
    R = torch.from_numpy(R0[None].astype(np.float32)).cuda().requires_grad_(True)
    s = torch.from_numpy((s_true + rng.choice([-1.0, 1.0], s_true.shape)).astype(np.float32))
    s = s.cuda().requires_grad_(True)
    opt = torch.optim.Adam([{"params": [R], "lr": 5e-3}, {"params": [s], "lr": 5e-2}])

    def loss_fn():
        y = tpa.project(vol, R, s, interp=interp, cutoff=D / 4)
        return (y - target).abs().pow(2).sum() / target.abs().pow(2).sum()

    with torch.no_grad():
        first = float(loss_fn())
    for _ in range(400):
        opt.zero_grad()
        loss = loss_fn()
        loss.backward()
        opt.step()
    with torch.no_grad():
        last = float(loss_fn())
    # only the first two columns act on q = (kx, ky, 0): the third is not observable
    R_err = np.abs(R.detach().cpu().numpy()[0][..., :2] - R_true[..., :2]).max()
    s_err = np.abs(s.detach().cpu().numpy() - s_true).max()
    assert last < 1e-3 * first, (first, last)
    assert R_err < 5e-3, R_err
    assert s_err < 0.05, s_err
