"""GPU: the padding kernels (bit-exact data movement) and the on-the-fly oversampling pipeline
at the compared sizes, D = 128 with factor 1 (cubic) and factor 2 (linear), checked against
the fp64 oracle on sampled pixels."""
import numpy as np
import pytest
import torch

from parity_util import TOL_FWD, dev, host, max_rel, oracle, rotations
from back_projection_fourier_b300 import autograd as tpa
from back_projection_fourier_b300 import tp

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ndim,D,factor,n", [(3, 6, 1, 2), (3, 10, 2, 1), (3, 8, 3, 2), (2, 34, 2, 3),
                                             (2, 2, 8, 1), (3, 130, 2, 1)])
def test_pad_and_crop_bit_exact(ndim, D, factor, n):
    rng = np.random.default_rng(D + factor)
    vol = rng.standard_normal((n,) + (D,) * ndim).astype(np.float32)
    p = tp.pad_volume(dev(vol), factor, ndim)
    np.testing.assert_array_equal(host(p), oracle.pad_volume(vol, factor).astype(np.float32))
    big = rng.standard_normal(p.shape).astype(np.float32)
    c = tp.crop_volume(dev(big), D, factor, ndim)
    np.testing.assert_array_equal(host(c), oracle.crop_volume(big, D).astype(np.float32))


def test_pad_empty():
    vol = torch.empty((0, 8, 8, 8), device="cuda")
    assert tp.pad_volume(vol, 2).shape == (0, 16, 16, 16)


@pytest.mark.parametrize("factor,interp", [(1, 1), (2, 0)])
def test_pipeline_d128_sampled(factor, interp):
    """D = 128 real-space volume, 64 poses, projected through the pipeline; 4000 sampled pixels
    against the oracle's own pipeline (numpy FFT in fp64, then per-pixel projection)."""
    rng = np.random.default_rng(7 + factor)
    D, n_pose = 128, 64
    vol = rng.standard_normal((1, D, D, D)).astype(np.float32)
    rot = rotations(rng, n_pose, 3)[None]
    shift = rng.uniform(-5, 5, (1, n_pose, 2)).astype(np.float32)
    with torch.no_grad():
        out = host(tpa.project_real(dev(vol), dev(rot), dev(shift), factor=factor, interp=interp))
    spec = oracle.oversampled_spectrum(vol, factor)
    items = rng.integers(0, n_pose, 4000)
    pix = rng.integers(0, D * (D // 2 + 1), 4000)
    ref = oracle.project_samples(3, spec, rot, items, pix, shift, Do=D, interp=interp,
                                 layout=oracle.FFTW, oversampling=float(factor))
    assert max_rel(out.reshape(n_pose, -1)[items, pix], ref) <= TOL_FWD
