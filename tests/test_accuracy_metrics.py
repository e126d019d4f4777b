"""CPU pins of the accuracy metrics (back_projection_fourier_b300.accuracy) and of the oracle's
exact projection, the ground truth of the accuracy comparison."""
import numpy as np
import pytest

from back_projection_fourier_b300 import accuracy, synth
from test_oracle_pins import crandn, random_rotations


def test_frc_of_scaled_copies():
    rng = np.random.default_rng(1)
    a = crandn(rng, (3, 16, 9))
    np.testing.assert_allclose(accuracy.frc(a, a), 1.0, atol=1e-12)
    np.testing.assert_allclose(accuracy.frc(a, 2.5 * a), 1.0, atol=1e-12)
    np.testing.assert_allclose(accuracy.frc(a, -a), -1.0, atol=1e-12)
    np.testing.assert_allclose(accuracy.frc(a, 1j * a), 0.0, atol=1e-12)


def test_frc_of_independent_noise_is_small():
    rng = np.random.default_rng(2)
    a, b = crandn(rng, (64, 32, 17)), crandn(rng, (64, 32, 17))
    f = accuracy.frc(a, b)
    n = np.bincount(accuracy.ring_index(32).ravel()) * 64
    assert np.all(np.abs(f[1:]) < 5 / np.sqrt(n[1:17]))


def test_frc_layouts_agree():
    rng = np.random.default_rng(3)
    a, b = crandn(rng, (2, 12, 7)), crandn(rng, (2, 12, 7))
    c = lambda x: np.fft.fftshift(x, axes=-2)
    np.testing.assert_allclose(accuracy.frc(c(a), c(b), accuracy.CENTERED), accuracy.frc(a, b),
                               atol=1e-12)


def test_attenuation_recovers_a_radial_gain():
    """a = the reference image multiplied by a gain that is constant on each radius bin."""
    rng = np.random.default_rng(4)
    D, nbins = 32, 8
    img = rng.standard_normal((5, D, D))
    yy, xx = np.indices((D, D)) - D // 2
    rr = np.sqrt(xx * xx + yy * yy)
    edges = np.linspace(0, D / 2, nbins + 1)
    want = rng.uniform(0.3, 1.0, nbins)
    w = np.ones((D, D))
    for i in range(nbins):
        w[(rr >= edges[i]) & (rr < edges[i + 1])] = want[i]
    spec = lambda x: np.fft.rfft2(np.fft.ifftshift(x, axes=(-2, -1)))
    e, gain = accuracy.real_space_attenuation(spec(img * w), spec(img), nbins=nbins)
    np.testing.assert_allclose(e, edges)
    np.testing.assert_allclose(gain, want, atol=1e-12)


# ------------------------------------------------------- exact projection ----

def test_exact_projection_identity_is_the_dft_of_the_z_sum(orc):
    rng = np.random.default_rng(5)
    D = 10
    v = rng.standard_normal((1, D, D, D))
    ex = orc.exact_projection(3, v, np.eye(3)[None, None])
    want = np.fft.rfft2(np.fft.ifftshift(v[0].sum(0)))
    keep = ex[0, 0] != 0
    assert keep.sum() > 0.7 * keep.size
    np.testing.assert_allclose(ex[0, 0][keep], want[keep], atol=1e-11 * np.abs(want).max())


def test_exact_projection_of_a_point(orc):
    """A single voxel at n0 has F(c) = exp(-2 pi i c.(n0 - D/2) / D) at any c."""
    rng = np.random.default_rng(6)
    D = 12
    n0 = np.array([7, 3, 9])   # (x, y, z)
    v = np.zeros((1, D, D, D))
    v[0, n0[2], n0[1], n0[0]] = 1.0
    R = random_rotations(rng, 3, 3)[None]
    ex = orc.exact_projection(3, v, R, cutoff=1e9)
    ky = np.fft.fftfreq(D, 1.0 / D)
    KY, KX = np.meshgrid(ky, np.arange(D // 2 + 1), indexing="ij")
    for p in range(3):
        c = np.einsum("ab,b...->a...", R[0, p][:, :2], np.stack([KX, KY]))
        want = np.exp(-2j * np.pi * np.einsum("a...,a->...", c, n0 - D // 2) / D)
        np.testing.assert_allclose(ex[0, p], want, atol=1e-12)


def test_exact_projection_shift_is_a_real_space_roll(orc):
    rng = np.random.default_rng(7)
    D = 12
    v = synth.ball_noise_volume(rng, D, margin=4)[None]
    s = np.array([[[2.0, -3.0]]])
    moved = np.roll(v, (-3, 2), axis=(2, 3))     # +2 in x, -3 in y
    a = orc.exact_projection(3, v, np.eye(3)[None, None], shift=s)
    b = orc.exact_projection(3, moved, np.eye(3)[None, None])
    np.testing.assert_allclose(a, b, atol=1e-11 * np.abs(b).max())


def test_pipeline_converges_at_the_interpolation_order(orc):
    """Relative L2 error of pad -> FFT -> sample against the exact projection as the padding
    factor f doubles: linear interpolation is second order (error / 4 per doubling), Keys'
    cubic third order (error / 8)."""
    rng = np.random.default_rng(8)
    D = 16
    v = synth.ball_noise_volume(rng, D)[None]
    R = random_rotations(rng, 3, 3)[None]
    ex = orc.exact_projection(3, v, R)
    err = {}
    for interp in (0, 1):
        for f in (2, 4, 8):
            a = orc.project_real(3, v, R, factor=f, interp=interp)
            err[interp, f] = np.linalg.norm(a - ex) / np.linalg.norm(ex)
    for f in (2, 4):
        assert 3.0 < err[0, f] / err[0, 2 * f] < 5.0, err
        assert 6.0 < err[1, f] / err[1, 2 * f] < 16.0, err


def test_exact_projection_2d(orc):
    rng = np.random.default_rng(9)
    D = 14
    v = rng.standard_normal((2, D, D))
    ex = orc.exact_projection(2, v, np.eye(2)[None, None])
    for r in range(2):
        want = np.fft.rfft2(np.fft.ifftshift(v[r]))
        keep = ex[r, 0] != 0
        np.testing.assert_allclose(ex[r, 0][keep], want[keep], atol=1e-11 * np.abs(want).max())
