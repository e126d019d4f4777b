"""The seeded input generator: each input has the distribution and structure the recipe
states (uniform rotations, CN(0, 1) upstream gradients, spectra of real volumes, the
CTF-like weights), and is reproducible from its seed alone.  CPU only."""
import numpy as np
import pytest

from back_projection_fourier_b300 import synth


class _FixedRng:
    """Stands in for a numpy Generator whose draws are chosen by the test."""

    def __init__(self, values):
        self.values = np.asarray(values, np.float64)

    def standard_normal(self, shape):
        return self.values.reshape(shape).copy()

    def uniform(self, lo, hi, n):
        return self.values.reshape(n).copy()


def test_quaternion_to_matrix_convention():
    """Hamilton convention: the unit quaternion (cos t/2, sin t/2 * axis) is the right-handed
    rotation by t about that axis; the identity quaternion gives the identity."""
    t = 0.7
    q = [[1, 0, 0, 0], [np.cos(t / 2), 0, 0, np.sin(t / 2)], [np.cos(t / 2), np.sin(t / 2), 0, 0]]
    R = synth.rotations_3d(_FixedRng(q), 3).astype(np.float64)
    c, s = np.cos(t), np.sin(t)
    np.testing.assert_allclose(R[0], np.eye(3), atol=1e-7)
    np.testing.assert_allclose(R[1], [[c, -s, 0], [s, c, 0], [0, 0, 1]], atol=1e-7)
    np.testing.assert_allclose(R[2], [[1, 0, 0], [0, c, -s], [0, s, c]], atol=1e-7)
    # an unnormalised draw is normalised first
    R2 = synth.rotations_3d(_FixedRng([[3.0, 0, 0, 0]]), 1)
    np.testing.assert_allclose(R2[0], np.eye(3), atol=1e-7)


def test_rotations_3d_are_uniform_on_so3():
    """Proper orthogonal matrices with the moments of the Haar measure on SO(3):
    E[tr R] = 0, E[tr(R)^2] = 1, and every column uniform on the sphere."""
    n = 40000
    R = synth.rotations_3d(np.random.default_rng(1), n)
    assert R.dtype == np.float32 and R.shape == (n, 3, 3)
    R = R.astype(np.float64)
    np.testing.assert_allclose(np.einsum("nji,njk->nik", R, R), np.broadcast_to(np.eye(3), R.shape),
                               atol=2e-6)
    np.testing.assert_allclose(np.linalg.det(R), 1.0, atol=2e-6)
    tr = np.trace(R, axis1=1, axis2=2)
    assert abs(tr.mean()) < 0.03                  # std of the mean 0.005
    assert abs((tr * tr).mean() - 1.0) < 0.05     # std of the mean 0.007
    for col in range(3):
        v = R[:, :, col]
        assert np.all(np.abs(v.mean(0)) < 0.02)
        np.testing.assert_allclose((v * v).mean(0), 1.0 / 3.0, atol=0.01)


def test_rotations_2d():
    th = np.array([0.0, np.pi / 2, 2.0])
    R = synth.rotations_2d(_FixedRng(th), 3).astype(np.float64)
    np.testing.assert_allclose(R[1], [[0, -1], [1, 0]], atol=1e-7)
    np.testing.assert_allclose(R[2], [[np.cos(2.0), -np.sin(2.0)], [np.sin(2.0), np.cos(2.0)]],
                               atol=1e-7)
    R = synth.rotations_2d(np.random.default_rng(2), 20000).astype(np.float64)
    np.testing.assert_allclose(np.linalg.det(R), 1.0, atol=1e-6)
    ang = np.arctan2(R[:, 1, 0], R[:, 0, 0])
    assert abs(np.cos(ang).mean()) < 0.03 and abs(np.sin(ang).mean()) < 0.03
    assert abs((np.cos(ang) ** 2).mean() - 0.5) < 0.02


def test_cn01_items_moments_and_reproducibility():
    """Real and imaginary parts N(0, 1/2), uncorrelated; any subset of items regenerates
    exactly from (seed, tag) alone, in any order; another tag draws other numbers."""
    n, shape = 600, (8, 5)
    z = synth.cn01_items(7, 1, n, shape).astype(np.complex128)
    assert z.shape == (n,) + shape
    np.testing.assert_allclose((z.real ** 2).mean(), 0.5, atol=0.02)
    np.testing.assert_allclose((z.imag ** 2).mean(), 0.5, atol=0.02)
    assert abs((z.real * z.imag).mean()) < 0.02 and abs(z.mean()) < 0.03
    assert abs((z * z).mean()) < 0.03             # circular: E[z^2] = 0
    items = [599, 3, 256, 255, 3]
    np.testing.assert_array_equal(synth.cn01_items(7, 1, n, shape, items=items), z[items])
    assert not np.array_equal(synth.cn01_items(7, 2, n, shape), z)


def test_volume_spectrum_is_the_unit_variance_spectrum_of_a_real_volume():
    D = 16
    V = synth.volume_spectrum(np.random.default_rng(3), D, layout=synth.FFTW).astype(np.complex128)
    assert V.shape == (D, D, D // 2 + 1)
    f = np.fft.irfftn(V, s=(D, D, D), axes=(0, 1, 2), norm="ortho")
    np.testing.assert_allclose(np.fft.rfftn(f, norm="ortho"), V, atol=1e-5)   # Hermitian planes
    assert abs(np.var(f) - 1.0) < 0.1
    Vc = synth.volume_spectrum(np.random.default_rng(3), D, layout=synth.CENTERED)
    np.testing.assert_array_equal(Vc, np.fft.fftshift(V.astype(np.complex64), axes=(0, 1)))
    # the falloff divides by max(|k|, 1)
    Vf = synth.volume_spectrum(np.random.default_rng(3), D, layout=synth.FFTW, falloff=True)
    k = np.fft.fftfreq(D, 1.0 / D)
    kk = np.sqrt(k[:, None, None] ** 2 + k[None, :, None] ** 2 + np.arange(D // 2 + 1) ** 2)
    np.testing.assert_allclose(Vf, V / np.maximum(kk, 1.0), rtol=1e-6, atol=1e-7)


def test_image_spectra_and_ball_volume():
    D = 12
    im = synth.image_spectra(np.random.default_rng(4), 3, D, layout=synth.FFTW).astype(np.complex128)
    f = np.fft.irfft2(im, s=(D, D), norm="ortho")
    np.testing.assert_allclose(np.fft.rfft2(f, norm="ortho"), im, atol=1e-5)
    v = synth.ball_noise_volume(np.random.default_rng(5), D, margin=2)
    r2 = ((np.indices(v.shape) - D // 2) ** 2).sum(0)
    assert np.all(v[r2 > (D // 2 - 2) ** 2] == 0) and np.all(v[r2 <= (D // 2 - 2) ** 2] != 0)


@pytest.mark.parametrize("layout", [synth.FFTW, synth.CENTERED])
def test_ctf_like_weights(layout):
    """1 - exp(-|k|^2/sigma^2) cos(gamma |k|^2): non-negative, zero at DC only, one far out."""
    D, sigma, gamma = 64, 10.0, 1e-3
    w = synth.ctf_like_weights(D, sigma, gamma, layout).astype(np.float64)
    assert w.shape == (D, D // 2 + 1) and np.all(w >= 0)
    dc_row = D // 2 if layout == synth.CENTERED else 0
    assert w[dc_row, 0] == 0 and np.count_nonzero(w == 0) == 1
    ky = D // 2 - 4 + (0 if layout == synth.CENTERED else D // 2)   # ky = -4 in either layout
    k2 = 16.0 + 9.0
    np.testing.assert_allclose(w[ky % D, 3], 1 - np.exp(-k2 / sigma ** 2) * np.cos(gamma * k2),
                               rtol=1e-6)
    assert abs(w[dc_row, D // 2] - 1.0) < 1e-4     # |k| = 32 >> sigma


def test_workloads_are_seeded_and_shaped():
    a = synth.make_workload("fwdbwd3d_d64_cubic_b4096", B=64)
    b = synth.make_workload("fwdbwd3d_d64_cubic_b4096", B=64)
    for x, y in ((a.rec, b.rec), (a.rot, b.rot), (a.shift, b.shift), (a.grad, b.grad)):
        np.testing.assert_array_equal(x, y)
    assert a.rec.shape == (1, 64, 64, 33) and a.rec.dtype == np.complex64
    assert a.rot.shape == (1, 64, 3, 3) and a.rot.dtype == np.float32
    assert a.shift.shape == (1, 64, 2) and np.all(np.abs(a.shift) <= 5.0)
    assert a.grad.shape == (1, 64, 64, 33) and a.grad.dtype == np.complex64
    r8 = synth.make_workload("fwdbwd3d_d128_cubic_r8_b16384", B=64)
    assert r8.rec.shape[0] == 8 and r8.rot.shape == (8, 8, 3, 3) and r8.grad.shape[:2] == (8, 8)
    ins = synth.make_workload("insert3d_d128_b16384", B=4)
    assert ins.rec is None and ins.weights.shape == (1, 4, 128, 65) and ins.shift is None
    im = synth.make_workload("rot2d_d256_cubic_b8192", B=5)
    assert im.rec.shape == (5, 256, 129) and im.rot.shape == (5, 1, 2, 2)
    with pytest.raises(ValueError):
        synth.make_workload("fwdbwd3d_d128_cubic_r8_b16384", B=12)
