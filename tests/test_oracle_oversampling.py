"""Pins of the oracle's on-the-fly oversampling pipeline (real-space zero padding, FFT,
sampling at c = factor * R q) against facts it does not compute itself: the DFT of a
zero-padded signal sampled every `factor` bins is the DFT of the signal; padding and
cropping are adjoint and crop(pad(v)) = v; the Fourier slice theorem for a volume centred at
D/2, with rotations of the cube applied to the real-space data; and central differences of
the pipeline for its gradient.  Sources: torch-projectors summaries (gist.science), Dutch
page, problem statement (oversampling = zero-filling in the spatial domain); French page,
results, interpolation comparison (cubic without padding against linear with padding on the
fly)."""
import numpy as np
import pytest

from test_oracle_pins import pixel_freqs, random_rotations, rdot, signed_permutations, crandn


def ball_volume(rng, D, k):
    """Random real data that vanish outside the ball of radius D/2 - 1 about the centre D/2,
    so that rotations about the centre keep every voxel inside the box."""
    f = rng.standard_normal((D,) * k)
    r = np.indices(f.shape) - D // 2
    f[(r ** 2).sum(0) > (D // 2 - 1) ** 2] = 0.0
    return f


def rotate_about_centre(f, R):
    """g[m] = f[c + R (m - c)], c = D/2 on every axis (vector order x, y[, z]).  The one face
    that maps outside the box (component +D/2) wraps onto the face at -D/2, where f (a ball
    volume) is zero either way."""
    D = f.shape[0]
    vec = (np.indices(f.shape) - D // 2)[::-1]
    src = (np.rint(np.einsum("ab,b...->a...", R, vec)).astype(np.int64) + D // 2) % D
    return f[tuple(src[::-1])]


@pytest.mark.parametrize("k", [2, 3])
@pytest.mark.parametrize("factor", [1, 2, 3])
def test_pad_crop_roundtrip_and_adjoint(orc, k, factor):
    rng = np.random.default_rng(50 + k + factor)
    D = 6
    v = rng.standard_normal((2,) + (D,) * k)
    p = orc.pad_volume(v, factor)
    assert p.shape == (2,) + (factor * D,) * k
    np.testing.assert_array_equal(orc.crop_volume(p, D), v)
    # every entry of v appears once, the rest are zeros
    assert np.count_nonzero(p) == np.count_nonzero(v)
    b = rng.standard_normal(p.shape)
    assert abs(np.sum(p * b) - np.sum(v * orc.crop_volume(b, D))) <= 1e-12 * np.abs(b).sum()
    # the centre voxel lands at index 0 of the padded box
    d = np.zeros((1,) + (D,) * k)
    d[(0,) + (D // 2,) * k] = 1.0
    assert orc.pad_volume(d, factor)[(0,) + (0,) * k] == 1.0


@pytest.mark.parametrize("k", [2, 3])
@pytest.mark.parametrize("factor", [2, 3])
def test_padded_spectrum_even_samples_are_the_unpadded_spectrum(orc, k, factor):
    rng = np.random.default_rng(60 + k)
    D = 8
    v = rng.standard_normal((1,) + (D,) * k)
    big = orc.oversampled_spectrum(v, factor)
    small = orc.oversampled_spectrum(v, 1)
    sub = big[(slice(None),) + (slice(None, None, factor),) * k]
    np.testing.assert_allclose(sub, small, rtol=0, atol=1e-11 * np.abs(small).max())


@pytest.mark.parametrize("factor,interp", [(1, 1), (2, 0), (2, 1), (3, 0)])
def test_centred_slice_theorem_through_the_pipeline(orc, factor, interp):
    """For every rotation of the cube the taps are exact grid points, so the pipeline must give
    rfft2 of the real-space projection (sum over z) of the volume rotated about its centre."""
    D = 10
    rng = np.random.default_rng(70)
    f = ball_volume(rng, D, 3)
    mats = signed_permutations(3)
    rot = np.stack(mats)[None]
    out = orc.project_real(3, f[None], rot, factor=factor, interp=interp, cutoff=1e9)
    ky, kx = pixel_freqs(D, 0)
    q = np.stack([kx, ky, np.zeros_like(kx)], 0).astype(np.float64)
    for p, R in enumerate(mats):
        img = rotate_about_centre(f, R).sum(axis=0)
        want = np.fft.rfft2(np.fft.ifftshift(img))
        c = np.einsum("ab,b...->a...", R, q)
        inside = np.all(np.abs(c) < D // 2, axis=0)
        np.testing.assert_allclose(out[0, p][inside], want[inside], rtol=0,
                                   atol=1e-11 * np.abs(want).max())


@pytest.mark.parametrize("factor,interp", [(1, 1), (2, 0)])
def test_centred_slice_theorem_2d(orc, factor, interp):
    D = 12
    rng = np.random.default_rng(71)
    f = ball_volume(rng, D, 2)
    mats = signed_permutations(2)
    rot = np.stack(mats)[None]
    out = orc.project_real(2, f[None], rot, factor=factor, interp=interp, cutoff=1e9)
    ky, kx = pixel_freqs(D, 0)
    q = np.stack([kx, ky], 0).astype(np.float64)
    for p, R in enumerate(mats):
        want = np.fft.rfft2(np.fft.ifftshift(rotate_about_centre(f, R)))
        c = np.einsum("ab,b...->a...", R, q)
        inside = np.all(np.abs(c) < D // 2, axis=0)
        np.testing.assert_allclose(out[0, p][inside], want[inside], rtol=0,
                                   atol=1e-11 * np.abs(want).max())


@pytest.mark.parametrize("ndim,factor,interp", [(3, 1, 1), (3, 2, 1), (2, 2, 1), (3, 2, 0)])
def test_pipeline_gradients_match_differences(orc, ndim, factor, interp):
    """L = Re<G, project_real(v)>: linear in v (the difference is exact), C1 in R for cubic."""
    D, n_pose = 8, 3
    rng = np.random.default_rng(80 + ndim + factor)
    v = rng.standard_normal((1,) + (D,) * ndim)
    R = random_rotations(rng, n_pose, ndim)[None]
    s = rng.uniform(-2, 2, (1, n_pose, 2))
    G = crandn(rng, (1, n_pose, D, D // 2 + 1))
    kw = dict(factor=factor, interp=interp)

    def L(v, R, s):
        return rdot(G, orc.project_real(ndim, v, R, s, **kw))

    gv, gR, gs = orc.project_real_backward(ndim, v, R, G, s, **kw)
    assert gv.shape == v.shape
    for _ in range(2):
        E = rng.standard_normal(v.shape)
        fd = (L(v + E, R, s) - L(v - E, R, s)) / 2
        assert abs(fd - np.sum(gv * E)) <= 1e-9 * max(1.0, abs(fd))
    h = 1e-6
    for idx in np.ndindex(s.shape):
        sp, sm = s.copy(), s.copy()
        sp[idx] += h
        sm[idx] -= h
        fd = (L(v, R, sp) - L(v, R, sm)) / (2 * h)
        assert abs(fd - gs[idx]) <= 1e-6 * max(1.0, abs(fd))
    if interp == 1:
        for idx in [(0, 0, 0, 0), (0, 1, 1, 0), (0, 2, ndim - 1, 1)]:
            Rp, Rm = R.copy(), R.copy()
            Rp[idx] += h
            Rm[idx] -= h
            fd = (L(v, Rp, s) - L(v, Rm, s)) / (2 * h)
            assert abs(fd - gR[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, gR[idx])
