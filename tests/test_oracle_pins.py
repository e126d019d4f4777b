"""Pins of the fp64 oracle against facts it does not compute itself.

Each test ties the oracle to something fixed outside it: the Fourier slice theorem and
the shift theorem evaluated with numpy's FFT, exact index permutations of the real-space
volume, Keys' kernel values derived by hand (tests/golden), polynomial reproduction,
the real-linear adjoint relation, central finite differences of the oracle's own forward
map, and Friedel symmetry of real inputs.  Sources: torch-projectors paper summaries
(gist.science), Method section bullets on the RFFT format, interpolation, Friedel
symmetry, the four operations and shifts; and the Hindi page's statement of the Fourier
slice theorem.
"""
import itertools
import os

import numpy as np
import pytest

from back_projection_fourier_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers ----

def full_freqs(D):
    return np.fft.fftfreq(D, 1.0 / D).astype(np.int64)


def to_layout(spec, axes, layout):
    return np.fft.fftshift(spec, axes=axes) if layout == synth.CENTERED else spec


def pixel_freqs(Do, layout):
    """(ky, kx) integer grids of the output image in `layout`."""
    ky = full_freqs(Do)
    if layout == synth.CENTERED:
        ky = np.fft.fftshift(ky)
    kx = np.arange(Do // 2 + 1)
    return np.meshgrid(ky, kx, indexing="ij")


def signed_permutations(k):
    """All k x k signed permutation matrices with det +1 (rotations of the square/cube)."""
    mats = []
    for perm in itertools.permutations(range(k)):
        for signs in itertools.product((1, -1), repeat=k):
            M = np.zeros((k, k))
            for r, c in enumerate(perm):
                M[r, c] = signs[r]
            if round(np.linalg.det(M)) == 1:
                mats.append(M)
    return mats


def random_rotations(rng, n, k):
    return synth.rotations_3d(rng, n).astype(np.float64) if k == 3 else \
        synth.rotations_2d(rng, n).astype(np.float64)


def crandn(rng, shape):
    return rng.standard_normal(shape) + 1j * rng.standard_normal(shape)


def rdot(a, b):
    """Re <a, b> = Re sum conj(a) b."""
    return float(np.real(np.vdot(a.ravel(), b.ravel())))


# ------------------------------------------------------------- the kernel ----

def test_keys_weights_match_hand_derivation(orc):
    rows = np.loadtxt(os.path.join(GOLDEN, "keys_weights.txt"))
    for row in rows:
        t, w, dw = orc.axis_weights(row[0], orc.CUBIC)
        assert t[0] == int(row[1])
        np.testing.assert_allclose(w, row[2:6], rtol=0, atol=1e-15)
        np.testing.assert_allclose(dw, row[6:10], rtol=0, atol=1e-15)


@pytest.mark.parametrize("interp", [0, 1])
def test_kernel_partition_of_unity_and_control_points(orc, interp):
    rng = np.random.default_rng(1)
    for c in rng.uniform(-20, 20, 200):
        t, w, dw = orc.axis_weights(c, interp)
        assert abs(w.sum() - 1.0) < 1e-14
        assert abs(dw.sum()) < 1e-13
        # the weights reproduce the coordinate itself (and, for cubic, its square)
        assert abs((w * t).sum() - c) < 1e-12
        if interp == 1:
            assert abs((w * t * t).sum() - c * c) < 1e-10
    for c in range(-5, 6):
        t, w, _ = orc.axis_weights(float(c), interp)
        assert np.array_equal(w, np.eye(len(w))[0 if interp == 0 else 1])


def test_cubic_kernel_is_c1(orc):
    """Derivative returned by the oracle equals the numerical derivative of its weights,
    also across the cell boundaries (C1 continuity)."""
    rng = np.random.default_rng(2)
    h = 1e-6
    cs = list(rng.uniform(-8, 8, 100)) + [1.0 + 1e-3, 2.0 - 1e-3, -1.0 + 2e-3]
    for c in cs:
        t, w, dw = orc.axis_weights(c, 1)
        num = []
        for k, ti in enumerate(t):
            def kern(x):
                tt, ww, _ = orc.axis_weights(x, 1)
                return sum(wv for tv, wv in zip(tt, ww) if tv == ti)
            num.append((kern(c + h) - kern(c - h)) / (2 * h))
        np.testing.assert_allclose(dw, num, atol=1e-8)


# ------------------------------------------------ Fourier slice theorem ----

def _rotated_real(f, R):
    """f_R[r] = f[R r mod D] for an integer matrix R (vector order x, y[, z])."""
    D = f.shape[0]
    k = f.ndim
    idx = np.indices(f.shape)          # axis order (z, y, x) or (y, x)
    vec = idx[::-1]                    # (x, y[, z])
    src = np.einsum("ab,b...->a...", R.astype(np.int64), vec) % D
    return f[tuple(src[::-1])] if k == 3 else f[src[1], src[0]]


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("interp", [0, 1])
def test_fourier_slice_theorem_3d(orc, layout, interp):
    """Projection of rfftn(f) along rotation R equals rfft2 of the real-space projection
    (sum over z) of the rotated volume f(R r), for every rotation of the cube, at every
    pixel whose sample coordinate lies strictly inside the stored band."""
    D = 12
    rng = np.random.default_rng(3)
    f = rng.standard_normal((D, D, D))
    V = to_layout(np.fft.rfftn(f), (0, 1), layout)
    mats = signed_permutations(3)
    rot = np.stack(mats)[None]
    out = orc.project(3, V[None], rot, interp=interp, layout=layout, cutoff=1e9)
    ky, kx = pixel_freqs(D, layout)
    q = np.stack([kx, ky, np.zeros_like(kx)], 0).astype(np.float64)
    for p, R in enumerate(mats):
        fr = _rotated_real(f, R)
        want = to_layout(np.fft.rfft2(fr.sum(axis=0)), (0,), layout)
        c = np.einsum("ab,b...->a...", R, q)
        inside = np.all(np.abs(c) < D // 2, axis=0)
        assert inside.sum() > 0.5 * inside.size
        np.testing.assert_allclose(out[0, p][inside], want[inside], rtol=0,
                                   atol=1e-12 * np.abs(want).max())


@pytest.mark.parametrize("layout", [0, 1])
def test_fourier_slice_theorem_2d(orc, layout):
    """2D->2D: rotating rfft2(f) by a rotation of the square equals rfft2(f(R r))."""
    D = 10
    rng = np.random.default_rng(4)
    f = rng.standard_normal((D, D))
    V = to_layout(np.fft.rfft2(f), (0,), layout)
    mats = signed_permutations(2)
    rot = np.stack(mats)[:, None]
    out = orc.project(2, np.repeat(V[None], len(mats), 0), rot, layout=layout, cutoff=1e9)
    ky, kx = pixel_freqs(D, layout)
    q = np.stack([kx, ky], 0).astype(np.float64)
    for r, R in enumerate(mats):
        want = to_layout(np.fft.rfft2(_rotated_real(f, R)), (0,), layout)
        c = np.einsum("ab,b...->a...", R, q)
        inside = np.all(np.abs(c) < D // 2, axis=0)
        np.testing.assert_allclose(out[r, 0][inside], want[inside], rtol=0,
                                   atol=1e-12 * np.abs(want).max())


def test_identity_projection_is_central_plane_everywhere(orc):
    """R = I samples the kz = 0 plane exactly, including the Nyquist row, and the
    cutoff zeroes exactly the pixels with kx^2 + ky^2 > rc^2."""
    D = 16
    rng = np.random.default_rng(5)
    f = rng.standard_normal((D, D, D))
    V = np.fft.fftshift(np.fft.rfftn(f), axes=(0, 1))
    want = np.fft.fftshift(np.fft.rfft2(f.sum(0)), axes=(0,))
    for rc in (-1.0, 5.5, 7.0, 100.0):
        out = orc.project(3, V[None], np.eye(3)[None, None], interp=1, cutoff=rc)[0, 0]
        ky, kx = pixel_freqs(D, 1)
        r = D / 2 if rc < 0 else rc
        keep = kx * kx + ky * ky <= r * r
        np.testing.assert_allclose(out[keep], want[keep], rtol=0, atol=1e-12 * abs(want).max())
        assert np.all(out[~keep] == 0)


@pytest.mark.parametrize("ndim,Dv,Do,o", [(3, 48, 32, 1.25), (2, 48, 32, 1.25), (3, 20, 32, 0.5),
                                          (2, 24, 40, 0.5)])
def test_default_cutoff_is_the_disk_inscribed_in_the_image(orc, ndim, Dv, Do, o):
    """Without a cutoff, the sampled pixels are exactly the integer points of the disk of
    radius Do/2 in the half plane of the image box, whatever the volume's box (smaller or
    larger than the image).  The disk is enumerated by brute force: 414 points at Do = 32.
    o keeps every sample of the disk inside the stored band, so each of them is non-zero."""
    rng = np.random.default_rng(Dv * 100 + Do)
    H = Dv // 2 + 1
    V = crandn(rng, (1, Dv, Dv, H) if ndim == 3 else (1, Dv, H))
    R = random_rotations(rng, 3, ndim)[None]
    y = orc.project(ndim, V, R, None, Do=Do, interp=1, oversampling=o)
    disk = np.array([[kx * kx + ky * ky <= (Do // 2) ** 2 for kx in range(Do // 2 + 1)]
                     for ky in range(-Do // 2, Do // 2)])     # centered rows
    if Do == 32:
        assert disk.sum() == 414
    assert np.all(y[..., ~disk] == 0)
    assert np.all(y[..., disk] != 0)


# ------------------------------------------------------- shift theorem ----

@pytest.mark.parametrize("ndim", [2, 3])
def test_shift_theorem_integer_shifts(orc, ndim):
    """An integer shift s with R = I equals np.roll of the real-space image by s."""
    D = 12
    rng = np.random.default_rng(6)
    f = rng.standard_normal((D,) * ndim)
    P = f.sum(0) if ndim == 3 else f
    V = np.fft.fftshift(np.fft.rfftn(f), axes=tuple(range(ndim - 1)))
    shifts = np.array([[0, 0], [1, 0], [0, 1], [3, -2], [-5, 4]], np.float64)
    rot = np.broadcast_to(np.eye(ndim), (len(shifts), ndim, ndim))
    if ndim == 3:
        out = orc.project(3, V[None], rot[None], shifts[None], cutoff=1e9)[0]
    else:
        out = orc.project(2, np.repeat(V[None], len(shifts), 0), rot[:, None],
                          shifts[:, None], cutoff=1e9)[:, 0]
    for n, (sx, sy) in enumerate(shifts):
        want = np.fft.fftshift(np.fft.rfft2(np.roll(P, (int(sy), int(sx)), axis=(0, 1))), axes=(0,))
        np.testing.assert_allclose(out[n], want, rtol=0, atol=1e-11 * np.abs(want).max())


@pytest.mark.parametrize("ndim", [2, 3])
def test_shift_theorem_oversampled(orc, ndim):
    """A real box g of size N zero-padded into the corner of a 2N box has, at even
    frequencies 2k, exactly the spectrum of g at k.  So the o = 2 projection of the padded
    spectrum (Dv = 2N, Do = N) with integer shift s equals the rfft2 of the N-box
    projection of g rolled by s: the phase ramp is taken over the image box Do."""
    N = 8
    rng = np.random.default_rng(12)
    g = rng.standard_normal((N,) * ndim)
    f = np.zeros((2 * N,) * ndim)
    f[(slice(0, N),) * ndim] = g
    P = g.sum(0) if ndim == 3 else g
    V = np.fft.fftshift(np.fft.rfftn(f), axes=tuple(range(ndim - 1)))
    shifts = np.array([[1, 0], [0, 1], [3, -2], [-5, 4]], np.float64)
    n = len(shifts)
    rot = np.broadcast_to(np.eye(ndim), (n, ndim, ndim))
    if ndim == 3:
        out = orc.project(3, V[None], rot[None], shifts[None], Do=N, oversampling=2.0,
                          cutoff=1e9)[0]
    else:
        out = orc.project(2, np.repeat(V[None], n, 0), rot[:, None], shifts[:, None], Do=N,
                          oversampling=2.0, cutoff=1e9)[:, 0]
    for m, (sx, sy) in enumerate(shifts):
        want = np.fft.fftshift(np.fft.rfft2(np.roll(P, (int(sy), int(sx)), axis=(0, 1))), axes=(0,))
        np.testing.assert_allclose(out[m], want, rtol=0, atol=1e-11 * np.abs(want).max())


# --------------------------------------------- polynomial reproduction ----

@pytest.mark.parametrize("ndim", [2, 3])
@pytest.mark.parametrize("interp", [0, 1])
@pytest.mark.parametrize("o", [1.0, 1.5])
def test_polynomial_reproduction(orc, ndim, interp, o):
    """Spectra that are polynomials of the frequency vector are sampled exactly where
    every tap lies in the stored half (t_x >= 0) and inside the band: linear polynomials
    by both kernels, quadratics by the cubic one.  Pins c = o R q and the tap weights."""
    D, Do = 24, 12
    rng = np.random.default_rng(7 + ndim + 10 * interp)
    H = D // 2 + 1
    fz = np.fft.fftshift(full_freqs(D))
    if ndim == 3:
        Z, Y, X = np.meshgrid(fz, fz, np.arange(H), indexing="ij")
        coords = [X, Y, Z]
    else:
        Y, X = np.meshgrid(fz, np.arange(H), indexing="ij")
        coords = [X, Y]
    a = crandn(rng, ndim)
    b = crandn(rng, (ndim, ndim)) if interp == 1 else np.zeros((ndim, ndim))
    beta = crandn(rng, ())
    V = beta + sum(a[i] * coords[i] for i in range(ndim))
    V = V + sum(b[i, j] * coords[i] * coords[j] for i in range(ndim) for j in range(ndim))
    R = random_rotations(rng, 6, ndim)
    out = orc.project(ndim, V[None], R[None], Do=Do, interp=interp, oversampling=o, cutoff=1e9)[0]
    ky, kx = pixel_freqs(Do, 1)
    q = np.stack([kx, ky] + ([np.zeros_like(kx)] if ndim == 3 else []), 0).astype(np.float64)
    checked = 0
    for p in range(6):
        c = o * np.einsum("ab,b...->a...", R[p], q)
        lo = np.floor(c) - (1 if interp == 1 else 0)
        hi = np.floor(c) + (2 if interp == 1 else 1)
        ok = (lo[0] >= 0) & (hi[0] <= D // 2)
        for i in range(1, ndim):
            ok &= (lo[i] >= -D // 2) & (hi[i] <= D // 2 - 1)
        want = beta + sum(a[i] * c[i] for i in range(ndim))
        want = want + sum(b[i, j] * c[i] * c[j] for i in range(ndim) for j in range(ndim))
        np.testing.assert_allclose(out[p][ok], want[ok], rtol=1e-12, atol=1e-10)
        checked += ok.sum()
    assert checked > 50


# --------------------------------------------------------- Friedel ----

@pytest.mark.parametrize("interp", [0, 1])
def test_friedel_hermitian_kx0_column(orc, interp):
    """For the rfft of a real volume, the kx = 0 column of every projection is Hermitian:
    y(0, -ky) = conj y(0, ky), wherever all taps avoid the Nyquist planes."""
    D = 16
    rng = np.random.default_rng(8)
    V = np.fft.fftshift(np.fft.rfftn(rng.standard_normal((D, D, D))), axes=(0, 1))
    R = random_rotations(rng, 5, 3)
    s = rng.uniform(-3, 3, (1, 5, 2))
    out = orc.project(3, V[None], R[None], s, interp=interp, cutoff=1e9)[0]
    for ky in range(1, D // 2 - 3):
        a = out[:, D // 2 + ky, 0]
        b = out[:, D // 2 - ky, 0]
        np.testing.assert_allclose(a, np.conj(b), rtol=0, atol=1e-12 * np.abs(out).max())


def test_layouts_agree_after_permutation(orc):
    rng = np.random.default_rng(9)
    D = 10
    Vc = crandn(rng, (2, D, D, D // 2 + 1))
    Vf = np.fft.ifftshift(Vc, axes=(1, 2))
    R = random_rotations(rng, 4, 3)
    s = rng.uniform(-2, 2, (1, 4, 2))
    yc = orc.project(3, Vc, R[None], s, layout=1)
    yf = orc.project(3, Vf, R[None], s, layout=0)
    np.testing.assert_allclose(np.fft.ifftshift(yc, axes=(2,)), yf, rtol=0, atol=1e-13)


# ---------------------------------------------------------- adjointness ----

CASES = [
    # ndim, interp, layout, o, Dv, Do, cutoff, shifted, n_rec, n_rot
    (3, 1, 1, 1.0, 10, 10, -1.0, True, 1, 1),
    (3, 0, 1, 1.0, 10, 10, 4.5, True, 1, 1),
    (3, 1, 0, 1.5, 12, 8, -1.0, True, 2, 2),
    (3, 0, 0, 1.0, 8, 8, 100.0, False, 2, 1),
    (2, 1, 1, 1.0, 12, 12, -1.0, True, 3, 3),
    (2, 0, 0, 1.5, 12, 8, 3.5, True, 2, 1),
    # image boxes larger than the volume: samples beyond the stored range read zero
    (3, 1, 1, 1.0, 8, 14, -1.0, True, 1, 1),
    (2, 0, 0, 1.0, 8, 16, -1.0, True, 2, 2),
]


@pytest.mark.parametrize("case", CASES)
def test_adjointness(orc, case):
    """Re <P V, Y> = Re <V, P^T Y> for non-Hermitian V and Y: the back-projection and the
    volume gradient are the exact real-linear transpose of the projection."""
    ndim, interp, layout, o, Dv, Do, rc, shifted, n_rec, n_rot = case
    rng = np.random.default_rng(hash(case) % 2**32)
    n_pose = 5
    H = Dv // 2 + 1
    shape = (n_rec, Dv, Dv, H) if ndim == 3 else (n_rec, Dv, H)
    V = crandn(rng, shape)
    R = random_rotations(rng, n_rot * n_pose, ndim).reshape(n_rot, n_pose, ndim, ndim)
    s = rng.uniform(-4, 4, (n_rot, n_pose, 2)) if shifted else None
    Y = crandn(rng, (n_rec, n_pose, Do, Do // 2 + 1))
    kw = dict(interp=interp, layout=layout, oversampling=o, cutoff=rc)
    PV = orc.project(ndim, V, R, s, Do=Do, **kw)
    PtY, _ = orc.backproject(ndim, Y, R, shift=s, Dv=Dv, **kw)
    g_rec, _, _ = orc.project_backward(ndim, V, R, Y, s, **kw, want_rot=False, want_shift=False)
    lhs, rhs = rdot(PV, Y), rdot(V, PtY)
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), np.abs(PV).sum())
    np.testing.assert_allclose(g_rec, PtY, rtol=0, atol=1e-13 * np.abs(PtY).max())


def test_adjoint_matrix_brute_force(orc):
    """Tiny case: the full real matrices of the projection and of the back-projection,
    probed column by column, are exact transposes of each other."""
    rng = np.random.default_rng(10)
    ndim, Dv, Do = 3, 4, 4
    H = Dv // 2 + 1
    R = random_rotations(rng, 2, 3)[None]
    s = rng.uniform(-2, 2, (1, 2, 2))
    nin = Dv * Dv * H
    nout = 2 * Do * (Do // 2 + 1)
    kw = dict(interp=1, layout=1, cutoff=-1.0, nthreads=1)
    A = np.zeros((2 * nout, 2 * nin))
    for e in range(2 * nin):
        V = np.zeros(nin, complex)
        V[e // 2] = 1.0 if e % 2 == 0 else 1j
        y = orc.project(3, V.reshape(1, Dv, Dv, H), R, s, **kw).ravel()
        A[0::2, e], A[1::2, e] = y.real, y.imag
    B = np.zeros((2 * nin, 2 * nout))
    for e in range(2 * nout):
        Y = np.zeros(nout, complex)
        Y[e // 2] = 1.0 if e % 2 == 0 else 1j
        v, _ = orc.backproject(3, Y.reshape(1, 2, Do, Do // 2 + 1), R, shift=s, Dv=Dv, **kw)
        v = v.ravel()
        B[0::2, e], B[1::2, e] = v.real, v.imag
    assert np.abs(A).max() > 0.1
    np.testing.assert_allclose(B, A.T, rtol=0, atol=1e-14)


@pytest.mark.parametrize("ndim", [2, 3])
def test_weight_volume_equals_insertion_of_real_weights(orc, ndim):
    """With no shift, inserting the real weight map as data gives a real volume equal to
    the weight volume: the weights use the same interpolation weights, with no phase
    and no conjugation on the mirrored taps."""
    rng = np.random.default_rng(11)
    D = 10
    n_pose = 4
    R = random_rotations(rng, n_pose, ndim)[None]
    wt = rng.uniform(0.2, 2.0, (1, n_pose, D, D // 2 + 1))
    vol, wvol = orc.backproject(ndim, wt.astype(complex), R, weights=wt, Dv=D, interp=1)
    np.testing.assert_allclose(vol.imag, 0, atol=1e-13)
    np.testing.assert_allclose(vol.real, wvol, rtol=0, atol=1e-13)
    _, w1 = orc.backproject(ndim, wt.astype(complex), R, weights=None, Dv=D, interp=1)
    vol1, _ = orc.backproject(ndim, np.ones_like(wt, complex), R, Dv=D, interp=1)
    np.testing.assert_allclose(vol1.real, w1, rtol=0, atol=1e-13)


# ---------------------------------------------------- finite differences ----

def _loss(orc, ndim, V, R, s, G, kw):
    return rdot(orc.project(ndim, V, R, s, **kw), G)


def _coords_clear_of_integers(R, Do, o, margin=1e-4):
    ky, kx = pixel_freqs(Do, 1)
    ndim = R.shape[-1]
    q = np.stack([kx, ky] + ([np.zeros_like(kx)] if ndim == 3 else []), 0).astype(np.float64)
    for Rm in R.reshape(-1, ndim, ndim):
        c = o * np.einsum("ab,b...->a...", Rm, q)
        fr = np.abs(c - np.round(c))
        keep = kx * kx + ky * ky <= (Do / 2) ** 2
        if (fr[:, keep] < margin).any():
            # the only integer coordinates allowed are the exact zeros at q = 0
            bad = (fr < margin) & keep[None] & (np.abs(c) > 1e-9)
            if bad.any():
                return False
    return True


@pytest.mark.parametrize("ndim,interp,n_rec,n_rot,o", [(3, 1, 1, 1, 1.0), (3, 0, 1, 1, 1.0),
                                                       (3, 1, 2, 1, 1.0), (2, 1, 2, 2, 1.0),
                                                       (2, 0, 1, 1, 1.0), (3, 1, 1, 1, 1.5),
                                                       (2, 0, 2, 1, 0.75)])
def test_rotation_and_shift_gradients_match_central_differences(orc, ndim, interp, n_rec, n_rot, o):
    D, n_pose = 10, 3
    H = D // 2 + 1
    seed = 20
    while True:
        rng = np.random.default_rng(seed)
        R = random_rotations(rng, n_rot * n_pose, ndim).reshape(n_rot, n_pose, ndim, ndim)
        if interp == 1 or _coords_clear_of_integers(R, D, o):
            break
        seed += 1
    shape = (n_rec, D, D, H) if ndim == 3 else (n_rec, D, H)
    V = crandn(rng, shape)
    s = rng.uniform(-3, 3, (n_rot, n_pose, 2))
    G = crandn(rng, (n_rec, n_pose, D, H))
    kw = dict(interp=interp, layout=1, oversampling=o, cutoff=-1.0)
    _, gR, gs = orc.project_backward(ndim, V, R, G, s, **kw)
    h = 1e-6
    for idx in np.ndindex(R.shape):
        if ndim == 3 and idx[-1] == 2:
            continue
        Rp, Rm = R.copy(), R.copy()
        Rp[idx] += h
        Rm[idx] -= h
        fd = (_loss(orc, ndim, V, Rp, s, G, kw) - _loss(orc, ndim, V, Rm, s, G, kw)) / (2 * h)
        assert abs(fd - gR[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, gR[idx])
    # the z column multiplies q_z = 0: its gradient is exactly zero
    if ndim == 3:
        assert np.all(gR[..., 2] == 0)
    for idx in np.ndindex(s.shape):
        sp, sm = s.copy(), s.copy()
        sp[idx] += h
        sm[idx] -= h
        fd = (_loss(orc, ndim, V, R, sp, G, kw) - _loss(orc, ndim, V, R, sm, G, kw)) / (2 * h)
        assert abs(fd - gs[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, gs[idx])


def test_gradient_of_volume_matches_directional_difference(orc):
    """dL/dV in PyTorch's complex convention: L(V + h E) - L(V - h E) = 2 h Re<grad, E>."""
    rng = np.random.default_rng(30)
    D = 8
    V = crandn(rng, (1, D, D, D // 2 + 1))
    R = random_rotations(rng, 3, 3)[None]
    s = rng.uniform(-2, 2, (1, 3, 2))
    G = crandn(rng, (1, 3, D, D // 2 + 1))
    kw = dict(interp=1, layout=1, cutoff=-1.0)
    gV, _, _ = orc.project_backward(3, V, R, G, s, **kw)
    for _ in range(3):
        E = crandn(rng, V.shape)
        h = 1e-3   # L is linear in V: the difference is exact up to rounding
        fd = (_loss(orc, 3, V + h * E, R, s, G, kw) - _loss(orc, 3, V - h * E, R, s, G, kw)) / (2 * h)
        assert abs(fd - rdot(gV, E)) <= 1e-9 * abs(fd)


@pytest.mark.parametrize("ndim,interp,layout,o,Dv,shifted,weighted,n_rec,n_rot",
                         [(3, 1, 1, 1.0, 10, True, True, 1, 1), (3, 0, 0, 1.0, 10, True, True, 1, 1),
                          (3, 1, 1, 1.0, 10, False, False, 2, 2),
                          (2, 1, 1, 1.5, 14, True, True, 2, 1), (2, 0, 1, 1.0, 10, True, False, 2, 2)])
def test_backproject_gradients_match_central_differences(orc, ndim, interp, layout, o, Dv, shifted,
                                                         weighted, n_rec, n_rot):
    """The insertion's backward (a composition of projections) against central differences
    of the insertion itself: L = Re<Gv, vol> + <GW, wvol>, with (vol, wvol) from backproject()."""
    Do, n_pose = 10, 3
    Ho = Do // 2 + 1
    seed = 40
    while True:
        rng = np.random.default_rng(seed)
        R = random_rotations(rng, n_rot * n_pose, ndim).reshape(n_rot, n_pose, ndim, ndim)
        if interp == 1 or _coords_clear_of_integers(R, Do, o):
            break
        seed += 1
    Hv = Dv // 2 + 1
    vshape = (n_rec, Dv, Dv, Hv) if ndim == 3 else (n_rec, Dv, Hv)
    P = crandn(rng, (n_rec, n_pose, Do, Ho))
    W = rng.uniform(0.2, 2.0, P.shape) if weighted else None
    s = rng.uniform(-3, 3, (n_rot, n_pose, 2)) if shifted else None
    Gv = crandn(rng, vshape)
    GW = rng.standard_normal(vshape)
    kw = dict(interp=interp, layout=layout, oversampling=o, cutoff=-1.0)

    def L(P, W, R, s):
        vol, wvol = orc.backproject(ndim, P, R, weights=W, shift=s, Dv=Dv, **kw)
        return rdot(Gv, vol) + float(np.sum(GW * wvol))

    gP, gW, gR, gs = orc.backproject_backward(ndim, P, R, Gv, GW, W, s, **kw)
    h = 1e-6
    for idx in np.ndindex(R.shape):
        if ndim == 3 and idx[-1] == 2:
            continue
        Rp, Rm = R.copy(), R.copy()
        Rp[idx] += h
        Rm[idx] -= h
        fd = (L(P, W, Rp, s) - L(P, W, Rm, s)) / (2 * h)
        assert abs(fd - gR[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, gR[idx])
    if ndim == 3:
        assert np.all(gR[..., 2] == 0)
    if shifted:
        for idx in np.ndindex(s.shape):
            sp, sm = s.copy(), s.copy()
            sp[idx] += h
            sm[idx] -= h
            fd = (L(P, W, R, sp) - L(P, W, R, sm)) / (2 * h)
            assert abs(fd - gs[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, gs[idx])
    else:
        assert np.all(gs == 0)
    # L is linear in P and in W: the differences are exact up to rounding
    Wb = W if weighted else np.ones(P.shape)
    for _ in range(2):
        E = crandn(rng, P.shape)
        fd = (L(P + E, W, R, s) - L(P - E, W, R, s)) / 2
        assert abs(fd - rdot(gP, E)) <= 1e-9 * max(1.0, abs(fd))
        F = rng.standard_normal(P.shape)
        fd = (L(P, Wb + F, R, s) - L(P, Wb - F, R, s)) / 2
        assert abs(fd - float(np.sum(gW * F))) <= 1e-9 * max(1.0, abs(fd))


def test_samples_match_full_projection(orc):
    rng = np.random.default_rng(31)
    D = 12
    V = crandn(rng, (2, D, D // 2 + 1))
    R = random_rotations(rng, 6, 2).reshape(2, 3, 2, 2)
    s = rng.uniform(-3, 3, (2, 3, 2))
    full = orc.project(2, V, R, s)
    items = rng.integers(0, 6, 50)
    pix = rng.integers(0, D * (D // 2 + 1), 50)
    vals = orc.project_samples(2, V, R, items, pix, s)
    np.testing.assert_array_equal(vals, full.reshape(6, -1)[items, pix])
