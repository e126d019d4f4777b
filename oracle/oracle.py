"""ctypes wrapper around oracle.c (plain fp64 C, OpenMP over items).

TEST INFRASTRUCTURE ONLY.  The oracle restates, from the torch-projectors paper
summaries (gist.science: Method section bullets on the RFFT half-spectrum format,
linear / Catmull-Rom interpolation, Friedel symmetry, the four projection operations,
shifts by phase modulation and gradients for inputs, rotations and shifts), what the
projection computes, one pixel and one tap at a time.  It shares no code with the CUDA
library and is never called by it.

Every wrapper takes numpy arrays (any float dtype; they are widened to fp64 /
complex128) and returns fresh numpy arrays.  ``nthreads`` defaults to every core this
process may run on.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

LINEAR, CUBIC = 0, 1
FFTW, CENTERED = 0, 1

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "liboracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so (gcc, -O2, no fast-math, no FMA contraction)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.{os.getpid()}")
        subprocess.run(
            ["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
             "-o", str(tmp), str(_SRC), "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # TP_ORACLE_LIB points the wrapper at another build of oracle.c; the mutation
        # tests use it to check that the pins reject deliberately broken oracles.
        alt = os.environ.get("TP_ORACLE_LIB")
        if not alt:
            build()
        lib = ctypes.CDLL(alt or str(_LIB))
        P, I, D, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_long
        lib.orc_project.argtypes = [I, P, I, I, P, I, I, P, I, P, I, I, I, D, D, I]
        lib.orc_project_samples.argtypes = [I, P, I, I, P, I, I, P, I, I, I, I, D, D, L, P, P, P, I]
        lib.orc_backproject.argtypes = [I, P, P, I, I, P, I, I, P, I, P, P, I, I, I, D, D, I]
        lib.orc_project_backward.argtypes = [I, P, I, I, P, I, I, P, I, P, I, P, P, P, I, I, D, D, I]
        lib.orc_axis_weights.argtypes = [D, I, P, P, P]
        for f in (lib.orc_project, lib.orc_project_samples, lib.orc_backproject,
                  lib.orc_project_backward, lib.orc_axis_weights):
            f.restype = I
        _lib = lib
    return _lib


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _c128(a):
    return np.ascontiguousarray(a, dtype=np.complex128)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def _dims(ndim, rec_shape, rot, shift):
    n_rec = rec_shape[0]
    Dv = rec_shape[1]
    k = ndim
    rot = _f64(rot)
    if rot.ndim != 4 or rot.shape[2:] != (k, k):
        raise ValueError("rot must be [n_rot][n_pose][k][k]")
    n_rot, n_pose = rot.shape[:2]
    n_sh = 1
    if shift is not None:
        shift = _f64(shift)
        if shift.ndim != 3 or shift.shape[1:] != (n_pose, 2):
            raise ValueError("shift must be [n_sh][n_pose][2]")
        n_sh = shift.shape[0]
    return n_rec, Dv, rot, n_rot, n_pose, shift, n_sh


def project(ndim, rec, rot, shift=None, Do=None, interp=CUBIC, layout=CENTERED,
            oversampling=1.0, cutoff=-1.0, nthreads=None):
    """Forward projection: [n_rec][n_pose][Do][Do/2+1] complex128."""
    rec = _c128(rec)
    n_rec, Dv, rot, n_rot, n_pose, shift, n_sh = _dims(ndim, rec.shape, rot, shift)
    Do = Dv if Do is None else Do
    out = np.zeros((n_rec, n_pose, Do, Do // 2 + 1), np.complex128)
    rc = _load().orc_project(ndim, _ptr(rec), n_rec, Dv, _ptr(rot), n_rot, n_pose, _ptr(shift),
                             n_sh, _ptr(out), Do, interp, layout, oversampling, cutoff,
                             nthreads or _cores())
    _check(rc, "project")
    return out


def project_samples(ndim, rec, rot, items, pix, shift=None, Do=None, interp=CUBIC,
                    layout=CENTERED, oversampling=1.0, cutoff=-1.0, nthreads=None):
    """Forward projection at (item, pixel) pairs only; item = r*n_pose + p, pix = i*H + j."""
    rec = _c128(rec)
    n_rec, Dv, rot, n_rot, n_pose, shift, n_sh = _dims(ndim, rec.shape, rot, shift)
    Do = Dv if Do is None else Do
    items = np.ascontiguousarray(items, dtype=np.int64)
    pix = np.ascontiguousarray(pix, dtype=np.int64)
    vals = np.zeros(items.shape[0], np.complex128)
    rc = _load().orc_project_samples(ndim, _ptr(rec), n_rec, Dv, _ptr(rot), n_rot, n_pose,
                                     _ptr(shift), n_sh, Do, interp, layout, oversampling, cutoff,
                                     items.shape[0], _ptr(items), _ptr(pix), _ptr(vals),
                                     nthreads or _cores())
    _check(rc, "project_samples")
    return vals


def backproject(ndim, proj, rot, weights=None, shift=None, Dv=None, interp=CUBIC,
                layout=CENTERED, oversampling=1.0, cutoff=-1.0, nthreads=None,
                want_weights=True):
    """Back-projection (insertion): returns (rec [n_rec][...] complex128, wrec float64 or None)."""
    proj = _c128(proj)
    n_rec, n_pose_p, Do = proj.shape[0], proj.shape[1], proj.shape[2]
    rot = _f64(rot)
    k = ndim
    n_rot, n_pose = rot.shape[:2]
    if n_pose != n_pose_p:
        raise ValueError("rot and proj disagree on n_pose")
    n_sh = 1
    if shift is not None:
        shift = _f64(shift)
        n_sh = shift.shape[0]
    if weights is not None:
        weights = _f64(weights)
        if weights.shape != proj.shape:
            raise ValueError("weights must have the projection shape")
    Dv = Do if Dv is None else Dv
    H = Dv // 2 + 1
    shape = (n_rec, Dv, Dv, H) if ndim == 3 else (n_rec, Dv, H)
    rec = np.zeros(shape, np.complex128)
    wrec = np.zeros(shape, np.float64) if want_weights else None
    rc = _load().orc_backproject(ndim, _ptr(proj), _ptr(weights), n_rec, Do, _ptr(rot), n_rot,
                                 n_pose, _ptr(shift), n_sh, _ptr(rec), _ptr(wrec), Dv, interp,
                                 layout, oversampling, cutoff, nthreads or _cores())
    _check(rc, "backproject")
    assert rot.shape[2:] == (k, k)
    return rec, wrec


def project_backward(ndim, rec, rot, grad_out, shift=None, interp=CUBIC, layout=CENTERED,
                     oversampling=1.0, cutoff=-1.0, nthreads=None, want_rec=True,
                     want_rot=True, want_shift=True):
    """Backward of project(): (grad_rec, grad_rot, grad_shift); unwanted ones are None."""
    rec = _c128(rec)
    n_rec, Dv, rot, n_rot, n_pose, shift, n_sh = _dims(ndim, rec.shape, rot, shift)
    grad_out = _c128(grad_out)
    Do = grad_out.shape[2]
    if grad_out.shape != (n_rec, n_pose, Do, Do // 2 + 1):
        raise ValueError("grad_out must be [n_rec][n_pose][Do][Do/2+1]")
    g_rec = np.zeros(rec.shape, np.complex128) if want_rec else None
    g_rot = np.zeros(rot.shape, np.float64) if want_rot else None
    g_sh = np.zeros((n_sh, n_pose, 2), np.float64) if want_shift else None
    rc = _load().orc_project_backward(ndim, _ptr(rec), n_rec, Dv, _ptr(rot), n_rot, n_pose,
                                      _ptr(shift), n_sh, _ptr(grad_out), Do, _ptr(g_rec),
                                      _ptr(g_rot), _ptr(g_sh), interp, layout, oversampling,
                                      cutoff, nthreads or _cores())
    _check(rc, "project_backward")
    return g_rec, g_rot, g_sh


def backproject_backward(ndim, proj, rot, grad_vol=None, grad_wvol=None, weights=None,
                         shift=None, interp=CUBIC, layout=CENTERED, oversampling=1.0,
                         cutoff=-1.0, nthreads=None):
    """Gradients of the insertion (vol, wvol) = backproject(proj, weights, rot, shift) for the
    upstream gradients grad_vol (complex) and grad_wvol (real); returns (grad_proj,
    grad_weights, grad_rot, grad_shift).  torch-projectors summaries, Method section,
    differentiation bullet: every operation is differentiable in its inputs, rotations and
    shifts.

    vol is real-linear in proj with the projection as its adjoint, so with
    L = Re<grad_vol, vol> + <grad_wvol, wvol>:
      grad_proj = P(grad_vol), and the data part's pose gradients are those of
      Re<P(grad_vol), proj>, i.e. project_backward with rec = grad_vol, grad_out = proj;
      wvol is linear in the weights with the same taps and no phase or conjugation, so
      grad_weights = the projection of grad_wvol without shift (real), and the weight
      part's rotation gradient is that of sum weights * P0(grad_wvol).
    The composition is pinned against central differences of backproject() itself."""
    proj = _c128(proj)
    Do = proj.shape[2]
    rot = _f64(rot)
    kw = dict(interp=interp, layout=layout, oversampling=oversampling, cutoff=cutoff,
              nthreads=nthreads)
    n_sh = 1 if shift is None else np.asarray(shift).shape[0]
    g_proj = np.zeros(proj.shape, np.complex128)
    g_rot = np.zeros(rot.shape, np.float64)
    g_sh = np.zeros((n_sh, rot.shape[1], 2), np.float64)
    g_w = np.zeros(proj.shape, np.float64)
    if grad_vol is not None:
        g_proj = project(ndim, grad_vol, rot, shift, Do=Do, **kw)
        _, gr, gs = project_backward(ndim, grad_vol, rot, proj, shift, want_rec=False, **kw)
        g_rot += gr
        if shift is not None:
            g_sh += gs
    if grad_wvol is not None:
        gw = _c128(np.asarray(grad_wvol, np.float64))
        g_w = project(ndim, gw, rot, None, Do=Do, **kw).real
        w = np.ones(proj.shape) if weights is None else _f64(weights)
        _, gr, _ = project_backward(ndim, gw, rot, w.astype(np.complex128), None, want_rec=False,
                                    want_shift=False, **kw)
        g_rot += gr
    return g_proj, g_w, g_rot, g_sh


def pad_volume(vol, factor: int):
    """Real-space zero padding for on-the-fly oversampling (Dutch page, problem statement:
    oversampling is zero-filling in the spatial domain; French page, interpolation
    comparison).  vol is [n][D]^k real with its centre at index D/2; the result is the
    [n][factor*D]^k box holding vol centred, zeros elsewhere, ifftshifted so that the centre
    sits at index 0 (np.pad, then np.fft.ifftshift over the spatial axes)."""
    vol = np.asarray(vol, np.float64)
    D = vol.shape[-1]
    k = vol.ndim - 1
    m = (factor - 1) * D // 2
    padded = np.pad(vol, [(0, 0)] + [(m, m)] * k)
    return np.fft.ifftshift(padded, axes=tuple(range(1, k + 1)))


def crop_volume(padded, D: int):
    """Adjoint and left inverse of pad_volume: undo the shift, cut the centred D box out."""
    padded = np.asarray(padded, np.float64)
    k = padded.ndim - 1
    P = padded.shape[-1]
    m = (P - D) // 2
    c = np.fft.fftshift(padded, axes=tuple(range(1, k + 1)))
    return c[(slice(None),) + (slice(m, m + D),) * k]


def oversampled_spectrum(vol, factor: int):
    """Half spectrum (FFTW order) of the padded volume: numpy's rfftn of pad_volume."""
    k = np.asarray(vol).ndim - 1
    return np.fft.rfftn(pad_volume(vol, factor), axes=tuple(range(1, k + 1)))


def project_real(ndim, vol, rot, shift=None, factor=1, interp=CUBIC, cutoff=-1.0, nthreads=None):
    """On-the-fly pipeline from a real-space volume of box D to its projections at box D:
    pad by `factor`, FFT, then sample the oversampled spectrum at c = factor * R q (FFTW
    layout).  factor = 1 with cubic weights and factor = 2 with linear weights are the two
    alternatives the pages compare."""
    D = np.asarray(vol).shape[-1]
    spec = oversampled_spectrum(vol, factor)
    return project(ndim, spec, rot, shift, Do=D, interp=interp, layout=FFTW,
                   oversampling=float(factor), cutoff=cutoff, nthreads=nthreads)


def project_real_backward(ndim, vol, rot, grad_out, shift=None, factor=1, interp=CUBIC,
                          cutoff=-1.0, nthreads=None):
    """Gradients of project_real for the upstream grad_out (PyTorch's complex convention):
    (grad_vol real, grad_rot, grad_shift).  With g the gradient of the half spectrum
    X_k = sum_n x_n exp(-2 pi i k.n / P), dL/dx_n = Re sum_k conj(g_k) exp(-2 pi i k.n / P)
    = Re(P^k * ifftn(g placed in the full spectrum, zeros in the other half))_n; the
    volume's gradient is then the adjoint of the padding (crop_volume)."""
    vol = np.asarray(vol, np.float64)
    D = vol.shape[-1]
    spec = oversampled_spectrum(vol, factor)
    g_spec, g_rot, g_sh = project_backward(ndim, spec, rot, grad_out, shift, interp=interp,
                                           layout=FFTW, oversampling=float(factor),
                                           cutoff=cutoff, nthreads=nthreads)
    P = factor * D
    axes = tuple(range(1, ndim + 1))
    full = np.zeros(vol.shape[:1] + (P,) * ndim, np.complex128)
    full[..., : P // 2 + 1] = g_spec
    g_x = np.real(np.fft.ifftn(full, axes=axes)) * float(P) ** ndim
    return crop_volume(g_x, D), g_rot, g_sh


def exact_projection(ndim, vol, rot, shift=None, Do=None, cutoff=-1.0):
    """Ground truth of the projection of a real-space volume: its Fourier transform evaluated
    exactly (no interpolation) at c = R q for every kept pixel,
        F(c) = sum_n v[n] exp(-2 pi i c . (n - D/2) / D),
    times the shift phase exp(-2 pi i (kx sx + ky sy) / Do), in FFTW layout.  This is the
    reference of the accuracy comparison (Spanish page, results, precision bullet: Fourier
    ring correlation and real-space intensity attenuation of cubic without oversampling
    against linear with 2x oversampling).  vol: [n][D]^ndim real, centre at index D/2; rot:
    [n_rot][n_pose][k][k]; shift as in project().  Cost D^ndim per pixel (matrix products
    over one axis at a time)."""
    vol = np.asarray(vol, np.float64)
    rot = np.asarray(rot, np.float64)
    n, D = vol.shape[0], vol.shape[-1]
    Do = D if Do is None else Do
    Ho = Do // 2 + 1
    n_rot, n_pose = rot.shape[:2]
    rc = Do / 2 if cutoff < 0 else cutoff
    ky = np.fft.fftfreq(Do, 1.0 / Do)
    KY, KX = np.meshgrid(ky, np.arange(Ho), indexing="ij")
    keep = KX * KX + KY * KY <= np.floor(rc * rc)
    q = np.stack([KX[keep], KY[keep]], 0)
    m = np.arange(D) - D // 2
    out = np.zeros((n, n_pose, Do, Ho), np.complex128)
    for r in range(n):
        for p in range(n_pose):
            R = rot[0 if n_rot == 1 else r, p]
            c = R[:, :2] @ q                      # (k, P): vector order x, y[, z]
            E = [np.exp(-2j * np.pi * np.outer(c[a], m) / D) for a in range(ndim)]
            if ndim == 3:
                t = vol[r].reshape(D * D, D) @ E[0].T            # (z*y, P)
                t = np.einsum("zyp,py->zp", t.reshape(D, D, -1), E[1])
                val = np.einsum("zp,pz->p", t, E[2])
            else:
                t = vol[r] @ E[0].T                               # (y, P)
                val = np.einsum("yp,py->p", t, E[1])
            if shift is not None:
                sh = np.asarray(shift, np.float64)
                s = sh[0 if sh.shape[0] == 1 else r, p]
                val = val * np.exp(-2j * np.pi * (q[0] * s[0] + q[1] * s[1]) / Do)
            img = np.zeros((Do, Ho), np.complex128)
            img[keep] = val
            out[r, p] = img
    return out


def axis_weights(c: float, interp=CUBIC):
    """Taps, kernel weights and kernel derivatives of one axis at coordinate c."""
    t = np.zeros(4, np.int64)
    w = np.zeros(4, np.float64)
    dw = np.zeros(4, np.float64)
    n = _load().orc_axis_weights(float(c), interp, _ptr(t), _ptr(w), _ptr(dw))
    return t[:n], w[:n], dw[:n]
