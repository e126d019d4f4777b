"""Differentiable PyTorch operators over libtp.so.

Every operation of the library is differentiable in its inputs, its rotation matrices and
its shifts, with the backward computed by the library's own kernels and nothing stored
but the forward's inputs (torch-projectors summaries, Method section, differentiation
bullet).  Each ``torch.autograd.Function`` here calls the ``tp_*`` entry points only:

  project(rec, rot, shift, Do, ...)           forward projection, 3D->2D or 2D->2D;
                                              backward = tp_project_backward
  backproject(proj, rot, shift, weights, ...) insertion (data, weight volume);
                                              backward = tp_backproject_backward
  pad_volume(vol, factor)                     real-space zero padding; backward = crop
  project_real(vol, rot, shift, factor, ...)  on-the-fly oversampling pipeline from a
                                              real-space volume: pad, FFT, project at
                                              c = factor * R q (Dutch page, problem
                                              statement; French page, interpolation
                                              comparison)

Complex tensors follow PyTorch's convention: the gradient of a real loss L with respect
to z is dL/dRe(z) + i dL/dIm(z), which is also the library's.  The FFT of the pipeline is
torch.fft (cuFFT), a library transform; every other step is a libtp.so kernel.
"""
from __future__ import annotations

import torch

from . import tp


def _opts(interp, layout, oversampling, cutoff):
    return tp.make_opts(interp, layout, oversampling, cutoff)


class _Project(torch.autograd.Function):
    @staticmethod
    def forward(ctx, rec, rot, shift, Do, opts):
        out = tp.project(rec, rot, shift, Do=Do, opts=opts)
        ctx.save_for_backward(rec, rot, shift)
        ctx.opts = opts
        return out

    @staticmethod
    def backward(ctx, grad):
        rec, rot, shift = ctx.saved_tensors
        want_rec, want_rot, want_shift = ctx.needs_input_grad[:3]
        want_shift = want_shift and shift is not None
        if not (want_rec or want_rot or want_shift):
            return None, None, None, None, None
        g_rec, g_rot, g_sh = tp.project_backward(rec, rot, grad.contiguous(), shift,
                                                 want_rec=want_rec, want_rot=want_rot,
                                                 want_shift=want_shift, opts=ctx.opts)
        return g_rec, g_rot, g_sh, None, None


class _Backproject(torch.autograd.Function):
    @staticmethod
    def forward(ctx, proj, weights, rot, shift, Dv, ndim, opts):
        vol, wvol = tp.backproject(proj, rot, shift, weights, Dv=Dv,
                                   want_weights=weights is not None, opts=opts, ndim=ndim)
        ctx.save_for_backward(proj, weights, rot, shift)
        ctx.opts, ctx.ndim = opts, ndim
        if wvol is None:
            return vol
        return vol, wvol

    @staticmethod
    def backward(ctx, g_vol, g_wvol=None):
        proj, weights, rot, shift = ctx.saved_tensors
        want_proj, want_w, want_rot, want_shift = ctx.needs_input_grad[:4]
        want_w = want_w and weights is not None
        want_shift = want_shift and shift is not None
        if not (want_proj or want_w or want_rot or want_shift):
            return (None,) * 7
        g_vol = None if g_vol is None else g_vol.contiguous()
        g_wvol = None if g_wvol is None else g_wvol.contiguous()
        if g_vol is None and g_wvol is None:
            return (None,) * 7
        g_proj, g_w, g_rot, g_sh = tp.backproject_backward(
            proj, rot, g_vol, g_wvol, shift, weights, want_proj=want_proj, want_weights=want_w,
            want_rot=want_rot, want_shift=want_shift, opts=ctx.opts, ndim=ctx.ndim)
        return g_proj, g_w, g_rot, g_sh, None, None, None


class _Pad(torch.autograd.Function):
    @staticmethod
    def forward(ctx, vol, factor, ndim):
        ctx.factor, ctx.ndim, ctx.D = factor, ndim, vol.shape[-1]
        return tp.pad_volume(vol, factor, ndim)

    @staticmethod
    def backward(ctx, grad):
        if not ctx.needs_input_grad[0]:
            return None, None, None
        return tp.crop_volume(grad.contiguous(), ctx.D, ctx.factor, ctx.ndim), None, None


def project(rec, rot, shift=None, Do=None, interp=tp.TP_CUBIC, layout=tp.TP_LAYOUT_CENTERED,
            oversampling=1.0, cutoff=-1.0):
    """Differentiable forward projection; rec [n_rec][D][D][D/2+1] (3D) or [n_rec][D][D/2+1]."""
    Do = rec.shape[1] if Do is None else int(Do)
    return _Project.apply(rec, rot, shift, Do, _opts(interp, layout, oversampling, cutoff))


def backproject(proj, rot, shift=None, weights=None, Dv=None, ndim=3, interp=tp.TP_CUBIC,
                layout=tp.TP_LAYOUT_CENTERED, oversampling=1.0, cutoff=-1.0):
    """Differentiable insertion: the reconstruction, plus the weight volume when weights are
    given (returned as a pair)."""
    Dv = proj.shape[2] if Dv is None else int(Dv)
    return _Backproject.apply(proj, weights, rot, shift, Dv, ndim,
                              _opts(interp, layout, oversampling, cutoff))


def pad_volume(vol, factor, ndim=3):
    """Differentiable real-space zero padding (centre moved to index 0)."""
    return _Pad.apply(vol, int(factor), ndim)


def oversampled_spectrum(vol, factor, ndim=3):
    """Half spectrum (FFTW order) of the volume zero-padded by `factor`."""
    padded = pad_volume(vol, factor, ndim)
    return torch.fft.rfftn(padded, dim=tuple(range(-ndim, 0)))


def project_real(vol, rot, shift=None, factor=1, interp=tp.TP_CUBIC, cutoff=-1.0, ndim=3):
    """On-the-fly pipeline from real-space volumes [n][D]^ndim (centre at D/2) to their
    projections at box D: pad by `factor`, FFT, project at c = factor * R q.  factor = 1 with
    cubic weights and factor = 2 with linear weights are the alternatives the pages compare."""
    D = vol.shape[-1]
    spec = oversampled_spectrum(vol, factor, ndim)
    return project(spec.contiguous(), rot, shift, Do=D, interp=interp, layout=tp.TP_LAYOUT_FFTW,
                   oversampling=float(factor), cutoff=cutoff)
