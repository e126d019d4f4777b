"""Accuracy metrics of projections against a reference (host-side analysis, numpy).

The pages compare cubic interpolation without oversampling against linear interpolation with
2x oversampling by Fourier ring correlation and by the real-space intensity attenuation of
the projections (Spanish page, results, precision bullet; French page, results, precision;
Dutch page, results, interpolation efficiency).  Both metrics here take batches of images as
rfft half spectra [..., Do, Do/2+1] in FFTW or centered layout.

  frc(a, b)                   per ring |k| = 0 .. Do/2 (rounded radius), summed over the batch:
                              Re sum a conj(b) / sqrt(sum |a|^2 sum |b|^2)
  real_space_attenuation(a, b) per real-space radius bin of the centred images:
                              sum a_real b_real / sum b_real^2, the least-squares gain of a
                              against the reference b (1 = no attenuation)
"""
from __future__ import annotations

import numpy as np

FFTW, CENTERED = 0, 1


def _fftw(spec, layout):
    spec = np.asarray(spec)
    return np.fft.ifftshift(spec, axes=-2) if layout == CENTERED else spec


def ring_index(Do: int) -> np.ndarray:
    """Rounded |k| of every pixel of a half-spectrum image in FFTW order."""
    ky = np.fft.fftfreq(Do, 1.0 / Do)
    KY, KX = np.meshgrid(ky, np.arange(Do // 2 + 1), indexing="ij")
    return np.rint(np.sqrt(KX * KX + KY * KY)).astype(np.int64)


def frc(a, b, layout=FFTW) -> np.ndarray:
    """Fourier ring correlation of a against b, rings 0 .. Do/2."""
    a, b = _fftw(a, layout), _fftw(b, layout)
    Do = a.shape[-2]
    kr = ring_index(Do)
    out = np.zeros(Do // 2 + 1)
    for k in range(Do // 2 + 1):
        m = kr == k
        aa, bb = a[..., m], b[..., m]
        num = np.real(np.sum(aa * np.conj(bb)))
        den = np.sqrt(np.sum(np.abs(aa) ** 2) * np.sum(np.abs(bb) ** 2))
        out[k] = num / den if den > 0 else 0.0
    return out


def real_images(spec, layout=FFTW) -> np.ndarray:
    """Real-space images, centre at index Do/2, from half spectra (inverse rfft2)."""
    s = _fftw(spec, layout)
    Do = s.shape[-2]
    return np.fft.fftshift(np.fft.irfft2(s, s=(Do, Do)), axes=(-2, -1))


def real_space_attenuation(a, b, layout=FFTW, nbins=8):
    """(bin edges in pixels, gain of a against b per radius bin of the centred images)."""
    ia, ib = real_images(a, layout), real_images(b, layout)
    Do = ia.shape[-1]
    yy, xx = np.indices((Do, Do)) - Do // 2
    rr = np.sqrt(xx * xx + yy * yy)
    edges = np.linspace(0.0, Do / 2, nbins + 1)
    gain = np.zeros(nbins)
    for i in range(nbins):
        m = (rr >= edges[i]) & (rr < edges[i + 1])
        den = np.sum(ib[..., m] ** 2)
        gain[i] = np.sum(ia[..., m] * ib[..., m]) / den if den > 0 else 0.0
    return edges, gain
