"""Seeded synthetic inputs for Fourier-slice projection workloads.

This module only draws random inputs; it holds none of the projection arithmetic, so
both the CUDA path and the CPU oracle can take their inputs from it.

Recipe (all host numpy, ``numpy.random.default_rng``):
  * volumes / images: real N(0, 1) samples, rfftn / rfft2 in fp64 with ``norm="ortho"``
    (unit-variance spectra), optional 1/max(|k|, 1) amplitude falloff, then the full
    (non-half) axes are put in the requested layout (centered = fftshift), cast to
    complex64;
  * 3D rotations: uniform on SO(3) from normalised 4-D Gaussian quaternions (w, x, y, z)
    converted with the Hamilton formula; 2D rotations from angles U[0, 2 pi);
  * shifts: U(-a, a) per component, fp32;
  * per-item complex arrays (upstream gradients, projections): CN(0, 1), real and
    imaginary parts N(0, 1/2), drawn directly in fp32 in chunks of ``CHUNK`` items, each
    chunk from its own stream ``default_rng([seed, tag, chunk])`` so that any item can be
    regenerated alone;
  * CTF-like weights: 1 - exp(-|k|^2 / sigma^2) * cos(gamma |k|^2), |k| in pixel
    frequency units, the same map for every item.
Seeds: 1000 + the workload number; draw order: volume/images, rotations, shifts,
upstream gradient / projections, weights.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

FFTW, CENTERED = 0, 1
LINEAR, CUBIC = 0, 1
CHUNK = 256


def _layout(spec: np.ndarray, full_axes, layout: int) -> np.ndarray:
    return np.fft.fftshift(spec, axes=full_axes) if layout == CENTERED else spec


def _kfreq(D: int):
    return np.fft.fftfreq(D, 1.0 / D)


def volume_spectrum(rng, D: int, layout=CENTERED, falloff=False) -> np.ndarray:
    """rfftn half-volume complex64 [D][D][D/2+1] of a real N(0,1) volume."""
    f = rng.standard_normal((D, D, D))
    spec = np.fft.rfftn(f, norm="ortho")
    if falloff:
        kz = _kfreq(D)[:, None, None]
        ky = _kfreq(D)[None, :, None]
        kx = np.arange(D // 2 + 1, dtype=np.float64)[None, None, :]
        spec = spec / np.maximum(np.sqrt(kx * kx + ky * ky + kz * kz), 1.0)
    return np.ascontiguousarray(_layout(spec, (0, 1), layout).astype(np.complex64))


def ball_noise_volume(rng, D: int, margin: int = 2, ndim: int = 3) -> np.ndarray:
    """Real-space N(0,1) noise inside the ball of radius D/2 - margin about the centre D/2 and
    zero outside ([D]^ndim, fp64): a synthetic volume whose rotations stay inside the box."""
    f = rng.standard_normal((D,) * ndim)
    r = np.indices(f.shape) - D // 2
    f[(r ** 2).sum(0) > (D // 2 - margin) ** 2] = 0.0
    return f


def image_spectra(rng, n: int, D: int, layout=CENTERED) -> np.ndarray:
    """rfft2 half-images complex64 [n][D][D/2+1] of real N(0,1) images."""
    out = np.empty((n, D, D // 2 + 1), np.complex64)
    for a in range(0, n, CHUNK):
        b = min(n, a + CHUNK)
        spec = np.fft.rfft2(rng.standard_normal((b - a, D, D)), norm="ortho")
        out[a:b] = _layout(spec, (1,), layout)
    return out


def rotations_3d(rng, n: int) -> np.ndarray:
    """Uniform SO(3) rotation matrices fp32 [n][3][3] (row-major)."""
    q = rng.standard_normal((n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    w, x, y, z = q.T
    R = np.empty((n, 3, 3))
    R[:, 0, 0] = 1 - 2 * (y * y + z * z)
    R[:, 0, 1] = 2 * (x * y - z * w)
    R[:, 0, 2] = 2 * (x * z + y * w)
    R[:, 1, 0] = 2 * (x * y + z * w)
    R[:, 1, 1] = 1 - 2 * (x * x + z * z)
    R[:, 1, 2] = 2 * (y * z - x * w)
    R[:, 2, 0] = 2 * (x * z - y * w)
    R[:, 2, 1] = 2 * (y * z + x * w)
    R[:, 2, 2] = 1 - 2 * (x * x + y * y)
    return R.astype(np.float32)


def rotations_2d(rng, n: int) -> np.ndarray:
    """In-plane rotations fp32 [n][2][2] with angles U[0, 2 pi)."""
    th = rng.uniform(0.0, 2.0 * np.pi, n)
    c, s = np.cos(th), np.sin(th)
    return np.stack([np.stack([c, -s], -1), np.stack([s, c], -1)], -2).astype(np.float32)


def shifts(rng, n: int, amp: float) -> np.ndarray:
    """Shifts fp32 [n][2] = (sx, sy), each U(-amp, amp)."""
    return rng.uniform(-amp, amp, (n, 2)).astype(np.float32)


def cn01_items(seed: int, tag: int, n_items: int, item_shape, items=None) -> np.ndarray:
    """CN(0,1) complex64 [len(items)][*item_shape]; chunk c of CHUNK items comes from
    default_rng([seed, tag, c]), so a subset of items is reproducible on its own."""
    item_shape = tuple(item_shape)
    per = int(np.prod(item_shape))
    items = np.arange(n_items) if items is None else np.asarray(items)
    out = np.empty((len(items),) + item_shape, np.complex64)
    flat = out.reshape(len(items), per)
    order = np.argsort(items, kind="stable")
    cache_c, cache = -1, None
    scale = np.float32(np.sqrt(0.5))
    for pos in order:
        it = int(items[pos])
        c = it // CHUNK
        if c != cache_c:
            m = min(CHUNK, n_items - c * CHUNK)
            g = np.random.default_rng([seed, tag, c])
            re = g.standard_normal((m, per), dtype=np.float32)
            im = g.standard_normal((m, per), dtype=np.float32)
            cache = (re * scale) + 1j * (im * scale)
            cache_c = c
        flat[pos] = cache[it - c * CHUNK]
    return out


def ctf_like_weights(D: int, sigma: float, gamma: float, layout=CENTERED) -> np.ndarray:
    """fp32 [D][D/2+1]: 1 - exp(-|k|^2/sigma^2) * cos(gamma |k|^2), rows in `layout`."""
    ky = _kfreq(D)[:, None]
    kx = np.arange(D // 2 + 1, dtype=np.float64)[None, :]
    k2 = kx * kx + ky * ky
    w = 1.0 - np.exp(-k2 / (sigma * sigma)) * np.cos(gamma * k2)
    return np.ascontiguousarray(_layout(w, (0,), layout).astype(np.float32))


@dataclass
class Workload:
    """Inputs of one workload.  Shapes follow the C ABI (see include/tp.h)."""

    name: str
    number: int
    ndim: int
    op: str                      # "fwd", "fwdbwd", "insert"
    interp: int
    D: int
    B: int
    rc: float
    layout: int = CENTERED
    n_rec: int = 1
    n_pose: int = 1
    rec: np.ndarray | None = None          # [n_rec][D][D][H] or [n_rec][D][H]
    rot: np.ndarray | None = None          # [n_rot][n_pose][k][k]
    shift: np.ndarray | None = None        # [n_sh][n_pose][2] or None
    grad: np.ndarray | None = None         # upstream grad / projections [n_rec][n_pose][D][H]
    weights: np.ndarray | None = None      # [n_rec][n_pose][D][H] fp32 or None
    extra: dict = field(default_factory=dict)

    @property
    def H(self) -> int:
        return self.D // 2 + 1


# name -> (number, ndim, op, interp, D, B, rc, shift amplitude, falloff[, n_rec])
# B counts projections; with n_rec > 1 (3D) each reconstruction has B / n_rec poses of its own.
WORKLOADS = {
    "fwd3d_d32_linear_b64": (1, 3, "fwd", LINEAR, 32, 64, 16.0, 0.0, False),
    "fwdbwd3d_d64_cubic_b4096": (2, 3, "fwdbwd", CUBIC, 64, 4096, 32.0, 5.0, False),
    "insert3d_d128_b16384": (3, 3, "insert", CUBIC, 128, 16384, 64.0, 0.0, False),
    "rot2d_d256_cubic_b8192": (4, 2, "fwdbwd", CUBIC, 256, 8192, 128.0, 8.0, False),
    "fwdbwd3d_d256_cubic_b50000": (5, 3, "fwdbwd", CUBIC, 256, 50000, 128.0, 10.0, True),
    "fwdbwd3d_d128_cubic_b16384": (6, 3, "fwdbwd", CUBIC, 128, 16384, 64.0, 5.0, False),
    "fwdbwd3d_d128_cubic_r8_b16384": (7, 3, "fwdbwd", CUBIC, 128, 16384, 64.0, 5.0, False, 8),
}


def make_workload(name: str, B: int | None = None, interp: int | None = None,
                  with_grad: bool = True, layout: int = CENTERED,
                  poses: tuple[int, int] | None = None) -> Workload:
    """Draw the inputs of a named workload; ``B`` overrides the batch (same recipe).

    ``poses = (a, b)`` keeps only poses a..b-1 of every reconstruction (3D workloads): the
    rotations, shifts, upstream gradients and weights of those poses, drawn exactly as in
    the whole batch (the per-item arrays regenerate those items alone), and ``B`` becomes
    the number of projections kept.  This is how one rank of a data-parallel run draws its
    shard of a larger batch without drawing the rest."""
    number, ndim, op, interp0, D, B0, rc, amp, falloff, *rest = WORKLOADS[name]
    n_rec = rest[0] if rest else 1
    B = B0 if B is None else B
    if B % n_rec:
        raise ValueError(f"batch {B} is not a multiple of the {n_rec} reconstructions")
    if poses is not None:
        if ndim != 3:
            raise ValueError("pose ranges apply to 3D workloads (2D items are images)")
        a, b = poses
        if not 0 <= a <= b <= B // n_rec:
            raise ValueError(f"pose range {poses} outside 0..{B // n_rec}")
    interp = interp0 if interp is None else interp
    seed = 1000 + number
    rng = np.random.default_rng(seed)
    H = D // 2 + 1
    wl = Workload(name, number, ndim, op, interp, D, B, rc, layout)
    if ndim == 3:
        wl.n_rec, wl.n_pose = n_rec, B // n_rec
        if op != "insert":
            wl.rec = np.stack([volume_spectrum(rng, D, layout, falloff) for _ in range(n_rec)])
        wl.rot = rotations_3d(rng, B).reshape(n_rec, B // n_rec, 3, 3)
    else:
        wl.n_rec, wl.n_pose = B, 1
        wl.rec = image_spectra(rng, B, D, layout)
        wl.rot = rotations_2d(rng, B)[:, None]
    if amp > 0:
        s = shifts(rng, B, amp)
        wl.shift = s.reshape(n_rec, B // n_rec, 2) if ndim == 3 else s[:, None]
    if (op == "insert" or (op == "fwdbwd" and with_grad)) and poses is None:
        g = cn01_items(seed, 1, B, (D, H))
        wl.grad = g.reshape(n_rec, B // n_rec, D, H) if ndim == 3 else g[:, None]
    if op == "insert":
        w = ctf_like_weights(D, 40.0, 1e-3, layout)
        wl.weights = np.broadcast_to(w, (wl.n_rec, wl.n_pose, D, H))
    wl.extra["shift_amp"] = amp
    wl.extra["falloff"] = falloff
    if poses is not None:
        a, b = poses
        n_pose = B // n_rec
        keep = lambda x: None if x is None else np.ascontiguousarray(x[:, a:b])  # noqa: E731
        wl.rot, wl.shift = keep(wl.rot), keep(wl.shift)
        if wl.weights is not None:
            wl.weights = np.broadcast_to(wl.weights[:1, :1], (n_rec, b - a, D, H))
        if op == "insert" or (op == "fwdbwd" and with_grad):
            items = (np.arange(n_rec)[:, None] * n_pose + np.arange(a, b)[None, :]).ravel()
            wl.grad = cn01_items(seed, 1, B, (D, H), items).reshape(n_rec, b - a, D, H)
        wl.n_pose = b - a
        wl.B = n_rec * (b - a)
        wl.extra["poses"] = (a, b)
        wl.extra["batch_total"] = B
    return wl
