"""Shared helpers of the GPU parity tests: upload seeded inputs, call the C ABI through the
binding, call the oracle on the same values, compare with the relative-to-max metric."""
import numpy as np
import torch

import oracle
from back_projection_fourier_b300 import tp

# Tolerances (max |gpu - oracle| / max |oracle| per output tensor): fp32 projection 1e-5;
# atomics-ordered back-projection and gradients 1e-4.
TOL_FWD = 1e-5
TOL_BWD = 1e-4


def max_rel(gpu, ref) -> float:
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu.astype(ref.dtype) - ref).max() / scale)


def dev(a, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return None if t is None else t.detach().cpu().numpy()


def opts(interp, layout=1, o=1.0, cutoff=-1.0):
    return tp.make_opts(interp, layout, o, cutoff)


def crandn32(rng, shape):
    return (rng.standard_normal(shape, dtype=np.float32)
            + 1j * rng.standard_normal(shape, dtype=np.float32)).astype(np.complex64)


def rotations(rng, n, k):
    from back_projection_fourier_b300 import synth
    return synth.rotations_3d(rng, n) if k == 3 else synth.rotations_2d(rng, n)


__all__ = ["oracle", "TOL_FWD", "TOL_BWD", "max_rel", "dev", "host", "opts", "crandn32",
           "rotations"]
