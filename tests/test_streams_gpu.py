"""Stream semantics of the C ABI: each call enqueues its output zeroing and its kernels on the
stream it is given (NULL: the legacy default stream; the binding passes the current torch
stream when none is named) and returns without synchronising.

Every check runs the same work on a side stream whose inputs are written there only after a
short GPU sleep: a call that launched anywhere else would read them before they exist.
"""
import numpy as np
import pytest
import torch

from parity_util import crandn32, dev, opts, rotations
from back_projection_fourier_b300 import tp

pytestmark = pytest.mark.gpu

D, N_POSE = 32, 33
SLEEP_CYCLES = 20_000_000     # about 10 ms of GPU time before the inputs are written


def _inputs(seed):
    rng = np.random.default_rng(seed)
    H = D // 2 + 1
    V = dev(crandn32(rng, (1, D, D, H)))
    R = dev(rotations(rng, N_POSE, 3).reshape(1, N_POSE, 3, 3))
    S = dev(rng.uniform(-5, 5, (1, N_POSE, 2)).astype(np.float32))
    G = dev(crandn32(rng, (1, N_POSE, D, H)))
    return V, R, S, G


def _step(V, R, S, G, op, ws, stream):
    """Forward, pose gradients and volume gradient, as three calls on one stream."""
    y = torch.empty_like(G)
    gR, gS, gV = torch.empty_like(R), torch.empty_like(S), torch.empty_like(V)
    tp.tp_project_3d_to_2d_ws(V, R, S, y, ws, op, stream)
    tp.tp_project_backward_ws(3, V, R, S, G, None, gR, gS, ws, op, stream)
    tp.tp_project_backward(3, V, R, S, G, gV, None, None, op, stream)
    return y, gR, gS, gV


def _rel(a, b):
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def _late_copies(s, *src):
    """Copies of src written on stream s after a GPU sleep there (allocated beforehand)."""
    dst = [torch.full_like(t, float("nan")) for t in src]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(SLEEP_CYCLES)
        for d, t in zip(dst, src):
            d.copy_(t)
    return dst


@pytest.mark.parametrize("how", ["object", "handle", "current"])
def test_calls_run_on_the_given_stream(how):
    V, R, S, G = _inputs(11)
    op = opts(1, 1)
    ref = _step(V, R, S, G, op, tp.workspace_for(V, op), None)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    V2, R2, S2, G2 = _late_copies(s, V, R, S, G)
    ws = tp.workspace_for(V, op)
    if how == "object":
        out = _step(V2, R2, S2, G2, op, ws, s)
    elif how == "handle":
        out = _step(V2, R2, S2, G2, op, ws, s.cuda_stream)
    else:
        with torch.cuda.stream(s):
            out = _step(V2, R2, S2, G2, op, ws, None)
    s.synchronize()
    assert torch.equal(out[0], ref[0])              # the forward has no atomics: bit for bit
    for a, b in zip(out[1:], ref[1:]):
        assert _rel(a, b) <= 1e-5                    # atomics: only the order of the sums differs


def test_zeroing_and_accumulation_are_ordered_on_the_stream():
    """Overwrite then accumulate on a side stream: twice the single insertion, with the
    weight volume, in 3D and in 2D."""
    rng = np.random.default_rng(12)
    s = torch.cuda.Stream()
    for ndim in (3, 2):
        H = D // 2 + 1
        P = dev(crandn32(rng, (2, 5, D, H)))
        W = dev(rng.uniform(0, 2, (2, 5, D, H)).astype(np.float32))
        R = dev(rotations(rng, 10, ndim).reshape(2, 5, ndim, ndim))
        shape = (2, D, D, H) if ndim == 3 else (2, D, H)
        ref_v, ref_w = tp.backproject(P, R, None, W, Dv=D, opts=opts(1, 1), ndim=ndim)
        torch.cuda.synchronize()
        P2, W2 = _late_copies(s, P, W)
        vol = torch.full(shape, float("nan"), dtype=torch.complex64, device="cuda")
        wvol = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        fn = tp.tp_backproject_2d_to_3d if ndim == 3 else tp.tp_backproject_2d_to_2d
        fn(P2, W2, R, None, vol, wvol, D, False, opts(1, 1), s)
        fn(P2, W2, R, None, vol, wvol, D, True, opts(1, 1), s)
        s.synchronize()
        assert _rel(vol, 2 * ref_v) <= 1e-5
        assert _rel(wvol, 2 * ref_w) <= 1e-5
