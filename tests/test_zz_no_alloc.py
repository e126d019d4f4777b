"""GPU check of tp_project_3d_to_2d_noalloc, the forward projection for callers that cannot
allocate device memory (their memory belongs to another allocator, or they run where a
cudaMalloc and its possible device synchronisation are not allowed) and so cannot pass a
workspace.  Its scratch is a fixed array that the library holds; two calls in a row, with
different inputs and the second smaller than the first, must each give bit for bit what the
workspace entry point tp_project_3d_to_2d_ws gives with a workspace of the caller's, so the
second call cannot be reading the first call's leftovers.  This file is collected last, so
that a run stopping at its first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

from back_projection_fourier_b300 import synth, tp

pytestmark = pytest.mark.gpu

TOL_FWD = 1e-5       # the forward projection's parity bar
SCRATCH_BYTES = 36704256


def max_rel(a, b):
    return float((a - b).abs().max() / b.abs().max())


def call_noalloc(V, R, S, Y, op):
    """Through the C ABI directly."""
    L = tp.lib()
    n_sh = 1 if S is None else S.shape[0]
    return L.tp_project_3d_to_2d_noalloc(
        ctypes.c_void_p(V.data_ptr()), V.shape[0], V.shape[1], ctypes.c_void_p(R.data_ptr()),
        R.shape[0], R.shape[1], None if S is None else ctypes.c_void_p(S.data_ptr()), n_sh,
        ctypes.c_void_p(Y.data_ptr()), Y.shape[2], ctypes.byref(op),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _inputs(rng, D, n_rec, n_pose):
    V = torch.from_numpy(np.stack([synth.volume_spectrum(rng, D) for _ in range(n_rec)])).cuda()
    R = torch.from_numpy(synth.rotations_3d(rng, n_pose * n_rec).reshape(n_rec, n_pose, 3, 3)).cuda()
    S = torch.from_numpy(synth.shifts(rng, n_pose * n_rec, 4.0).reshape(n_rec, n_pose, 2)).cuda()
    Y = torch.empty((n_rec, n_pose, D, D // 2 + 1), dtype=torch.complex64, device="cuda")
    return V, R, S, Y


# (D, n_rec) of the first call, then of the second: the second grouped copy is smaller, so
# the first call's bytes lie right beyond (and around) the extent the second one writes.
@pytest.mark.parametrize("interp,calls", [(tp.TP_CUBIC, [(128, 1), (64, 1)]),
                                          (tp.TP_LINEAR, [(64, 3), (32, 2)])])
def test_two_calls_equal_the_workspace_path(interp, calls):
    rng = np.random.default_rng(17 + interp)
    op = tp.make_opts(interp, tp.TP_LAYOUT_CENTERED, 1.0, -1.0)
    for k, (D, n_rec) in enumerate(calls):
        need = tp.tp_workspace_size(3, n_rec, D, op)
        assert 0 < need <= SCRATCH_BYTES
        V, R, S, Y = _inputs(rng, D, n_rec, 40)
        assert call_noalloc(V, R, S, Y, op) == 0, k
        # the same grouped path with a workspace of the caller's: the same taps, weights and
        # summation order, so the results are equal bit for bit
        ref = torch.empty_like(Y)
        tp.tp_project_3d_to_2d_ws(V, R, S, ref, torch.empty(need, dtype=torch.uint8, device="cuda"),
                                  op)
        torch.cuda.synchronize()
        assert torch.equal(Y, ref), k
        # and within the forward bar of the plain entry point
        assert max_rel(Y, tp.project(V, R, S, opts=op)) <= TOL_FWD, k


def test_sizes_beyond_the_scratch_are_rejected():
    op = tp.make_opts(tp.TP_CUBIC, tp.TP_LAYOUT_CENTERED, 1.0, -1.0)
    assert tp.tp_workspace_size(3, 1, 130, op) > SCRATCH_BYTES
    assert tp.tp_workspace_size(3, 2, 128, op) > SCRATCH_BYTES
    V = torch.zeros((1, 130, 130, 66), dtype=torch.complex64, device="cuda")
    R = torch.zeros((1, 2, 3, 3), device="cuda")
    Y = torch.empty((1, 2, 130, 66), dtype=torch.complex64, device="cuda")
    assert call_noalloc(V, R, None, Y, op) == 2          # TP_ERR_SHAPE, nothing enqueued
