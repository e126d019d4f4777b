"""Thin Python binding of libtp.so (include/tp.h), argument marshalling only.

Every ``tp_*`` function here has the name of the C entry point it calls, takes torch
tensors on the current CUDA device (complex64 spectra, float32 rotations / shifts /
weights, C-contiguous) and derives the sizes from their shapes.  All the arithmetic runs
in the CUDA kernels of libtp.so; there is no CPU or PyTorch fallback: importing this
module fails when the library has not been built.

The functional helpers at the end (``project``, ``backproject``, ``project_backward``,
``backproject_backward``, ``pad_volume``, ``crop_volume``) allocate the outputs with torch
and call the ``tp_*`` functions.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import torch

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "libtp.so"
HEADER = PKG.parent / "include" / "tp.h"

TP_LINEAR, TP_CUBIC = 0, 1
TP_LAYOUT_FFTW, TP_LAYOUT_CENTERED = 0, 1
STATUS = {0: "TP_OK", 1: "TP_ERR_NULL", 2: "TP_ERR_SHAPE", 3: "TP_ERR_VALUE", 4: "TP_ERR_CUDA"}


class tp_opts(ctypes.Structure):
    _fields_ = [("interp", ctypes.c_int), ("layout", ctypes.c_int),
                ("oversampling", ctypes.c_float), ("cutoff", ctypes.c_float)]


class TPError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib().tp_status_string(status).decode()}")


def _load() -> ctypes.CDLL:
    if not LIB_PATH.exists():
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m back_projection_fourier_b300.build` "
            "(there is no fallback implementation)")
    L = ctypes.CDLL(str(LIB_PATH))
    P, I = ctypes.c_void_p, ctypes.c_int
    O = ctypes.POINTER(tp_opts)
    L.tp_project_3d_to_2d.argtypes = [P, I, I, P, I, I, P, I, P, I, O, P]
    L.tp_project_2d_to_2d.argtypes = [P, I, I, P, I, I, P, I, P, I, O, P]
    L.tp_backproject_2d_to_3d.argtypes = [P, P, I, I, P, I, I, P, I, P, P, I, I, O, P]
    L.tp_backproject_2d_to_2d.argtypes = [P, P, I, I, P, I, I, P, I, P, P, I, I, O, P]
    L.tp_project_backward.argtypes = [I, P, I, I, P, I, I, P, I, P, I, P, P, P, O, P]
    L.tp_project_backward_fused.argtypes = [I, P, I, I, P, I, I, P, I, P, I, P, P, P, O, P]
    L.tp_backproject_backward.argtypes = [I, P, P, I, I, P, I, I, P, I, P, P, I, P, P, P, P, O, P]
    Z = ctypes.c_size_t
    L.tp_workspace_size.argtypes = [I, I, I, O]
    L.tp_workspace_size.restype = Z
    L.tp_project_3d_to_2d_ws.argtypes = [P, I, I, P, I, I, P, I, P, I, P, Z, O, P]
    L.tp_project_backward_ws.argtypes = [I, P, I, I, P, I, I, P, I, P, I, P, P, P, P, Z, O, P]
    L.tp_project_3d_to_2d_noalloc.argtypes = [P, I, I, P, I, I, P, I, P, I, O, P]
    L.tp_pad_volume.argtypes = [I, P, I, I, I, P, P]
    L.tp_crop_volume.argtypes = [I, P, I, I, I, P, P]
    L.tp_status_string.argtypes = [I]
    L.tp_status_string.restype = ctypes.c_char_p
    for f in (L.tp_project_3d_to_2d, L.tp_project_2d_to_2d, L.tp_backproject_2d_to_3d,
              L.tp_backproject_2d_to_2d, L.tp_project_backward, L.tp_backproject_backward,
              L.tp_pad_volume, L.tp_crop_volume, L.tp_project_3d_to_2d_ws,
              L.tp_project_backward_ws, L.tp_project_3d_to_2d_noalloc,
              L.tp_project_backward_fused):
        f.restype = I
    return L


_LIB = _load()


def lib() -> ctypes.CDLL:
    return _LIB


def header_symbols() -> list[str]:
    """Names of the functions include/tp.h declares."""
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^\s*(?:tp_status|const char\*|size_t)\s+(tp_\w+)\s*\(", text,
                                 re.M)))


# ------------------------------------------------------------- marshalling ----

def make_opts(interp=TP_CUBIC, layout=TP_LAYOUT_CENTERED, oversampling=1.0, cutoff=-1.0):
    return tp_opts(int(interp), int(layout), float(oversampling), float(cutoff))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, dtype, name):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _sz(t, i):
    """Size of axis i of t, or -1 (no such axis, or no tensor): a size that fails every check."""
    return t.shape[i] if t is not None and t.dim() > i else -1


def _rec_shape(n_rec, D, ndim):
    return (n_rec, D, D, D // 2 + 1) if ndim == 3 else (n_rec, D, D // 2 + 1)


def _img_shape(n_rec, n_pose, Do):
    return (n_rec, n_pose, Do, Do // 2 + 1)


def _check(*items):
    """items: (tensor or None, dtype, name, expected shape).  Every shape is checked before any
    dtype or device, so a tensor whose shape disagrees with the sizes the call passes to the
    library is refused on any device: the kernels index the buffers by those sizes."""
    for t, _, name, shape in items:
        if t is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    for t, dtype, name, _ in items:
        _need(t, dtype, name)


def _rs(rot, shift, k):
    """(n_rot, n_pose, n_sh) and the check items of rot [n_rot][n_pose][k][k] and shift
    [n_sh][n_pose][2]."""
    n_rot, n_pose = _sz(rot, 0), _sz(rot, 1)
    n_sh = 1 if shift is None else _sz(shift, 0)
    items = [(rot, torch.float32, "rot", (n_rot, n_pose, k, k)),
             (shift, torch.float32, "shift", (n_sh, n_pose, 2))]
    return n_rot, n_pose, n_sh, items


def _gshift(grad_shift, shift, n_sh, n_pose):
    """Check item of a shift gradient: [n_sh][n_pose][2], or [1][n_pose][2] without shift."""
    return (grad_shift, torch.float32, "grad_shift", (n_sh if shift is not None else 1, n_pose, 2))


def _call(status: int, what: str):
    if status != 0:
        raise TPError(status, what)


def _opts(opts):
    return ctypes.byref(opts if opts is not None else make_opts())


# ------------------------------------------------------- C entry points ----

def _project_checks(ndim, vol, rot, shift, out, vname):
    n_rot, n_pose, n_sh, items = _rs(rot, shift, ndim)
    n_rec, Dv, Do = _sz(vol, 0), _sz(vol, 1), _sz(out, 2)
    _check((vol, torch.complex64, vname, _rec_shape(n_rec, Dv, ndim)),
           (out, torch.complex64, "out", _img_shape(n_rec, n_pose, Do)), *items)
    return n_rec, Dv, n_rot, n_pose, n_sh, Do


def tp_project_3d_to_2d(vol, rot, shift, out, opts=None, stream=None):
    n_rec, Dv, n_rot, n_pose, n_sh, Do = _project_checks(3, vol, rot, shift, out, "vol")
    _call(_LIB.tp_project_3d_to_2d(_ptr(vol), n_rec, Dv, _ptr(rot), n_rot, n_pose,
                                   _ptr(shift), n_sh, _ptr(out), Do, _opts(opts),
                                   _stream(stream)), "tp_project_3d_to_2d")


def tp_project_2d_to_2d(img, rot, shift, out, opts=None, stream=None):
    n_rec, Dv, n_rot, n_pose, n_sh, Do = _project_checks(2, img, rot, shift, out, "img")
    _call(_LIB.tp_project_2d_to_2d(_ptr(img), n_rec, Dv, _ptr(rot), n_rot, n_pose,
                                   _ptr(shift), n_sh, _ptr(out), Do, _opts(opts),
                                   _stream(stream)), "tp_project_2d_to_2d")


def _backproject_checks(ndim, proj, weights, rot, shift, vol_out, wvol_out, Dv, names):
    n_rot, n_pose, n_sh, items = _rs(rot, shift, ndim)
    ref = proj if proj is not None else weights   # proj may be absent when only weights go in
    n_rec, Do = _sz(ref, 0), _sz(ref, 2)
    img, rec = _img_shape(n_rec, n_pose, Do), _rec_shape(n_rec, int(Dv), ndim)
    _check((proj, torch.complex64, "proj", img), (weights, torch.float32, "weights", img),
           (vol_out, torch.complex64, names[0], rec), (wvol_out, torch.float32, names[1], rec),
           *items)
    return n_rec, Do, n_rot, n_pose, n_sh


def tp_backproject_2d_to_3d(proj, weights, rot, shift, vol_out, wvol_out, Dv, accumulate=False,
                            opts=None, stream=None):
    n_rec, Do, n_rot, n_pose, n_sh = _backproject_checks(3, proj, weights, rot, shift, vol_out,
                                                         wvol_out, Dv, ("vol_out", "wvol_out"))
    _call(_LIB.tp_backproject_2d_to_3d(_ptr(proj), _ptr(weights), n_rec, Do,
                                       _ptr(rot), n_rot, n_pose, _ptr(shift), n_sh, _ptr(vol_out),
                                       _ptr(wvol_out), int(Dv), int(bool(accumulate)), _opts(opts),
                                       _stream(stream)), "tp_backproject_2d_to_3d")


def tp_backproject_2d_to_2d(proj, weights, rot, shift, img_out, wimg_out, Dv, accumulate=False,
                            opts=None, stream=None):
    n_rec, Do, n_rot, n_pose, n_sh = _backproject_checks(2, proj, weights, rot, shift, img_out,
                                                         wimg_out, Dv, ("img_out", "wimg_out"))
    _call(_LIB.tp_backproject_2d_to_2d(_ptr(proj), _ptr(weights), n_rec, Do,
                                       _ptr(rot), n_rot, n_pose, _ptr(shift), n_sh, _ptr(img_out),
                                       _ptr(wimg_out), int(Dv), int(bool(accumulate)), _opts(opts),
                                       _stream(stream)), "tp_backproject_2d_to_2d")


def _backward_checks(ndim, rec, rot, shift, grad_out, grad_rec, grad_rot, grad_shift):
    n_rot, n_pose, n_sh, items = _rs(rot, shift, ndim)
    n_rec, Dv, Do = _sz(rec, 0), _sz(rec, 1), _sz(grad_out, 2)
    rshape = _rec_shape(n_rec, Dv, ndim)
    _check((rec, torch.complex64, "rec", rshape),
           (grad_out, torch.complex64, "grad_out", _img_shape(n_rec, n_pose, Do)),
           (grad_rec, torch.complex64, "grad_rec", rshape),
           (grad_rot, torch.float32, "grad_rot", (n_rot, n_pose, ndim, ndim)),
           _gshift(grad_shift, shift, n_sh, n_pose), *items)
    return n_rec, Dv, n_rot, n_pose, n_sh, Do


def tp_project_backward(ndim, rec, rot, shift, grad_out, grad_rec, grad_rot, grad_shift,
                        opts=None, stream=None):
    n_rec, Dv, n_rot, n_pose, n_sh, Do = _backward_checks(ndim, rec, rot, shift, grad_out,
                                                          grad_rec, grad_rot, grad_shift)
    _call(_LIB.tp_project_backward(int(ndim), _ptr(rec), n_rec, Dv, _ptr(rot), n_rot,
                                   n_pose, _ptr(shift), n_sh, _ptr(grad_out), Do,
                                   _ptr(grad_rec), _ptr(grad_rot), _ptr(grad_shift), _opts(opts),
                                   _stream(stream)), "tp_project_backward")


def tp_project_backward_fused(ndim, rec, rot, shift, grad_out, grad_rec, grad_rot, grad_shift,
                              opts=None, stream=None):
    n_rec, Dv, n_rot, n_pose, n_sh, Do = _backward_checks(ndim, rec, rot, shift, grad_out,
                                                          grad_rec, grad_rot, grad_shift)
    _call(_LIB.tp_project_backward_fused(int(ndim), _ptr(rec), n_rec, Dv, _ptr(rot), n_rot,
                                         n_pose, _ptr(shift), n_sh, _ptr(grad_out), Do,
                                         _ptr(grad_rec), _ptr(grad_rot), _ptr(grad_shift),
                                         _opts(opts), _stream(stream)), "tp_project_backward_fused")


def tp_backproject_backward(ndim, proj, weights, rot, shift, grad_vol, grad_wvol, grad_proj,
                            grad_weights, grad_rot, grad_shift, opts=None, stream=None):
    n_rot, n_pose, n_sh, items = _rs(rot, shift, ndim)
    ref = next((t for t in (proj, grad_proj, grad_weights, weights) if t is not None), None)
    vref = grad_vol if grad_vol is not None else grad_wvol
    if ref is None or vref is None:
        raise ValueError("the image size needs one of proj, grad_proj, grad_weights, weights and "
                         "the volume size one of grad_vol, grad_wvol")
    n_rec, Do, Dv = _sz(ref, 0), _sz(ref, 2), _sz(vref, 1)
    img, vol = _img_shape(n_rec, n_pose, Do), _rec_shape(n_rec, Dv, ndim)
    _check((proj, torch.complex64, "proj", img), (weights, torch.float32, "weights", img),
           (grad_vol, torch.complex64, "grad_vol", vol),
           (grad_wvol, torch.float32, "grad_wvol", vol),
           (grad_proj, torch.complex64, "grad_proj", img),
           (grad_weights, torch.float32, "grad_weights", img),
           (grad_rot, torch.float32, "grad_rot", (n_rot, n_pose, ndim, ndim)),
           _gshift(grad_shift, shift, n_sh, n_pose), *items)
    _call(_LIB.tp_backproject_backward(int(ndim), _ptr(proj), _ptr(weights), n_rec,
                                       Do, _ptr(rot), n_rot, n_pose, _ptr(shift), n_sh,
                                       _ptr(grad_vol), _ptr(grad_wvol), Dv,
                                       _ptr(grad_proj), _ptr(grad_weights), _ptr(grad_rot),
                                       _ptr(grad_shift), _opts(opts), _stream(stream)),
          "tp_backproject_backward")


def tp_workspace_size(ndim, n_rec, Dv, opts=None) -> int:
    return int(_LIB.tp_workspace_size(int(ndim), int(n_rec), int(Dv), _opts(opts)))


def _ws(workspace):
    if workspace is None:
        return None, 0
    if workspace.dtype != torch.uint8 or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA uint8 tensor")
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel()


def tp_project_3d_to_2d_ws(vol, rot, shift, out, workspace, opts=None, stream=None):
    n_rec, Dv, n_rot, n_pose, n_sh, Do = _project_checks(3, vol, rot, shift, out, "vol")
    wp, wb = _ws(workspace)
    _call(_LIB.tp_project_3d_to_2d_ws(_ptr(vol), n_rec, Dv, _ptr(rot), n_rot,
                                      n_pose, _ptr(shift), n_sh, _ptr(out), Do, wp, wb,
                                      _opts(opts), _stream(stream)), "tp_project_3d_to_2d_ws")


def tp_project_backward_ws(ndim, rec, rot, shift, grad_out, grad_rec, grad_rot, grad_shift,
                           workspace, opts=None, stream=None):
    n_rec, Dv, n_rot, n_pose, n_sh, Do = _backward_checks(ndim, rec, rot, shift, grad_out,
                                                          grad_rec, grad_rot, grad_shift)
    wp, wb = _ws(workspace)
    _call(_LIB.tp_project_backward_ws(int(ndim), _ptr(rec), n_rec, Dv, _ptr(rot),
                                      n_rot, n_pose, _ptr(shift), n_sh, _ptr(grad_out),
                                      Do, _ptr(grad_rec), _ptr(grad_rot),
                                      _ptr(grad_shift), wp, wb, _opts(opts), _stream(stream)),
          "tp_project_backward_ws")


def tp_project_3d_to_2d_noalloc(vol, rot, shift, out, opts=None, stream=None):
    n_rec, Dv, n_rot, n_pose, n_sh, Do = _project_checks(3, vol, rot, shift, out, "vol")
    _call(_LIB.tp_project_3d_to_2d_noalloc(_ptr(vol), n_rec, Dv, _ptr(rot), n_rot,
                                           n_pose, _ptr(shift), n_sh, _ptr(out), Do,
                                           _opts(opts), _stream(stream)),
          "tp_project_3d_to_2d_noalloc")


def tp_pad_volume(ndim, vol, factor, out, stream=None):
    n, D, P = _sz(vol, 0), _sz(vol, ndim), int(factor) * _sz(vol, ndim)
    _check((vol, torch.float32, "vol", (n,) + (D,) * ndim),
           (out, torch.float32, "out", (n,) + (P,) * ndim))
    _call(_LIB.tp_pad_volume(int(ndim), _ptr(vol), n, D, int(factor),
                             _ptr(out), _stream(stream)), "tp_pad_volume")


def tp_crop_volume(ndim, padded, factor, out, stream=None):
    n, D, P = _sz(out, 0), _sz(out, ndim), int(factor) * _sz(out, ndim)
    _check((padded, torch.float32, "padded", (n,) + (P,) * ndim),
           (out, torch.float32, "out", (n,) + (D,) * ndim))
    _call(_LIB.tp_crop_volume(int(ndim), _ptr(padded), n, D, int(factor),
                              _ptr(out), _stream(stream)), "tp_crop_volume")


def tp_status_string(status: int) -> str:
    return _LIB.tp_status_string(int(status)).decode()


# -------------------------------------------------------- functional API ----

def project(rec, rot, shift=None, Do=None, opts=None, stream=None):
    """Forward projection (3D->2D when rec is [n_rec][D][D][H], 2D->2D when [n_rec][D][H])."""
    ndim = rec.dim() - 1
    Do = rec.shape[1] if Do is None else int(Do)
    out = torch.empty((rec.shape[0], rot.shape[1], Do, Do // 2 + 1), dtype=torch.complex64,
                      device=rec.device)
    (tp_project_3d_to_2d if ndim == 3 else tp_project_2d_to_2d)(rec, rot, shift, out, opts, stream)
    return out


def backproject(proj, rot, shift=None, weights=None, Dv=None, want_weights=True, opts=None,
                stream=None, ndim=3):
    """Back-projection (insertion) into fresh zeroed outputs: (rec, weight rec or None)."""
    Dv = proj.shape[2] if Dv is None else int(Dv)
    H = Dv // 2 + 1
    shape = (proj.shape[0], Dv, Dv, H) if ndim == 3 else (proj.shape[0], Dv, H)
    rec = torch.empty(shape, dtype=torch.complex64, device=proj.device)
    wrec = torch.empty(shape, dtype=torch.float32, device=proj.device) if want_weights else None
    fn = tp_backproject_2d_to_3d if ndim == 3 else tp_backproject_2d_to_2d
    fn(proj, weights, rot, shift, rec, wrec, Dv, False, opts, stream)
    return rec, wrec


def project_backward(rec, rot, grad_out, shift=None, want_rec=True, want_rot=True,
                     want_shift=True, opts=None, stream=None, fused=False):
    """Backward of the projection in one call: (grad_rec, grad_rot, grad_shift), each None when
    not wanted.  fused=True takes tp_project_backward_fused (one kernel pass where it applies)."""
    ndim = rec.dim() - 1
    g_rec = torch.empty_like(rec) if want_rec else None
    g_rot = torch.empty_like(rot) if want_rot else None
    n_sh = shift.shape[0] if shift is not None else 1
    g_sh = torch.empty((n_sh, rot.shape[1], 2), dtype=torch.float32, device=rec.device) \
        if want_shift else None
    (tp_project_backward_fused if fused else tp_project_backward)(
        ndim, rec, rot, shift, grad_out, g_rec, g_rot, g_sh, opts, stream)
    return g_rec, g_rot, g_sh


def backproject_backward(proj, rot, grad_vol, grad_wvol=None, shift=None, weights=None,
                         want_proj=True, want_weights=True, want_rot=True, want_shift=True,
                         opts=None, stream=None, ndim=3):
    """Backward of the insertion: (grad_proj, grad_weights, grad_rot, grad_shift), each None
    when not wanted (grad_weights also when weights is None)."""
    g_proj = torch.empty_like(proj) if want_proj else None
    g_w = torch.empty(proj.shape, dtype=torch.float32, device=proj.device) \
        if want_weights and weights is not None else None
    g_rot = torch.empty_like(rot) if want_rot else None
    n_sh = shift.shape[0] if shift is not None else 1
    g_sh = torch.empty((n_sh, rot.shape[1], 2), dtype=torch.float32, device=proj.device) \
        if want_shift else None
    tp_backproject_backward(ndim, proj, weights, rot, shift, grad_vol, grad_wvol, g_proj, g_w,
                            g_rot, g_sh, opts, stream)
    return g_proj, g_w, g_rot, g_sh


def pad_volume(vol, factor, ndim=3, stream=None):
    """Zero-pad [n][D]^ndim real data by `factor`, centre moved to index 0."""
    P = int(factor) * vol.shape[-1]
    out = torch.empty((vol.shape[0],) + (P,) * ndim, dtype=torch.float32, device=vol.device)
    tp_pad_volume(ndim, vol, factor, out, stream)
    return out


def crop_volume(padded, D, factor, ndim=3, stream=None):
    """Adjoint of pad_volume: the [n][D]^ndim box back out of the padded array."""
    out = torch.empty((padded.shape[0],) + (int(D),) * ndim, dtype=torch.float32,
                      device=padded.device)
    tp_crop_volume(ndim, padded, factor, out, stream)
    return out


def workspace_for(rec, opts=None):
    """A workspace (CUDA uint8 tensor) for the 3D gathers over `rec`, or None when unused."""
    n = tp_workspace_size(rec.dim() - 1, rec.shape[0], rec.shape[1], opts)
    return torch.empty(n, dtype=torch.uint8, device=rec.device) if n else None
