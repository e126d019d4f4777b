"""C-ABI checks that need no GPU: the library loads, exports every function the header
declares, and rejects bad arguments on the host (before any CUDA call) with the status
the header documents."""
import ctypes
import math
import subprocess

import pytest

from back_projection_fourier_b300 import build as tp_build

tp_build.build()
from back_projection_fourier_b300 import tp  # noqa: E402

L = tp.lib()
FAKE = 0x10000          # aligned, never dereferenced: validation fails first
MIS = 0x10004           # 4-byte aligned, not 8-byte aligned


def test_header_symbols_are_exported():
    names = tp.header_symbols()
    assert set(names) == {"tp_project_3d_to_2d", "tp_backproject_2d_to_3d", "tp_project_2d_to_2d",
                          "tp_backproject_2d_to_2d", "tp_project_backward", "tp_backproject_backward",
                          "tp_pad_volume", "tp_crop_volume", "tp_status_string",
                          "tp_workspace_size", "tp_project_3d_to_2d_ws", "tp_project_backward_ws",
                          "tp_project_3d_to_2d_noalloc", "tp_project_backward_fused"}
    for n in names:
        assert hasattr(L, n), n
    dyn = subprocess.run(["nm", "-D", "--defined-only", str(tp.LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in dyn.splitlines() if " T " in line}
    assert set(names) <= exported


def test_status_strings():
    for code, name in tp.STATUS.items():
        assert tp.tp_status_string(code).startswith(name)
    assert "UNKNOWN" in tp.tp_status_string(99)


def opts(interp=1, layout=1, o=1.0, cutoff=-1.0):
    return ctypes.byref(tp.make_opts(interp, layout, o, cutoff))


def proj3(vol=FAKE, n_rec=1, Dv=8, rot=FAKE, n_rot=1, n_pose=2, shift=None, n_sh=1, out=FAKE,
          Do=8, o=None):
    return L.tp_project_3d_to_2d(vol, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, out, Do,
                                 o if o is not None else opts(), None)


def test_project_argument_errors():
    assert proj3(vol=None) == 1
    assert proj3(rot=None) == 1
    assert proj3(out=None) == 1
    assert proj3(Dv=7) == 2
    assert proj3(Do=0) == 2
    assert proj3(Dv=2048) == 2
    assert proj3(n_rec=-1) == 2
    assert proj3(n_pose=-3) == 2
    assert proj3(n_rec=3, n_rot=2) == 2
    assert proj3(n_rec=3, n_rot=3, shift=FAKE, n_sh=2) == 2
    assert proj3(o=opts(interp=2)) == 3
    assert proj3(o=opts(layout=-1)) == 3
    assert proj3(o=opts(o=0.0)) == 3
    assert proj3(o=opts(o=-1.0)) == 3
    assert proj3(o=opts(o=math.inf)) == 3
    assert proj3(o=opts(cutoff=math.nan)) == 3
    assert proj3(vol=MIS) == 3
    assert proj3(out=MIS) == 3
    # empty batches are valid and enqueue nothing
    assert proj3(n_rec=0, vol=None, rot=None, out=None) == 0
    assert proj3(n_pose=0, vol=None, rot=None, out=None) == 0
    assert L.tp_project_2d_to_2d(FAKE, 1, 40000, FAKE, 1, 1, None, 1, FAKE, 8, None, None) == 2


def test_backproject_argument_errors():
    bp = L.tp_backproject_2d_to_3d
    assert bp(FAKE, None, 1, 8, FAKE, 1, 2, None, 1, FAKE, None, 8, 2, opts(), None) == 3
    assert bp(None, None, 1, 8, FAKE, 1, 2, None, 1, FAKE, None, 8, 0, opts(), None) == 1
    assert bp(FAKE, None, 1, 8, None, 1, 2, None, 1, FAKE, None, 8, 0, opts(), None) == 1
    assert bp(FAKE, None, 1, 9, FAKE, 1, 2, None, 1, FAKE, None, 8, 0, opts(), None) == 2
    assert bp(FAKE, None, 1, 8, FAKE, 1, 2, None, 1, MIS, None, 8, 0, opts(), None) == 3
    assert bp(FAKE, None, 0, 8, FAKE, 1, 2, None, 1, FAKE, None, 8, 0, opts(), None) == 0
    bp2 = L.tp_backproject_2d_to_2d
    assert bp2(FAKE, None, 2, 8, FAKE, 3, 1, None, 1, FAKE, None, 8, 0, opts(), None) == 2


@pytest.mark.parametrize("entry", ["tp_project_backward", "tp_project_backward_fused"])
def test_backward_argument_errors(entry):
    bw = getattr(L, entry)
    assert bw(4, FAKE, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, FAKE, None, None, opts(), None) == 3
    assert bw(3, FAKE, 1, 8, FAKE, 1, 2, None, 1, None, 8, FAKE, None, None, opts(), None) == 1
    assert bw(3, None, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, None, FAKE, None, opts(), None) == 1
    assert bw(3, None, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, FAKE, FAKE, None, opts(), None) == 1
    assert bw(3, FAKE, 1, 8, FAKE, 1, 2, None, 1, FAKE, 6, FAKE, None, None, opts(cutoff=math.inf), None) == 3
    assert bw(2, FAKE, 2, 8, FAKE, 1, 2, FAKE, 3, FAKE, 8, FAKE, None, None, opts(), None) == 2
    assert bw(3, FAKE, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, MIS, FAKE, None, opts(), None) == 3


def test_backproject_backward_argument_errors():
    bb = L.tp_backproject_backward
    # ndim, proj, weights, n_rec, Do, rot, n_rot, n_pose, shift, n_sh, grad_vol, grad_wvol, Dv,
    # grad_proj, grad_weights, grad_rot, grad_shift, opts, stream
    args = [3, FAKE, None, 1, 8, FAKE, 1, 2, None, 1, FAKE, None, 8, FAKE, None, FAKE, None, opts(), None]

    def call(**kw):
        a = list(args)
        names = ["ndim", "proj", "weights", "n_rec", "Do", "rot", "n_rot", "n_pose", "shift", "n_sh",
                 "grad_vol", "grad_wvol", "Dv", "grad_proj", "grad_weights", "grad_rot", "grad_shift",
                 "opts"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return bb(*a)

    assert call(ndim=1) == 3
    assert call(rot=None) == 1
    assert call(proj=None) == 1                      # data part of grad_rot needs proj
    assert call(Dv=7) == 2
    assert call(Do=4096) == 2
    assert call(n_rec=2, n_rot=3) == 2
    assert call(opts=opts(interp=5)) == 3
    assert call(proj=MIS) == 3
    assert call(grad_vol=MIS) == 3
    assert call(grad_proj=MIS) == 3
    assert call(grad_wvol=FAKE + 2) == 3
    assert call(grad_weights=FAKE + 1) == 3


@pytest.mark.parametrize("fn", ["tp_pad_volume", "tp_crop_volume"])
def test_pad_argument_errors(fn):
    f = getattr(L, fn)
    assert f(4, FAKE, 1, 8, 2, FAKE, None) == 3
    assert f(3, FAKE, 1, 8, 0, FAKE, None) == 3
    assert f(3, FAKE, 1, 8, 9, FAKE, None) == 3
    assert f(3, FAKE, 1, 7, 2, FAKE, None) == 2
    assert f(3, FAKE, -1, 8, 2, FAKE, None) == 2
    assert f(3, FAKE, 1, 768, 2, FAKE, None) == 2     # padded box beyond the 3D limit
    assert f(3, None, 1, 8, 2, FAKE, None) == 1
    assert f(3, FAKE, 1, 8, 2, None, None) == 1
    assert f(3, FAKE + 2, 1, 8, 2, FAKE, None) == 3
    assert f(3, None, 0, 8, 2, None, None) == 0


def test_workspace_size():
    # cubic D = 128: rows of 64 + 4 = 68 groups padded to 70 (2 mod 4), planes of 128 * 70
    # groups padded to 8961 (1 mod 4), 4 taps of 8 bytes a group
    assert tp.tp_workspace_size(3, 1, 128, tp.make_opts(1)) == 128 * 8961 * 4 * 8
    # linear D = 64: rows of 32 + 2 = 34 groups (already 2 mod 8), planes of 64 * 34 = 2176
    # groups padded to 2177 (1 mod 8), 2 taps a group
    assert tp.tp_workspace_size(3, 2, 64, tp.make_opts(0)) == 2 * 64 * 2177 * 2 * 8
    assert tp.tp_workspace_size(2, 1, 128, tp.make_opts(1)) == 0      # 2D: not used
    assert tp.tp_workspace_size(3, 1, 7, tp.make_opts(1)) == 0        # odd box
    assert tp.tp_workspace_size(3, 1, 1024, tp.make_opts(1)) == 0     # 32-bit offsets
    assert tp.tp_workspace_size(3, 1, 128, tp.make_opts(5)) == 0      # bad interp
    per = 1020 * (1020 * 514 + 1) * 4 * 8                             # bytes of one volume's copy
    assert tp.tp_workspace_size(3, 2**29, 1020, tp.make_opts(1)) == per * 2**29
    assert tp.tp_workspace_size(3, 1, 1022, tp.make_opts(1)) == 0     # 32-bit offsets: just over
    assert tp.tp_workspace_size(3, 2**31 - 1, 1020, tp.make_opts(1)) == 0   # would overflow
    assert tp.tp_workspace_size(3, -1, 128, tp.make_opts(1)) == 0


def test_workspace_argument_errors():
    need = tp.tp_workspace_size(3, 1, 8, tp.make_opts())
    pw = L.tp_project_3d_to_2d_ws
    assert pw(FAKE, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, FAKE, need - 8, opts(), None) == 2
    assert pw(FAKE, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, FAKE + 16, need, opts(), None) == 3
    assert pw(FAKE, 1, 7, FAKE, 1, 2, None, 1, FAKE, 8, FAKE, need, opts(), None) == 2
    assert pw(None, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, FAKE, need, opts(), None) == 1
    bw = L.tp_project_backward_ws
    assert bw(3, FAKE, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, None, FAKE, None, FAKE, 1, opts(), None) == 2
    assert bw(3, FAKE, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, None, FAKE, None, FAKE + 8, need, opts(),
              None) == 3
    assert bw(3, None, 1, 8, FAKE, 1, 2, None, 1, FAKE, 8, None, FAKE, None, FAKE, need, opts(),
              None) == 1


def test_binding_rejects_bad_tensors():
    import torch
    vol = torch.zeros((1, 8, 8, 5), dtype=torch.complex64)
    rot = torch.zeros((1, 2, 3, 3))
    out = torch.zeros((1, 2, 8, 5), dtype=torch.complex64)
    with pytest.raises(TypeError):
        tp.tp_project_3d_to_2d(vol, rot, None, out)          # CPU tensors
    with pytest.raises(TypeError):
        tp.tp_project_3d_to_2d(vol.real.contiguous(), rot, None, out)


def _z(shape, complex_=False):
    import torch
    return torch.zeros(shape, dtype=torch.complex64 if complex_ else torch.float32)


def test_binding_checks_every_shape_before_the_device():
    """The binding passes sizes taken from some tensors' shapes; every other tensor must
    agree with them exactly, or the kernels would index past it.  A disagreeing shape is a
    ValueError on any device; consistent CPU tensors get as far as the device check."""
    vol, rot, sh, out = _z((2, 8, 8, 5), True), _z((2, 3, 3, 3)), _z((1, 3, 2)), _z((2, 3, 8, 5), True)
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_project_3d_to_2d(vol, rot, sh, out)
    for bad in [dict(out=_z((2, 2, 8, 5), True)),            # pose count
                dict(out=_z((1, 3, 8, 5), True)),            # reconstruction count
                dict(out=_z((2, 3, 8, 4), True)),            # half axis of the image
                dict(vol=_z((2, 8, 8, 4), True)),            # half axis of the volume
                dict(vol=_z((2, 8, 6, 5), True)),            # not a cube
                dict(rot=_z((2, 3, 3, 2))),                  # matrix shape
                dict(sh=_z((1, 2, 2))),                      # shifts for fewer poses
                dict(sh=_z((1, 3, 3))),                      # three shift components
                dict(sh=_z((3,)))]:                          # wrong rank
        a = {**dict(vol=vol, rot=rot, sh=sh, out=out), **bad}
        with pytest.raises(ValueError, match="must have shape"):
            tp.tp_project_3d_to_2d(a["vol"], a["rot"], a["sh"], a["out"])
        with pytest.raises(ValueError, match="must have shape"):
            tp.tp_project_3d_to_2d_ws(a["vol"], a["rot"], a["sh"], a["out"], None)
        with pytest.raises(ValueError, match="must have shape"):
            tp.tp_project_3d_to_2d_noalloc(a["vol"], a["rot"], a["sh"], a["out"])
    # 2D: images [n_rec][D][D/2+1], rotations 2 x 2
    img, rot2 = _z((2, 8, 5), True), _z((2, 3, 2, 2))
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_project_2d_to_2d(img, rot2, sh, out)
    with pytest.raises(ValueError, match="must have shape"):
        tp.tp_project_2d_to_2d(img, rot, sh, out)            # 3 x 3 matrices
    # backward: gradients shaped like their inputs; the shift gradient [1][n_pose][2] without shift
    gR, gS1 = _z((2, 3, 3, 3)), _z((1, 3, 2))
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_project_backward(3, vol, rot, None, out, vol, gR, gS1)
    for args in [(vol, rot, None, out, _z((2, 8, 8, 4), True), gR, gS1),
                 (vol, rot, None, out, vol, _z((1, 3, 3, 3)), gS1),
                 (vol, rot, None, out, vol, gR, _z((2, 3, 2))),
                 (vol, rot, sh, _z((2, 3, 8, 4), True), vol, gR, gS1)]:
        with pytest.raises(ValueError, match="must have shape"):
            tp.tp_project_backward(3, *args)
        with pytest.raises(ValueError, match="must have shape"):
            tp.tp_project_backward_ws(3, *args, None)
        with pytest.raises(ValueError, match="must have shape"):
            tp.tp_project_backward_fused(3, *args)


def test_binding_checks_insertion_and_padding_shapes():
    proj, w = _z((2, 3, 8, 5), True), _z((2, 3, 8, 5))
    rot = _z((1, 3, 3, 3))
    vol, wvol = _z((2, 12, 12, 7), True), _z((2, 12, 12, 7))
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_backproject_2d_to_3d(proj, w, rot, None, vol, wvol, 12)
    with pytest.raises(TypeError, match="CUDA"):                 # weights only: no data image
        tp.tp_backproject_2d_to_3d(None, w, rot, None, None, wvol, 12)
    for args in [(proj, _z((2, 3, 8, 4)), rot, None, vol, wvol, 12),
                 (proj, w, rot, None, vol, wvol, 10),             # Dv disagrees with the outputs
                 (proj, w, rot, None, vol, _z((1, 12, 12, 7)), 12),
                 (proj, w, _z((1, 2, 3, 3)), None, vol, wvol, 12)]:
        with pytest.raises(ValueError, match="must have shape"):
            tp.tp_backproject_2d_to_3d(*args)
    img, wimg = _z((2, 12, 7), True), _z((2, 12, 7))
    rot2 = _z((2, 3, 2, 2))
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_backproject_2d_to_2d(proj, w, rot2, None, img, wimg, 12)
    with pytest.raises(ValueError, match="must have shape"):
        tp.tp_backproject_2d_to_2d(proj, w, rot2, None, vol, wimg, 12)
    # backward of the insertion
    gR = _z((1, 3, 3, 3))
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_backproject_backward(3, proj, w, rot, None, vol, wvol, proj, w, gR, None)
    with pytest.raises(ValueError, match="must have shape"):
        tp.tp_backproject_backward(3, proj, w, rot, None, vol, _z((2, 12, 12, 6)), proj, w, gR, None)
    with pytest.raises(ValueError, match="must have shape"):
        tp.tp_backproject_backward(3, proj, w, rot, None, vol, wvol, _z((2, 4, 8, 5), True), w, gR,
                                   None)
    with pytest.raises(ValueError, match="image size"):
        tp.tp_backproject_backward(3, None, None, rot, None, vol, wvol, None, None, gR, None)
    # padding: out is factor * D on every axis, and the adjoint the other way round
    v, X = _z((1, 6, 6, 6)), _z((1, 12, 12, 12))
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_pad_volume(3, v, 2, X)
    with pytest.raises(TypeError, match="CUDA"):
        tp.tp_crop_volume(3, X, 2, v)
    with pytest.raises(ValueError, match="must have shape"):
        tp.tp_pad_volume(3, v, 2, _z((1, 12, 12, 10)))
    with pytest.raises(ValueError, match="must have shape"):
        tp.tp_crop_volume(3, _z((1, 12, 12, 12)), 3, v)
    with pytest.raises(ValueError, match="must have shape"):
        tp.tp_pad_volume(2, _z((1, 6, 5)), 2, _z((1, 12, 10)))


def test_header_is_plain_c_and_links(tmp_path):
    """include/tp.h compiles as strict C99 and a C program links against libtp.so with every
    declared function referenced; the calls it makes return before any CUDA call (argument
    validation, status strings, workspace sizes), so no GPU is needed."""
    import os

    pkg = os.path.dirname(tp.LIB_PATH)
    refs = ",\n    ".join(f"(void (*)(void)){name}" for name in tp.header_symbols())
    (tmp_path / "t.c").write_text(f"""#include <stdio.h>
#include "tp.h"
static void (*const every_entry[])(void) = {{
    {refs}
}};
int main(void) {{
    tp_opts o = {{TP_CUBIC, TP_LAYOUT_CENTERED, 1.0f, -1.0f}};
    printf("%s\\n", tp_status_string(TP_ERR_SHAPE));
    printf("%d\\n", (int)tp_project_3d_to_2d(NULL, 1, 7, NULL, 1, 1, NULL, 1, NULL, 8, &o, NULL));
    printf("%d\\n", (int)tp_project_2d_to_2d(NULL, 1, 8, NULL, 1, 1, NULL, 1, NULL, 8, NULL, NULL));
    printf("%zu\\n", tp_workspace_size(3, 1, 128, &o));
    printf("%d\\n", (int)(sizeof every_entry / sizeof every_entry[0]));
    return 0;
}}
""")
    exe = tmp_path / "t"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(os.path.dirname(pkg), "include"), str(tmp_path / "t.c"),
                    "-L", pkg, "-ltp", f"-Wl,-rpath,{pkg}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0].startswith("TP_ERR_SHAPE")
    assert out[1] == "2"                    # odd volume box
    assert out[2] == "1"                    # valid sizes, one item, NULL pointers: TP_ERR_NULL
    assert out[3] == str(128 * 8961 * 4 * 8)
    assert out[4] == str(len(tp.header_symbols()))


def test_peaks_library_exports_and_validates(tmp_path):
    """libtp_peaks.so (include/tp_peaks.h) exports what its header declares, the header is
    plain C99, and bad arguments are refused on the host (status 1) before any CUDA call."""
    import os
    import re

    from back_projection_fourier_b300 import peaks

    hdr = os.path.join(os.path.dirname(os.path.dirname(tp.LIB_PATH)), "include", "tp_peaks.h")
    names = sorted(set(re.findall(r"^\s*(?:int|size_t)\s+(tp_peak_\w+)\s*\(", open(hdr).read(), re.M)))
    assert names == ["tp_peak_run", "tp_peak_scratch_bytes"]
    dyn = subprocess.run(["nm", "-D", "--defined-only", str(peaks.LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in dyn.splitlines() if " T " in line}
    assert set(names) <= exported
    P = peaks._lib()
    need = P.tp_peak_scratch_bytes()
    assert need >= (8 << 20)
    o, b = ctypes.c_double(), ctypes.c_double()
    for kind, ptr, size, ctas, iters in [(0, None, need, 1, 1),          # NULL scratch
                                         (0, FAKE, need - 1, 1, 1),      # too small
                                         (0, FAKE + 16, need, 1, 1),     # not 256-aligned
                                         (0, FAKE, need, 0, 1),          # no CTAs
                                         (0, FAKE, need, 1, 0),          # no iterations
                                         (99, FAKE, need, 1, 1)]:        # unknown kind
        assert P.tp_peak_run(kind, ptr, size, ctas, iters, None, ctypes.byref(o), ctypes.byref(b)) == 1
    pkg = os.path.dirname(peaks.LIB_PATH)
    (tmp_path / "p.c").write_text("""#include <stdio.h>
#include "tp_peaks.h"
int main(void) {
    double o = 0, b = 0;
    printf("%d\\n", tp_peak_run(TP_PEAK_FMA, NULL, tp_peak_scratch_bytes(), 1, 1, NULL, &o, &b));
    return 0;
}
""")
    exe = tmp_path / "p"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.dirname(hdr), str(tmp_path / "p.c"), "-L", pkg, "-ltp_peaks",
                    f"-Wl,-rpath,{pkg}", "-o", str(exe)], check=True)
    assert subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout == "1\n"
