"""Host-side arithmetic of the benchmark (CPU): the counts its roofline figures rest on, and
the hash that decides whether stored counter captures still describe the kernels."""
import numpy as np
import pytest

import bench
from back_projection_fourier_b300 import synth


@pytest.mark.parametrize("D,count", [(32, 414), (64, 1636), (128, 6490), (256, 25844)])
def test_kept_pixels_match_enumeration(D, count):
    """Pixels of the half plane with kx^2 + ky^2 <= (D/2)^2, enumerated one by one."""
    brute = sum(1 for ky in range(-D // 2, D // 2) for kx in range(D // 2 + 1)
                if kx * kx + ky * ky <= (D // 2) ** 2)
    assert brute == count
    wl = synth.Workload("t", 0, 3, "fwdbwd", synth.CUBIC, D, 1, D / 2)
    assert bench.kept_pixels(wl) == count


def test_algorithmic_bytes_of_the_headline_step():
    """Per projection: a 128 x 65 complex64 image (66 560 B) and a pose of 9 + 2 floats (44 B);
    per launch the 128 x 128 x 65 complex64 volume (8.52 MB)."""
    wl = synth.make_workload(bench.DEFAULT_WORKLOAD, B=16, with_grad=False)
    b = bench.hbm_bytes(wl)
    vol = 128 * 128 * 65 * 8
    assert b["forward"] == 16 * (66560 + 44) + vol
    assert b["grad_pose"] == 16 * (66560 + 88) + vol
    assert b["grad_volume"] == 16 * (66560 + 44) + vol
    assert bench.metric_for(wl) == bench.METRIC


def test_kernel_hash_ignores_comments_only(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ["k.cu"])
    src.write_text("int f(int x) {\n    return x + 1;\n}\n")
    h0 = bench.kernel_hash()
    src.write_text("// the successor\nint f(int x) {  // of x\n\n    return x + 1;\n}\n")
    assert bench.kernel_hash() == h0
    src.write_text("int f(int x) {\n    return x + 2;\n}\n")
    assert bench.kernel_hash() != h0
