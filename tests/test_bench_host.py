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


def test_relevant_roofline_arithmetic():
    """T_roof of each kernel is the largest of its measured-peak times; frac = T_roof / time.
    Fake peaks and times, checked by hand: the forward's 6490 x 16 x 64 taps of 8 B at
    1e13 B/s take 5.3 ms of L1 time against 0.1 ms of FP32 and HBM time."""
    wl = synth.make_workload(bench.DEFAULT_WORKLOAD, B=16, with_grad=False)
    taps = 6490 * 16 * 64
    pk = {"sms": 148, "l1_load": {"bytes_per_s": 1e13}, "l1_gather8": {"ops_per_s": 1e11},
          "l1_gather32": {"ops_per_s": 2e11}, "smem_rmw": {"ops_per_s": 2e12},
          "smem_rmw_random": {"ops_per_s": 1e12}, "smem_red": {"ops_per_s": 5e11},
          "l2_red": {"ops_per_s": 2e11}, "fma": {"ops_per_s": 7e13}}
    kms = {"forward": 10.0, "grad_pose": 20.0, "grad_volume": 40.0}
    hbm = bench.hbm_bytes(wl)
    r = bench.relevant_roofline(wl, kms, hbm, 6400.0, pk, 2000.0)
    assert r["forward"]["bound"] == "l1_load"
    assert r["forward"]["t_roof_ms"] == pytest.approx(1e3 * taps * 8 / 1e13)
    assert r["forward"]["frac"] == pytest.approx(taps * 8 / 1e13 / 10e-3)
    assert r["forward"]["row_gather_frac"] == pytest.approx(taps / 4 / 2e11 / 10e-3)
    assert r["grad_volume"]["bound"] == "smem_rmw"
    assert r["grad_volume"]["t_roof_ms"] == pytest.approx(1e3 * taps / 2e12)
    assert r["per_sm_per_clk"]["l1_load_B"] == pytest.approx(1e13 / (2000e6 * 148))
    assert bench.relevant_roofline(wl, kms, hbm, 6400.0, None, 2000.0) is None


def test_shared_atomic_context_of_the_linear_insertion():
    """The linear 3D scatter adds each of a pixel's 8 taps with shared float atomics: 3 per tap
    with the weights (data re, im and weight).  Its context fraction sets those atomics
    against the shared atomic rate; the bound stays the read-modify-write one (1.5 per tap).
    The cubic tile scatter issues no shared atomics and has no such figure."""
    wl = synth.make_workload("insert3d_d128_b16384", B=16, interp=synth.LINEAR, with_grad=False)
    taps = 6490 * 16 * 8
    pk = {"sms": 148, "l1_load": {"bytes_per_s": 1e13}, "l1_gather8": {"ops_per_s": 1e11},
          "l1_gather32": {"ops_per_s": 2e11}, "smem_rmw": {"ops_per_s": 2e12},
          "smem_rmw_random": {"ops_per_s": 1e12}, "smem_red": {"ops_per_s": 5e11},
          "l2_red": {"ops_per_s": 2e11}, "fma": {"ops_per_s": 7e13}}
    hbm = {"insertion": 1e6}
    r = bench.relevant_roofline(wl, {"insertion": 2.0}, hbm, 6400.0, pk, 2000.0)
    assert r["insertion"]["bound"] == "smem_rmw"
    assert r["insertion"]["t_roof_ms"] == pytest.approx(1e3 * (taps * 3 // 2) / 2e12)
    assert r["insertion"]["smem_red_frac"] == pytest.approx(3 * taps / 5e11 / 2e-3)
    wc = synth.make_workload("insert3d_d128_b16384", B=16, interp=synth.CUBIC, with_grad=False)
    rc = bench.relevant_roofline(wc, {"insertion": 2.0}, hbm, 6400.0, pk, 2000.0)
    assert "smem_red_frac" not in rc["insertion"]


def test_one_pass_backward_bytes_and_label():
    """The one-pass backward reads the upstream gradient and the poses once, reads the volume
    and writes its gradient: per projection 66 560 + 88 B, per launch twice the volume.  Its
    step is labelled in the config that both arms share."""
    wl = synth.make_workload(bench.DEFAULT_WORKLOAD, B=16, with_grad=False)
    b = bench.hbm_bytes(wl)
    vol = 128 * 128 * 65 * 8
    assert b["backward_fused"] == 16 * (66560 + 88) + 2 * vol
    assert "one-pass" in bench.workload_config(wl, "l2", True)["step"]
    assert "one-pass" not in bench.workload_config(wl, "l2")["step"]
