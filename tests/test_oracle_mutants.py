"""The pins must reject a broken oracle.

Each case copies oracle.c, plants one plausible mistake (a transposed operand, a dropped
conjugation, a wrong sign, a wrong index or constant), compiles the copy on the CPU and
runs the pin suite against it in a subprocess.  The pins pass on the real oracle
(test_oracle_pins.py) and must fail on every mutant.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "rotation_transposed": ("px.c[a] += g->o * R[a * k + b] * q[b]", "px.c[a] += g->o * R[b * k + a] * q[b]"),
    "oversampling_dropped": ("px.c[a] += g->o * R[a * k + b] * q[b]", "px.c[a] += R[a * k + b] * q[b]"),
    "mirror_read_not_conjugated": ("val = mirror ? conj(V[off]) : V[off];", "val = V[off];"),
    "mirror_keeps_y": ("        ty = -ty;\n", ""),
    "mirror_scatter_not_conjugated": ("R[off] += mirror ? conj(w * val) : w * val;", "R[off] += w * val;"),
    "phase_sign": ("cexp(-2.0 * M_PI * I * turns)", "cexp(2.0 * M_PI * I * turns)"),
    "phase_uses_rec_box": ("/ (double)g->Do;\n        px.phase", "/ (double)g->Dv;\n        px.phase"),
    "backproject_phase_not_conjugated": ("proj[e] * conj(px.phase)", "proj[e] * px.phase"),
    "keys_a": ("const double a = -0.5;\n    double u = fabs(d);\n", "const double a = -0.75;\n    double u = fabs(d);\n"),
    "cubic_taps_off_by_one": ("long first = interp == ORC_LINEAR ? b : b - 1;", "long first = interp == ORC_LINEAR ? b : b - 2;"),
    "centered_index": ("if (layout == ORC_CENTERED) return f + D / 2;", "if (layout == ORC_CENTERED) return f + D / 2 - 1;"),
    "x_range": ("if (tx > g->Dv / 2) return -1;", "if (tx >= g->Dv / 2) return -1;"),
    "cutoff_strict": ("<= g->rc2;", "< g->rc2;"),
    "dv_y_uses_x_derivative": ("dv[1] += wz[a] * dwy[b] * wx[k] * val;", "dv[1] += wz[a] * wy[b] * dwx[k] * val;"),
    "grad_rot_transposed": ("item_grot[it * k * k + a * k + b]", "item_grot[it * k * k + b * k + a]"),
    "grad_shift_sign": ("(-2.0 * M_PI * I * q[b] / (double)g.Do)", "(2.0 * M_PI * I * q[b] / (double)g.Do)"),
    "weights_ignore_pixel_weight": ("if (W) W[off] += w * wt;", "if (W) W[off] += w;"),
    "linear_derivative_sign": ("if (d >= 0.0 && d < 1.0) return -1.0;", "if (d >= 0.0 && d < 1.0) return 1.0;"),
    "cubic_derivative_outer": ("return s * (3.0 * a * u * u - 10.0 * a * u + 8.0 * a);",
                               "return s * (3.0 * a * u * u - 10.0 * a * u + 7.0 * a);"),
    "x0_plane_mirrored": ("*mirror = tx < 0;", "*mirror = tx <= 0;"),
    "mirror_keeps_z": ("        tz = -tz;\n    }", "    }"),
    "shift_axes_swapped": ("(double)px.kx * s[0] + (double)px.ky * s[1]",
                           "(double)px.kx * s[1] + (double)px.ky * s[0]"),
    "fftw_nyquist_row_positive": ("return i < D / 2 ? i : i - D;", "return i <= D / 2 ? i : i - D;"),
    "default_cutoff_uses_rec_box": ("cutoff = cutoff < 0.0 ? 0.5 * Do : cutoff;",
                                    "cutoff = cutoff < 0.0 ? 0.5 * Dv : cutoff;"),
    "grad_rot_drops_oversampling": ("+= g.o * q[b] * creal(conj(gp) * dv[a]);",
                                    "+= q[b] * creal(conj(gp) * dv[a]);"),
    "weights_skip_mirrored": ("if (W) W[off] += w * wt;", "if (W && !mirror) W[off] += w * wt;"),
    "linear_tent_curved": ("return u < 1.0 ? 1.0 - u : 0.0;", "return u < 1.0 ? 1.0 - u * u : 0.0;"),
    "dv_z_conjugated": ("dv[2] += dwz[a] * wy[b] * wx[k] * val;",
                        "dv[2] += dwz[a] * wy[b] * wx[k] * conj(val);"),
    "cubic_inner_perturbed": ("if (u <= 1.0) return (a + 2.0) * u * u * u - (a + 3.0) * u * u + 1.0;",
                              "if (u <= 1.0) return (a + 2.0) * u * u * u - (a + 3.0) * u * u + 1.0"
                              " + 0.01 * u * (1.0 - u);"),
}


def _run_pins(source, tmp_path):
    """Compile `source` as the oracle library and run the pin suite against it."""
    mutant_c = tmp_path / "mutant.c"
    mutant_so = tmp_path / "libmutant.so"
    mutant_c.write_text(source)
    subprocess.run(["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC",
                    "-shared", "-o", str(mutant_so), str(mutant_c), "-lm"], check=True)
    env = dict(os.environ, TP_ORACLE_LIB=str(mutant_so), OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unmutated_copy_passes_the_pins(tmp_path):
    """Control: the same route with the oracle's own source passes, so a failure below is
    the planted mistake's doing and not the route's."""
    r = _run_pins(open(SRC).read(), tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    r = _run_pins(src.replace(old, new), tmp_path)
    assert r.returncode != 0, f"pins accepted mutant {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
