"""The pins must reject a broken oracle: the Python half (padding, the insertion's backward,
the on-the-fly pipeline's backward, the exact projection).

Each case copies the oracle package, plants one plausible mistake in oracle.py and runs the
pins that cover those functions in a subprocess started inside the copy, so that `import
oracle` finds the mutated package first.  The pins pass on the real oracle and must fail on
every mutant.  (test_oracle_mutants.py does the same for oracle.c.)
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = [os.path.join(ROOT, "tests", f)
        for f in ("test_oracle_pins.py", "test_oracle_oversampling.py", "test_accuracy_metrics.py")]

MUTANTS = {
    "pad_off_centre": ("padded = np.pad(vol, [(0, 0)] + [(m, m)] * k)",
                       "padded = np.pad(vol, [(0, 0)] + [(m + 1, m - 1)] * k)"),
    "pad_not_shifted": ("    return np.fft.ifftshift(padded, axes=tuple(range(1, k + 1)))",
                        "    return padded"),
    "insertion_grad_proj_drops_shift": ("g_proj = project(ndim, grad_vol, rot, shift, Do=Do, **kw)",
                                        "g_proj = project(ndim, grad_vol, rot, None, Do=Do, **kw)"),
    "insertion_grad_weights_shifted": ("g_w = project(ndim, gw, rot, None, Do=Do, **kw).real",
                                       "g_w = project(ndim, gw, rot, shift, Do=Do, **kw).real"),
    "pipeline_backward_drops_box_volume": (
        "g_x = np.real(np.fft.ifftn(full, axes=axes)) * float(P) ** ndim",
        "g_x = np.real(np.fft.ifftn(full, axes=axes))"),
    "exact_projection_sign": (
        "E = [np.exp(-2j * np.pi * np.outer(c[a], m) / D) for a in range(ndim)]",
        "E = [np.exp(2j * np.pi * np.outer(c[a], m) / D) for a in range(ndim)]"),
    "exact_projection_uncentred": (
        "    m = np.arange(D) - D // 2\n    out = np.zeros((n, n_pose, Do, Ho), np.complex128)",
        "    m = np.arange(D)\n    out = np.zeros((n, n_pose, Do, Ho), np.complex128)"),
}


def _run_pins(source, tmp_path):
    """Copy the oracle package with `source` as its oracle.py and run the pins against it."""
    pkg = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg,
                    ignore=shutil.ignore_patterns("*.so", "*.so.*", "__pycache__"))
    (pkg / "oracle.py").write_text(source)
    env = dict(os.environ, PYTHONPATH=f"{tmp_path}{os.pathsep}{ROOT}", OMP_NUM_THREADS="2")
    env.pop("TP_ORACLE_LIB", None)
    probe = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"],
                           cwd=tmp_path, env=env, capture_output=True, text=True, timeout=120)
    assert probe.stdout.strip().startswith(str(tmp_path)), probe.stdout + probe.stderr
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           *PINS], cwd=tmp_path, env=env, capture_output=True, text=True,
                          timeout=900)


def test_unmutated_copy_passes_the_pins(tmp_path):
    """Control: the copied package with the oracle's own source passes the same pins."""
    r = _run_pins(open(os.path.join(ROOT, "oracle", "oracle.py")).read(), tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_python_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "oracle.py")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    r = _run_pins(src.replace(old, new), tmp_path)
    assert r.returncode != 0, f"pins accepted mutant {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
