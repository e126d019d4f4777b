"""fp64 CPU oracle for differentiable Fourier-slice projection.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product path never imports this package.
"""
from .oracle import (  # noqa: F401
    build,
    project,
    project_samples,
    backproject,
    project_backward,
    backproject_backward,
    pad_volume,
    crop_volume,
    oversampled_spectrum,
    project_real,
    project_real_backward,
    exact_projection,
    axis_weights,
    LINEAR,
    CUBIC,
    FFTW,
    CENTERED,
)
