"""B300-native differentiable Fourier-slice projection.

The compute lives in ``libtp.so`` (CUDA, sm_103a) behind the C ABI declared in
``include/tp.h``; ``back_projection_fourier_b300.tp`` is its thin Python binding and
``back_projection_fourier_b300.synth`` draws seeded synthetic inputs.  Importing the
package itself loads nothing native; importing ``.tp`` does, and fails loudly when the
library is missing.
"""
