// kernels.h -- internal launchers of libtp.so (C++ only; the public ABI is include/tp.h).
#pragma once

#include <cuda_runtime.h>

#include "tp_device.cuh"

namespace tp {

// Each launcher enqueues on `stream` and returns cudaGetLastError().  Arguments have been
// validated by the ABI layer; `sms` is the device's SM count (grid sizing).
// `grouped` (3D only; NULL = read rec directly): the grouped copy of rec written by
// launch_expand_groups, read by the gathers' fast path.
cudaError_t launch_project(int ndim, int interp, const Geom& g, const void* rec,
                           const float* rot, const float* shift, void* out, int sms,
                           cudaStream_t stream, const void* grouped = nullptr);

// fused: the volume, rotation and shift gradients in one pass of the tile scatter where that
// kernel applies (3D cubic, every output wanted); elsewhere the two kernels as without it.
cudaError_t launch_backward(int ndim, int interp, const Geom& g, const void* rec,
                            const float* rot, const float* shift, const void* grad_out,
                            void* grad_rec, float* grad_rot, float* grad_shift, int sms,
                            cudaStream_t stream, const void* grouped = nullptr,
                            bool fused = false);

// Grouped copy of the volumes for the gathers: n_rec * Dv * g.gplane groups of NT complex taps,
// NT = 4 (cubic) / 2 (linear); see expand_groups_kernel.
cudaError_t launch_expand_groups(int interp, const Geom& g, const void* rec, void* grouped, int sms,
                                 cudaStream_t stream);

cudaError_t launch_backproject(int ndim, int interp, const Geom& g, const void* proj,
                               const float* weights, const float* rot, const float* shift,
                               void* vol_out, float* wvol_out, int sms, cudaStream_t stream);

// Weight-volume part of the back-projection's backward (see tp_backproject_backward).
cudaError_t launch_weights_grad(int ndim, int interp, const Geom& g, const float* grad_wvol,
                                const float* weights, const float* rot, float* grad_weights,
                                float* grad_rot, int sms, cudaStream_t stream);

// Real-space zero padding by an integer factor with the centre moved to index 0, and its
// adjoint (pad.cu).  vol / out are [n][D]^ndim and [n][factor*D]^ndim fp32.
cudaError_t launch_pad(int ndim, const float* vol, int n, int D, int factor, float* out, int sms,
                       cudaStream_t stream);
cudaError_t launch_crop(int ndim, const float* padded, int n, int D, int factor, float* out,
                        int sms, cudaStream_t stream);

}  // namespace tp
