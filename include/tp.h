/*
 * tp.h -- C ABI of libtp.so: differentiable Fourier-slice projection on one NVIDIA B300
 * (sm_103a).
 *
 * The operations are those of the torch-projectors paper summaries (gist.science):
 *   - Method section, operations list: 3D->2D forward projection (central slice theorem),
 *     2D->3D backward projection (accumulation into a 3D volume), 2D->2D forward (rotation
 *     of 2D Fourier data) and 2D->2D backward (accumulation into a 2D reconstruction);
 *     every operation supports rotation, translation by phase modulation and weight
 *     accumulation ("useful for CTF correction");
 *   - Method section, RFFT bullet: data are PyTorch/FFTW rfft half spectra;
 *   - Method section, interpolation bullet: linear (bilinear / trilinear) or cubic
 *     Catmull-Rom (Keys kernel, a = -0.5);
 *   - Method section, Friedel bullet: F(-k) = conj F(k) of real functions, handled without
 *     double counting on the zero-frequency axis;
 *   - Method section, differentiation bullet: gradients for the inputs, the rotation
 *     matrices and the shifts, computed without stored intermediates;
 *   - Dutch page, Method section: shifts are applied by Fourier phase modulation.
 *
 * Definition (the pages give no formulas; this is the plainest reading they support):
 *   Output pixel (i, j) of an image of box Do has kx = j in [0, Do/2] and ky = the frequency
 *   of row i.  It is kept iff kx^2 + ky^2 <= rc^2, else it is 0.  A kept pixel samples the
 *   reconstruction at c = o * R * q, q = (kx, ky, 0) (3D) or (kx, ky) (2D), R row-major
 *   with vector order (x, y, z) <-> tensor axes (last, middle, first):
 *       v(c) = sum_t w(c - t) V_ext(t)        (separable weights, taps floor(c)+{0,1} for
 *                                              linear, floor(c)+{-1,0,1,2} for cubic)
 *       V_ext(t) = V[t] if t_x >= 0, conj(V[-t]) if t_x < 0, and 0 where the stored
 *                  frequency lies outside x in [0, Dv/2], y, z in [-Dv/2, Dv/2 - 1]
 *       y = v(c) * exp(-2 pi i (kx sx + ky sy) / Do)
 *   Back-projection is the exact real-linear transpose of this map under
 *   <a, b> = Re sum conj(a) b; the weight accumulation scatters a real per-pixel weight
 *   with the same interpolation weights (no phase, no conjugation).
 *
 * Layout (all arrays C-contiguous; complex = interleaved (re, im) fp32, 8-byte aligned):
 *   3D reconstruction  [n_rec][Dv][Dv][Dv/2+1]   axes (z, y, x); x is the half axis
 *   2D reconstruction  [n_rec][Dv][Dv/2+1]       axes (y, x)
 *   images             [n_rec][n_pose][Do][Do/2+1]
 *   rot                [n_rot][n_pose][k][k] fp32, k = 3 (3D) or 2 (2D), n_rot in {1, n_rec};
 *                      n_rot = 1 shares one set of poses between all reconstructions
 *   shift              [n_sh][n_pose][2] fp32 (sx, sy) in image pixels, n_sh in {1, n_rec};
 *                      NULL means no shift
 *   weights            fp32 with the image shape; NULL means weight 1
 *   Full (non-half) axes are in FFTW order (index i holds i for i < D/2, else i - D) or
 *   centered order (index i holds i - D/2), chosen by tp_opts.layout for every array.
 *
 * Ownership and execution: every pointer is a caller-owned DEVICE pointer on the current
 * CUDA device.  The library allocates no device memory and keeps no state between calls.
 * Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and
 * the call returns without synchronising.  Outputs must not alias inputs.
 *
 * Errors: arguments are checked on the host before anything is enqueued; a rejected call
 * enqueues nothing.  TP_ERR_CUDA reports a launch error (cudaGetLastError after the
 * launches).  Errors of the asynchronous execution itself surface at the caller's next
 * synchronisation.  No exception crosses the ABI and no kernel traps.
 *
 * Limits: Dv, Do even, 2 <= D; 3D boxes up to 1024, 2D boxes up to 32768; n_rec, n_pose,
 * n_rot, n_sh >= 0; n_rec * n_pose images of Do*(Do/2+1) pixels each (64-bit offsets).
 */
#ifndef TP_H
#define TP_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tp_status {
    TP_OK = 0,
    TP_ERR_NULL = 1,  /* a required pointer is NULL */
    TP_ERR_SHAPE = 2, /* a size is negative, odd, too large, or n_rot / n_sh mismatch */
    TP_ERR_VALUE = 3, /* bad interp / layout, non-positive or non-finite oversampling,
                         non-finite cutoff, ndim not 2 or 3, accumulate not 0 or 1 */
    TP_ERR_CUDA = 4   /* a CUDA launch or memset failed */
} tp_status;

enum { TP_LINEAR = 0, TP_CUBIC = 1 };
enum { TP_LAYOUT_FFTW = 0, TP_LAYOUT_CENTERED = 1 };

/* Options shared by every call; a NULL tp_opts* means
 * { TP_CUBIC, TP_LAYOUT_CENTERED, 1.0f, -1.0f }. */
typedef struct tp_opts {
    int interp;         /* TP_LINEAR or TP_CUBIC */
    int layout;         /* TP_LAYOUT_FFTW or TP_LAYOUT_CENTERED */
    float oversampling; /* o > 0: sample coordinate scale (Dv = o * Do for a padded volume) */
    float cutoff;       /* rc in image frequency units; < 0 means Do / 2 */
} tp_opts;

/* 3D->2D forward projection (central slices).  Operations list, "3D -> 2D forward".
 *   vol   [n_rec][Dv][Dv][Dv/2+1] complex (read)
 *   out   [n_rec][n_pose][Do][Do/2+1] complex (overwritten; pixels beyond rc are 0) */
tp_status tp_project_3d_to_2d(const void* vol, int n_rec, int Dv, const float* rot, int n_rot,
                              int n_pose, const float* shift, int n_sh, void* out, int Do,
                              const tp_opts* opts, void* stream);

/* 2D->3D back-projection (insertion), the adjoint of tp_project_3d_to_2d, plus the weight
 * accumulation.  Operations list, "2D -> 3D backward".
 *   proj      [n_rec][n_pose][Do][Do/2+1] complex (read); data are multiplied by
 *             conj(phase) and scattered with the transpose of the forward weights
 *   weights   fp32 image-shaped per-pixel weights (read; NULL = 1)
 *   vol_out   [n_rec][Dv][Dv][Dv/2+1] complex (NULL = skip the data)
 *   wvol_out  [n_rec][Dv][Dv][Dv/2+1] fp32 (NULL = skip the weights)
 *   accumulate 1 adds into the outputs; 0 zeroes them first */
tp_status tp_backproject_2d_to_3d(const void* proj, const float* weights, int n_rec, int Do,
                                  const float* rot, int n_rot, int n_pose, const float* shift,
                                  int n_sh, void* vol_out, float* wvol_out, int Dv,
                                  int accumulate, const tp_opts* opts, void* stream);

/* 2D->2D forward (rotation of 2D Fourier data).  Operations list, "2D -> 2D forward".
 *   img   [n_rec][Dv][Dv/2+1] complex (read); rot [n_rot][n_pose][2][2]
 *   out   [n_rec][n_pose][Do][Do/2+1] complex (overwritten) */
tp_status tp_project_2d_to_2d(const void* img, int n_rec, int Dv, const float* rot, int n_rot,
                              int n_pose, const float* shift, int n_sh, void* out, int Do,
                              const tp_opts* opts, void* stream);

/* 2D->2D backward (accumulation into a 2D reconstruction), the adjoint of
 * tp_project_2d_to_2d, plus the weight accumulation.  Operations list, "2D -> 2D backward".
 *   img_out [n_rec][Dv][Dv/2+1] complex, wimg_out fp32 (each NULL = skip); other arguments
 *   as in tp_backproject_2d_to_3d */
tp_status tp_backproject_2d_to_2d(const void* proj, const float* weights, int n_rec, int Do,
                                  const float* rot, int n_rot, int n_pose, const float* shift,
                                  int n_sh, void* img_out, float* wimg_out, int Dv,
                                  int accumulate, const tp_opts* opts, void* stream);

/* Fused backward of tp_project_3d_to_2d (ndim = 3) or tp_project_2d_to_2d (ndim = 2) for
 * the upstream gradient grad_out = dL/dRe(out) + i dL/dIm(out).  Differentiation bullet.
 *   grad_rec   reconstruction-shaped complex: the transpose of the projection applied to
 *              grad_out (overwritten; NULL = skip)
 *   grad_rot   [n_rot][n_pose][k][k] fp32: dL/dR[a][b] = sum o q_b Re(conj(g') dv/dc_a),
 *              g' = grad_out * conj(phase); summed over reconstructions when n_rot = 1;
 *              the z column (3D) is 0 because q_z = 0 (overwritten; NULL = skip)
 *   grad_shift [n_sh][n_pose][2] fp32: dL/ds = sum Re(conj(grad_out) y (-2 pi i k / Do)),
 *              summed over reconstructions when n_sh = 1 (overwritten; NULL = skip).
 *              When shift is NULL, n_sh is ignored and grad_shift, if given, is
 *              [1][n_pose][2] and is set to 0 */
tp_status tp_project_backward(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                              int n_rot, int n_pose, const float* shift, int n_sh,
                              const void* grad_out, int Do, void* grad_rec, float* grad_rot,
                              float* grad_shift, const tp_opts* opts, void* stream);

/* tp_project_backward in one kernel pass.  The pages' CUDA backend computes each operation in
 * a single kernel call without stored intermediates (nl page, Belangrijkste Bijdragen, item 1;
 * Methodologie, Differentiatie bullet).  For ndim = 3 with cubic interpolation, when grad_rec
 * and grad_rot or grad_shift are requested, one kernel reads grad_out once and emits the
 * volume, rotation and shift gradients together: the lanes of the volume-gradient scatter also
 * read the volume at their taps and sum the pose terms.  In every other case the call is
 * tp_project_backward.  Arguments, layouts, results and errors as tp_project_backward; the
 * results agree with it to rounding (the summation order differs).  On B300 the one-pass
 * kernel is slower than tp_project_backward's two kernels: the extra per-tap work goes to a
 * kernel that is already bound by instruction issue and by the shared-memory pipe. */
tp_status tp_project_backward_fused(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                                    int n_rot, int n_pose, const float* shift, int n_sh,
                                    const void* grad_out, int Do, void* grad_rec, float* grad_rot,
                                    float* grad_shift, const tp_opts* opts, void* stream);

/* Optional workspace of the 3D gathers.  tp_project_3d_to_2d_ws and tp_project_backward_ws
 * are tp_project_3d_to_2d and tp_project_backward with a caller-owned device workspace; the
 * results are the same (the same taps, weights and summation order).  The call first writes
 * a grouped copy of the volumes into the workspace -- for every row and every start
 * x = -(NT-1) .. Dv/2 the NT taps x .. x+NT-1 of that row, NT = 4 (cubic) or 2 (linear),
 * zeros past x = Dv/2 and the conjugate Friedel mirror left of x = 0 -- and the gathers then
 * read each row of taps with one aligned vector load instead of several unaligned ones, also
 * for the pixels whose taps straddle the x = 0 plane.  Layout: per volume Dv planes of P
 * groups, a plane holding Dv rows of R groups, a group NT complex values; R = Dv/2 + NT
 * padded up to 2 modulo 16/NT and P = Dv * R padded up to 1 modulo 16/NT (padding that
 * spreads the rows a warp loads over the L1 banks).  It costs about NT times the volumes'
 * memory and one pass over them per call; it pays when many poses share the volumes.
 * This is a B300 layout choice; the pages have no counterpart.
 *
 * tp_workspace_size returns the bytes needed (n_rec * Dv * P * NT * 8), or 0
 * when the workspace would not be used (ndim = 2, invalid sizes or options, or NT times one
 * volume's elements >= 2^31).  A NULL workspace runs the plain path; so does any workspace
 * when tp_workspace_size is 0 for these arguments (the workspace is then ignored).
 * Errors, in addition to the plain call's: TP_ERR_SHAPE when a non-NULL workspace is
 * smaller than tp_workspace_size, TP_ERR_VALUE when it is not 32-byte aligned.  The workspace must
 * not overlap any argument; its contents are scratch (undefined after the call), and two
 * calls in flight at once need two workspaces. */
size_t tp_workspace_size(int ndim, int n_rec, int Dv, const tp_opts* opts);

tp_status tp_project_3d_to_2d_ws(const void* vol, int n_rec, int Dv, const float* rot, int n_rot,
                                 int n_pose, const float* shift, int n_sh, void* out, int Do,
                                 void* workspace, size_t workspace_bytes, const tp_opts* opts,
                                 void* stream);

tp_status tp_project_backward_ws(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                                 int n_rot, int n_pose, const float* shift, int n_sh,
                                 const void* grad_out, int Do, void* grad_rec, float* grad_rot,
                                 float* grad_shift, void* workspace, size_t workspace_bytes,
                                 const tp_opts* opts, void* stream);

/* tp_project_3d_to_2d with the workspace path, for callers that cannot allocate device
 * memory and cannot pass a workspace: code whose device memory belongs entirely to another
 * allocator (a framework's caching allocator, a fixed-budget memory pool) and code on a
 * latency-critical path that must not call cudaMalloc, which can synchronise the device.
 * The pages have no counterpart; this is a property of the library, not of the method.
 *   Arguments, layouts and results as tp_project_3d_to_2d.  The grouped copy of the volumes
 *   goes into a fixed scratch array of 36704256 bytes (one Dv = 128 volume with cubic taps)
 *   that the library holds in device memory on every GPU that loads it, until the process
 *   exits.  Sizes whose grouped copy needs more (tp_workspace_size above 36704256) return
 *   TP_ERR_SHAPE before anything is enqueued.  The call allocates nothing.
 *   The first call on a device, with that device current, looks up the array's device
 *   address (cudaGetSymbolAddress) and keeps it, per process and per device ordinal, for
 *   the later calls.  Make that first call on each device before any stream capture.  The
 *   address is not looked up again after a cudaDeviceReset (which unloads the library's
 *   device code and with it the array), so a process must not call this entry point on a
 *   device it has reset.
 *   All calls share the one array and each overwrites what it reads, so calls whose work
 *   overlaps on the GPU (other streams, other host threads) race and must be ordered by
 *   the caller. */
tp_status tp_project_3d_to_2d_noalloc(const void* vol, int n_rec, int Dv, const float* rot,
                                      int n_rot, int n_pose, const float* shift, int n_sh,
                                      void* out, int Do, const tp_opts* opts, void* stream);

/* Backward of tp_backproject_2d_to_3d (ndim = 3) or tp_backproject_2d_to_2d (ndim = 2): the
 * gradients of the back-projection itself, for upstream gradients grad_vol (complex,
 * reconstruction-shaped) of the data volume and grad_wvol (fp32, reconstruction-shaped) of
 * the weight volume; either may be NULL (= 0).  Differentiation bullet ("all operations
 * support gradients for inputs, rotations and shifts").  With vol = P^T(proj):
 *   grad_proj    image-shaped complex = P(grad_vol), the forward projection of grad_vol
 *                (overwritten; NULL = skip)
 *   grad_weights image-shaped fp32 = the real interpolation of grad_wvol at every pixel
 *                (Friedel mirror without conjugation, no phase; overwritten; NULL = skip)
 *   grad_rot     [n_rot][n_pose][k][k]: d/dR of Re<P(grad_vol), proj> plus, with grad_wvol,
 *                d/dR of sum weights * interp(grad_wvol) (overwritten; NULL = skip)
 *   grad_shift   [n_sh][n_pose][2] (or [1][n_pose][2] without shift): d/ds of
 *                Re<P(grad_vol), proj> (overwritten; NULL = skip)
 * Layouts and shapes as in tp_backproject_2d_to_3d / tp_backproject_2d_to_2d (n_rec, Do
 * describe proj, Dv the volumes).  proj is needed for grad_rot / grad_shift of the data
 * part; weights (NULL = 1) for the weight part of grad_rot.  The caller owns every
 * buffer; nothing is allocated.  Errors: TP_ERR_NULL when rot is NULL, or proj is NULL
 * while grad_vol and grad_rot / grad_shift are given (n_rec * n_pose > 0); TP_ERR_SHAPE /
 * TP_ERR_VALUE as for the forward; TP_ERR_CUDA when a launch fails. */
tp_status tp_backproject_backward(int ndim, const void* proj, const float* weights, int n_rec,
                                  int Do, const float* rot, int n_rot, int n_pose,
                                  const float* shift, int n_sh, const void* grad_vol,
                                  const float* grad_wvol, int Dv, void* grad_proj,
                                  float* grad_weights, float* grad_rot, float* grad_shift,
                                  const tp_opts* opts, void* stream);

/* Real-space zero padding for on-the-fly oversampling.  Dutch page, problem statement
 * (oversampling is zero-filling in the spatial domain and needs Fourier transforms on
 * every pass); Spanish page, results, comparison bullet; French page, interpolation
 * comparison (linear with on-the-fly padding and extra FFTs against cubic without).
 *   vol  [n_rec][D][D][D] (ndim = 3) or [n_rec][D][D] (ndim = 2) fp32 real-space data
 *        whose centre is at index D/2 on every axis (read)
 *   out  [n_rec][P][P][P] or [n_rec][P][P] fp32, P = factor * D (overwritten): the volume
 *        centred in the P box, zeros elsewhere, with the centre moved to index 0 (the
 *        ifftshift of the padded box), so that a real-to-complex FFT of out is the
 *        oversampled half spectrum in FFTW order; sampling it at c = factor * R q
 *        (tp_opts.oversampling = factor, layout TP_LAYOUT_FFTW) gives the projection of
 *        the volume at box D.  factor = 1 is the plain ifftshift.
 * D even >= 2, 1 <= factor <= 8, P within the box limit of the projection (1024 in 3D,
 * 32768 in 2D).  Errors: TP_ERR_VALUE for ndim / factor / misaligned pointers,
 * TP_ERR_SHAPE for sizes, TP_ERR_NULL for a NULL pointer with n_rec > 0. */
tp_status tp_pad_volume(int ndim, const float* vol, int n_rec, int D, int factor, float* out,
                        void* stream);

/* Adjoint of tp_pad_volume (and its left inverse): out [n_rec][D]^ndim = the entries of
 * padded [n_rec][P]^ndim that tp_pad_volume filled from the volume.  It is the gradient
 * of the padding for an upstream gradient `padded`.  Arguments and errors as in
 * tp_pad_volume. */
tp_status tp_crop_volume(int ndim, const float* padded, int n_rec, int D, int factor, float* out,
                         void* stream);

/* Static, NUL-terminated name of a status code (never NULL). */
const char* tp_status_string(tp_status status);

#ifdef __cplusplus
}
#endif

#endif /* TP_H */
