// tp_abi.cu -- the extern "C" entry points of libtp.so declared in include/tp.h:
// argument validation on the host, derived geometry, output zeroing and the launches.
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <climits>

#include "../../include/tp.h"
#include "kernels.h"

namespace {

constexpr int kMaxBox3 = 1024;
constexpr int kMaxBox2 = 32768;

struct Opts {
    int interp = TP_CUBIC;
    int layout = TP_LAYOUT_CENTERED;
    float o = 1.0f;
    float cutoff = -1.0f;
};

tp_status read_opts(const tp_opts* in, Opts& o)
{
    if (in) {
        o.interp = in->interp;
        o.layout = in->layout;
        o.o = in->oversampling;
        o.cutoff = in->cutoff;
    }
    if (o.interp != TP_LINEAR && o.interp != TP_CUBIC) return TP_ERR_VALUE;
    if (o.layout != TP_LAYOUT_FFTW && o.layout != TP_LAYOUT_CENTERED) return TP_ERR_VALUE;
    if (!(o.o > 0.0f) || !std::isfinite(o.o)) return TP_ERR_VALUE;
    if (!std::isfinite(o.cutoff)) return TP_ERR_VALUE;
    return TP_OK;
}

bool box_ok(int D, int ndim)
{
    return D >= 2 && (D % 2) == 0 && D <= (ndim == 3 ? kMaxBox3 : kMaxBox2);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shapes shared by every call.  `need_*` says whether the pointer is required.
tp_status check_common(int ndim, int n_rec, int Dv, int Do, int n_rot, int n_pose,
                       const float* shift, int n_sh)
{
    if (ndim != 2 && ndim != 3) return TP_ERR_VALUE;
    if (n_rec < 0 || n_pose < 0) return TP_ERR_SHAPE;
    if (!box_ok(Dv, ndim) || !box_ok(Do, ndim)) return TP_ERR_SHAPE;
    if (n_rot != 1 && n_rot != n_rec) return TP_ERR_SHAPE;
    if (shift && n_sh != 1 && n_sh != n_rec) return TP_ERR_SHAPE;
    return TP_OK;
}

tp::Geom make_geom(int ndim, int n_rec, int Dv, int n_rot, int n_pose, const float* shift,
                   int n_sh, int Do, const Opts& o)
{
    tp::Geom g;
    g.n_rec = n_rec;
    g.n_pose = n_pose;
    g.rot_shared = n_rot == 1;
    g.sh_shared = n_sh == 1;
    g.Dv = Dv;
    g.Hv = Dv / 2 + 1;
    g.halfv = Dv / 2;
    g.Do = Do;
    g.Ho = Do / 2 + 1;
    g.halfo = Do / 2;
    g.centered = o.layout == TP_LAYOUT_CENTERED;
    g.has_shift = shift != nullptr;
    g.o_is_one = o.o == 1.0f;
    g.o = o.o;
    g.Do_f = (float)Do;
    g.inv_Do = 1.0f / (float)Do;
    // kx^2 + ky^2 <= rc^2  <=>  kx^2 + ky^2 <= floor(rc^2) for integer kx, ky; rc^2 of an
    // fp32 rc is exact in double.
    const double rc = o.cutoff < 0.0f ? 0.5 * Do : (double)o.cutoff;
    const double rc2 = std::floor(rc * rc);
    g.rc2 = rc2 >= (double)INT_MAX ? INT_MAX : (int)rc2;
    g.rec_elems = ndim == 3 ? (long long)Dv * Dv * g.Hv : (long long)Dv * g.Hv;
    g.img_elems = (long long)Do * g.Ho;
    const tp::GroupPitch gp = tp::group_pitch(Dv, o.interp == TP_CUBIC ? 4 : 2);
    g.grow = gp.row;
    g.gplane = gp.plane;
    return g;
}

int sm_count()
{
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

// Bytes of the grouped-volume workspace of the 3D gathers (0: not used).  The gathers index
// it with 32-bit offsets, so NT * (elements of one volume) must stay below 2^31.
size_t grouped_bytes(int ndim, int n_rec, int Dv, int interp)
{
    if (ndim != 3 || n_rec <= 0 || !box_ok(Dv, 3)) return 0;
    const long long nt = interp == TP_CUBIC ? 4 : 2;
    const long long per = tp::grouped_volume_elems(Dv, (int)nt);
    if (per >= (1LL << 31)) return 0;
    if ((long long)n_rec > (LLONG_MAX / 8) / per) return 0;  // beyond any device memory
    return (size_t)(per * n_rec * 8);
}

// Checks a caller's workspace; sets `use` when the gathers will read the grouped copy.
tp_status check_workspace(int ndim, int n_rec, int Dv, int interp, const void* ws, size_t ws_bytes,
                          bool& use)
{
    use = false;
    if (!ws) return TP_OK;
    const size_t need = grouped_bytes(ndim, n_rec, Dv, interp);
    if (need == 0) return TP_OK;
    if (ws_bytes < need) return TP_ERR_SHAPE;
    if (!aligned(ws, 32)) return TP_ERR_VALUE;
    use = true;
    return TP_OK;
}

tp_status project_impl(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                       int n_rot, int n_pose, const float* shift, int n_sh, void* out, int Do,
                       const tp_opts* opts, void* stream, void* ws = nullptr, size_t ws_bytes = 0)
{
    Opts o;
    tp_status st = read_opts(opts, o);
    if (st != TP_OK) return st;
    st = check_common(ndim, n_rec, Dv, Do, n_rot, n_pose, shift, n_sh);
    if (st != TP_OK) return st;
    bool use_ws = false;
    st = check_workspace(ndim, n_rec, Dv, o.interp, ws, ws_bytes, use_ws);
    if (st != TP_OK) return st;
    const long long n_items = (long long)n_rec * n_pose;
    if (n_items == 0) return TP_OK;
    if (!rec || !rot || !out) return TP_ERR_NULL;
    if (!aligned(rec, 8) || !aligned(out, 8) || !aligned(rot, 4) || (shift && !aligned(shift, 4)))
        return TP_ERR_VALUE;
    const tp::Geom g = make_geom(ndim, n_rec, Dv, n_rot, n_pose, shift, n_sh, Do, o);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sms = sm_count();
    cudaError_t e = cudaSuccess;
    if (use_ws) e = tp::launch_expand_groups(o.interp, g, rec, ws, sms, s);
    if (e == cudaSuccess)
        e = tp::launch_project(ndim, o.interp, g, rec, rot, shift, out, sms, s, use_ws ? ws : nullptr);
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

tp_status backproject_impl(int ndim, const void* proj, const float* weights, int n_rec, int Do,
                           const float* rot, int n_rot, int n_pose, const float* shift, int n_sh,
                           void* vol_out, float* wvol_out, int Dv, int accumulate,
                           const tp_opts* opts, void* stream)
{
    Opts o;
    tp_status st = read_opts(opts, o);
    if (st != TP_OK) return st;
    st = check_common(ndim, n_rec, Dv, Do, n_rot, n_pose, shift, n_sh);
    if (st != TP_OK) return st;
    if (accumulate != 0 && accumulate != 1) return TP_ERR_VALUE;
    const long long n_items = (long long)n_rec * n_pose;
    if (n_rec > 0 && !vol_out && !wvol_out) return TP_OK;
    if (n_items > 0) {
        if (!rot || (vol_out && !proj)) return TP_ERR_NULL;
        if ((proj && !aligned(proj, 8)) || (weights && !aligned(weights, 4)) || !aligned(rot, 4) ||
            (shift && !aligned(shift, 4)))
            return TP_ERR_VALUE;
    }
    if ((vol_out && !aligned(vol_out, 8)) || (wvol_out && !aligned(wvol_out, 4)))
        return TP_ERR_VALUE;
    const tp::Geom g = make_geom(ndim, n_rec, Dv, n_rot, n_pose, shift, n_sh, Do, o);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!accumulate && n_rec > 0) {
        const size_t elems = (size_t)g.rec_elems * (size_t)n_rec;
        if (vol_out && cudaMemsetAsync(vol_out, 0, elems * 8, s) != cudaSuccess) return TP_ERR_CUDA;
        if (wvol_out && cudaMemsetAsync(wvol_out, 0, elems * 4, s) != cudaSuccess) return TP_ERR_CUDA;
    }
    if (n_items == 0) return TP_OK;
    const cudaError_t e = tp::launch_backproject(ndim, o.interp, g, proj, weights, rot, shift,
                                                 vol_out, wvol_out, sm_count(), s);
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// The backward of the projection; `fused` selects the one-pass kernel where it exists.
tp_status project_backward_impl(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                                int n_rot, int n_pose, const float* shift, int n_sh,
                                const void* grad_out, int Do, void* grad_rec, float* grad_rot,
                                float* grad_shift, void* workspace, size_t workspace_bytes,
                                const tp_opts* opts, void* stream, bool fused)
{
    Opts o;
    tp_status st = read_opts(opts, o);
    if (st != TP_OK) return st;
    st = check_common(ndim, n_rec, Dv, Do, n_rot, n_pose, shift, n_sh);
    if (st != TP_OK) return st;
    bool use_ws = false;
    st = check_workspace(ndim, n_rec, Dv, o.interp, workspace, workspace_bytes, use_ws);
    if (st != TP_OK) return st;
    const long long n_items = (long long)n_rec * n_pose;
    const bool want_grad = grad_rot || (grad_shift && shift);
    if (n_items > 0 && (grad_rec || want_grad)) {
        if (!grad_out || !rot || (want_grad && !rec)) return TP_ERR_NULL;
        if (!aligned(grad_out, 8) || !aligned(rot, 4) || (rec && !aligned(rec, 8)) ||
            (shift && !aligned(shift, 4)))
            return TP_ERR_VALUE;
    }
    if ((grad_rec && !aligned(grad_rec, 8)) || (grad_rot && !aligned(grad_rot, 4)) ||
        (grad_shift && !aligned(grad_shift, 4)))
        return TP_ERR_VALUE;
    const tp::Geom g = make_geom(ndim, n_rec, Dv, n_rot, n_pose, shift, n_sh, Do, o);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int k2 = ndim * ndim;
    const size_t n_sh_rows = shift ? (size_t)n_sh : 1;
    if (grad_rec && n_rec > 0 &&
        cudaMemsetAsync(grad_rec, 0, (size_t)g.rec_elems * n_rec * 8, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (grad_rot && cudaMemsetAsync(grad_rot, 0, (size_t)n_rot * n_pose * k2 * 4, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (grad_shift && cudaMemsetAsync(grad_shift, 0, n_sh_rows * n_pose * 2 * 4, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (n_items == 0 || (!grad_rec && !want_grad)) return TP_OK;
    const int sms = sm_count();
    use_ws = use_ws && want_grad;  // only the pose-gradient gather reads the grouped copy
    cudaError_t e = cudaSuccess;
    if (use_ws) e = tp::launch_expand_groups(o.interp, g, rec, workspace, sms, s);
    if (e == cudaSuccess)
        e = tp::launch_backward(ndim, o.interp, g, rec, rot, shift, grad_out, grad_rec, grad_rot,
                                grad_shift, sms, s, use_ws ? workspace : nullptr, fused);
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

}  // namespace

extern "C" {

tp_status tp_project_3d_to_2d(const void* vol, int n_rec, int Dv, const float* rot, int n_rot,
                              int n_pose, const float* shift, int n_sh, void* out, int Do,
                              const tp_opts* opts, void* stream)
{
    return project_impl(3, vol, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, out, Do, opts, stream);
}

tp_status tp_project_3d_to_2d_ws(const void* vol, int n_rec, int Dv, const float* rot, int n_rot,
                                 int n_pose, const float* shift, int n_sh, void* out, int Do,
                                 void* workspace, size_t workspace_bytes, const tp_opts* opts,
                                 void* stream)
{
    return project_impl(3, vol, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, out, Do, opts, stream,
                        workspace, workspace_bytes);
}

size_t tp_workspace_size(int ndim, int n_rec, int Dv, const tp_opts* opts)
{
    Opts o;
    if (read_opts(opts, o) != TP_OK) return 0;
    return grouped_bytes(ndim, n_rec, Dv, o.interp);
}

tp_status tp_project_2d_to_2d(const void* img, int n_rec, int Dv, const float* rot, int n_rot,
                              int n_pose, const float* shift, int n_sh, void* out, int Do,
                              const tp_opts* opts, void* stream)
{
    return project_impl(2, img, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, out, Do, opts, stream);
}

tp_status tp_backproject_2d_to_3d(const void* proj, const float* weights, int n_rec, int Do,
                                  const float* rot, int n_rot, int n_pose, const float* shift,
                                  int n_sh, void* vol_out, float* wvol_out, int Dv,
                                  int accumulate, const tp_opts* opts, void* stream)
{
    return backproject_impl(3, proj, weights, n_rec, Do, rot, n_rot, n_pose, shift, n_sh, vol_out,
                            wvol_out, Dv, accumulate, opts, stream);
}

tp_status tp_backproject_2d_to_2d(const void* proj, const float* weights, int n_rec, int Do,
                                  const float* rot, int n_rot, int n_pose, const float* shift,
                                  int n_sh, void* img_out, float* wimg_out, int Dv,
                                  int accumulate, const tp_opts* opts, void* stream)
{
    return backproject_impl(2, proj, weights, n_rec, Do, rot, n_rot, n_pose, shift, n_sh, img_out,
                            wimg_out, Dv, accumulate, opts, stream);
}

tp_status tp_project_backward(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                              int n_rot, int n_pose, const float* shift, int n_sh,
                              const void* grad_out, int Do, void* grad_rec, float* grad_rot,
                              float* grad_shift, const tp_opts* opts, void* stream)
{
    return tp_project_backward_ws(ndim, rec, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, grad_out,
                                  Do, grad_rec, grad_rot, grad_shift, nullptr, 0, opts, stream);
}

tp_status tp_project_backward_fused(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                                    int n_rot, int n_pose, const float* shift, int n_sh,
                                    const void* grad_out, int Do, void* grad_rec, float* grad_rot,
                                    float* grad_shift, const tp_opts* opts, void* stream)
{
    return project_backward_impl(ndim, rec, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, grad_out,
                                 Do, grad_rec, grad_rot, grad_shift, nullptr, 0, opts, stream, true);
}

tp_status tp_project_backward_ws(int ndim, const void* rec, int n_rec, int Dv, const float* rot,
                                 int n_rot, int n_pose, const float* shift, int n_sh,
                                 const void* grad_out, int Do, void* grad_rec, float* grad_rot,
                                 float* grad_shift, void* workspace, size_t workspace_bytes,
                                 const tp_opts* opts, void* stream)
{
    return project_backward_impl(ndim, rec, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, grad_out,
                                 Do, grad_rec, grad_rot, grad_shift, workspace, workspace_bytes,
                                 opts, stream, false);
}

tp_status tp_backproject_backward(int ndim, const void* proj, const float* weights, int n_rec,
                                  int Do, const float* rot, int n_rot, int n_pose,
                                  const float* shift, int n_sh, const void* grad_vol,
                                  const float* grad_wvol, int Dv, void* grad_proj,
                                  float* grad_weights, float* grad_rot, float* grad_shift,
                                  const tp_opts* opts, void* stream)
{
    Opts o;
    tp_status st = read_opts(opts, o);
    if (st != TP_OK) return st;
    st = check_common(ndim, n_rec, Dv, Do, n_rot, n_pose, shift, n_sh);
    if (st != TP_OK) return st;
    const long long n_items = (long long)n_rec * n_pose;
    // the data part needs grad_vol (and proj for the pose gradients); NULL upstream = 0
    const bool data_pose = grad_vol && (grad_rot || (grad_shift && shift));
    const bool wts_part = grad_wvol && (grad_weights || grad_rot);
    if (n_items > 0) {
        if (!rot || (data_pose && !proj)) return TP_ERR_NULL;
        if (!aligned(rot, 4) || (proj && !aligned(proj, 8)) || (grad_vol && !aligned(grad_vol, 8)) ||
            (grad_wvol && !aligned(grad_wvol, 4)) || (weights && !aligned(weights, 4)) ||
            (shift && !aligned(shift, 4)))
            return TP_ERR_VALUE;
    }
    if ((grad_proj && !aligned(grad_proj, 8)) || (grad_weights && !aligned(grad_weights, 4)) ||
        (grad_rot && !aligned(grad_rot, 4)) || (grad_shift && !aligned(grad_shift, 4)))
        return TP_ERR_VALUE;
    const tp::Geom g = make_geom(ndim, n_rec, Dv, n_rot, n_pose, shift, n_sh, Do, o);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int k2 = ndim * ndim;
    const size_t n_sh_rows = shift ? (size_t)n_sh : 1;
    const size_t img_bytes = (size_t)g.img_elems * (size_t)n_items;
    if (grad_rot && cudaMemsetAsync(grad_rot, 0, (size_t)n_rot * n_pose * k2 * 4, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (grad_shift && cudaMemsetAsync(grad_shift, 0, n_sh_rows * n_pose * 2 * 4, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (grad_proj && !grad_vol && cudaMemsetAsync(grad_proj, 0, img_bytes * 8, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (grad_weights && !grad_wvol && cudaMemsetAsync(grad_weights, 0, img_bytes * 4, s) != cudaSuccess)
        return TP_ERR_CUDA;
    if (n_items == 0) return TP_OK;
    const int sms = sm_count();
    cudaError_t e = cudaSuccess;
    // Re<grad_vol, P^T proj> = Re<P grad_vol, proj>: the projection of grad_vol is the
    // gradient for proj, and its pose gradients against proj are those of the insertion
    if (grad_proj && grad_vol)
        e = tp::launch_project(ndim, o.interp, g, grad_vol, rot, shift, grad_proj, sms, s);
    if (e == cudaSuccess && data_pose)
        e = tp::launch_backward(ndim, o.interp, g, grad_vol, rot, shift, proj, nullptr, grad_rot,
                                grad_shift, sms, s);
    if (e == cudaSuccess && wts_part)
        e = tp::launch_weights_grad(ndim, o.interp, g, grad_wvol, weights, rot, grad_weights, grad_rot,
                                    sms, s);
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

namespace {

constexpr int kMaxPadFactor = 8;

tp_status check_pad(int ndim, const void* a, const void* b, int n_rec, int D, int factor)
{
    if (ndim != 2 && ndim != 3) return TP_ERR_VALUE;
    if (factor < 1 || factor > kMaxPadFactor) return TP_ERR_VALUE;
    if (n_rec < 0 || D < 2 || (D % 2) != 0) return TP_ERR_SHAPE;
    if (!box_ok((long long)factor * D > INT_MAX ? -1 : factor * D, ndim)) return TP_ERR_SHAPE;
    if (n_rec == 0) return TP_OK;
    if (!a || !b) return TP_ERR_NULL;
    if (!aligned(a, 4) || !aligned(b, 4)) return TP_ERR_VALUE;
    return TP_OK;
}

}  // namespace

tp_status tp_pad_volume(int ndim, const float* vol, int n_rec, int D, int factor, float* out,
                        void* stream)
{
    const tp_status st = check_pad(ndim, vol, out, n_rec, D, factor);
    if (st != TP_OK || n_rec == 0) return st;
    const cudaError_t e = tp::launch_pad(ndim, vol, n_rec, D, factor, out, sm_count(),
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

tp_status tp_crop_volume(int ndim, const float* padded, int n_rec, int D, int factor, float* out,
                         void* stream)
{
    const tp_status st = check_pad(ndim, padded, out, n_rec, D, factor);
    if (st != TP_OK || n_rec == 0) return st;
    const cudaError_t e = tp::launch_crop(ndim, padded, n_rec, D, factor, out, sm_count(),
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

const char* tp_status_string(tp_status status)
{
    switch (status) {
    case TP_OK: return "TP_OK";
    case TP_ERR_NULL: return "TP_ERR_NULL: a required pointer is NULL";
    case TP_ERR_SHAPE: return "TP_ERR_SHAPE: a size is negative, odd, too large or mismatched";
    case TP_ERR_VALUE: return "TP_ERR_VALUE: an option or flag is out of range, or a pointer is misaligned";
    case TP_ERR_CUDA: return "TP_ERR_CUDA: a CUDA launch or memset failed";
    }
    return "TP_ERR_UNKNOWN: not a tp_status value";
}

}  // extern "C"
