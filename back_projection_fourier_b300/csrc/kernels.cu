// kernels.cu -- forward projection, fused backward and back-projection kernels.
//
// Operations (torch-projectors paper summaries, gist.science, Method section, list of
// operations): 3D->2D forward (central slice theorem), 2D->3D backward (accumulation in a
// 3D volume), 2D->2D forward (rotation of 2D Fourier data) and 2D->2D backward
// (accumulation into a 2D reconstruction); gradients for inputs, rotations and shifts
// without stored intermediates (differentiation bullet); shifts by phase modulation.
//
// Work decomposition: a CTA owns one item (reconstruction r, pose p) -- or 1/splits of
// its pixels when items are too few to fill the GPU -- and stages the item's rotation and
// shift once.  Threads stride over the item's pixels in row-major (ky, kx) order, so
// image reads and writes are coalesced; the volume is read through the read-only path
// and stays L2-resident (a D = 256 half volume is 68 MB of a 126 MB L2).
#include "kernels.h"
#include "tp_device.cuh"

namespace tp {

namespace {

constexpr int kThreads = 256;

struct ItemRange {
    long long item;
    int r, p, part;
};

__device__ __forceinline__ ItemRange item_of(const Geom& g, long long w, int splits)
{
    ItemRange ir;
    ir.item = w / splits;
    ir.part = (int)(w - ir.item * splits);
    ir.r = (int)(ir.item / g.n_pose);
    ir.p = (int)(ir.item - (long long)ir.r * g.n_pose);
    return ir;
}

// ------------------------------------------------------------------ forward ----

template <int NDIM, int INTERP>
__global__ void __launch_bounds__(kThreads) project_kernel(
    const float2* __restrict__ rec, const float* __restrict__ rot,
    const float* __restrict__ shift, float2* __restrict__ out, Geom g, int splits,
    long long n_work)
{
    const int npix = (int)g.img_elems;
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        ItemParams<NDIM> ip;
        load_item<NDIM>(g, rot, shift, ir.r, ir.p, ip);
        const float2* V = rec + (long long)ir.r * g.rec_elems;
        float2* y = out + ir.item * g.img_elems;
        for (int pix = ir.part * kThreads + threadIdx.x; pix < npix; pix += splits * kThreads) {
            int i, j;
            split_pixel(pix, g.Ho, i, j);
            const int ky = row_freq(i, g.Do, g.halfo, g.centered), kx = j;
            float2 val = make_float2(0.f, 0.f);
            if (kx * kx + ky * ky <= g.rc2) {
                PixelTaps<NDIM, INTERP, false> t;
                t.init(g, ip.R, (float)kx, (float)ky);
                gather<NDIM, INTERP, false>(V, g, t, val, nullptr);
                if (g.has_shift)
                    val = cmul(val, shift_phase((float)kx, (float)ky, ip.sx, ip.sy, g.Do_f, g.inv_Do));
            }
            y[pix] = val;
        }
    }
}

// ----------------------------------------------------------------- backward ----

// Sum of a per-thread value over the CTA, valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0)
        for (int k = 0; k < kThreads / 32; ++k) s += red[k];
    return s;
}

template <int NDIM, int INTERP, bool WANT_REC, bool WANT_GRAD>
__global__ void __launch_bounds__(kThreads) backward_kernel(
    const float2* __restrict__ rec, const float* __restrict__ rot,
    const float* __restrict__ shift, const float2* __restrict__ gout,
    float2* __restrict__ grec, float* __restrict__ grot, float* __restrict__ gsh, Geom g,
    int splits, long long n_work)
{
    constexpr int NG = NDIM * 2 + 2;  // dL/dR[a][0..1] for a < NDIM, then dL/ds[0..1]
    __shared__ float red[kThreads / 32];
    const int npix = (int)g.img_elems;
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        ItemParams<NDIM> ip;
        load_item<NDIM>(g, rot, shift, ir.r, ir.p, ip);
        const float2* V = rec + (long long)ir.r * g.rec_elems;
        float2* G = WANT_REC ? grec + (long long)ir.r * g.rec_elems : nullptr;
        const float2* gy = gout + ir.item * g.img_elems;
        float acc[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) acc[k] = 0.f;
        for (int pix = ir.part * kThreads + threadIdx.x; pix < npix; pix += splits * kThreads) {
            int i, j;
            split_pixel(pix, g.Ho, i, j);
            const int ky = row_freq(i, g.Do, g.halfo, g.centered), kx = j;
            if (kx * kx + ky * ky > g.rc2) continue;
            float2 gp = __ldg(gy + pix);  // g' = g conj(phase)
            if (g.has_shift)
                gp = cmul_conj(gp, shift_phase((float)kx, (float)ky, ip.sx, ip.sy, g.Do_f, g.inv_Do));
            PixelTaps<NDIM, INTERP, WANT_GRAD> t;
            t.init(g, ip.R, (float)kx, (float)ky);
            if constexpr (WANT_GRAD) {
                float2 v, dv[3];
                gather<NDIM, INTERP, true>(V, g, t, v, dv);
                // Re(conj(g') dv/dc_a) times q_b; Im(conj(g') v) times q_b for the shifts
#pragma unroll
                for (int a = 0; a < NDIM; ++a) {
                    const float cr = gp.x * dv[a].x + gp.y * dv[a].y;
                    acc[2 * a] = fmaf(cr, (float)kx, acc[2 * a]);
                    acc[2 * a + 1] = fmaf(cr, (float)ky, acc[2 * a + 1]);
                }
                const float ci = gp.x * v.y - gp.y * v.x;
                acc[2 * NDIM] = fmaf(ci, (float)kx, acc[2 * NDIM]);
                acc[2 * NDIM + 1] = fmaf(ci, (float)ky, acc[2 * NDIM + 1]);
            }
            if constexpr (WANT_REC) scatter<NDIM, INTERP, WANT_GRAD>(G, nullptr, g, t, gp, 0.f);
        }
        if constexpr (WANT_GRAD) {
            const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
            const long long si = (long long)(g.sh_shared ? 0 : ir.r) * g.n_pose + ir.p;
            const float two_pi_over_Do = 6.283185307179586f * g.inv_Do;
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const float s = block_sum(acc[k], red);
                if (threadIdx.x == 0) {
                    if (k < 2 * NDIM) {
                        if (grot) atomicAdd(grot + ri * NDIM * NDIM + (k / 2) * NDIM + (k % 2), g.o * s);
                    } else if (gsh && g.has_shift) {
                        atomicAdd(gsh + si * 2 + (k - 2 * NDIM), two_pi_over_Do * s);
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------ back-projection ----

template <int NDIM, int INTERP>
__global__ void __launch_bounds__(kThreads) backproject_kernel(
    const float2* __restrict__ proj, const float* __restrict__ weights,
    const float* __restrict__ rot, const float* __restrict__ shift,
    float2* __restrict__ vout, float* __restrict__ wout, Geom g, int splits, long long n_work)
{
    const int npix = (int)g.img_elems;
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        ItemParams<NDIM> ip;
        load_item<NDIM>(g, rot, shift, ir.r, ir.p, ip);
        float2* G = vout ? vout + (long long)ir.r * g.rec_elems : nullptr;
        float* W = wout ? wout + (long long)ir.r * g.rec_elems : nullptr;
        const float2* py = proj + ir.item * g.img_elems;
        const float* pw = weights ? weights + ir.item * g.img_elems : nullptr;
        for (int pix = ir.part * kThreads + threadIdx.x; pix < npix; pix += splits * kThreads) {
            int i, j;
            split_pixel(pix, g.Ho, i, j);
            const int ky = row_freq(i, g.Do, g.halfo, g.centered), kx = j;
            if (kx * kx + ky * ky > g.rc2) continue;
            float2 val = G ? __ldg(py + pix) : make_float2(0.f, 0.f);
            if (G && g.has_shift)
                val = cmul_conj(val, shift_phase((float)kx, (float)ky, ip.sx, ip.sy, g.Do_f, g.inv_Do));
            const float wt = pw ? __ldg(pw + pix) : 1.0f;
            PixelTaps<NDIM, INTERP, false> t;
            t.init(g, ip.R, (float)kx, (float)ky);
            scatter<NDIM, INTERP, false>(G, W, g, t, val, wt);
        }
    }
}

// ------------------------------------------------------------------ launches ----

struct LaunchShape {
    int splits;
    long long n_work;
    unsigned grid;
};

LaunchShape launch_shape(const Geom& g, int sms)
{
    const long long n_items = (long long)g.n_rec * g.n_pose;
    const long long per_item = (g.img_elems + kThreads - 1) / kThreads;  // thread-rows
    const long long target = 8LL * sms;  // CTAs for a full wave at 8 CTAs / SM
    long long splits = 1;
    if (n_items < target) splits = (target + n_items - 1) / n_items;
    if (splits > per_item) splits = per_item;
    if (splits < 1) splits = 1;
    LaunchShape s;
    s.splits = (int)splits;
    s.n_work = n_items * splits;
    const long long cap = 64LL * sms * 8;
    s.grid = (unsigned)(s.n_work < cap ? s.n_work : cap);
    return s;
}

}  // namespace

cudaError_t launch_project(int ndim, int interp, const Geom& g, const void* rec,
                           const float* rot, const float* shift, void* out, int sms,
                           cudaStream_t stream)
{
    const LaunchShape s = launch_shape(g, sms);
    if (s.n_work == 0) return cudaSuccess;
    auto R = static_cast<const float2*>(rec);
    auto Y = static_cast<float2*>(out);
    if (ndim == 3 && interp == kCubic)
        project_kernel<3, kCubic><<<s.grid, kThreads, 0, stream>>>(R, rot, shift, Y, g, s.splits, s.n_work);
    else if (ndim == 3)
        project_kernel<3, kLinear><<<s.grid, kThreads, 0, stream>>>(R, rot, shift, Y, g, s.splits, s.n_work);
    else if (interp == kCubic)
        project_kernel<2, kCubic><<<s.grid, kThreads, 0, stream>>>(R, rot, shift, Y, g, s.splits, s.n_work);
    else
        project_kernel<2, kLinear><<<s.grid, kThreads, 0, stream>>>(R, rot, shift, Y, g, s.splits, s.n_work);
    return cudaGetLastError();
}

template <int NDIM, int INTERP>
static void launch_backward_t(const LaunchShape& s, const Geom& g, const float2* R,
                              const float* rot, const float* shift, const float2* G,
                              float2* grec, float* grot, float* gsh, cudaStream_t stream)
{
    const bool want_grad = grot || (gsh && g.has_shift);
    if (grec && want_grad)
        backward_kernel<NDIM, INTERP, true, true><<<s.grid, kThreads, 0, stream>>>(
            R, rot, shift, G, grec, grot, gsh, g, s.splits, s.n_work);
    else if (grec)
        backward_kernel<NDIM, INTERP, true, false><<<s.grid, kThreads, 0, stream>>>(
            R, rot, shift, G, grec, grot, gsh, g, s.splits, s.n_work);
    else if (want_grad)
        backward_kernel<NDIM, INTERP, false, true><<<s.grid, kThreads, 0, stream>>>(
            R, rot, shift, G, grec, grot, gsh, g, s.splits, s.n_work);
}

cudaError_t launch_backward(int ndim, int interp, const Geom& g, const void* rec,
                            const float* rot, const float* shift, const void* grad_out,
                            void* grad_rec, float* grad_rot, float* grad_shift, int sms,
                            cudaStream_t stream)
{
    const LaunchShape s = launch_shape(g, sms);
    if (s.n_work == 0) return cudaSuccess;
    auto R = static_cast<const float2*>(rec);
    auto G = static_cast<const float2*>(grad_out);
    auto GR = static_cast<float2*>(grad_rec);
    if (ndim == 3 && interp == kCubic)
        launch_backward_t<3, kCubic>(s, g, R, rot, shift, G, GR, grad_rot, grad_shift, stream);
    else if (ndim == 3)
        launch_backward_t<3, kLinear>(s, g, R, rot, shift, G, GR, grad_rot, grad_shift, stream);
    else if (interp == kCubic)
        launch_backward_t<2, kCubic>(s, g, R, rot, shift, G, GR, grad_rot, grad_shift, stream);
    else
        launch_backward_t<2, kLinear>(s, g, R, rot, shift, G, GR, grad_rot, grad_shift, stream);
    return cudaGetLastError();
}

cudaError_t launch_backproject(int ndim, int interp, const Geom& g, const void* proj,
                               const float* weights, const float* rot, const float* shift,
                               void* vol_out, float* wvol_out, int sms, cudaStream_t stream)
{
    const LaunchShape s = launch_shape(g, sms);
    if (s.n_work == 0 || (!vol_out && !wvol_out)) return cudaSuccess;
    auto P = static_cast<const float2*>(proj);
    auto VO = static_cast<float2*>(vol_out);
    if (ndim == 3 && interp == kCubic)
        backproject_kernel<3, kCubic><<<s.grid, kThreads, 0, stream>>>(P, weights, rot, shift, VO, wvol_out, g, s.splits, s.n_work);
    else if (ndim == 3)
        backproject_kernel<3, kLinear><<<s.grid, kThreads, 0, stream>>>(P, weights, rot, shift, VO, wvol_out, g, s.splits, s.n_work);
    else if (interp == kCubic)
        backproject_kernel<2, kCubic><<<s.grid, kThreads, 0, stream>>>(P, weights, rot, shift, VO, wvol_out, g, s.splits, s.n_work);
    else
        backproject_kernel<2, kLinear><<<s.grid, kThreads, 0, stream>>>(P, weights, rot, shift, VO, wvol_out, g, s.splits, s.n_work);
    return cudaGetLastError();
}

}  // namespace tp
