// pad.cu -- real-space zero padding for on-the-fly oversampling, and its adjoint.
//
// Oversampling a reconstruction means zero-filling it in real space to a larger box and
// transforming again, every pass (Dutch page, problem statement; Spanish page, results,
// comparison bullet; French page, interpolation comparison: "padding on the fly, with
// additional FFTs").  A real-space volume of box D has its centre at index D/2 on every
// axis.  pad writes the factor*D box that holds the volume centred and zeros elsewhere,
// already moved so that the centre sits at index 0 (the ifftshift that a real-to-complex
// FFT of centred data needs), so one FFT of the result is the oversampled spectrum in
// FFTW order.  factor = 1 is the plain ifftshift.  crop is the adjoint (and the left
// inverse) of pad: it gathers the D box back out of a padded array.
#include <cstdint>

#include "kernels.h"

namespace tp {
namespace {

constexpr int kPadThreads = 256;

// Source index along one axis of the padded, origin-moved box P = factor * D, or -1 in
// the zero band.  Index u < D/2 holds volume index u + D/2 (frequency-0 side of the
// centre); u >= P - D/2 holds u - (P - D/2).
__device__ __forceinline__ int src_of(int u, int D, int P)
{
    const int h = D / 2;
    if (u < h) return u + h;
    if (u >= P - h) return u - (P - h);
    return -1;
}

// Where volume index i lands in the padded box (inverse of src_of).
__device__ __forceinline__ int dst_of(int i, int D, int P)
{
    const int h = D / 2;
    return i >= h ? i - h : i + P - h;
}

// One CTA per output row (n, z, y) at a time, threads along x: coalesced stores of the
// padded box (the larger array), gathered loads from the volume row.
__global__ void __launch_bounds__(kPadThreads) pad_kernel(const float* __restrict__ vol,
                                                          float* __restrict__ out, int ndim, int D,
                                                          int P, long long n_rows)
{
    for (long long row = blockIdx.x; row < n_rows; row += gridDim.x) {
        // row = (n * P + z) * P + y in 3D, n * P + y in 2D
        const int y = (int)(row % P);
        long long rest = row / P;
        int sz = 0;
        if (ndim == 3) {
            sz = src_of((int)(rest % P), D, P);
            rest /= P;
        }
        const long long n = rest;
        const int sy = src_of(y, D, P);
        float* o = out + row * P;
        if (sy < 0 || sz < 0) {
            for (int x = threadIdx.x; x < P; x += kPadThreads) o[x] = 0.0f;
            continue;
        }
        const long long srow = ndim == 3 ? ((n * D + sz) * D + sy) : (n * D + sy);
        const float* s = vol + srow * D;
        for (int x = threadIdx.x; x < P; x += kPadThreads) {
            const int sx = src_of(x, D, P);
            o[x] = sx >= 0 ? __ldg(s + sx) : 0.0f;
        }
    }
}

// One CTA per volume row, threads along x: coalesced stores of the D box.
__global__ void __launch_bounds__(kPadThreads) crop_kernel(const float* __restrict__ padded,
                                                           float* __restrict__ out, int ndim, int D,
                                                           int P, long long n_rows)
{
    for (long long row = blockIdx.x; row < n_rows; row += gridDim.x) {
        const int y = (int)(row % D);
        long long rest = row / D;
        int pz = 0;
        if (ndim == 3) {
            pz = dst_of((int)(rest % D), D, P);
            rest /= D;
        }
        const long long n = rest;
        const int py = dst_of(y, D, P);
        const long long prow = ndim == 3 ? ((n * P + pz) * P + py) : (n * P + py);
        const float* s = padded + prow * P;
        float* o = out + row * D;
        for (int x = threadIdx.x; x < D; x += kPadThreads) o[x] = __ldg(s + dst_of(x, D, P));
    }
}

unsigned rows_grid(long long n_rows, int sms)
{
    const long long cap = 16LL * sms;
    return (unsigned)(n_rows < cap ? n_rows : cap);
}

}  // namespace

cudaError_t launch_pad(int ndim, const float* vol, int n, int D, int factor, float* out, int sms,
                       cudaStream_t stream)
{
    const int P = factor * D;
    long long n_rows = (long long)n * P;
    if (ndim == 3) n_rows *= P;
    if (n_rows == 0) return cudaSuccess;
    pad_kernel<<<rows_grid(n_rows, sms), kPadThreads, 0, stream>>>(vol, out, ndim, D, P, n_rows);
    return cudaGetLastError();
}

cudaError_t launch_crop(int ndim, const float* padded, int n, int D, int factor, float* out,
                        int sms, cudaStream_t stream)
{
    const int P = factor * D;
    long long n_rows = (long long)n * D;
    if (ndim == 3) n_rows *= D;
    if (n_rows == 0) return cudaSuccess;
    crop_kernel<<<rows_grid(n_rows, sms), kPadThreads, 0, stream>>>(padded, out, ndim, D, P,
                                                                      n_rows);
    return cudaGetLastError();
}

}  // namespace tp
