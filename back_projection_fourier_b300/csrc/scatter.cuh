// scatter.cuh -- back-projection (the adjoint of the projection) by owner computes.
//
// The transpose of the forward map scatters, for every kept pixel q of every item, the
// value w(c - t) g'(q) into tap t when t_x >= 0 and conj(w(c - t) g'(q)) into -t when
// t_x < 0 (Friedel symmetry of the half spectrum; torch-projectors summaries, Method
// section, Friedel bullet; the insertion "accumulates into the 3D volume", operations
// list).  Scattering tap by tap costs one L2 atomic per tap.  Here instead a thread owns
// a segment of one volume row -- (u_z, u_y) fixed, u_x in [X0, X0 + W) -- for one item and
// gathers every contribution that lands in it:
//   direct:   pixels with |c_y - u_y| < s, |c_z - u_z| < s and c_x within s of the segment
//             (s = kernel support: 2 cubic, 1 linear), weight w(c - u);
//   mirrored: pixels whose -c satisfies the same (their taps t = -u have t_x < 0), adding
//             conj(w(-c - u) g'), only for u_x >= 1.
// Those pixels form a small parallelogram of the image (three linear strips in (kx, ky)),
// which is enumerated line by line.  The segment is accumulated in the thread's private
// slice of shared memory, without atomics, and then added to the volume with one vector
// reduction per pair of elements.  Per item the contributions land in the thin slab of
// voxels the slice crosses, so the global reductions drop from one per tap (64 per pixel
// for cubic 3D) to about one per touched voxel pair.
#pragma once

#include "tp_device.cuh"

namespace tp {

// Interpolation kernel as a function of the distance d (zero outside the support).
template <int INTERP>
__device__ __forceinline__ float kernel_w(float d)
{
    const float u = fabsf(d);
    if constexpr (INTERP == kCubic) {
        const float inner = (1.5f * u - 2.5f) * u * u + 1.0f;
        const float outer = ((-0.5f * u + 2.5f) * u - 4.0f) * u + 2.0f;
        return u < 1.0f ? inner : (u < 2.0f ? outer : 0.0f);
    } else {
        return fmaxf(1.0f - u, 0.0f);
    }
}

// |a kx + b ky - m| < h
struct Strip {
    float a, b, m, h;
};

// Lines ky of the parallelogram cut out of the kept half-disk by up to three strips.  The
// ky range comes from the pair of strips with the largest determinant (the three (a, b)
// rows are two orthonormal columns of a rotation, so one pair has |det| >= 1/sqrt(3));
// each line's kx interval is the intersection of the strips' intervals, widened by a
// hair so that rounding never drops a pixel whose weight is not zero.
template <int NS, typename Visit>
__device__ __forceinline__ void for_each_pixel(const Strip* st, const Geom& g, Visit&& visit)
{
    int pi = 0, pj = 1;
    float best = fabsf(st[0].a * st[1].b - st[1].a * st[0].b);
    if constexpr (NS == 3) {
        const float d02 = fabsf(st[0].a * st[2].b - st[2].a * st[0].b);
        const float d12 = fabsf(st[1].a * st[2].b - st[2].a * st[1].b);
        if (d02 > best) { best = d02; pi = 0; pj = 2; }
        if (d12 > best) { best = d12; pi = 1; pj = 2; }
    }
    const Strip si = st[pi], sj = st[pj];
    const float det = si.a * sj.b - sj.a * si.b;
    const float inv = 1.0f / det;
    const float kc = (si.a * sj.m - sj.a * si.m) * inv;
    const float kr = (fabsf(si.a) * sj.h + fabsf(sj.a) * si.h) * fabsf(inv);
    const int rc = (int)sqrtf((float)g.rc2) + 1;
    int ky0 = (int)ceilf(kc - kr - 1e-3f), ky1 = (int)floorf(kc + kr + 1e-3f);
    ky0 = max(ky0, max(-g.halfo, -rc));
    ky1 = min(ky1, min(g.halfo - 1, rc));
    float inva[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) inva[k] = fabsf(st[k].a) > 1e-7f ? 1.0f / st[k].a : 0.0f;
    for (int ky = ky0; ky <= ky1; ++ky) {
        const int m = g.rc2 - ky * ky;
        if (m < 0) continue;
        int kmax = (int)sqrtf((float)m);
        if (kmax * kmax > m) --kmax;
        if ((kmax + 1) * (kmax + 1) <= m) ++kmax;
        kmax = min(kmax, g.halfo);
        float lo = 0.0f, hi = (float)kmax;
        bool empty = false;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const float r = st[k].m - st[k].b * (float)ky;
            if (inva[k] != 0.0f) {
                const float t1 = (r - st[k].h) * inva[k], t2 = (r + st[k].h) * inva[k];
                lo = fmaxf(lo, fminf(t1, t2));
                hi = fminf(hi, fmaxf(t1, t2));
            } else if (fabsf(r) >= st[k].h) {
                empty = true;
            }
        }
        if (empty) continue;
        const int k0 = max(0, (int)ceilf(lo - 1e-3f));
        const int k1 = min(kmax, (int)floorf(hi + 1e-3f));
        for (int kx = k0; kx <= k1; ++kx) visit(kx, ky);
    }
}

}  // namespace tp

namespace tp {

constexpr int kSegW = 16;  // volume row segment owned by one thread

// Range of B.q over the disk |q| <= rho cut by the strip |A.q - m| < h, as [lo, hi];
// returns false when the strip misses the disk.  The extremes of a linear function over
// that convex set lie at the disk's own extremes (if inside the strip) or at the ends of
// the two chords A.q = m +- h.
__device__ __forceinline__ bool strip_range(float A0, float A1, float B0, float B1, float m, float h,
                                            float rho, float& lo, float& hi)
{
    const float aa2 = A0 * A0 + A1 * A1, bb = sqrtf(B0 * B0 + B1 * B1);
    lo = 3.0e38f;
    hi = -3.0e38f;
    if (aa2 < 1e-12f) {
        if (fabsf(m) >= h) return false;
        lo = -rho * bb;
        hi = rho * bb;
        return true;
    }
    if (bb > 0.f) {
        const float ab = (A0 * B0 + A1 * B1) / bb;  // A.q at q = rho B / |B|
        if (fabsf(rho * ab - m) < h) hi = rho * bb;
        if (fabsf(-rho * ab - m) < h) lo = -rho * bb;
    } else {
        lo = hi = 0.f;
    }
    const float aa = sqrtf(aa2);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const float t = e ? m + h : m - h;
        const float rr = rho * rho - t * t / aa2;
        if (rr < 0.f) continue;
        const float L = sqrtf(rr);
        // q = t A / |A|^2 +- L A_perp / |A|
        const float q0 = t * A0 / aa2, q1 = t * A1 / aa2;
        const float d0 = -A1 / aa, d1 = A0 / aa;
        const float v0 = B0 * q0 + B1 * q1, dv = L * (B0 * d0 + B1 * d1);
        lo = fminf(lo, fminf(v0 - dv, v0 + dv));
        hi = fmaxf(hi, fmaxf(v0 - dv, v0 + dv));
    }
    return lo <= hi;
}

}  // namespace tp

namespace tp {

// Lines of the parallelogram cut out of the kept half-disk by NS strips: calls
// line(ky, image row, k0, k1) for every image line with a non-empty kx interval.  The ky
// range is the intersection of the ranges implied by every pair of strips whose
// determinant is not negligible (the (a, b) rows are two orthonormal columns of a
// rotation, so at least one pair has |det| >= 1/sqrt(3)).  Interval ends are widened by a
// hair so that rounding never drops a pixel whose weight is not zero.
template <int NS, typename Line>
__device__ __forceinline__ void for_each_line(const Strip* st, const Geom& g, const int* kmaxt,
                                              Line&& line)
{
    float kylo = -3.0e38f, kyhi = 3.0e38f;
#pragma unroll
    for (int p = 0; p < (NS == 3 ? 3 : 1); ++p) {
        const Strip si = st[p == 2 ? 1 : 0], sj = st[p == 0 ? 1 : 2];
        const float det = si.a * sj.b - sj.a * si.b;
        if (fabsf(det) < 1e-4f) continue;
        const float inv = 1.0f / det;
        const float kc = (si.a * sj.m - sj.a * si.m) * inv;
        const float kr = (fabsf(si.a) * sj.h + fabsf(sj.a) * si.h) * fabsf(inv);
        kylo = fmaxf(kylo, kc - kr);
        kyhi = fminf(kyhi, kc + kr);
    }
    const int ky0 = max((int)ceilf(fmaxf(kylo, -1.0e6f) - 1e-3f), -g.halfo);
    const int ky1 = min((int)floorf(fminf(kyhi, 1.0e6f) + 1e-3f), g.halfo - 1);
    float inva[NS], r0[NS], bb[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        inva[k] = fabsf(st[k].a) > 1e-7f ? 1.0f / st[k].a : 0.0f;
        r0[k] = st[k].m;
        bb[k] = st[k].b;
    }
    for (int ky = ky0; ky <= ky1; ++ky) {
        const int irow = g.centered ? ky + g.halfo : (ky < 0 ? ky + g.Do : ky);
        const int kmax = kmaxt[irow];
        if (kmax < 0) continue;
        float lo = 0.0f, hi = (float)kmax;
        bool empty = false;
#pragma unroll
        for (int k = 0; k < NS; ++k) {
            const float r = fmaf(-bb[k], (float)ky, r0[k]);
            if (inva[k] != 0.0f) {
                const float t1 = (r - st[k].h) * inva[k], t2 = (r + st[k].h) * inva[k];
                lo = fmaxf(lo, fminf(t1, t2));
                hi = fminf(hi, fmaxf(t1, t2));
            } else if (fabsf(r) >= st[k].h) {
                empty = true;
            }
        }
        if (empty) continue;
        const int k0 = max(0, (int)ceilf(lo - 1e-3f));
        const int k1 = min(kmax, (int)floorf(hi + 1e-3f));
        if (k0 <= k1) line(ky, irow, k0, k1);
    }
}

}  // namespace tp
