// tp_device.cuh -- device-side building blocks shared by the projection kernels.
//
// Method (torch-projectors paper summaries, gist.science, Method section): rfft half
// spectra in FFTW/PyTorch conventions; linear or Catmull-Rom (Keys a = -0.5) cubic
// interpolation; Friedel symmetry F(-k) = conj F(k); rotation of the sample coordinate;
// shifts by Fourier phase modulation.
//
// Numerics.  The sample coordinate c = o * (R q) is formed as an unevaluated sum
// hi + lo of two floats with error-free products and sums (Dekker / Knuth; the FMA
// form of TwoProduct), so that frac(c) is exact to ~1e-7 even at |c| ~ 128-512, where a
// plain fp32 product would already be off by ~1e-5.  The shift phase is reduced the same
// way to a turn count in [-1/2, 1/2] before sincospif.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tp {

constexpr int kLinear = 0;
constexpr int kCubic = 1;

// Number of taps per axis.
template <int INTERP>
struct Taps {
    static constexpr int N = INTERP == kCubic ? 4 : 2;
    static constexpr int first = INTERP == kCubic ? -1 : 0;  // first tap relative to floor(c)
};

// Pitches of the gathers' grouped copy of a 3D volume, in groups of NT taps (8 NT bytes).
// A row holds at least Hv + NT - 1 groups (starts x = -(NT - 1) .. Dv/2) and a plane at least
// Dv rows.  Each is padded up to a fixed residue modulo the groups in a 128-byte line
// (16 / NT): the residues set where the y and z neighbours of a tap row fall within their
// cache lines, and so how the rows that the lanes of a warp load spread over the L1 data
// banks.  Measured at D = 128, cubic, 16 384 poses (forward + pose gradients): residues
// (row, plane) = (2, 1) 9.50 ms, (1, 2) 9.52, (1, 0) 10.14, (0, 0) -- every row starting a
// cache line -- 10.88.
#ifndef TP_GROUP_ROW_RES
#define TP_GROUP_ROW_RES 2
#endif
#ifndef TP_GROUP_PLANE_RES
#define TP_GROUP_PLANE_RES 1
#endif
struct GroupPitch {
    int row, plane;
};

__host__ __device__ constexpr int pad_to_residue(int n, int m, int res)
{
    return n + ((res - n) % m + m) % m;
}

__host__ __device__ constexpr GroupPitch group_pitch(int Dv, int nt)
{
    return {pad_to_residue(Dv / 2 + nt, 16 / nt, TP_GROUP_ROW_RES),
            pad_to_residue(Dv * pad_to_residue(Dv / 2 + nt, 16 / nt, TP_GROUP_ROW_RES), 16 / nt,
                           TP_GROUP_PLANE_RES)};
}

// Complex elements of one volume's grouped copy.
__host__ __device__ constexpr long long grouped_volume_elems(int Dv, int nt)
{
    return (long long)Dv * group_pitch(Dv, nt).plane * nt;
}

// Launch-wide geometry of one call, passed by value.
struct Geom {
    int n_rec, n_pose;
    int rot_shared, sh_shared;  // 1 when n_rot == 1 (resp. n_sh == 1)
    int Dv, Hv, halfv;          // reconstruction box, half-axis length, Dv / 2
    int Do, Ho, halfo;          // image box
    int centered;               // layout of every full axis
    int has_shift;
    int o_is_one;
    float o;
    float Do_f, inv_Do;
    int rc2;                    // keep pixel iff kx^2 + ky^2 <= rc2 (integer)
    long long rec_elems;        // elements of one reconstruction
    long long img_elems;        // elements of one image (Do * Ho)
    int grow, gplane;           // grouped copy (3D): group_pitch(Dv, NT of the call)
};

// ---------------------------------------------------------------- indexing -----

// Frequency held at storage row i of a full axis (image side).
__device__ __forceinline__ int row_freq(int i, int D, int half, int centered)
{
    return centered ? i - half : (i < half ? i : i - D);
}

// Storage index of frequency f on a full axis of length D, or -1 when f lies outside
// [-D/2, D/2 - 1] (that sample of the extended spectrum is zero).
__device__ __forceinline__ int full_index(int f, int D, int half, int centered)
{
    const bool ok = (unsigned)(f + half) < (unsigned)D;
    const int i = centered ? f + half : (f < 0 ? f + D : f);
    return ok ? i : -1;
}

// Linear pixel index p of an image with Ho columns -> (row, column).
__device__ __forceinline__ void split_pixel(int p, int Ho, int& i, int& j)
{
    i = (int)((unsigned)p / (unsigned)Ho);
    j = p - i * Ho;
}

// ------------------------------------------------------ error-free arithmetic --

struct dfloat {
    float hi, lo;
};

__device__ __forceinline__ dfloat two_prod(float a, float b)
{
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ dfloat two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

// r0 * x + r1 * y as hi + lo (error below 2^-46 relative).
__device__ __forceinline__ dfloat dot2(float r0, float x, float r1, float y)
{
    const dfloat p = two_prod(r0, x);
    const dfloat q = two_prod(r1, y);
    const dfloat s = two_sum(p.hi, q.hi);
    return {s.hi, __fadd_rn(__fadd_rn(p.lo, q.lo), s.lo)};
}

// o * (hi + lo) as hi + lo (exact up to the rounding of the low part); c itself when o = 1.
__device__ __forceinline__ dfloat scale_coord(dfloat c, float o, int o_is_one)
{
    if (!o_is_one) {
        const dfloat h = two_prod(o, c.hi);
        c = {h.hi, __fmaf_rn(o, c.lo, h.lo)};
    }
    return c;
}

// floor and fraction of hi + lo (already scaled).  frac is in [0, 1]; the value 1 can only
// come from rounding of an fp32 fraction just below 1, and both the kernels and their
// derivatives are continuous there (cubic) or take the neighbouring cell's value (linear),
// so either reading samples the same interpolant.
__device__ __forceinline__ void floor_split(dfloat c, int& base, float& frac)
{
    // Beyond +-2^23 every tap lies outside any supported box; clamping keeps the integer
    // tap indices far from overflow for any input (a NaN coordinate clamps too, and its
    // NaN weights propagate to the output without touching memory out of range).
    c.hi = fminf(fmaxf(c.hi, -8388608.0f), 8388608.0f);
    float fl = floorf(c.hi);
    float fr = __fadd_rn(__fsub_rn(c.hi, fl), c.lo);
    if (fr < 0.f) {
        fl -= 1.f;
        fr = __fadd_rn(fr, 1.f);
    } else if (fr >= 1.f) {
        fl += 1.f;
        fr = __fsub_rn(fr, 1.f);
    }
    base = (int)fl;
    frac = fr;
}

// floor and fraction of o * (hi + lo).
__device__ __forceinline__ void floor_frac(dfloat c, float o, int o_is_one, int& base, float& frac)
{
    floor_split(scale_coord(c, o, o_is_one), base, frac);
}

// ----------------------------------------------------------------- weights -----

// Interpolation weights of the taps floor(c) + first + k as polynomials in f = frac(c),
// and their derivatives d/dc.  Linear: (1 - f, f).  Cubic: Keys' convolution kernel with
// a = -1/2 evaluated at distances f + 1, f, f - 1, f - 2.
template <int INTERP>
__device__ __forceinline__ void weights(float f, float* w)
{
    if constexpr (INTERP == kCubic) {
        w[0] = f * (f * (-0.5f * f + 1.0f) - 0.5f);
        w[1] = f * f * (1.5f * f - 2.5f) + 1.0f;
        w[2] = f * (f * (-1.5f * f + 2.0f) + 0.5f);
        w[3] = f * f * (0.5f * f - 0.5f);
    } else {
        w[0] = 1.0f - f;
        w[1] = f;
    }
}

template <int INTERP>
__device__ __forceinline__ void dweights(float f, float* d)
{
    if constexpr (INTERP == kCubic) {
        d[0] = f * (-1.5f * f + 2.0f) - 0.5f;
        d[1] = f * (4.5f * f - 5.0f);
        d[2] = f * (-4.5f * f + 4.0f) + 0.5f;
        d[3] = f * (1.5f * f - 1.0f);
    } else {
        d[0] = -1.0f;
        d[1] = 1.0f;
    }
}

// ------------------------------------------------------------------- phase -----

// exp(-2 pi i (kx sx + ky sy) / Do), with the turn count reduced exactly before the
// sine and cosine are taken.
__device__ __forceinline__ float2 shift_phase(float kx, float ky, float sx, float sy,
                                              float Do_f, float inv_Do)
{
    const dfloat s = dot2(sx, kx, sy, ky);
    const float th = __fmul_rn(s.hi, inv_Do);
    const float res = __fmaf_rn(-th, Do_f, s.hi);  // s.hi - th * Do, exact
    const float tl = __fmul_rn(__fadd_rn(res, s.lo), inv_Do);
    const float n = rintf(th);
    const float t = __fadd_rn(__fsub_rn(th, n), tl);
    float sn, cs;
    sincospif(2.0f * t, &sn, &cs);
    return make_float2(cs, -sn);
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b)
{
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// a * conj(b)
__device__ __forceinline__ float2 cmul_conj(float2 a, float2 b)
{
    return make_float2(a.x * b.x + a.y * b.y, a.y * b.x - a.x * b.y);
}

// ------------------------------------------------------------ tap geometry -----

// Everything one output pixel needs to touch its taps: the tap origin on each axis, the
// storage index of every direct (t) and mirrored (-t) full-axis tap, and the weights.
template <int NDIM, int INTERP, bool DERIV>
struct PixelTaps {
    static constexpr int NT = Taps<INTERP>::N;
    static constexpr int NZ = NDIM == 3 ? NT : 1;
    int t0x;             // first x tap (may be negative: mirrored)
    int iyd[NT], iym[NT];  // row index of direct / mirrored y taps (-1 = zero)
    int izd[NZ], izm[NZ];  // plane index of direct / mirrored z taps (3D)
    float wx[NT], wy[NT], wz[NZ];
    float dx[DERIV ? NT : 1], dy[DERIV ? NT : 1], dz[DERIV ? NZ : 1];

    // c = o * R q for q = (kx, ky[, 0]); R row-major k x k in shared/registers.
    __device__ __forceinline__ void init(const Geom& g, const float* R, float kx, float ky)
    {
        int b;
        float f;
        constexpr int K = NDIM;
        // x
        floor_frac(dot2(R[0], kx, R[1], ky), g.o, g.o_is_one, b, f);
        t0x = b + Taps<INTERP>::first;
        weights<INTERP>(f, wx);
        if constexpr (DERIV) dweights<INTERP>(f, dx);
        // y
        floor_frac(dot2(R[K], kx, R[K + 1], ky), g.o, g.o_is_one, b, f);
        weights<INTERP>(f, wy);
        if constexpr (DERIV) dweights<INTERP>(f, dy);
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const int t = b + Taps<INTERP>::first + k;
            iyd[k] = full_index(t, g.Dv, g.halfv, g.centered);
            iym[k] = full_index(-t, g.Dv, g.halfv, g.centered);
        }
        if constexpr (NDIM == 3) {
            floor_frac(dot2(R[6], kx, R[7], ky), g.o, g.o_is_one, b, f);
            weights<INTERP>(f, wz);
            if constexpr (DERIV) dweights<INTERP>(f, dz);
#pragma unroll
            for (int k = 0; k < NT; ++k) {
                const int t = b + Taps<INTERP>::first + k;
                izd[k] = full_index(t, g.Dv, g.halfv, g.centered);
                izm[k] = full_index(-t, g.Dv, g.halfv, g.centered);
            }
        } else {
            izd[0] = 0;
            izm[0] = 0;
            wz[0] = 1.0f;
            if constexpr (DERIV) dz[0] = 0.0f;
        }
    }

    // Element offset of the row (z tap a, y tap b) within one reconstruction for the
    // direct (mirror = false) or mirrored taps; -1 when that row is outside the band.
    __device__ __forceinline__ int row(const Geom& g, int a, int b, bool mirror) const
    {
        const int iz = mirror ? izm[a] : izd[a];
        const int iy = mirror ? iym[b] : iyd[b];
        return (iz | iy) < 0 ? -1 : (iz * g.Dv + iy) * g.Hv;
    }
};

}  // namespace tp

namespace tp {

// ------------------------------------------------------------ gather / scatter --

// v = sum_t w(c - t) V_ext(t) over the pixel's taps and, when DERIV, dv[a] = dv/dc_a.
// Each x tap is read directly (t_x >= 0) or from the conjugate mirror (t_x < 0); the
// mirror also negates the y and z taps, whose row offsets come precomputed in `t`.
template <int NDIM, int INTERP, bool DERIV>
__device__ __forceinline__ void gather(const float2* __restrict__ V, const Geom& g,
                                       const PixelTaps<NDIM, INTERP, DERIV>& t, float2& v,
                                       float2* dv)
{
    constexpr int NT = Taps<INTERP>::N;
    constexpr int NZ = NDIM == 3 ? NT : 1;
    v = make_float2(0.f, 0.f);
    if constexpr (DERIV) {
        dv[0] = dv[1] = dv[2] = make_float2(0.f, 0.f);
    }
    // y rows outer, z planes inner: the order of the fast path's gather_fast, so a pixel
    // gives the same bits on either path when both read the same tap values
#pragma unroll
    for (int b = 0; b < NT; ++b) {
#pragma unroll
        for (int a = 0; a < NZ; ++a) {
            const int rd = t.row(g, a, b, false);
            const int rm = t.row(g, a, b, true);
            float2 rs = make_float2(0.f, 0.f), rsd = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < NT; ++k) {
                const int tx = t.t0x + k;
                const bool m = tx < 0;
                const int ax = m ? -tx : tx;
                const int r = m ? rm : rd;
                float2 val = make_float2(0.f, 0.f);
                if (r >= 0 && ax <= g.halfv) val = __ldg(V + r + ax);
                if (m) val.y = -val.y;
                rs.x = fmaf(t.wx[k], val.x, rs.x);
                rs.y = fmaf(t.wx[k], val.y, rs.y);
                if constexpr (DERIV) {
                    rsd.x = fmaf(t.dx[k], val.x, rsd.x);
                    rsd.y = fmaf(t.dx[k], val.y, rsd.y);
                }
            }
            const float wzy = t.wz[a] * t.wy[b];
            v.x = fmaf(wzy, rs.x, v.x);
            v.y = fmaf(wzy, rs.y, v.y);
            if constexpr (DERIV) {
                dv[0].x = fmaf(wzy, rsd.x, dv[0].x);
                dv[0].y = fmaf(wzy, rsd.y, dv[0].y);
                const float wzdy = t.wz[a] * t.dy[b];
                dv[1].x = fmaf(wzdy, rs.x, dv[1].x);
                dv[1].y = fmaf(wzdy, rs.y, dv[1].y);
                if constexpr (NDIM == 3) {
                    const float dzwy = t.dz[a] * t.wy[b];
                    dv[2].x = fmaf(dzwy, rs.x, dv[2].x);
                    dv[2].y = fmaf(dzwy, rs.y, dv[2].y);
                }
            }
        }
    }
}

// Real-volume variant of gather() for the weight volume: V_ext(t) = W[t] (t_x >= 0) or
// W[-t] (t_x < 0) -- the Friedel mirror of a real array needs no conjugation.
template <int NDIM, int INTERP, bool DERIV>
__device__ __forceinline__ void gather_real(const float* __restrict__ Wv, const Geom& g,
                                            const PixelTaps<NDIM, INTERP, DERIV>& t, float& v,
                                            float* dv)
{
    constexpr int NT = Taps<INTERP>::N;
    constexpr int NZ = NDIM == 3 ? NT : 1;
    v = 0.f;
    if constexpr (DERIV) dv[0] = dv[1] = dv[2] = 0.f;
#pragma unroll
    for (int a = 0; a < NZ; ++a) {
#pragma unroll
        for (int b = 0; b < NT; ++b) {
            const int rd = t.row(g, a, b, false);
            const int rm = t.row(g, a, b, true);
            float rs = 0.f, rsd = 0.f;
#pragma unroll
            for (int k = 0; k < NT; ++k) {
                const int tx = t.t0x + k;
                const bool m = tx < 0;
                const int ax = m ? -tx : tx;
                const int r = m ? rm : rd;
                const float val = (r >= 0 && ax <= g.halfv) ? __ldg(Wv + r + ax) : 0.f;
                rs = fmaf(t.wx[k], val, rs);
                if constexpr (DERIV) rsd = fmaf(t.dx[k], val, rsd);
            }
            const float wzy = t.wz[a] * t.wy[b];
            v = fmaf(wzy, rs, v);
            if constexpr (DERIV) {
                dv[0] = fmaf(wzy, rsd, dv[0]);
                dv[1] = fmaf(t.wz[a] * t.dy[b], rs, dv[1]);
                if constexpr (NDIM == 3) dv[2] = fmaf(t.dz[a] * t.wy[b], rs, dv[2]);
            }
        }
    }
}

// Transpose of gather(): G[t] += w(c - t) val for t_x >= 0 and G[-t] += conj(w(c - t) val)
// for t_x < 0; W (real) receives w(c - t) wt on the same element, without conjugation.
// Either destination may be null.
template <int NDIM, int INTERP, bool DERIV>
__device__ __forceinline__ void scatter(float2* __restrict__ G, float* __restrict__ W,
                                        const Geom& g, const PixelTaps<NDIM, INTERP, DERIV>& t,
                                        float2 val, float wt)
{
    constexpr int NT = Taps<INTERP>::N;
    constexpr int NZ = NDIM == 3 ? NT : 1;
#pragma unroll
    for (int a = 0; a < NZ; ++a) {
#pragma unroll
        for (int b = 0; b < NT; ++b) {
            const int rd = t.row(g, a, b, false);
            const int rm = t.row(g, a, b, true);
            const float wzy = t.wz[a] * t.wy[b];
#pragma unroll
            for (int k = 0; k < NT; ++k) {
                const int tx = t.t0x + k;
                const bool m = tx < 0;
                const int ax = m ? -tx : tx;
                const int r = m ? rm : rd;
                if (r >= 0 && ax <= g.halfv) {
                    const float w = wzy * t.wx[k];
                    if (G) atomicAdd(G + r + ax, make_float2(w * val.x, m ? -w * val.y : w * val.y));
                    if (W) atomicAdd(W + r + ax, w * wt);
                }
            }
        }
    }
}

// Per-item parameters staged once per CTA: rotation (k x k) and shift.
template <int NDIM>
struct ItemParams {
    float R[NDIM * NDIM];
    float sx, sy;
};

template <int NDIM>
__device__ __forceinline__ void load_item(const Geom& g, const float* __restrict__ rot,
                                          const float* __restrict__ shift, int r, int p,
                                          ItemParams<NDIM>& ip)
{
    const long long ri = (long long)(g.rot_shared ? 0 : r) * g.n_pose + p;
#pragma unroll
    for (int k = 0; k < NDIM * NDIM; ++k) ip.R[k] = __ldg(rot + ri * NDIM * NDIM + k);
    ip.sx = ip.sy = 0.f;
    if (g.has_shift) {
        const long long si = (long long)(g.sh_shared ? 0 : r) * g.n_pose + p;
        ip.sx = __ldg(shift + si * 2);
        ip.sy = __ldg(shift + si * 2 + 1);
    }
}

}  // namespace tp
