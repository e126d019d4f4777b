// gather.cuh -- fast interpolation gather for pixels whose taps are all read directly.
//
// Effective frame.  For a pixel with c_x < 0 the sample is taken at c' = -c and
// conjugated: with a symmetric kernel, v(c) = conj(sum_u w(c' - u) Z(u)) where Z(u) = V[u]
// for u_x > 0 (Friedel symmetry of the half spectrum, F(-k) = conj F(k); torch-projectors
// summaries, Method section, Friedel bullet).  So every pixel whose effective taps satisfy
// 1 <= u_x <= Dv/2 reads V[u] directly, whatever the sign of c_x; only pixels whose taps
// touch the x = 0 plane (|c_x| < 2 for cubic) or the x = Dv/2 edge need the per-tap rule.
// y / z taps outside the stored band get weight 0 and read a valid row instead.
//
// Rows of 4 (cubic) or 2 (linear) consecutive x taps are read as aligned vector windows:
//   WIN = 1: one 8-byte load per tap;
//   WIN = 2: 16-byte loads of an even-aligned window (6 elements for cubic);
//   WIN = 4: 32-byte loads of a 4-aligned window (8 elements for cubic).
// The window's alignment shift depends only on the y row (the z plane stride Dv*Hv is a
// multiple of the window for WIN = 2, and of 4 elements when Dv % 4 == 0, which the host
// requires for WIN = 4), so the shifted x weights are formed once per y tap.
//   WIN = kGrouped: rows read from the grouped copy of the volume (see expand_groups in
//   kernels.cu), where group i of a row holds the NT taps i .. i + NT - 1: one aligned
//   32-byte (cubic) or 16-byte (linear) load per row, always within one sector.  Its rows
//   also hold the groups starting at x = -(NT - 1) .. -1, whose taps left of x = 0 are the
//   conjugate mirror values, so pixels near the x = 0 plane read it in the original frame.
#pragma once

#include "tp_device.cuh"

namespace tp {

constexpr int kGrouped = 8;  // WIN tag of the grouped-row reader

__device__ __forceinline__ float4 ldg_v4(const float2* p)
{
    return __ldg(reinterpret_cast<const float4*>(p));
}

// 32-byte read-only load (ld.global.nc.v8.f32); p must be 32-byte aligned.
__device__ __forceinline__ void ldg_v8(const float2* p, float* e)
{
    asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(e[0]), "=f"(e[1]), "=f"(e[2]), "=f"(e[3]), "=f"(e[4]), "=f"(e[5]),
                   "=f"(e[6]), "=f"(e[7])
                 : "l"(p));
}

// Per-pixel tap data of the fast path (effective frame).
template <int NDIM, int INTERP, bool DERIV>
struct FastTaps {
    static constexpr int NT = Taps<INTERP>::N;
    static constexpr int NZ = NDIM == 3 ? NT : 1;
    int x0;            // first x tap (>= 1; >= -(NT - 1) on the grouped copy)
    int zoff[NZ];      // iz * Dv * row length (0 for 2D)
    int yrow[NT];      // iy * row length
    float wx[NT], wy[NT], wz[NZ];
    float dx[DERIV ? NT : 1], dy[DERIV ? NT : 1], dz[DERIV ? NZ : 1];
};

// Set up the effective-frame taps of a pixel.  Returns false when the pixel needs the
// general per-tap path.  `flip` is set when the sample is conjugated.
//   EXT = false (volume read in place): every pixel with c_x < 0 is flipped, and the pixel is
//   fast when its taps lie in 1 <= x <= Dv/2.
//   EXT = true (grouped copy, whose rows also hold the mirrored taps x = -(NT-1) .. -1):
//   only pixels with o c_x <= -NT/2 are flipped, which puts their first tap at x >= 1, and
//   the rest are read in the original frame, first tap x >= -(NT - 1).  A tap left of x = 0
//   then reads the mirrored row (-y, -z); when a direct y or z tap of such a pixel lies
//   outside the stored band its mirror may not, and the pixel takes the general path.
template <int NDIM, int INTERP, bool DERIV, bool EXT>
__device__ __forceinline__ bool fast_taps(const Geom& g, const float* R, float kx, float ky,
                                          FastTaps<NDIM, INTERP, DERIV>& t, bool& flip)
{
    constexpr int NT = Taps<INTERP>::N;
    constexpr int K = NDIM;
    const int hv = EXT ? g.grow : g.Hv;  // row pitch in elements (groups)
    dfloat cx = dot2(R[0], kx, R[1], ky);
    dfloat cy = dot2(R[K], kx, R[K + 1], ky);
    int b;
    float f;
    if constexpr (EXT) {
        // decided on o c_x: negation commutes exactly with the scaling by o
        cx = scale_coord(cx, g.o, g.o_is_one);
        constexpr float T = -0.5f * NT;
        flip = cx.hi < T || (cx.hi == T && cx.lo <= 0.f);
        if (flip) {
            cx = {-cx.hi, -cx.lo};
            cy = {-cy.hi, -cy.lo};
        }
        floor_split(cx, b, f);
    } else {
        flip = cx.hi < 0.f || (cx.hi == 0.f && cx.lo < 0.f);
        if (flip) {
            cx = {-cx.hi, -cx.lo};
            cy = {-cy.hi, -cy.lo};
        }
        floor_frac(cx, g.o, g.o_is_one, b, f);
    }
    t.x0 = b + Taps<INTERP>::first;
    if (t.x0 < (EXT ? 1 - NT : 1) || t.x0 + NT - 1 > g.halfv) return false;
    weights<INTERP>(f, t.wx);
    if constexpr (DERIV) dweights<INTERP>(f, t.dx);
    floor_frac(cy, g.o, g.o_is_one, b, f);
    weights<INTERP>(f, t.wy);
    if constexpr (DERIV) dweights<INTERP>(f, t.dy);
    bool outside = false;  // a direct y or z tap outside the stored band
#pragma unroll
    for (int k = 0; k < NT; ++k) {
        const int iy = full_index(b + Taps<INTERP>::first + k, g.Dv, g.halfv, g.centered);
        if (iy < 0) {
            t.wy[k] = 0.f;
            if constexpr (DERIV) t.dy[k] = 0.f;
            outside = true;
        }
        t.yrow[k] = (iy < 0 ? 0 : iy) * hv;
    }
    if constexpr (NDIM == 3) {
        dfloat cz = dot2(R[6], kx, R[7], ky);
        if (flip) cz = {-cz.hi, -cz.lo};
        floor_frac(cz, g.o, g.o_is_one, b, f);
        weights<INTERP>(f, t.wz);
        if constexpr (DERIV) dweights<INTERP>(f, t.dz);
        const int plane = EXT ? g.gplane : g.Dv * g.Hv;
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const int iz = full_index(b + Taps<INTERP>::first + k, g.Dv, g.halfv, g.centered);
            if (iz < 0) {
                t.wz[k] = 0.f;
                if constexpr (DERIV) t.dz[k] = 0.f;
                outside = true;
            }
            t.zoff[k] = (iz < 0 ? 0 : iz) * plane;
        }
    } else {
        t.zoff[0] = 0;
        t.wz[0] = 1.f;
        if constexpr (DERIV) t.dz[0] = 0.f;
    }
    return !(EXT && outside && t.x0 < 0);
}

// Row sums over the x taps of one row: rs = sum_k wx[k] V[row + x0 + k] and, with DERIV,
// rsd = sum_k dx[k] V[...].  `ws` / `wds` are the window-shifted weights of this y row.
template <int INTERP, int WIN, bool DERIV>
struct RowReader;

// One 8-byte load per tap.
template <int INTERP, bool DERIV>
struct RowReader<INTERP, 1, DERIV> {
    static constexpr int NT = Taps<INTERP>::N;
    static constexpr int NW = NT;
    __device__ __forceinline__ static int shift(const float2*, int) { return 0; }
    __device__ __forceinline__ static void shifted(int, const float* w, float* ws)
    {
#pragma unroll
        for (int k = 0; k < NT; ++k) ws[k] = w[k];
    }
    __device__ __forceinline__ static void read(const float2* __restrict__ p, int, const float* ws,
                                                const float* wds, float2& rs, float2& rsd)
    {
        rs = make_float2(0.f, 0.f);
        rsd = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const float2 e = __ldg(p + k);
            rs.x = fmaf(ws[k], e.x, rs.x);
            rs.y = fmaf(ws[k], e.y, rs.y);
            if constexpr (DERIV) {
                rsd.x = fmaf(wds[k], e.x, rsd.x);
                rsd.y = fmaf(wds[k], e.y, rsd.y);
            }
        }
    }
};

// 16-byte loads of the even-aligned window [p - s, p - s + NT + 2).
template <int INTERP, bool DERIV>
struct RowReader<INTERP, 2, DERIV> {
    static constexpr int NT = Taps<INTERP>::N;
    static constexpr int NW = NT + 1;  // window elements that can carry a weight
    __device__ __forceinline__ static int shift(const float2* p, int)
    {
        return (int)((reinterpret_cast<uintptr_t>(p) >> 3) & 1);
    }
    __device__ __forceinline__ static void shifted(int s, const float* w, float* ws)
    {
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const float a = j < NT ? w[j] : 0.f;
            const float b = j >= 1 ? w[j - 1] : 0.f;
            ws[j] = s ? b : a;
        }
    }
    __device__ __forceinline__ static void read(const float2* __restrict__ p, int s,
                                                const float* ws, const float* wds, float2& rs,
                                                float2& rsd)
    {
        const float2* q = p - s;
        float e[2 * (NT + 2)];
#pragma unroll
        for (int c = 0; c < NT / 2; ++c) {
            const float4 v = ldg_v4(q + 2 * c);
            e[4 * c] = v.x;
            e[4 * c + 1] = v.y;
            e[4 * c + 2] = v.z;
            e[4 * c + 3] = v.w;
        }
        e[2 * NT] = e[2 * NT + 1] = e[2 * NT + 2] = e[2 * NT + 3] = 0.f;
        if (s) {
            const float4 v = ldg_v4(q + NT);
            e[2 * NT] = v.x;
            e[2 * NT + 1] = v.y;
        }
        rs = make_float2(0.f, 0.f);
        rsd = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            rs.x = fmaf(ws[j], e[2 * j], rs.x);
            rs.y = fmaf(ws[j], e[2 * j + 1], rs.y);
            if constexpr (DERIV) {
                rsd.x = fmaf(wds[j], e[2 * j], rsd.x);
                rsd.y = fmaf(wds[j], e[2 * j + 1], rsd.y);
            }
        }
    }
};

// 32-byte loads of the 4-aligned window [p - s, p - s + 8).
template <int INTERP, bool DERIV>
struct RowReader<INTERP, 4, DERIV> {
    static constexpr int NT = Taps<INTERP>::N;
    static constexpr int NW = NT + 3;
    __device__ __forceinline__ static int shift(const float2* p, int)
    {
        return (int)((reinterpret_cast<uintptr_t>(p) >> 3) & 3);
    }
    __device__ __forceinline__ static void shifted(int s, const float* w, float* ws)
    {
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const float a0 = j < NT ? w[j] : 0.f;
            const float a1 = (j >= 1 && j - 1 < NT) ? w[j - 1] : 0.f;
            const float a2 = (j >= 2 && j - 2 < NT) ? w[j - 2] : 0.f;
            const float a3 = (j >= 3 && j - 3 < NT) ? w[j - 3] : 0.f;
            ws[j] = s == 0 ? a0 : (s == 1 ? a1 : (s == 2 ? a2 : a3));
        }
    }
    __device__ __forceinline__ static void read(const float2* __restrict__ p, int s,
                                                const float* ws, const float* wds, float2& rs,
                                                float2& rsd)
    {
        const float2* q = p - s;
        float e[16];
        ldg_v8(q, e);
#pragma unroll
        for (int k = 8; k < 16; ++k) e[k] = 0.f;
        if (s + NT > 4) ldg_v8(q + 4, e + 8);
        rs = make_float2(0.f, 0.f);
        rsd = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            rs.x = fmaf(ws[j], e[2 * j], rs.x);
            rs.y = fmaf(ws[j], e[2 * j + 1], rs.y);
            if constexpr (DERIV) {
                rsd.x = fmaf(wds[j], e[2 * j], rsd.x);
                rsd.y = fmaf(wds[j], e[2 * j + 1], rsd.y);
            }
        }
    }
};

// Grouped rows: p points at a group of NT consecutive taps (32-byte aligned for cubic,
// 16-byte aligned for linear).
template <int INTERP, bool DERIV>
struct RowReader<INTERP, kGrouped, DERIV> {
    static constexpr int NT = Taps<INTERP>::N;
    static constexpr int NW = NT;
    __device__ __forceinline__ static int shift(const float2*, int) { return 0; }
    __device__ __forceinline__ static void shifted(int, const float* w, float* ws)
    {
#pragma unroll
        for (int k = 0; k < NT; ++k) ws[k] = w[k];
    }
    __device__ __forceinline__ static void read(const float2* __restrict__ p, int, const float* ws,
                                                const float* wds, float2& rs, float2& rsd)
    {
        float e[2 * NT];
        if constexpr (NT == 4) {
            ldg_v8(p, e);
        } else {
            const float4 v = ldg_v4(p);
            e[0] = v.x;
            e[1] = v.y;
            e[2] = v.z;
            e[3] = v.w;
        }
        rs = make_float2(0.f, 0.f);
        rsd = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            rs.x = fmaf(ws[j], e[2 * j], rs.x);
            rs.y = fmaf(ws[j], e[2 * j + 1], rs.y);
            if constexpr (DERIV) {
                rsd.x = fmaf(wds[j], e[2 * j], rsd.x);
                rsd.y = fmaf(wds[j], e[2 * j + 1], rsd.y);
            }
        }
    }
};

// v (and dv when DERIV) in the effective frame: sum over rows (z tap a, y tap b).  With
// WIN = kGrouped, V is the item's grouped volume (NT elements per voxel).
template <int NDIM, int INTERP, int WIN, bool DERIV>
__device__ __forceinline__ void gather_fast(const float2* __restrict__ V,
                                            const FastTaps<NDIM, INTERP, DERIV>& t, float2& v,
                                            float2* dv)
{
    using RR = RowReader<INTERP, WIN, DERIV>;
    constexpr int NT = Taps<INTERP>::N;
    constexpr int NZ = NDIM == 3 ? NT : 1;
    v = make_float2(0.f, 0.f);
    if constexpr (DERIV) dv[0] = dv[1] = dv[2] = make_float2(0.f, 0.f);
    constexpr int M = WIN == kGrouped ? NT : 1;  // elements per voxel of V
    // the grouped copy's rows start at x = -(NT - 1)
    const float2* Vx = V + M * (t.x0 + (WIN == kGrouped ? NT - 1 : 0));
#pragma unroll
    for (int b = 0; b < NT; ++b) {
        // the window shift depends on the y row only (plane strides keep the alignment)
        const int s = RR::shift(Vx + t.yrow[b], 0);
        float ws[RR::NW], wds[DERIV ? RR::NW : 1];
        RR::shifted(s, t.wx, ws);
        if constexpr (DERIV) RR::shifted(s, t.dx, wds);
#pragma unroll
        for (int a = 0; a < NZ; ++a) {
            float2 rs, rsd;
            RR::read(Vx + M * (t.zoff[a] + t.yrow[b]), s, ws, wds, rs, rsd);
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

}  // namespace tp
