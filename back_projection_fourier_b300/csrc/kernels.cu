// kernels.cu -- forward projection, backward gradients and back-projection kernels.
//
// Operations (torch-projectors paper summaries, gist.science, Method section, list of
// operations): 3D->2D forward (central slice theorem), 2D->3D backward (accumulation in a
// 3D volume), 2D->2D forward (rotation of 2D Fourier data) and 2D->2D backward
// (accumulation into a 2D reconstruction); gradients for inputs, rotations and shifts
// without stored intermediates (differentiation bullet); shifts by phase modulation.
//
// Gather kernels (forward projection; rotation / shift gradients).  A CTA owns one work
// unit at a time (grid-stride): an item (reconstruction r, pose p), or a chunk of one item's
// pixels when the batch has fewer items than resident CTAs.  Threads walk only the kept
// pixels (kx^2 + ky^2 <= rc^2) through a per-CTA table of row offsets, in row-major order,
// so image reads and writes stay coalesced.  Pixels whose taps are all read directly (the
// vast majority, see gather.cuh) take the fast path, reading each row of taps either from
// the volume in aligned vector windows or, with a workspace, from the grouped copy in one
// aligned load; the others -- taps on the x = 0 plane or past x = Dv/2 -- are queued in
// shared memory and evaluated densely with the exact per-tap rule, so they do not make whole
// warps diverge (with the grouped copy, whose rows also hold the mirrored taps left of x = 0,
// only taps past x = Dv/2 and a few band-edge cases remain).  The volume (and its grouped copy
// at D <= 128) stays L2-resident: a D = 256 half volume is 68 MB of a 126 MB L2.
//
// Scatter kernels (volume gradient, insertion).  3D cubic: scatter_tile_kernel, a warp per
// 4 x 4 pixel tile with a private shared-memory box, lanes on a pixel's 64 taps; its POSE
// instance is the one-pass backward.  3D linear: scatter_lane_kernel, a pixel per lane.  2D
// cubic with weights: scatter_tile2d_kernel, a tile per half-warp.  Other 2D: the
// owner-computes scatter_rows_kernel.  Boxes beyond the shared tables: backproject_kernel.
#include "gather.cuh"
#include "kernels.h"
#include "scatter.cuh"

// Width of the vector window used by the gather fast path: 1 (8-byte taps), 2 (16-byte
// loads) or 4 (32-byte loads).
#ifndef TP_GATHER_WIN
#define TP_GATHER_WIN 2
#endif

namespace tp {

namespace {

constexpr int kThreads = 256;
// The pose-gradient gather runs in CTAs of 128 threads: at its 128 registers per thread that
// is 4 CTAs per SM (4 items in flight) instead of 2, with cheaper per-item reductions.
constexpr int kPoseThreads = 128;
// The 3D forward gather: CTAs of 192 threads, 4 per SM (24 warps): cheaper CTA barriers
// around its shared slow-pixel queue than 256 x 3, with the same registers per thread.
constexpr int kFwd3Threads = 192;
#ifndef TP_ROWS_THREADS
#define TP_ROWS_THREADS 256
#endif
// The 2D owner-computes scatter: CTAs of this many threads, a thread per output row segment
// (128 measured the same, 64 slower).
constexpr int kRowsThreads = TP_ROWS_THREADS;
constexpr int kMaxTableRows = 4096;  // image boxes up to this size use the kept-pixel table

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

// ------------------------------------------------------------ shared tables ----

__device__ __forceinline__ int isqrt_floor(int m)
{
    int k = (int)sqrtf((float)m);
    while (k > 0 && k * k > m) --k;
    while ((k + 1) * (k + 1) <= m) ++k;
    return k;
}

// Kept pixels of image row i: kx in [0, count).
__device__ __forceinline__ int row_kept(const Geom& g, int i)
{
    const int ky = row_freq(i, g.Do, g.halfo, g.centered);
    const int m = g.rc2 - ky * ky;
    if (m < 0) return 0;
    const int k = isqrt_floor(m);
    return (k < g.halfo ? k : g.halfo) + 1;
}

// rowstart[i] = kept pixels in rows < i, for i = 0..Do (exclusive scan over a CTA of BT).
template <int BT = kThreads>
__device__ void build_rowstart(const Geom& g, int* rowstart, int* scratch)
{
    const int per = (g.Do + BT - 1) / BT;
    const int i0 = threadIdx.x * per;
    int sum = 0;
    for (int k = 0; k < per; ++k)
        if (i0 + k < g.Do) sum += row_kept(g, i0 + k);
    // inclusive warp scan, then the warp totals
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < BT / 32; ++w) {
            const int t = scratch[w];
            scratch[w] = acc;
            acc += t;
        }
    }
    __syncthreads();
    int run = scratch[warp] + inc - sum;
    for (int k = 0; k < per; ++k)
        if (i0 + k < g.Do) {
            rowstart[i0 + k] = run;
            run += row_kept(g, i0 + k);
        }
    if (threadIdx.x == BT - 1) rowstart[g.Do] = run;
    __syncthreads();
}

// Slow-path queue of one warp: 64 shared-memory slots of (row << 16) | kx.  The warp appends
// its slow pixels (one ballot) and evaluates them 32 at a time, one per lane, so they do not
// make the warp diverge; the rest are drained at the end of the work unit.  Warp-synchronous:
// the pixel loops need no CTA-wide barrier.
constexpr int kWarpQueue = 64;

struct WarpQueue {
    int* slots;  // this warp's kWarpQueue slots
    int count;   // entries waiting (the same in every lane)

    __device__ __forceinline__ void push(bool slow, int row, int kx)
    {
        const unsigned mask = __ballot_sync(0xffffffffu, slow);
        const int lane = threadIdx.x & 31;
        if (slow) slots[count + __popc(mask & ((1u << lane) - 1))] = (row << 16) | kx;
        count += __popc(mask);
        __syncwarp();
    }
};

// Slow-path queue of a whole CTA (kept for the 3D forward, whose warps gain from staying
// on neighbouring image rows): the CTA appends its slow pixels and, at CTA barriers,
// evaluates them one round of threads at a time.
struct CtaQueue {
    int* slots;  // [kWarpQueue * warps of the CTA] = [2 * threads]
    int* count;  // shared counter
};

__device__ __forceinline__ void cta_enqueue(CtaQueue q, bool slow, int row, int kx)
{
    const unsigned mask = __ballot_sync(0xffffffffu, slow);
    if (!mask) return;
    const int lane = threadIdx.x & 31;
    int base = 0;
    if (lane == __ffs(mask) - 1) base = atomicAdd(q.count, __popc(mask));
    base = __shfl_sync(0xffffffffu, base, __ffs(mask) - 1);
    if (slow) q.slots[base + __popc(mask & ((1u << lane) - 1))] = (row << 16) | kx;
}

// Sum of a per-thread value over the CTA of BT threads, valid in thread 0.
template <int BT = kThreads>
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
        for (int k = 0; k < BT / 32; ++k) s += red[k];
    return s;
}

// Work split of one item's kept pixels over `splits` CTAs: chunks of whole CTA rounds.
template <int BT = kThreads>
__device__ __forceinline__ int kept_chunk(int nkept, int splits)
{
    return ((nkept + splits - 1) / splits + BT - 1) / BT * BT;
}

// Image row holding kept pixel n0: the largest row r < Do with rowstart[r] <= n0.
__device__ __forceinline__ int row_of_kept(const int* rowstart, int Do, int n0)
{
    int lo = 0, hi = Do - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (rowstart[mid] <= n0)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// ------------------------------------------------------- per-pixel evaluation ----

// Exact per-tap evaluation in the original frame (any pixel).
template <int NDIM, int INTERP, bool DERIV>
__device__ __forceinline__ void eval_general(const Geom& g, const float2* __restrict__ V,
                                             const float* R, int kx, int ky, float2& v,
                                             float2* dv)
{
    PixelTaps<NDIM, INTERP, DERIV> t;
    t.init(g, R, (float)kx, (float)ky);
    gather<NDIM, INTERP, DERIV>(V, g, t, v, dv);
}

// Effective-frame evaluation; false when the pixel needs the general path.
template <int NDIM, int INTERP, int WIN, bool DERIV>
__device__ __forceinline__ bool eval_fast(const Geom& g, const float2* __restrict__ V,
                                          const float* R, int kx, int ky, float2& v, float2* dv)
{
    FastTaps<NDIM, INTERP, DERIV> t;
    bool flip;
    if (!fast_taps<NDIM, INTERP, DERIV, WIN == kGrouped>(g, R, (float)kx, (float)ky, t, flip))
        return false;
    gather_fast<NDIM, INTERP, WIN, DERIV>(V, t, v, dv);
    if (flip) {
        // v(c) = conj(v'(-c)); dv/dc = -conj(dv'/dc')
        v.y = -v.y;
        if constexpr (DERIV) {
#pragma unroll
            for (int a = 0; a < 3; ++a) dv[a].x = -dv[a].x;
        }
    }
    return true;
}

// Separable shift twiddles of one item (2D gathers): tw[kx] = phase(kx, 0) for kx < Ho and
// tw[Ho + row] = phase(0, ky(row)) for the Do rows, so that a pixel's phase is one complex
// product of two table entries instead of a phase evaluation (each factor is computed with the
// exact turn reduction of shift_phase).  Two buffers alternate by work unit; the barrier after
// each build also orders the previous unit's reads of the other buffer before its next build.
constexpr int kMaxTwiddleRows = 1024;  // tables of at most 2 x (513 + 1024) entries, 24.6 KB

__host__ __device__ __forceinline__ bool use_twiddles(const Geom& g, int ndim)
{
    return ndim == 2 && g.Do <= kMaxTwiddleRows;
}

__device__ __forceinline__ float2* twiddle_table(int* after_queues)
{
    // 8-byte aligned start after the int tables
    const uintptr_t a = (reinterpret_cast<uintptr_t>(after_queues) + 7) & ~(uintptr_t)7;
    return reinterpret_cast<float2*>(a);
}

template <int BT>
__device__ __forceinline__ void build_twiddles(const Geom& g, float sx, float sy, float2* tw)
{
    for (int k = threadIdx.x; k < g.Ho + g.Do; k += BT)
        tw[k] = k < g.Ho ? shift_phase((float)k, 0.f, sx, sy, g.Do_f, g.inv_Do)
                         : shift_phase(0.f, (float)row_freq(k - g.Ho, g.Do, g.halfo, g.centered), sx,
                                       sy, g.Do_f, g.inv_Do);
    __syncthreads();
}

// ------------------------------------------------------------------ forward ----

template <int NDIM, int INTERP, int WIN>
__global__ void __launch_bounds__(NDIM == 3 ? kFwd3Threads : kThreads, 4) project_kernel(
    const float2* __restrict__ rec, const float* __restrict__ rot,
    const float* __restrict__ shift, float2* __restrict__ out, Geom g, int splits, long long n_work,
    const float2* __restrict__ grouped)
{
    constexpr int BT = NDIM == 3 ? kFwd3Threads : kThreads;  // threads of the CTA
    extern __shared__ int smem[];
    int* rowstart = smem;                    // [Do + 1]
    int* qslots = smem + g.Do + 1;           // [kWarpQueue per warp]
    __shared__ int scratch[BT / 32];
    __shared__ int qcount;
    build_rowstart<BT>(g, rowstart, scratch);
    if (threadIdx.x == 0) qcount = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    WarpQueue q{qslots + (threadIdx.x >> 5) * kWarpQueue, 0};  // 2D
    const CtaQueue cq{qslots, &qcount};                         // 3D
    const int nkept = rowstart[g.Do];
    const int npix = (int)g.img_elems;
    const int chunk = kept_chunk<BT>(nkept, splits);
    float2* const tw0 = twiddle_table(qslots + kWarpQueue * (BT / 32));  // 2D: [2][Ho + Do]
    int unit = 0;

    // work unit = (item, part): part takes one chunk of the item's kept pixels
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x, ++unit) {
        const ItemRange ir = item_of(g, w, splits);
        ItemParams<NDIM> ip;
        load_item<NDIM>(g, rot, shift, ir.r, ir.p, ip);
        float2* const tw = tw0 + (unit & 1) * (g.Ho + g.Do);
        const bool twid = use_twiddles(g, NDIM) && g.has_shift;
        if (twid) build_twiddles<BT>(g, ip.sx, ip.sy, tw);
        const float2* V = rec + (long long)ir.r * g.rec_elems;
        const float2* VG =
            WIN == kGrouped ? grouped + (long long)ir.r * g.Dv * g.gplane * Taps<INTERP>::N : V;
        float2* y = out + ir.item * g.img_elems;
        // pixels beyond the cutoff are zero
        for (int p = ir.part * BT + threadIdx.x; p < npix; p += splits * BT) {
            int i, j;
            split_pixel(p, g.Ho, i, j);
            if (j >= rowstart[i + 1] - rowstart[i]) y[p] = make_float2(0.f, 0.f);
        }
        auto finish = [&](int row, int kx, float2 val) {
            if (twid) {
                val = cmul(val, cmul(tw[kx], tw[g.Ho + row]));
            } else if (g.has_shift) {
                const int ky = row_freq(row, g.Do, g.halfo, g.centered);
                val = cmul(val, shift_phase((float)kx, (float)ky, ip.sx, ip.sy, g.Do_f, g.inv_Do));
            }
            y[row * g.Ho + kx] = val;
        };
        const int b0 = ir.part * chunk, b1 = min(nkept, b0 + chunk);
        int row = b0 < nkept ? row_of_kept(rowstart, g.Do, b0) : 0;
        for (int base = b0; base < b1; base += BT) {
            const int n = base + threadIdx.x;
            bool slow = false;
            int kx = 0;
            if (n < b1) {
                while (rowstart[row + 1] <= n) ++row;
                kx = n - rowstart[row];
                const int ky = row_freq(row, g.Do, g.halfo, g.centered);
                float2 v;
                if (eval_fast<NDIM, INTERP, WIN, false>(g, WIN == kGrouped ? VG : V, ip.R, kx, ky, v,
                                                        nullptr))
                    finish(row, kx, v);
                else
                    slow = true;
            }
            if constexpr (NDIM == 3) {
                // 3D: the CTA's warps stay on neighbouring image rows, which share L1 lines of
                // the volume; slow pixels wait in one CTA queue, drained a round at a time
                cta_enqueue(cq, slow, row, kx);
                __syncthreads();
                if (qcount >= BT) {
                    const int e = cq.slots[qcount - BT + threadIdx.x];
                    const int qrow = e >> 16, qkx = e & 0xffff;
                    float2 v;
                    eval_general<NDIM, INTERP, false>(g, V, ip.R, qkx,
                                                      row_freq(qrow, g.Do, g.halfo, g.centered), v, nullptr);
                    finish(qrow, qkx, v);
                    __syncthreads();
                    if (threadIdx.x == 0) qcount -= BT;
                    __syncthreads();
                }
            } else {
                // 2D: each warp runs free with its own queue
                q.push(slow, row, kx);
                if (q.count >= 32) {
                    const int e = q.slots[q.count - 32 + lane];
                    const int qrow = e >> 16, qkx = e & 0xffff;
                    float2 v;
                    eval_general<NDIM, INTERP, false>(g, V, ip.R, qkx,
                                                      row_freq(qrow, g.Do, g.halfo, g.centered), v, nullptr);
                    finish(qrow, qkx, v);
                    q.count -= 32;
                    __syncwarp();
                }
            }
        }
        if constexpr (NDIM == 3) {
            if (threadIdx.x < qcount) {
                const int e = cq.slots[threadIdx.x];
                const int qrow = e >> 16, qkx = e & 0xffff;
                float2 v;
                eval_general<NDIM, INTERP, false>(g, V, ip.R, qkx,
                                                  row_freq(qrow, g.Do, g.halfo, g.centered), v, nullptr);
                finish(qrow, qkx, v);
            }
            __syncthreads();
            if (threadIdx.x == 0) qcount = 0;
            __syncthreads();
        } else {
            if (lane < q.count) {
                const int e = q.slots[lane];
                const int qrow = e >> 16, qkx = e & 0xffff;
                float2 v;
                eval_general<NDIM, INTERP, false>(g, V, ip.R, qkx,
                                                  row_freq(qrow, g.Do, g.halfo, g.centered), v, nullptr);
                finish(qrow, qkx, v);
            }
            q.count = 0;
            __syncwarp();
        }
    }
}

// Any image size: one thread per pixel slot, exact per-tap rule (used when the image has
// more rows than the kept-pixel table holds).
template <int NDIM, int INTERP>
__global__ void __launch_bounds__(kThreads) project_kernel_any(
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
                eval_general<NDIM, INTERP, false>(g, V, ip.R, kx, ky, val, nullptr);
                if (g.has_shift)
                    val = cmul(val, shift_phase((float)kx, (float)ky, ip.sx, ip.sy, g.Do_f, g.inv_Do));
            }
            y[pix] = val;
        }
    }
}

// ------------------------------------------------- rotation / shift gradients ----

// Per pixel: g' = g conj(phase); dL/dR[a][b] += o q_b Re(conj(g') dv/dc_a) and
// dL/ds_b += (2 pi / Do) q_b Im(conj(g') v), with q = (kx, ky).
template <int NDIM>
__device__ __forceinline__ void accumulate_grad(float* acc, float2 gp, float2 v, const float2* dv,
                                                int kx, int ky)
{
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

template <int NDIM, int INTERP, int WIN>
__global__ void __launch_bounds__(kPoseThreads, 4) grad_pose_kernel(
    const float2* __restrict__ rec, const float* __restrict__ rot,
    const float* __restrict__ shift, const float2* __restrict__ gout,
    float* __restrict__ grot, float* __restrict__ gsh, Geom g, int splits, long long n_work,
    const float2* __restrict__ grouped)
{
    constexpr int NG = NDIM * 2 + 2;
    extern __shared__ int smem[];
    int* rowstart = smem;
    int* qslots = smem + g.Do + 1;           // [kWarpQueue per warp]
    __shared__ int scratch[kPoseThreads / 32];
    // per-warp sums of the item's terms, double-buffered by work-unit parity: one barrier per
    // work unit orders the writes before the sums, and the next unit writes the other buffer
    constexpr int NWP = kPoseThreads / 32;
    __shared__ float red[2][NG][NWP];
    int parity = 0;
    build_rowstart<kPoseThreads>(g, rowstart, scratch);
    const int lane = threadIdx.x & 31;
    WarpQueue q{qslots + (threadIdx.x >> 5) * kWarpQueue, 0};
    const int nkept = rowstart[g.Do];
    const int chunk = kept_chunk<kPoseThreads>(nkept, splits);
    float2* const tw0 = twiddle_table(qslots + kWarpQueue * (kPoseThreads / 32));  // 2D
    int unit = 0;

    // work unit = (item, part): part sums one chunk of the item's kept pixels
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x, ++unit) {
        const ItemRange ir = item_of(g, w, splits);
        ItemParams<NDIM> ip;
        load_item<NDIM>(g, rot, shift, ir.r, ir.p, ip);
        float2* const tw = tw0 + (unit & 1) * (g.Ho + g.Do);
        const bool twid = use_twiddles(g, NDIM) && g.has_shift;
        if (twid) build_twiddles<kPoseThreads>(g, ip.sx, ip.sy, tw);
        const float2* V = rec + (long long)ir.r * g.rec_elems;
        const float2* VG =
            WIN == kGrouped ? grouped + (long long)ir.r * g.Dv * g.gplane * Taps<INTERP>::N : V;
        const float2* gy = gout + ir.item * g.img_elems;
        float acc[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) acc[k] = 0.f;
        auto add = [&](int row, int kx, float2 v, const float2* dv) {
            const int ky = row_freq(row, g.Do, g.halfo, g.centered);
            float2 gp = __ldg(gy + row * g.Ho + kx);
            if (twid)
                gp = cmul_conj(gp, cmul(tw[kx], tw[g.Ho + row]));
            else if (g.has_shift)
                gp = cmul_conj(gp, shift_phase((float)kx, (float)ky, ip.sx, ip.sy, g.Do_f, g.inv_Do));
            accumulate_grad<NDIM>(acc, gp, v, dv, kx, ky);
        };
        const int b0 = ir.part * chunk, b1 = min(nkept, b0 + chunk);
        int row = b0 < nkept ? row_of_kept(rowstart, g.Do, b0) : 0;
        for (int base = b0; base < b1; base += kPoseThreads) {
            const int n = base + threadIdx.x;
            bool slow = false;
            int kx = 0;
            if (n < b1) {
                while (rowstart[row + 1] <= n) ++row;
                kx = n - rowstart[row];
                const int ky = row_freq(row, g.Do, g.halfo, g.centered);
                float2 v, dv[3];
                if (eval_fast<NDIM, INTERP, WIN, true>(g, WIN == kGrouped ? VG : V, ip.R, kx, ky, v, dv))
                    add(row, kx, v, dv);
                else
                    slow = true;
            }
            q.push(slow, row, kx);
            if (q.count >= 32) {
                const int e = q.slots[q.count - 32 + lane];
                const int qrow = e >> 16, qkx = e & 0xffff;
                float2 v, dv[3];
                eval_general<NDIM, INTERP, true>(g, V, ip.R, qkx,
                                                 row_freq(qrow, g.Do, g.halfo, g.centered), v, dv);
                add(qrow, qkx, v, dv);
                q.count -= 32;
                __syncwarp();
            }
        }
        if (lane < q.count) {
            const int e = q.slots[lane];
            const int qrow = e >> 16, qkx = e & 0xffff;
            float2 v, dv[3];
            eval_general<NDIM, INTERP, true>(g, V, ip.R, qkx,
                                             row_freq(qrow, g.Do, g.halfo, g.centered), v, dv);
            add(qrow, qkx, v, dv);
        }
        q.count = 0;
        __syncwarp();
        // per-item sums; several reconstructions may share one pose's parameters
        const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
        const long long si = (long long)(g.sh_shared ? 0 : ir.r) * g.n_pose + ir.p;
        const float two_pi_over_Do = 6.283185307179586f * g.inv_Do;
#pragma unroll
        for (int k = 0; k < NG; ++k) {
            float v = acc[k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[parity][k][threadIdx.x >> 5] = v;
        }
        __syncthreads();
        // thread k < NG adds term k over the warps
        if (threadIdx.x < NG) {
            const int k = threadIdx.x;
            float s = 0.f;
#pragma unroll
            for (int wi = 0; wi < NWP; ++wi) s += red[parity][k][wi];
            if (k < 2 * NDIM) {
                if (grot) atomicAdd(grot + ri * NDIM * NDIM + (k / 2) * NDIM + (k % 2), g.o * s);
            } else if (gsh && g.has_shift) {
                atomicAdd(gsh + si * 2 + (k - 2 * NDIM), two_pi_over_Do * s);
            }
        }
        parity ^= 1;
    }
}

// Any image size: general per-tap path, one thread per pixel slot.
template <int NDIM, int INTERP>
__global__ void __launch_bounds__(kThreads) grad_pose_kernel_any(
    const float2* __restrict__ rec, const float* __restrict__ rot,
    const float* __restrict__ shift, const float2* __restrict__ gout,
    float* __restrict__ grot, float* __restrict__ gsh, Geom g, int splits, long long n_work)
{
    constexpr int NG = NDIM * 2 + 2;
    __shared__ float red[kThreads / 32];
    const int npix = (int)g.img_elems;
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        ItemParams<NDIM> ip;
        load_item<NDIM>(g, rot, shift, ir.r, ir.p, ip);
        const float2* V = rec + (long long)ir.r * g.rec_elems;
        const float2* gy = gout + ir.item * g.img_elems;
        float acc[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) acc[k] = 0.f;
        for (int pix = ir.part * kThreads + threadIdx.x; pix < npix; pix += splits * kThreads) {
            int i, j;
            split_pixel(pix, g.Ho, i, j);
            const int ky = row_freq(i, g.Do, g.halfo, g.centered), kx = j;
            if (kx * kx + ky * ky > g.rc2) continue;
            float2 gp = __ldg(gy + pix);
            if (g.has_shift)
                gp = cmul_conj(gp, shift_phase((float)kx, (float)ky, ip.sx, ip.sy, g.Do_f, g.inv_Do));
            float2 v, dv[3];
            eval_general<NDIM, INTERP, true>(g, V, ip.R, kx, ky, v, dv);
            accumulate_grad<NDIM>(acc, gp, v, dv, kx, ky);
        }
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

// ------------------------------------------------------------ back-projection ----

// Scatter of every kept pixel of every item (data g conj(phase) and / or real weights):
// the transpose of the forward projection.  Used for the volume gradient too.
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

// Owner-computes back-projection (see scatter.cuh).  A CTA takes one item at a time; its
// threads own row segments of the volume (3D: rows (u_z, u_y); 2D: rows u_y) and gather
// the item's contributions to them.  DATA: proj * conj(phase) into vout (complex);
// WTS: the real per-pixel weights into wout.
constexpr int kMaxScatterBox = 1024;

template <int INTERP>
struct SegMargin {
    // Candidates have c_x within s of the segment [X0, X0 + W), so their taps lie in
    // [X0 - ML + 1, X0 + W + ML - 1); one spare slot on each side absorbs rounding.
    static constexpr int ML = INTERP == kCubic ? 5 : 3;
    static constexpr int AW = kSegW + 2 * ML;
};

template <int NDIM, int INTERP, bool DATA, bool WTS, int BT>
__global__ void __launch_bounds__(BT) scatter_rows_kernel(
    const float2* __restrict__ proj, const float* __restrict__ wts,
    const float* __restrict__ rot, const float* __restrict__ shift,
    float2* __restrict__ vout, float* __restrict__ wout, Geom g, long long n_items)
{
    // the 3D row scan below counts at most 4 z planes per thread
    static_assert(NDIM == 2 || 4 * BT >= kMaxScatterBox, "3D needs 4 * BT >= the largest box");
    constexpr int NT = Taps<INTERP>::N;
    constexpr int FIRST = Taps<INTERP>::first;
    constexpr float S = INTERP == kCubic ? 2.0f : 1.0f;
    constexpr int W = kSegW;
    constexpr int ML = SegMargin<INTERP>::ML;
    constexpr int AW = SegMargin<INTERP>::AW;
    extern __shared__ __align__(16) unsigned char sm_raw[];
    // [acc: AW x BT float2][wacc: AW x BT float][twx: Ho][twy: Do][kmax: Do]
    // [rowtab: Dv+1][ylo: Dv]
    float2* acc = reinterpret_cast<float2*>(sm_raw);
    float* wacc = reinterpret_cast<float*>(acc + (DATA ? AW * BT : 0));
    float2* twx = reinterpret_cast<float2*>(wacc + (WTS ? AW * BT : 0));
    float2* twy = twx + g.Ho;
    int* kmaxt = reinterpret_cast<int*>(twy + g.Do);
    int* rowtab = kmaxt + g.Do;
    int* ylo = rowtab + g.Dv + 1;
    __shared__ int scratch[BT / 32];
    __shared__ float Rs[9];
    __shared__ float2 sh;

    for (int j = 0; j < AW; ++j) {
        if (DATA) acc[j * BT + threadIdx.x] = make_float2(0.f, 0.f);
        if (WTS) wacc[j * BT + threadIdx.x] = 0.f;
    }
    // last kept kx of every image row (-1: none)
    for (int i = threadIdx.x; i < g.Do; i += BT) {
        const int ky = row_freq(i, g.Do, g.halfo, g.centered);
        kmaxt[i] = row_kept(g, i) - 1;
        (void)ky;
    }
    const float rho = sqrtf((float)g.rc2) + 1e-3f;

    for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
        const ItemRange ir = item_of(g, item, 1);
        if (threadIdx.x < NDIM * NDIM) {
            const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
            Rs[threadIdx.x] = g.o * __ldg(rot + ri * NDIM * NDIM + threadIdx.x);
        }
        if (threadIdx.x == 0) {
            sh = make_float2(0.f, 0.f);
            if (g.has_shift) {
                const long long si = (long long)(g.sh_shared ? 0 : ir.r) * g.n_pose + ir.p;
                sh = make_float2(__ldg(shift + si * 2), __ldg(shift + si * 2 + 1));
            }
        }
        __syncthreads();
        // separable shift twiddles: conj(phase(kx, ky)) = conj(twx[kx]) * conj(twy[row])
        if (DATA && g.has_shift) {
            for (int k = threadIdx.x; k < g.Ho; k += BT) {
                const float2 t = shift_phase((float)k, 0.f, sh.x, sh.y, g.Do_f, g.inv_Do);
                twx[k] = make_float2(t.x, -t.y);
            }
            for (int i = threadIdx.x; i < g.Do; i += BT) {
                const float2 t = shift_phase(0.f, (float)row_freq(i, g.Do, g.halfo, g.centered), sh.x,
                                             sh.y, g.Do_f, g.inv_Do);
                twy[i] = make_float2(t.x, -t.y);
            }
        }
        // rows that can receive contributions
        int nrows;
        if constexpr (NDIM == 3) {
            // per z plane, the y range of the slice's disk cut by the strip |c_z - u_z| < s
            const int per = (g.Dv + BT - 1) / BT;
            const int i0 = threadIdx.x * per;
            int cnt[4] = {0, 0, 0, 0};
            int sum = 0;
            for (int k = 0; k < per && k < 4; ++k) {
                const int iz = i0 + k;
                if (iz >= g.Dv) break;
                const float uz = (float)row_freq(iz, g.Dv, g.halfv, g.centered);
                float lo, hi;
                int y0 = 0, y1 = -1;
                if (strip_range(Rs[6], Rs[7], Rs[3], Rs[4], uz, S, rho, lo, hi)) {
                    y0 = max(-g.halfv, (int)floorf(lo - S) - 1);
                    y1 = min(g.halfv - 1, (int)ceilf(hi + S) + 1);
                }
                ylo[iz] = y0;
                cnt[k] = max(0, y1 - y0 + 1);
                sum += cnt[k];
            }
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            int inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += v;
            }
            if (lane == 31) scratch[warp] = inc;
            __syncthreads();
            if (threadIdx.x == 0) {
                int a = 0;
                for (int w = 0; w < BT / 32; ++w) {
                    const int t = scratch[w];
                    scratch[w] = a;
                    a += t;
                }
            }
            __syncthreads();
            int run = scratch[warp] + inc - sum;
            for (int k = 0; k < per && k < 4; ++k) {
                const int iz = i0 + k;
                if (iz >= g.Dv) break;
                rowtab[iz] = run;
                run += cnt[k];
            }
            if (threadIdx.x == BT - 1) rowtab[g.Dv] = run;
            __syncthreads();
            nrows = rowtab[g.Dv];
        } else {
            float lo, hi;
            int y0 = 0, y1 = -1;
            if (strip_range(0.f, 0.f, Rs[2], Rs[3], 0.f, 1.f, rho, lo, hi)) {
                y0 = max(-g.halfv, (int)floorf(lo - S) - 1);
                y1 = min(g.halfv - 1, (int)ceilf(hi + S) + 1);
            }
            nrows = max(0, y1 - y0 + 1);
            if (threadIdx.x == 0) ylo[0] = y0;
            __syncthreads();
        }
        const float2* py = DATA ? proj + ir.item * g.img_elems : nullptr;
        const float* pw = (WTS && wts) ? wts + ir.item * g.img_elems : nullptr;  // NULL: weight 1
        float2* G = DATA ? vout + (long long)ir.r * g.rec_elems : nullptr;
        float* Wt = WTS ? wout + (long long)ir.r * g.rec_elems : nullptr;
        // In-plane geometry.  (c_y[, c_z]) = M q; the kx of the plane point with
        // (c_y, c_z) = (u_y, u_z) tells which pixels (direct, kx >= 0, or mirrored) feed a row.
        const float nx = Rs[2], ny = Rs[5], nz = Rs[8];
        float mdet, kxa, kxb, ekx;  // kx* = kxa * u_y + kxb * u_z; ekx: half-extent in kx
        if constexpr (NDIM == 3) {
            mdet = Rs[3] * Rs[7] - Rs[4] * Rs[6];
            kxa = Rs[7] / mdet;
            kxb = -Rs[4] / mdet;
            ekx = S * (fabsf(kxa) + fabsf(kxb)) + 1.0f;
        } else {
            mdet = 1.0f;
            kxa = kxb = 0.f;
            ekx = 3.0e38f;  // 2D rows take both sides
        }
        const bool sides_known = NDIM == 3 && fabsf(mdet) > 1e-3f;
        // ky ranges of the parallelogram from each pair of strips: pairs (x,y), (x,z), (y,z)
        int iz = 0;
        for (int n = threadIdx.x; n < nrows; n += BT) {
            int uz = 0, uy;
            if constexpr (NDIM == 3) {
                while (rowtab[iz + 1] <= n) ++iz;
                uz = row_freq(iz, g.Dv, g.halfv, g.centered);
                uy = ylo[iz] + (n - rowtab[iz]);
            } else {
                uy = ylo[0] + n;
            }
            const int iy = full_index(uy, g.Dv, g.halfv, g.centered);
            const int izs = NDIM == 3 ? full_index(uz, g.Dv, g.halfv, g.centered) : 0;
            const long long roff = ((long long)izs * g.Dv + iy) * g.Hv;
            // x extent of the contributions to this row
            int xlo = 0, xhi = g.halfv;
            if constexpr (NDIM == 3) {
                if (fabsf(nx) > 1e-4f) {
                    // direct taps (c_x near xc) and mirrored ones (pixels with c_x near -xc,
                    // target -t_x) both land within xc +- (delta + s)
                    const float xc = -(ny * (float)uy + nz * (float)uz) / nx;
                    const float dl = S * (fabsf(ny) + fabsf(nz)) / fabsf(nx) + S + 1.0f;
                    xlo = max(0, (int)floorf(xc - dl));
                    xhi = min(g.halfv, (int)ceilf(xc + dl));
                }
            } else {
                float lo, hi;
                if (strip_range(Rs[2], Rs[3], Rs[0], Rs[1], (float)uy, S, rho, lo, hi)) {
                    // c_x of the direct pixels lies in [lo, hi]; the mirrored pixels (c_y near
                    // -u_y) have -c_x in the same interval, by the symmetry q -> -q of the disk
                    xlo = max(0, (int)floorf(lo - S) - 1);
                    xhi = min(g.halfv, (int)ceilf(hi + S) + 1);
                } else {
                    xhi = -1;
                }
            }
            // which sides can contribute: direct pixels sit near kx*, mirrored ones near -kx*
            bool do_direct = true, do_mirror = true;
            if (sides_known) {
                const float ks = kxa * (float)uy + kxb * (float)uz;
                do_direct = ks + ekx >= 0.f;
                do_mirror = -ks + ekx >= 0.f;
            }
            for (int X0 = xlo; X0 <= xhi; X0 += W) {
                const float xm = (float)X0 + 0.5f * (float)(W - 1);
                const float xh = 0.5f * (float)(W - 1) + S;
                for (int pass = 0; pass < 2; ++pass) {
                    // pass 0: direct taps t = u; pass 1: mirrored taps t = -u (u_x >= 1)
                    if (pass == 0 ? !do_direct : !do_mirror) continue;
                    const float sg = pass ? -1.0f : 1.0f;
                    const bool skip_x0 = pass == 1 && X0 == 0;  // x = 0 has no mirrored taps
                    Strip st[3];
                    st[0] = {Rs[0], Rs[1], sg * xm, xh};
                    st[1] = {Rs[NDIM], Rs[NDIM + 1], sg * (float)uy, S};
                    if constexpr (NDIM == 3) st[2] = {Rs[6], Rs[7], sg * (float)uz, S};
                    for_each_line<NDIM>(st, g, kmaxt, [&](int ky, int irow, int k0, int k1) {
                        const float fky = (float)ky;
                        const float cx0 = Rs[1] * fky, cy0 = Rs[NDIM + 1] * fky;
                        const float cz0 = NDIM == 3 ? Rs[7] * fky : 0.f;
                        const float2* prow = DATA ? py + irow * g.Ho : nullptr;
                        const float* wrow = pw ? pw + irow * g.Ho : nullptr;
                        const float2 tyv = (DATA && g.has_shift) ? twy[irow] : make_float2(1.f, 0.f);
                        for (int kx = k0; kx <= k1; ++kx) {
                            const float fkx = (float)kx;
                            const float cx = sg * fmaf(Rs[0], fkx, cx0);
                            float w = kernel_w<INTERP>(sg * fmaf(Rs[NDIM], fkx, cy0) - (float)uy);
                            if constexpr (NDIM == 3)
                                w *= kernel_w<INTERP>(sg * fmaf(Rs[6], fkx, cz0) - (float)uz);
                            float2 s = make_float2(0.f, 0.f);
                            float sw = 0.f;
                            if constexpr (DATA) {
                                float2 v = __ldg(prow + kx);
                                if (g.has_shift) v = cmul(v, cmul(twx[kx], tyv));
                                s = make_float2(w * v.x, sg * w * v.y);  // conj when mirrored
                            }
                            if constexpr (WTS) sw = wrow ? w * __ldg(wrow + kx) : w;
                            const float fl = floorf(cx);
                            float wx[NT];
                            weights<INTERP>(cx - fl, wx);
                            int j0 = (int)fl + FIRST - X0 + ML;
                            j0 = min(max(j0, 0), AW - NT);  // never outside the thread's slots
#pragma unroll
                            for (int k = 0; k < NT; ++k) {
                                const float wk = (skip_x0 && j0 + k == ML) ? 0.f : wx[k];
                                if constexpr (DATA) {
                                    float2& a = acc[(j0 + k) * BT + threadIdx.x];
                                    a.x = fmaf(wk, s.x, a.x);
                                    a.y = fmaf(wk, s.y, a.y);
                                }
                                if constexpr (WTS) {
                                    float& b = wacc[(j0 + k) * BT + threadIdx.x];
                                    b = fmaf(wk, sw, b);
                                }
                            }
                        }
                    });
                }
                // add the finished segment to the volume and clear the accumulator
                for (int j = 0; j < ML; ++j) {
                    if (DATA) acc[j * BT + threadIdx.x] = make_float2(0.f, 0.f);
                    if (WTS) wacc[j * BT + threadIdx.x] = 0.f;
                    if (DATA) acc[(ML + W + j) * BT + threadIdx.x] = make_float2(0.f, 0.f);
                    if (WTS) wacc[(ML + W + j) * BT + threadIdx.x] = 0.f;
                }
                const int nown = min(W, g.halfv - X0 + 1);
                if constexpr (DATA) {
                    for (int j = 0; j < nown;) {
                        float2* dst = G + roff + X0 + j;
                        float2& a = acc[(ML + j) * BT + threadIdx.x];
                        if (j + 1 < nown && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                            float2& b = acc[(ML + j + 1) * BT + threadIdx.x];
                            if (a.x != 0.f || a.y != 0.f || b.x != 0.f || b.y != 0.f)
                                atomicAdd(reinterpret_cast<float4*>(dst), make_float4(a.x, a.y, b.x, b.y));
                            a = make_float2(0.f, 0.f);
                            b = make_float2(0.f, 0.f);
                            j += 2;
                        } else {
                            if (a.x != 0.f || a.y != 0.f) atomicAdd(dst, a);
                            a = make_float2(0.f, 0.f);
                            j += 1;
                        }
                    }
                    for (int j = nown; j < W; ++j) acc[(ML + j) * BT + threadIdx.x] = make_float2(0.f, 0.f);
                }
                if constexpr (WTS) {
                    for (int j = 0; j < W; ++j) {
                        float& b = wacc[(ML + j) * BT + threadIdx.x];
                        if (j < nown && b != 0.f) atomicAdd(Wt + roff + X0 + j, b);
                        b = 0.f;
                    }
                }
            }
        }
        __syncthreads();
    }
}

// Warp-tile back-projection for cubic 3D.  A warp takes a 4 x 4 tile of kept pixels of one
// item and accumulates the tile's taps in a private box of shared memory that covers the
// tile's footprint (the axis-aligned box of its taps in the effective frame, at most 9^3
// voxels for o = 1).  The warp walks the tile's pixels one at a time with its lanes on the
// pixel's 64 taps (two per lane); one pixel's taps are distinct voxels, so the
// lanes read-modify-write shared memory without atomics and __syncwarp orders successive
// pixels.  The box rows have a pitch of 12 voxels: a half-warp's 16 taps (4 y rows x 4 x
// taps, 8-byte values) then fall in 16 distinct bank pairs.  The finished box is added to
// the volume with coalesced vector reductions, one per voxel touched by the tile instead
// of one per tap.  Pixels with c_x < 0 are handled in the effective frame (c' = -c,
// conjugate value; see gather.cuh) in a second pass over the tile; pixels whose taps reach
// the x <= 0 planes take the exact per-tap rule, and tiles whose box would overflow (large
// oversampling) use direct vector atomics.
constexpr int kBoxPitch = 12;

// Box of one warp (cubic; the linear 3D scatter is scatter_lane_kernel).  Pitch 12: every
// 4 x 4 tile at o = 1 spans at most 9 voxels per axis, so 81 rows would hold all of them.
// 72 rows hold all but about 1 in 10^4 tile passes (NY * NZ = 8 x 9 is common, more is rare)
// and, with no static shared memory, fit exactly four CTAs of 7 warps per SM; with the weight
// box, 64 rows (all but 0.6 %: the common 8 x 9 boxes take the per-tap path) fit three CTAs of
// 7 warps instead of 6.  Larger tiles (o > 1) take the per-tap path.
template <bool WTS>
struct BoxDims {
    static constexpr int PITCH = kBoxPitch;
    static constexpr int ROWS = WTS ? 64 : 72;
    static constexpr int CAP = PITCH * ROWS;
};

// Threads of one scatter_tile_kernel CTA: 7 warps, so that four CTAs (three with the weight
// box) fit in the SM's 228 KB of shared memory.
constexpr int kTileThreads = 224;
constexpr int kTilePix = 16;                        // 4 x 4 pixels

// One record per pixel, stored contiguously (array of structs): gx gy wt base (one 16-byte
// broadcast load) | wx[4] | wy[4] | wz in the order 0, 2, 1, 3, so that the z weights of a
// lane's two planes a and a + 2 are one 8-byte load (the tap loop forms wz * wy) | fx fy fz.
// base < 0 flags the per-tap path and holds ~base.  With the pose gradients (POSE) the record
// also holds the derivative weights (z in the order 0, 2, 1, 3) and, for reading the volume at
// the taps, the element offset iy * Hv + x0 of each y tap row and iz * Dv * Hv of each z tap
// plane (order 0, 2, 1, 3), kOutside when the tap lies outside the stored band.
template <bool POSE>
struct TileRecT {
    enum : int { GX = 0, GY = 1, WT = 2, BASE = 3, WX = 4, WY = 8, WZ = 12, FX = 16, FY = 17, FZ = 18 };
    enum : int { DWX = 20, DWY = 24, DWZ = 28, YO = 32, ZO = 36 };
    enum : int {
        STRIDE = POSE ? 40 : 20,    // 16-byte aligned records
        WORDS = STRIDE * kTilePix,  // a multiple of 4: 16-byte aligned records
    };
};
using TileRec = TileRecT<false>;
// Offset of a tap row or plane outside the stored band: any sum of offsets that includes it
// stays negative (valid offsets are below 2^30 for every supported box).
constexpr int kOutside = -(1 << 30);
// CTAs of the fused backward (volume and pose gradients): 6 warps, whose larger records still
// let four CTAs fit in shared memory.
constexpr int kTileThreadsPose = 192;

// POSE: the one-pass backward.  Besides the volume gradient the kernel forms the rotation and
// shift gradients: every lane reads the volume at its two taps of the pixel (effective frame,
// the exact Friedel rule on the per-tap path), and accumulates, over the item's pixels, the
// terms o q_b Re(conj(g') dv/dc_a) and (2 pi / Do) q_b Im(conj(g') v) of each tap; a warp
// reduction and one atomic per term per warp finish the item.  The launch bound asks for four
// CTAs per SM only with POSE (80 registers); 0 leaves the other instances unconstrained.
template <int INTERP, bool DATA, bool WTS, bool POSE = false>
__global__ void __launch_bounds__(POSE ? kTileThreadsPose : kTileThreads, POSE ? 4 : 0)
scatter_tile_kernel(const float2* __restrict__ proj, const float* __restrict__ wts,
                    const float* __restrict__ rot, const float* __restrict__ shift,
                    float2* __restrict__ vout, float* __restrict__ wout, Geom g, int splits,
                    long long n_work, const float2* __restrict__ vol = nullptr,
                    float* __restrict__ grot = nullptr, float* __restrict__ gsh = nullptr)
{
    static_assert(INTERP == kCubic, "the linear 3D scatter is scatter_lane_kernel");
    static_assert(!POSE || (DATA && !WTS), "the fused backward scatters data only");
    using TR = TileRecT<POSE>;
    constexpr int NT = Taps<INTERP>::N;
    constexpr int FIRST = Taps<INTERP>::first;
    constexpr int TPL = 2;                 // taps per lane: 64 taps on 32 lanes
    constexpr int NWARP = (POSE ? kTileThreadsPose : kTileThreads) / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    extern __shared__ __align__(16) unsigned char sm_raw[];
    using BX = BoxDims<WTS>;
    constexpr int CAP = BX::CAP, PITCH = BX::PITCH, ROWS = BX::ROWS;
    // per warp: acc[CAP] float2 | wacc[CAP] float | records (TR::WORDS words)
    float2* acc = reinterpret_cast<float2*>(sm_raw) + warp * (DATA ? CAP : 0);
    float* wacc = reinterpret_cast<float*>(reinterpret_cast<float2*>(sm_raw) + NWARP * (DATA ? CAP : 0)) +
                  warp * (WTS ? CAP : 0);
    float* recf = reinterpret_cast<float*>(reinterpret_cast<float2*>(sm_raw) + NWARP * (DATA ? CAP : 0)) +
                  NWARP * (WTS ? CAP : 0) + warp * TR::WORDS;
    int* reci = reinterpret_cast<int*>(recf);
    static_assert(TR::WORDS % 4 == 0 && (CAP * 4) % 16 == 0, "16-byte aligned records");
    static_assert(TR::WORDS >= ROWS, "the record space holds the flush's row table");

    for (int e = lane; e < CAP; e += 32) {
        if (DATA) acc[e] = make_float2(0.f, 0.f);
        if (WTS) wacc[e] = 0.f;
    }
    // this lane's taps: tap index q = lane + 32 m -> (a, b, k) = (z, y, x) offsets
    int ta[TPL], tb[TPL];
    const int tk = lane % NT;
#pragma unroll
    for (int m = 0; m < TPL; ++m) {
        const int q = lane + 32 * m;
        ta[m] = q / (NT * NT);
        tb[m] = (q / NT) % NT;
    }
    const int tiles_x = (g.Ho + 3) / 4, tiles_y = (g.Do + 3) / 4;
    const int ntiles = tiles_x * tiles_y;

    // work unit = (item, part): part takes every splits-th round of NWARP tiles.  Every thread
    // reads the item's rotation (scaled by o) and shift into registers itself: the kernel needs
    // no static shared memory (its whole budget goes to the boxes) and no barrier between items.
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        float Rs[9];
        {
            const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
#pragma unroll
            for (int k = 0; k < 9; ++k) Rs[k] = g.o * __ldg(rot + ri * 9 + k);
        }
        float2 sh = make_float2(0.f, 0.f);
        if (g.has_shift) {
            const long long si = (long long)(g.sh_shared ? 0 : ir.r) * g.n_pose + ir.p;
            sh = make_float2(__ldg(shift + si * 2), __ldg(shift + si * 2 + 1));
        }
        const float2* py = DATA ? proj + ir.item * g.img_elems : nullptr;
        const float* pw = (WTS && wts) ? wts + ir.item * g.img_elems : nullptr;  // NULL: weight 1
        float2* G = DATA ? vout + (long long)ir.r * g.rec_elems : nullptr;
        float* Wt = WTS ? wout + (long long)ir.r * g.rec_elems : nullptr;
        const float2* V = POSE ? vol + (long long)ir.r * g.rec_elems : nullptr;
        // pose-gradient terms of this lane: o-free d/dR[a][b] (a = x, y, z; b = kx, ky) and
        // the shift's two
        float pacc[POSE ? 8 : 1];
#pragma unroll
        for (int k = 0; k < (POSE ? 8 : 1); ++k) pacc[k] = 0.f;

        for (int tile = ir.part * NWARP + warp; tile < ntiles; tile += splits * NWARP) {
            const int ti = tile / tiles_x, tj = tile - ti * tiles_x;
            // ---- per-pixel set-up: lane l < 16 owns pixel (row 4 ti + l / 4, kx 4 tj + l % 4)
            const int prow = 4 * ti + (lane >> 2), pkx = 4 * tj + (lane & 3);
            bool kept = false;
            int ky = 0;
            float cx = 0.f, cy = 0.f, cz = 0.f;
            if (lane < kTilePix && prow < g.Do && pkx < g.Ho) {
                ky = row_freq(prow, g.Do, g.halfo, g.centered);
                kept = pkx * pkx + ky * ky <= g.rc2;
                const float fkx = (float)pkx, fky = (float)ky;
                cx = fmaf(Rs[0], fkx, Rs[1] * fky);
                cy = fmaf(Rs[3], fkx, Rs[4] * fky);
                cz = fmaf(Rs[6], fkx, Rs[7] * fky);
            }
            const unsigned kept_mask = __ballot_sync(0xffffffffu, kept);
            if (!kept_mask) continue;
            const bool neg = cx < 0.f;
            const unsigned neg_mask = __ballot_sync(0xffffffffu, kept && neg);
            // value of the pixel: g' = g conj(phase), its weight
            float2 gp = make_float2(0.f, 0.f);
            float wt = 1.f;
            if (kept) {
                if (DATA) {
                    gp = __ldg(py + prow * g.Ho + pkx);
                    if (g.has_shift)
                        gp = cmul_conj(gp, shift_phase((float)pkx, (float)ky, sh.x, sh.y, g.Do_f, g.inv_Do));
                }
                if (WTS && pw) wt = __ldg(pw + prow * g.Ho + pkx);
            }
            for (int pass = 0; pass < 2; ++pass) {
                const unsigned pmask = pass ? neg_mask : (kept_mask & ~neg_mask);
                if (!pmask) continue;
                const bool mine = (pmask >> lane) & 1u;
                const float sg = pass ? -1.f : 1.f;
                // effective coordinates, clamped like floor_frac: beyond 2^23 every tap is
                // outside any box and the integer extents below stay far from overflow
                const float lim = 8388608.0f;
                const float ex = fminf(fmaxf(sg * cx, -lim), lim);
                const float ey = fminf(fmaxf(sg * cy, -lim), lim);
                const float ez = fminf(fmaxf(sg * cz, -lim), lim);
                const float flx = floorf(ex), fly = floorf(ey), flz = floorf(ez);
                const int fx = (int)flx, fy = (int)fly, fz = (int)flz;
                // box of this pass's taps
                const int big = 1 << 28;
                const int x0 = __reduce_min_sync(0xffffffffu, mine ? fx : big) + FIRST;
                const int y0 = __reduce_min_sync(0xffffffffu, mine ? fy : big) + FIRST;
                const int z0 = __reduce_min_sync(0xffffffffu, mine ? fz : big) + FIRST;
                const int x1 = __reduce_max_sync(0xffffffffu, mine ? fx : -big) + FIRST + NT - 1;
                const int y1 = __reduce_max_sync(0xffffffffu, mine ? fy : -big) + FIRST + NT - 1;
                const int z1 = __reduce_max_sync(0xffffffffu, mine ? fz : -big) + FIRST + NT - 1;
                const int NX = x1 - x0 + 1, NY = y1 - y0 + 1, NZ = z1 - z0 + 1;
                const bool boxed = NX <= PITCH && NY <= ROWS && NZ <= ROWS && NY * NZ <= ROWS;
                // records of this pass's pixels
                if (mine) {
                    float wx_[NT], wy_[NT], wz_[NT];
                    weights<INTERP>(ex - flx, wx_);
                    weights<INTERP>(ey - fly, wy_);
                    weights<INTERP>(ez - flz, wz_);
                    float* rf = recf + lane * TR::STRIDE;
                    int* ri = reci + lane * TR::STRIDE;
                    *reinterpret_cast<float4*>(rf + TR::WX) = make_float4(wx_[0], wx_[1], wx_[2], wx_[3]);
                    *reinterpret_cast<float4*>(rf + TR::WY) = make_float4(wy_[0], wy_[1], wy_[2], wy_[3]);
                    *reinterpret_cast<float4*>(rf + TR::WZ) = make_float4(wz_[0], wz_[2], wz_[1], wz_[3]);
                    rf[TR::WT] = wt;
                    // effective value: conj(g') on the mirrored pass (weights are real)
                    rf[TR::GX] = gp.x;
                    rf[TR::GY] = sg * gp.y;
                    // the box offset of the pixel's first tap (below CAP); 0 without a box, so
                    // that the per-tap flag ~base below is negative whatever the extents (the
                    // product would overflow for extents near the 2^23 clamp)
                    const int base = boxed ? ((fz + FIRST - z0) * NY + (fy + FIRST - y0)) * PITCH + (fx + FIRST - x0)
                                           : 0;
                    // (POSE: taps past x = Dv/2 also take the per-tap path, where the volume
                    // reads follow the exact rule)
                    ri[TR::BASE] = (fx + FIRST <= 0 || !boxed || (POSE && fx + FIRST + NT - 1 > g.halfv))
                                       ? ~base
                                       : base;
                    ri[TR::FX] = fx;
                    ri[TR::FY] = fy;
                    ri[TR::FZ] = fz;
                    if constexpr (POSE) {
                        float dx_[NT], dy_[NT], dz_[NT];
                        dweights<INTERP>(ex - flx, dx_);
                        dweights<INTERP>(ey - fly, dy_);
                        dweights<INTERP>(ez - flz, dz_);
                        *reinterpret_cast<float4*>(rf + TR::DWX) = make_float4(dx_[0], dx_[1], dx_[2], dx_[3]);
                        *reinterpret_cast<float4*>(rf + TR::DWY) = make_float4(dy_[0], dy_[1], dy_[2], dy_[3]);
                        *reinterpret_cast<float4*>(rf + TR::DWZ) = make_float4(dz_[0], dz_[2], dz_[1], dz_[3]);
                        int yo[NT], zo[NT];
#pragma unroll
                        for (int k = 0; k < NT; ++k) {
                            const int iy = full_index(fy + FIRST + k, g.Dv, g.halfv, g.centered);
                            const int iz = full_index(fz + FIRST + k, g.Dv, g.halfv, g.centered);
                            yo[k] = iy < 0 ? kOutside : iy * g.Hv + fx + FIRST;
                            zo[k] = iz < 0 ? kOutside : iz * g.Dv * g.Hv;
                        }
                        *reinterpret_cast<int4*>(ri + TR::YO) = make_int4(yo[0], yo[1], yo[2], yo[3]);
                        *reinterpret_cast<int4*>(ri + TR::ZO) = make_int4(zo[0], zo[2], zo[1], zo[3]);
                    }
                }
                __syncwarp();
                int toff[TPL];
#pragma unroll
                for (int m = 0; m < TPL; ++m) toff[m] = (ta[m] * NY + tb[m]) * PITCH + tk;
                // ---- scatter: one pixel at a time, lanes on its taps
                for (unsigned pm = pmask; pm; pm &= pm - 1) {
                    const int j = __ffs(pm) - 1;
                    {
                        const float* rf = recf + j * TR::STRIDE;
                        const int* ri = reci + j * TR::STRIDE;
                        const float4 head = *reinterpret_cast<const float4*>(rf);
                        const float2 gv = make_float2(head.x, head.y);
                        const float wtv = head.z;
                        const float wxk = rf[TR::WX + tk];
                        const int rb = __float_as_int(head.w);
                        const int base = rb < 0 ? ~rb : rb;
                        // z planes ta[0] and ta[0] + 2 of y row tb[0]
                        const float2 zp = *reinterpret_cast<const float2*>(rf + TR::WZ + 2 * ta[0]);
                        const float wyb = rf[TR::WY + tb[0]];
                        const float wzy[TPL] = {zp.x * wyb, zp.y * wyb};
                        float2 vv[POSE ? TPL : 1];  // the volume at this lane's taps (POSE)
                        if (rb >= 0) {
                            if constexpr (POSE) {
                                // taps at 1 <= x <= Dv/2: direct reads, zero outside the band
                                const int yo = ri[TR::YO + tb[0]];
                                const int2 zo = *reinterpret_cast<const int2*>(ri + TR::ZO + 2 * ta[0]);
                                const int o0 = zo.x + yo + tk, o1 = zo.y + yo + tk;
                                vv[0] = o0 >= 0 ? __ldg(V + o0) : make_float2(0.f, 0.f);
                                vv[1] = o1 >= 0 ? __ldg(V + o1) : make_float2(0.f, 0.f);
                            }
#pragma unroll
                            for (int m = 0; m < TPL; ++m) {
                                const float w = wzy[m] * wxk;
                                const int e = base + toff[m];
                                if (DATA) {
                                    float2 a = acc[e];
                                    a.x = fmaf(w, gv.x, a.x);
                                    a.y = fmaf(w, gv.y, a.y);
                                    acc[e] = a;
                                }
                                if (WTS) wacc[e] = fmaf(w, wtv, wacc[e]);
                            }
                        } else {
                            // taps on the x <= 0 planes (exact per-tap rule), or no box
                            const int pfx = ri[TR::FX];
                            const int pfy = ri[TR::FY];
                            const int pfz = ri[TR::FZ];
#pragma unroll
                            for (int m = 0; m < TPL; ++m) {
                                const float w = wzy[m] * wxk;
                                const int ux = pfx + FIRST + tk;
                                const bool direct = ux >= 1 || (ux == 0 && pass == 0);
                                if constexpr (POSE) {
                                    // the value of the extended spectrum at this tap
                                    int vx = ux, vy = pfy + FIRST + tb[m], vz = pfz + FIRST + ta[m];
                                    if (!direct) {
                                        vx = -vx;
                                        vy = -vy;
                                        vz = -vz;
                                    }
                                    const int iy = full_index(vy, g.Dv, g.halfv, g.centered);
                                    const int iz = full_index(vz, g.Dv, g.halfv, g.centered);
                                    float2 val = make_float2(0.f, 0.f);
                                    if (vx >= 0 && vx <= g.halfv && iy >= 0 && iz >= 0)
                                        val = __ldg(V + ((long long)iz * g.Dv + iy) * g.Hv + vx);
                                    if (!direct) val.y = -val.y;
                                    vv[m] = val;
                                }
                                if (direct && boxed) {
                                    const int e = base + toff[m];
                                    if (DATA) {
                                        float2 a = acc[e];
                                        a.x = fmaf(w, gv.x, a.x);
                                        a.y = fmaf(w, gv.y, a.y);
                                        acc[e] = a;
                                    }
                                    if (WTS) wacc[e] = fmaf(w, wtv, wacc[e]);
                                } else {
                                    // target u (direct) or -u (mirrored, conjugate value)
                                    int vx = ux, vy = pfy + FIRST + tb[m], vz = pfz + FIRST + ta[m];
                                    float vim = gv.y;
                                    if (!direct) {
                                        vx = -vx;
                                        vy = -vy;
                                        vz = -vz;
                                        vim = -vim;
                                    }
                                    const int iy = full_index(vy, g.Dv, g.halfv, g.centered);
                                    const int iz = full_index(vz, g.Dv, g.halfv, g.centered);
                                    if (vx >= 0 && vx <= g.halfv && iy >= 0 && iz >= 0) {
                                        const long long off = ((long long)iz * g.Dv + iy) * g.Hv + vx;
                                        if (DATA) atomicAdd(G + off, make_float2(w * gv.x, w * vim));
                                        if (WTS) atomicAdd(Wt + off, w * wtv);
                                    }
                                }
                            }
                        }
                        if constexpr (POSE) {
                            // this lane's share of Re(conj(h) dv'/dc'_a) and Im(conj(h) v') (h
                            // the record's value, v' the effective-frame sample; separable
                            // weights), times q_b and the pass sign (dv/dc = -conj(dv'/dc'),
                            // v = conj(v') on the mirrored pass)
                            const float dwxk = rf[TR::DWX + tk];
                            const float dwyb = rf[TR::DWY + tb[0]];
                            const float2 dzp = *reinterpret_cast<const float2*>(rf + TR::DWZ + 2 * ta[0]);
                            float tre[TPL], tim[TPL];
#pragma unroll
                            for (int m = 0; m < TPL; ++m) {
                                tre[m] = fmaf(gv.x, vv[m].x, gv.y * vv[m].y);
                                tim[m] = fmaf(gv.x, vv[m].y, -gv.y * vv[m].x);
                            }
                            const float za = fmaf(zp.x, tre[0], zp.y * tre[1]);
                            const float zd = fmaf(dzp.x, tre[0], dzp.y * tre[1]);
                            const float zi = fmaf(zp.x, tim[0], zp.y * tim[1]);
                            const float wyx = wyb * wxk;
                            const float sx = wyb * dwxk * za, sy = dwyb * wxk * za;
                            const float sz = wyx * zd, ss = wyx * zi;
                            const float qx = sg * (float)(4 * tj + (j & 3));
                            const float qy = sg * (float)row_freq(4 * ti + (j >> 2), g.Do, g.halfo, g.centered);
                            pacc[0] = fmaf(sx, qx, pacc[0]);
                            pacc[1] = fmaf(sx, qy, pacc[1]);
                            pacc[2] = fmaf(sy, qx, pacc[2]);
                            pacc[3] = fmaf(sy, qy, pacc[3]);
                            pacc[4] = fmaf(sz, qx, pacc[4]);
                            pacc[5] = fmaf(sz, qy, pacc[5]);
                            pacc[6] = fmaf(ss, qx, pacc[6]);
                            pacc[7] = fmaf(ss, qy, pacc[7]);
                        }
                    }
                    __syncwarp();
                }
                // ---- add the box to the volume (read and clear).  The records are dead
                // now: their space holds the global offset of every box row (-1 outside the
                // band).  Entries e < NX * NY * NZ map to row r = e / NX and column e % NX by
                // exact multiply-shift (e < 2^10, NX, NY <= 81); only non-zero entries are
                // added and cleared.
                if (boxed) {
                    const int nrows = NY * NZ;
                    const unsigned my = (65536u + NY - 1) / NY;
                    int* rowoff = reci;
                    for (int r = lane; r < nrows; r += 32) {
                        const int zi = (int)(((unsigned)r * my) >> 16);
                        const int iy = full_index(y0 + r - zi * NY, g.Dv, g.halfv, g.centered);
                        const int iz = full_index(z0 + zi, g.Dv, g.halfv, g.centered);
                        rowoff[r] = (iy >= 0 && iz >= 0) ? (iz * g.Dv + iy) * g.Hv : -1;
                    }
                    __syncwarp();
                    const unsigned mx = (65536u + NX - 1) / NX;
                    const int nused = nrows * NX;
                    for (int e = lane; e < nused; e += 32) {
                        const int r = (int)(((unsigned)e * mx) >> 16);
                        const int xi = e - r * NX;
                        const int be = r * PITCH + xi;
                        const int ux = x0 + xi;
                        bool hit = false;
                        float2 a = make_float2(0.f, 0.f);
                        float b = 0.f;
                        if (DATA) {
                            a = acc[be];
                            hit = a.x != 0.f || a.y != 0.f;
                        }
                        if (WTS) {
                            b = wacc[be];
                            hit = hit || b != 0.f;
                        }
                        if (hit) {
                            const int ro = rowoff[r];
                            if (ro >= 0 && ux >= 0 && ux <= g.halfv) {
                                if (DATA && (a.x != 0.f || a.y != 0.f)) atomicAdd(G + ro + ux, a);
                                if (WTS && b != 0.f) atomicAdd(Wt + ro + ux, b);
                            }
                            if (DATA) acc[be] = make_float2(0.f, 0.f);
                            if (WTS) wacc[be] = 0.f;
                        }
                    }
                }
                __syncwarp();
            }
        }
        if constexpr (POSE) {
            // the warp's sums for this item: one atomic per term
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float v = pacc[k];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                pacc[k] = v;
            }
            if (lane == 0) {
                const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
                const long long si = (long long)(g.sh_shared ? 0 : ir.r) * g.n_pose + ir.p;
                if (grot) {
#pragma unroll
                    for (int k = 0; k < 6; ++k) atomicAdd(grot + ri * 9 + (k / 2) * 3 + (k % 2), g.o * pacc[k]);
                }
                if (gsh && g.has_shift) {
                    const float two_pi_over_Do = 6.283185307179586f * g.inv_Do;
                    atomicAdd(gsh + si * 2, two_pi_over_Do * pacc[6]);
                    atomicAdd(gsh + si * 2 + 1, two_pi_over_Do * pacc[7]);
                }
            }
        }
    }
}

// Cubic 2D insertion with weights (data and weight images together).  A half-warp takes a
// 4 x 4 pixel tile with its own shared-memory box over the tile's tap footprint, so a warp
// adds two pixels at a time, one per half-warp, with plain read-modify-writes: the 16 lanes
// of a half-warp sit on the 16 taps of its pixel (distinct voxels), and __syncwarp orders
// successive pixels.  Box rows have a pitch of 12 voxels, so a pixel's 4 tap rows fall in 4
// distinct groups of 8 banks.  As in the 3D tile scatter, pixels with c_x < 0 go in a
// second pass in the effective frame (c' = -c, conjugate value); pixels whose taps reach
// x <= 0 take the exact per-tap rule (mirrored taps by global atomics), tiles whose box
// would overflow (o > 1) add every tap by atomics, and the box is added to the image with
// one vector reduction per touched voxel.
constexpr int kTile2Pitch = 12;
constexpr int kTile2Rows = 10;  // a 4 x 4 tile at o = 1 spans at most 9 rows
constexpr int kTile2Threads = 256;

// Record of one pixel: gx gy wt base (one 16-byte load) | wx[4] | wy[4] | fx fy.  base < 0
// flags the per-tap path and holds ~base.
struct Tile2Rec {
    enum : int { GX = 0, GY = 1, WT = 2, BASE = 3, WX = 4, WY = 8, FX = 12, FY = 13, STRIDE = 16 };
};

template <bool DATA, bool WTS>
__global__ void __launch_bounds__(kTile2Threads) scatter_tile2d_kernel(
    const float2* __restrict__ proj, const float* __restrict__ wts,
    const float* __restrict__ rot, const float* __restrict__ shift,
    float2* __restrict__ vout, float* __restrict__ wout, Geom g, int splits, long long n_work)
{
    using TR = Tile2Rec;
    constexpr int NT = 4, FIRST = -1;
    constexpr int PITCH = kTile2Pitch, ROWS = kTile2Rows, CAP = PITCH * ROWS;
    constexpr int NWARP = kTile2Threads / 32;
    constexpr unsigned kFull = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = lane >> 4, l = lane & 15;  // half-warp, lane within it
    const int hw = warp * 2 + h;             // half-warp of the CTA
    extern __shared__ __align__(16) unsigned char sm_raw[];
    // per half-warp: acc[CAP] float2 | wacc[CAP] float | records [16][STRIDE]
    float2* acc = reinterpret_cast<float2*>(sm_raw) + hw * (DATA ? CAP : 0);
    float* wbase = reinterpret_cast<float*>(reinterpret_cast<float2*>(sm_raw) + 2 * NWARP * (DATA ? CAP : 0));
    float* wacc = wbase + hw * (WTS ? CAP : 0);
    float* recf = wbase + 2 * NWARP * (WTS ? CAP : 0) + hw * kTilePix * TR::STRIDE;
    int* reci = reinterpret_cast<int*>(recf);

    for (int e = l; e < CAP; e += 16) {
        if (DATA) acc[e] = make_float2(0.f, 0.f);
        if (WTS) wacc[e] = 0.f;
    }
    // this lane's tap: row tb, column tk of the pixel's 4 x 4 taps
    const int tb = l >> 2, tk = l & 3;
    const int toff = tb * PITCH + tk;
    const int tiles_x = (g.Ho + 3) / 4, tiles_y = (g.Do + 3) / 4;
    const int ntiles = tiles_x * tiles_y;

    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        float Rs[4];
        {
            const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
#pragma unroll
            for (int k = 0; k < 4; ++k) Rs[k] = g.o * __ldg(rot + ri * 4 + k);
        }
        float2 sh = make_float2(0.f, 0.f);
        if (g.has_shift) {
            const long long si = (long long)(g.sh_shared ? 0 : ir.r) * g.n_pose + ir.p;
            sh = make_float2(__ldg(shift + si * 2), __ldg(shift + si * 2 + 1));
        }
        const float2* py = DATA ? proj + ir.item * g.img_elems : nullptr;
        const float* pw = (WTS && wts) ? wts + ir.item * g.img_elems : nullptr;  // NULL: weight 1
        float2* G = DATA ? vout + (long long)ir.r * g.rec_elems : nullptr;
        float* Wt = WTS ? wout + (long long)ir.r * g.rec_elems : nullptr;

        // tiles in pairs: half-warp h of the warp takes tile t2 + h
        for (int t2 = (ir.part * NWARP + warp) * 2; t2 < ntiles; t2 += splits * NWARP * 2) {
            const int tile = t2 + h;
            const bool tvalid = tile < ntiles;
            const int ti = tvalid ? tile / tiles_x : 0, tj = tvalid ? tile - ti * tiles_x : 0;
            const int prow = 4 * ti + (l >> 2), pkx = 4 * tj + (l & 3);
            bool kept = false;
            int ky = 0;
            float cx = 0.f, cy = 0.f;
            if (tvalid && prow < g.Do && pkx < g.Ho) {
                ky = row_freq(prow, g.Do, g.halfo, g.centered);
                kept = pkx * pkx + ky * ky <= g.rc2;
                const float fkx = (float)pkx, fky = (float)ky;
                cx = fmaf(Rs[0], fkx, Rs[1] * fky);
                cy = fmaf(Rs[2], fkx, Rs[3] * fky);
            }
            const unsigned kept_mask = __ballot_sync(kFull, kept);
            if (!kept_mask) continue;
            const unsigned neg_mask = __ballot_sync(kFull, kept && cx < 0.f);
            float2 gp = make_float2(0.f, 0.f);
            float wt = 1.f;
            if (kept) {
                if (DATA) {
                    gp = __ldg(py + prow * g.Ho + pkx);
                    if (g.has_shift)
                        gp = cmul_conj(gp, shift_phase((float)pkx, (float)ky, sh.x, sh.y, g.Do_f, g.inv_Do));
                }
                if (WTS && pw) wt = __ldg(pw + prow * g.Ho + pkx);
            }
            for (int pass = 0; pass < 2; ++pass) {
                const unsigned wmask = pass ? neg_mask : (kept_mask & ~neg_mask);
                if (!wmask) continue;
                const unsigned pmask = (wmask >> (16 * h)) & 0xffffu;  // this half's pixels
                const bool mine = (pmask >> l) & 1u;
                const float sg = pass ? -1.f : 1.f;
                // effective coordinates, clamped like floor_frac
                const float lim = 8388608.0f;
                const float ex = fminf(fmaxf(sg * cx, -lim), lim);
                const float ey = fminf(fmaxf(sg * cy, -lim), lim);
                const float flx = floorf(ex), fly = floorf(ey);
                const int fx = (int)flx, fy = (int)fly;
                // box of this half's pass: reductions within the half-warp
                const int big = 1 << 28;
                int mnx = mine ? fx : big, mny = mine ? fy : big;
                int mxx = mine ? fx : -big, mxy = mine ? fy : -big;
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) {
                    mnx = min(mnx, __shfl_xor_sync(kFull, mnx, o));
                    mny = min(mny, __shfl_xor_sync(kFull, mny, o));
                    mxx = max(mxx, __shfl_xor_sync(kFull, mxx, o));
                    mxy = max(mxy, __shfl_xor_sync(kFull, mxy, o));
                }
                const int x0 = mnx + FIRST, y0 = mny + FIRST;
                const int NX = mxx - mnx + NT, NY = mxy - mny + NT;
                const bool boxed = pmask != 0 && NX <= PITCH && NY <= ROWS;
                if (mine) {
                    float wx_[NT], wy_[NT];
                    weights<kCubic>(ex - flx, wx_);
                    weights<kCubic>(ey - fly, wy_);
                    float* rf = recf + l * TR::STRIDE;
                    int* ri = reci + l * TR::STRIDE;
                    *reinterpret_cast<float4*>(rf + TR::WX) = make_float4(wx_[0], wx_[1], wx_[2], wx_[3]);
                    *reinterpret_cast<float4*>(rf + TR::WY) = make_float4(wy_[0], wy_[1], wy_[2], wy_[3]);
                    // the box offset of the first tap; 0 without a box (the flag stays negative)
                    const int base = boxed ? (fy + FIRST - y0) * PITCH + (fx + FIRST - x0) : 0;
                    *reinterpret_cast<float4*>(rf) =
                        make_float4(gp.x, sg * gp.y, wt, __int_as_float((fx + FIRST <= 0 || !boxed) ? ~base : base));
                    ri[TR::FX] = fx;
                    ri[TR::FY] = fy;
                }
                __syncwarp();
                // both halves step together for as many pixels as the fuller one has
                const int cnt = __popc(pmask);
                const int cmax = max(cnt, __shfl_xor_sync(kFull, cnt, 16));
                unsigned m = pmask;
                for (int it = 0; it < cmax; ++it) {
                    if (m) {
                        const int j = __ffs(m) - 1;
                        m &= m - 1;
                        const float* rf = recf + j * TR::STRIDE;
                        const int* ri = reci + j * TR::STRIDE;
                        const float4 head = *reinterpret_cast<const float4*>(rf);
                        const float2 gv = make_float2(head.x, head.y);
                        const float wtv = head.z;
                        const int rb = __float_as_int(head.w);
                        const float w = rf[TR::WY + tb] * rf[TR::WX + tk];
                        if (rb >= 0) {
                            const int e = rb + toff;
                            if (DATA) {
                                float2 a = acc[e];
                                a.x = fmaf(w, gv.x, a.x);
                                a.y = fmaf(w, gv.y, a.y);
                                acc[e] = a;
                            }
                            if (WTS) wacc[e] = fmaf(w, wtv, wacc[e]);
                        } else {
                            // taps on the x <= 0 column (exact per-tap rule), or no box
                            const int base = ~rb;
                            const int ux = ri[TR::FX] + FIRST + tk;
                            const bool direct = ux >= 1 || (ux == 0 && pass == 0);
                            if (direct && boxed) {
                                const int e = base + toff;
                                if (DATA) {
                                    float2 a = acc[e];
                                    a.x = fmaf(w, gv.x, a.x);
                                    a.y = fmaf(w, gv.y, a.y);
                                    acc[e] = a;
                                }
                                if (WTS) wacc[e] = fmaf(w, wtv, wacc[e]);
                            } else {
                                // target u (direct) or -u (mirrored, conjugate value)
                                int vx = ux, vy = ri[TR::FY] + FIRST + tb;
                                float vim = gv.y;
                                if (!direct) {
                                    vx = -vx;
                                    vy = -vy;
                                    vim = -vim;
                                }
                                const int iy = full_index(vy, g.Dv, g.halfv, g.centered);
                                if (vx >= 0 && vx <= g.halfv && iy >= 0) {
                                    const int off = iy * g.Hv + vx;
                                    if (DATA) atomicAdd(G + off, make_float2(w * gv.x, w * vim));
                                    if (WTS) atomicAdd(Wt + off, w * wtv);
                                }
                            }
                        }
                    }
                    __syncwarp();
                }
                // add the half's box to the image (read and clear the non-zero entries)
                if (boxed) {
                    const int nused = NX * NY;
                    const unsigned mx = (65536u + NX - 1) / NX;
                    for (int e = l; e < nused; e += 16) {
                        const int r = (int)(((unsigned)e * mx) >> 16);
                        const int xi = e - r * NX;
                        const int be = r * PITCH + xi;
                        float2 a = make_float2(0.f, 0.f);
                        float b = 0.f;
                        bool hit = false;
                        if (DATA) {
                            a = acc[be];
                            hit = a.x != 0.f || a.y != 0.f;
                        }
                        if (WTS) {
                            b = wacc[be];
                            hit = hit || b != 0.f;
                        }
                        if (hit) {
                            const int iy = full_index(y0 + r, g.Dv, g.halfv, g.centered);
                            const int ux = x0 + xi;
                            if (iy >= 0 && ux >= 0 && ux <= g.halfv) {
                                if (DATA && (a.x != 0.f || a.y != 0.f)) atomicAdd(G + iy * g.Hv + ux, a);
                                if (WTS && b != 0.f) atomicAdd(Wt + iy * g.Hv + ux, b);
                            }
                            if (DATA) acc[be] = make_float2(0.f, 0.f);
                            if (WTS) wacc[be] = 0.f;
                        }
                    }
                }
                __syncwarp();
            }
        }
    }
}

// Lane-per-pixel back-projection for linear 3D.  With 8 taps per pixel, the tile scatter's
// lanes-on-taps mapping keeps only 8 lanes busy and pays its per-pixel record and loop costs 4
// times over.  Here a warp takes an 8 x 4 tile of kept pixels, one pixel per lane, with the
// pixel's weights in registers; every lane adds its 8 taps to the warp's private box of shared
// memory with shared-memory float atomics (two pixels of the tile may share a voxel), and the
// box is then added to the volume like the tile scatter's (row-offset table, one reduction per
// non-zero voxel).  The box is dense, NX x NY x NZ voxels over the tile's footprint in the
// effective frame (pixels with c_x < 0 in a second pass at c' = -c, conjugated; see
// gather.cuh): at most 10 x 10 x 10 at o = 1, 264 voxels on average; tiles needing more than
// kLaneCap voxels (about 2 in 10^4 at o = 1), wider than 16 voxels, or with taps on the x <= 0
// planes take the exact per-tap rule with global atomics.
constexpr int kLaneCap = 512;   // box voxels of one warp
constexpr int kLaneRows = 96;   // box rows NY * NZ

template <bool DATA, bool WTS>
__host__ __device__ constexpr size_t lane_warp_bytes()
{
    return (DATA ? (size_t)kLaneCap * 8 : 0) + (WTS ? (size_t)kLaneCap * 4 : 0) + (size_t)kLaneRows * 4;
}

template <bool DATA, bool WTS>
__global__ void __launch_bounds__(kThreads) scatter_lane_kernel(
    const float2* __restrict__ proj, const float* __restrict__ wts,
    const float* __restrict__ rot, const float* __restrict__ shift,
    float2* __restrict__ vout, float* __restrict__ wout, Geom g, int splits, long long n_work)
{
    constexpr int NWARP = kThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    extern __shared__ __align__(16) unsigned char sm_raw[];
    unsigned char* mine = sm_raw + warp * lane_warp_bytes<DATA, WTS>();
    float2* acc = reinterpret_cast<float2*>(mine);
    float* wacc = reinterpret_cast<float*>(mine + (DATA ? kLaneCap * 8 : 0));
    int* rowoff = reinterpret_cast<int*>(mine + (DATA ? kLaneCap * 8 : 0) + (WTS ? kLaneCap * 4 : 0));
    __shared__ float Rs[9];
    __shared__ float2 sh;

    for (int e = lane; e < kLaneCap; e += 32) {
        if (DATA) acc[e] = make_float2(0.f, 0.f);
        if (WTS) wacc[e] = 0.f;
    }
    const int tiles_x = (g.Ho + 7) / 8, tiles_y = (g.Do + 3) / 4;
    const int ntiles = tiles_x * tiles_y;
    const int big = 1 << 28;

    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        __syncthreads();
        if (threadIdx.x < 9) {
            const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
            Rs[threadIdx.x] = g.o * __ldg(rot + ri * 9 + threadIdx.x);
        }
        if (threadIdx.x == 0) {
            sh = make_float2(0.f, 0.f);
            if (g.has_shift) {
                const long long si = (long long)(g.sh_shared ? 0 : ir.r) * g.n_pose + ir.p;
                sh = make_float2(__ldg(shift + si * 2), __ldg(shift + si * 2 + 1));
            }
        }
        __syncthreads();
        const float2* py = DATA ? proj + ir.item * g.img_elems : nullptr;
        const float* pw = (WTS && wts) ? wts + ir.item * g.img_elems : nullptr;  // NULL: weight 1
        float2* G = DATA ? vout + (long long)ir.r * g.rec_elems : nullptr;
        float* Wt = WTS ? wout + (long long)ir.r * g.rec_elems : nullptr;

        for (int tile = ir.part * NWARP + warp; tile < ntiles; tile += splits * NWARP) {
            const int ti = tile / tiles_x, tj = tile - ti * tiles_x;
            // lane l owns pixel (row 4 ti + l / 8, kx 8 tj + l % 8)
            const int prow = 4 * ti + (lane >> 3), pkx = 8 * tj + (lane & 7);
            bool kept = false;
            int ky = 0;
            float cx = 0.f, cy = 0.f, cz = 0.f;
            if (prow < g.Do && pkx < g.Ho) {
                ky = row_freq(prow, g.Do, g.halfo, g.centered);
                kept = pkx * pkx + ky * ky <= g.rc2;
                const float fkx = (float)pkx, fky = (float)ky;
                cx = fmaf(Rs[0], fkx, Rs[1] * fky);
                cy = fmaf(Rs[3], fkx, Rs[4] * fky);
                cz = fmaf(Rs[6], fkx, Rs[7] * fky);
            }
            const unsigned kept_mask = __ballot_sync(0xffffffffu, kept);
            if (!kept_mask) continue;
            const unsigned neg_mask = __ballot_sync(0xffffffffu, kept && cx < 0.f);
            float2 gp = make_float2(0.f, 0.f);
            float wt = 1.f;
            if (kept) {
                if (DATA) {
                    gp = __ldg(py + prow * g.Ho + pkx);
                    if (g.has_shift)
                        gp = cmul_conj(gp, shift_phase((float)pkx, (float)ky, sh.x, sh.y, g.Do_f, g.inv_Do));
                }
                if (WTS && pw) wt = __ldg(pw + prow * g.Ho + pkx);
            }
            for (int pass = 0; pass < 2; ++pass) {
                const unsigned pmask = pass ? neg_mask : (kept_mask & ~neg_mask);
                if (!pmask) continue;
                const bool mine_px = (pmask >> lane) & 1u;
                const float sg = pass ? -1.f : 1.f;
                // effective coordinates, clamped like floor_frac (integer extents stay small)
                const float lim = 8388608.0f;
                const float ex = fminf(fmaxf(sg * cx, -lim), lim);
                const float ey = fminf(fmaxf(sg * cy, -lim), lim);
                const float ez = fminf(fmaxf(sg * cz, -lim), lim);
                const float flx = floorf(ex), fly = floorf(ey), flz = floorf(ez);
                const int fx = (int)flx, fy = (int)fly, fz = (int)flz;
                // box of this pass's taps (floor and floor + 1 on each axis)
                const int x0 = __reduce_min_sync(0xffffffffu, mine_px ? fx : big);
                const int y0 = __reduce_min_sync(0xffffffffu, mine_px ? fy : big);
                const int z0 = __reduce_min_sync(0xffffffffu, mine_px ? fz : big);
                const int NX = __reduce_max_sync(0xffffffffu, mine_px ? fx : -big) + 2 - x0;
                const int NY = __reduce_max_sync(0xffffffffu, mine_px ? fy : -big) + 2 - y0;
                const int NZ = __reduce_max_sync(0xffffffffu, mine_px ? fz : -big) + 2 - z0;
                const bool boxed = NX <= 16 && NY <= kLaneRows && NZ <= kLaneRows && NY * NZ <= kLaneRows &&
                                   NX * NY * NZ <= kLaneCap;
                if (mine_px) {
                    const float frx = ex - flx, fry = ey - fly, frz = ez - flz;
                    const float wxs[2] = {1.f - frx, frx}, wys[2] = {1.f - fry, fry}, wzs[2] = {1.f - frz, frz};
                    // effective value: conj(g') on the mirrored pass (weights are real)
                    const float vx = gp.x, vy = sg * gp.y;
#pragma unroll
                    for (int a = 0; a < 2; ++a)
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const float wzy = wzs[a] * wys[b];
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const float wgt = wzy * wxs[k];
                                const int ux = fx + k;
                                const bool direct = ux >= 1 || (ux == 0 && pass == 0);
                                if (direct && boxed) {
                                    const int e = ((fz + a - z0) * NY + (fy + b - y0)) * NX + (ux - x0);
                                    if (DATA) {
                                        atomicAdd(&acc[e].x, wgt * vx);
                                        atomicAdd(&acc[e].y, wgt * vy);
                                    }
                                    if (WTS) atomicAdd(&wacc[e], wgt * wt);
                                } else {
                                    // target u (direct) or -u (mirrored, conjugate value)
                                    int tx = ux, ty = fy + b, tz = fz + a;
                                    float tim = vy;
                                    if (!direct) {
                                        tx = -tx;
                                        ty = -ty;
                                        tz = -tz;
                                        tim = -tim;
                                    }
                                    const int iy = full_index(ty, g.Dv, g.halfv, g.centered);
                                    const int iz = full_index(tz, g.Dv, g.halfv, g.centered);
                                    if (tx >= 0 && tx <= g.halfv && iy >= 0 && iz >= 0) {
                                        const long long off = ((long long)iz * g.Dv + iy) * g.Hv + tx;
                                        if (DATA) atomicAdd(G + off, make_float2(wgt * vx, wgt * tim));
                                        if (WTS) atomicAdd(Wt + off, wgt * wt);
                                    }
                                }
                            }
                        }
                }
                __syncwarp();
                // ---- add the box to the volume (read and clear); rows r = zi * NY + yi, entries
                // e = r * NX + xi (exact multiply-shift: e < 512 with NX <= 16, r < 96 with
                // NY <= 96); only non-zero entries are added and cleared
                if (boxed) {
                    const int nrows = NY * NZ;
                    const unsigned my = (65536u + NY - 1) / NY;
                    for (int r = lane; r < nrows; r += 32) {
                        const int zi = (int)(((unsigned)r * my) >> 16);
                        const int iy = full_index(y0 + r - zi * NY, g.Dv, g.halfv, g.centered);
                        const int iz = full_index(z0 + zi, g.Dv, g.halfv, g.centered);
                        rowoff[r] = (iy >= 0 && iz >= 0) ? (iz * g.Dv + iy) * g.Hv : -1;
                    }
                    __syncwarp();
                    const unsigned mx = (65536u + NX - 1) / NX;
                    const int nused = nrows * NX;
                    for (int e = lane; e < nused; e += 32) {
                        const int r = (int)(((unsigned)e * mx) >> 16);
                        const int ux = x0 + (e - r * NX);
                        bool hit = false;
                        float2 c = make_float2(0.f, 0.f);
                        float b = 0.f;
                        if (DATA) {
                            c = acc[e];
                            hit = c.x != 0.f || c.y != 0.f;
                        }
                        if (WTS) {
                            b = wacc[e];
                            hit = hit || b != 0.f;
                        }
                        if (hit) {
                            const int ro = rowoff[r];
                            if (ro >= 0 && ux >= 0 && ux <= g.halfv) {
                                if (DATA && (c.x != 0.f || c.y != 0.f)) atomicAdd(G + ro + ux, c);
                                if (WTS && b != 0.f) atomicAdd(Wt + ro + ux, b);
                            }
                            if (DATA) acc[e] = make_float2(0.f, 0.f);
                            if (WTS) wacc[e] = 0.f;
                        }
                    }
                }
                __syncwarp();
            }
        }
    }
}

// Weight-volume part of the back-projection's backward: per kept pixel the real
// interpolation v of the upstream weight-volume gradient (that is dL/d weight) and, for the
// rotation gradient, weight * o q_b dv/dc_a summed per item (exact per-tap path).
template <int NDIM, int INTERP, bool WANT_W, bool WANT_ROT>
__global__ void __launch_bounds__(kThreads) weights_grad_kernel(
    const float* __restrict__ gw, const float* __restrict__ weights, const float* __restrict__ rot,
    float* __restrict__ gweights, float* __restrict__ grot, Geom g, int splits, long long n_work)
{
    __shared__ float red[kThreads / 32];
    const int npix = (int)g.img_elems;
    for (long long w = blockIdx.x; w < n_work; w += gridDim.x) {
        const ItemRange ir = item_of(g, w, splits);
        ItemParams<NDIM> ip;
        load_item<NDIM>(g, rot, nullptr, ir.r, ir.p, ip);
        const float* Wv = gw + (long long)ir.r * g.rec_elems;
        const float* pw = weights ? weights + ir.item * g.img_elems : nullptr;
        float* gwo = WANT_W ? gweights + ir.item * g.img_elems : nullptr;
        float acc[2 * NDIM];
#pragma unroll
        for (int k = 0; k < 2 * NDIM; ++k) acc[k] = 0.f;
        for (int pix = ir.part * kThreads + threadIdx.x; pix < npix; pix += splits * kThreads) {
            int i, j;
            split_pixel(pix, g.Ho, i, j);
            const int ky = row_freq(i, g.Do, g.halfo, g.centered), kx = j;
            if (kx * kx + ky * ky > g.rc2) {
                if (WANT_W) gwo[pix] = 0.f;
                continue;
            }
            PixelTaps<NDIM, INTERP, WANT_ROT> t;
            t.init(g, ip.R, (float)kx, (float)ky);
            float v, dv[3];
            gather_real<NDIM, INTERP, WANT_ROT>(Wv, g, t, v, dv);
            if (WANT_W) gwo[pix] = v;
            if constexpr (WANT_ROT) {
                const float wt = pw ? __ldg(pw + pix) : 1.f;
#pragma unroll
                for (int a = 0; a < NDIM; ++a) {
                    acc[2 * a] = fmaf(wt * dv[a], (float)kx, acc[2 * a]);
                    acc[2 * a + 1] = fmaf(wt * dv[a], (float)ky, acc[2 * a + 1]);
                }
            }
        }
        if constexpr (WANT_ROT) {
            const long long ri = (long long)(g.rot_shared ? 0 : ir.r) * g.n_pose + ir.p;
#pragma unroll
            for (int k = 0; k < 2 * NDIM; ++k) {
                const float s = block_sum(acc[k], red);
                if (threadIdx.x == 0) atomicAdd(grot + ri * NDIM * NDIM + (k / 2) * NDIM + (k % 2), g.o * s);
            }
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

// Grouped copy of the volumes for the gathers: for every volume row (z, y) and every group
// start x = -(NT - 1) .. Dv/2 the NT taps x .. x + NT - 1 of the extended spectrum -- V[z][y][x]
// for 0 <= x <= Dv/2, zero beyond, and for x < 0 the conjugate mirror conj V[-z][-y][-x]
// (Friedel symmetry of the half spectrum; zero when -z or -y is outside the stored band or
// -x > Dv/2), the value the per-tap rule reads there.  Group (z, y, x) sits at group index
// z * pplane + y * prow + x + NT - 1 of its volume (pitches from group_pitch; the padding
// groups are written as zeros), and a row's taps are then one aligned vector load.  A thread
// per group (IDX: 32-bit index arithmetic when the groups fit, else 64-bit).
template <int NT, typename IDX>
__global__ void __launch_bounds__(kThreads) expand_groups_kernel(const float2* __restrict__ V,
                                                                  float2* __restrict__ Q, int Dv,
                                                                  int Hv, int halfv, int centered,
                                                                  int prow, int pplane,
                                                                  IDX n_groups)
{
    constexpr int LEAD = NT - 1;  // groups ahead of x = 0
    const IDX P = (IDX)pplane, D = (IDX)Dv;
    // consecutive threads write consecutive groups
    for (IDX i = (IDX)blockIdx.x * kThreads + threadIdx.x; i < n_groups;
         i += (IDX)gridDim.x * kThreads) {
        const IDX zr = i / P;  // r * Dv + z
        const int j = (int)(i - zr * P);
        const int iy = j / prow;
        const int x0 = j - iy * prow - LEAD;
        float2 e[NT];
#pragma unroll
        for (int k = 0; k < NT; ++k) e[k] = make_float2(0.f, 0.f);
        if (iy < Dv) {
            const IDX r = zr / D;
            const int iz = (int)(zr - r * D);
            const float2* v = V + ((long long)zr * Dv + iy) * Hv;
            const float2* vm = nullptr;  // the mirrored row (-z, -y), when x0 < 0
            if (x0 < 0) {
                const int iym = full_index(-row_freq(iy, Dv, halfv, centered), Dv, halfv, centered);
                const int izm = full_index(-row_freq(iz, Dv, halfv, centered), Dv, halfv, centered);
                if ((iym | izm) >= 0) vm = V + (((long long)r * Dv + izm) * Dv + iym) * Hv;
            }
#pragma unroll
            for (int k = 0; k < NT; ++k) {
                const int x = x0 + k;
                if (x >= 0) {
                    if (x <= halfv) e[k] = __ldg(v + x);
                } else if (vm && -x <= halfv) {
                    e[k] = __ldg(vm - x);
                    e[k].y = -e[k].y;
                }
            }
        }
        float4* q = reinterpret_cast<float4*>(Q + (long long)i * NT);
#pragma unroll
        for (int k = 0; k < NT; k += 2) q[k / 2] = make_float4(e[k].x, e[k].y, e[k + 1].x, e[k + 1].y);
    }
}

// Splits of one item over CTAs so that a small batch still fills `target` CTAs: at most
// `max_parts` (the item's units of work), at least 1.
long long item_splits(long long n_items, long long target, long long max_parts)
{
    long long splits = 1;
    if (n_items > 0 && n_items < target) splits = (target + n_items - 1) / n_items;
    if (splits > max_parts) splits = max_parts;
    return splits < 1 ? 1 : splits;
}

// Table kernels: one CTA per (item, part) at a time, grid = a few waves of resident CTAs.
struct TableShape {
    unsigned grid;
    size_t smem;
    int splits;
    long long n_work;
};

TableShape table_shape(const Geom& g, int sms, int ctas_per_sm, int threads, int ndim)
{
    const long long n_items = (long long)g.n_rec * g.n_pose;
    const long long max_parts = (g.img_elems + threads - 1) / threads;
    TableShape t;
    t.splits = (int)item_splits(n_items, (long long)ctas_per_sm * sms, max_parts);
    t.n_work = n_items * t.splits;
    const long long cap = 16LL * sms;  // persistent-style: the table is built once per CTA
    t.grid = (unsigned)(t.n_work < cap ? t.n_work : cap);
    t.smem = (size_t)(g.Do + 1 + kWarpQueue * (threads / 32)) * sizeof(int);  // table + warp queues
    if (use_twiddles(g, ndim)) t.smem += 8 + 2 * (size_t)(g.Ho + g.Do) * sizeof(float2);  // aligned
    return t;
}

bool use_table(const Geom& g) { return g.Do <= kMaxTableRows; }

// Widest aligned window the volume layout allows: 32-byte windows need the z-plane
// stride Dv * Hv to be a multiple of 4 elements (Dv % 4 == 0).
int window_for(const Geom& g, int ndim) { return (ndim == 2 || g.Dv % 4 == 0) ? TP_GATHER_WIN : 2; }

template <int NDIM, int INTERP, int WIN>
void launch_project_table(const Geom& g, const float2* R, const float* rot, const float* shift,
                          float2* Y, const float2* grouped, int sms, cudaStream_t stream)
{
    constexpr int BT = NDIM == 3 ? kFwd3Threads : kThreads;
    const TableShape t = table_shape(g, sms, 4, BT, NDIM);
    project_kernel<NDIM, INTERP, WIN><<<t.grid, BT, t.smem, stream>>>(
        R, rot, shift, Y, g, t.splits, t.n_work, grouped);
}

template <int NDIM, int INTERP>
void launch_project_t(const Geom& g, const float2* R, const float* rot, const float* shift,
                      float2* Y, const float2* grouped, int sms, cudaStream_t stream)
{
    if (!use_table(g)) {
        const LaunchShape s = launch_shape(g, sms);
        project_kernel_any<NDIM, INTERP><<<s.grid, kThreads, 0, stream>>>(R, rot, shift, Y, g,
                                                                           s.splits, s.n_work);
        return;
    }
    if (grouped)
        launch_project_table<NDIM, INTERP, kGrouped>(g, R, rot, shift, Y, grouped, sms, stream);
    else if (window_for(g, NDIM) == 4)
        launch_project_table<NDIM, INTERP, 4>(g, R, rot, shift, Y, nullptr, sms, stream);
    else if (window_for(g, NDIM) == 2)
        launch_project_table<NDIM, INTERP, 2>(g, R, rot, shift, Y, nullptr, sms, stream);
    else
        launch_project_table<NDIM, INTERP, 1>(g, R, rot, shift, Y, nullptr, sms, stream);
}

template <int NDIM, int INTERP, int WIN>
void launch_grad_table(const Geom& g, const float2* R, const float* rot, const float* shift,
                       const float2* G, float* grot, float* gsh, const float2* grouped, int sms,
                       cudaStream_t stream)
{
    const TableShape t = table_shape(g, sms, 4, kPoseThreads, NDIM);
    grad_pose_kernel<NDIM, INTERP, WIN><<<t.grid, kPoseThreads, t.smem, stream>>>(
        R, rot, shift, G, grot, gsh, g, t.splits, t.n_work, grouped);
}

template <int NDIM, int INTERP>
void launch_grad_t(const Geom& g, const float2* R, const float* rot, const float* shift,
                   const float2* G, float* grot, float* gsh, const float2* grouped, int sms,
                   cudaStream_t stream)
{
    if (!use_table(g)) {
        const LaunchShape s = launch_shape(g, sms);
        grad_pose_kernel_any<NDIM, INTERP><<<s.grid, kThreads, 0, stream>>>(
            R, rot, shift, G, grot, gsh, g, s.splits, s.n_work);
        return;
    }
    if (grouped)
        launch_grad_table<NDIM, INTERP, kGrouped>(g, R, rot, shift, G, grot, gsh, grouped, sms, stream);
    else if (window_for(g, NDIM) == 4)
        launch_grad_table<NDIM, INTERP, 4>(g, R, rot, shift, G, grot, gsh, nullptr, sms, stream);
    else if (window_for(g, NDIM) == 2)
        launch_grad_table<NDIM, INTERP, 2>(g, R, rot, shift, G, grot, gsh, nullptr, sms, stream);
    else
        launch_grad_table<NDIM, INTERP, 1>(g, R, rot, shift, G, grot, gsh, nullptr, sms, stream);
}

template <int NDIM, int INTERP, bool DATA, bool WTS>
void launch_scatter_rows(const Geom& g, const float2* P, const float* weights, const float* rot,
                         const float* shift, float2* VO, float* WO, int sms, cudaStream_t stream)
{
    constexpr int AW = SegMargin<INTERP>::AW;
    const size_t smem = (DATA ? (size_t)AW * kRowsThreads * 8 : 0) + (WTS ? (size_t)AW * kRowsThreads * 4 : 0) +
                        (size_t)(g.Ho + g.Do) * 8 + (size_t)(g.Do + 2 * g.Dv + 1) * 4;
    auto kern = scatter_rows_kernel<NDIM, INTERP, DATA, WTS, kRowsThreads>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const long long n_items = (long long)g.n_rec * g.n_pose;
    const long long cap = 8LL * sms * kThreads / kRowsThreads;
    const unsigned grid = (unsigned)(n_items < cap ? n_items : cap);
    kern<<<grid, kRowsThreads, smem, stream>>>(P, weights, rot, shift, VO, WO, g, n_items);
}

template <int INTERP, bool DATA, bool WTS, bool POSE>
void launch_scatter_tile_t(const Geom& g, const float2* P, const float* weights, const float* rot,
                           const float* shift, float2* VO, float* WO, int sms, cudaStream_t stream,
                           const float2* vol, float* grot, float* gsh)
{
    constexpr size_t box_cap = BoxDims<WTS>::CAP;
    const size_t per_warp = (DATA ? box_cap * 8 : 0) + (WTS ? box_cap * 4 : 0) +
                            (size_t)TileRecT<POSE>::WORDS * 4;
    constexpr int threads = POSE ? kTileThreadsPose : kTileThreads, nwarp = threads / 32;
    const size_t smem = per_warp * nwarp;
    auto kern = scatter_tile_kernel<INTERP, DATA, WTS, POSE>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const long long n_items = (long long)g.n_rec * g.n_pose;
    const long long ntiles = (long long)((g.Ho + 3) / 4) * ((g.Do + 3) / 4);
    const int splits = (int)item_splits(n_items, 3LL * sms, (ntiles + nwarp - 1) / nwarp);
    const long long n_work = n_items * splits;
    const long long cap = 8LL * sms;
    const unsigned grid = (unsigned)(n_work < cap ? n_work : cap);
    kern<<<grid, threads, smem, stream>>>(P, weights, rot, shift, VO, WO, g, splits, n_work, vol,
                                          grot, gsh);
}

template <int INTERP, bool DATA, bool WTS>
void launch_scatter_tile(const Geom& g, const float2* P, const float* weights, const float* rot,
                         const float* shift, float2* VO, float* WO, int sms, cudaStream_t stream)
{
    launch_scatter_tile_t<INTERP, DATA, WTS, false>(g, P, weights, rot, shift, VO, WO, sms, stream,
                                                    nullptr, nullptr, nullptr);
}

template <bool DATA, bool WTS>
void launch_scatter_tile2d(const Geom& g, const float2* P, const float* weights, const float* rot,
                           const float* shift, float2* VO, float* WO, int sms, cudaStream_t stream)
{
    constexpr size_t cap = (size_t)kTile2Pitch * kTile2Rows;
    constexpr int nwarp = kTile2Threads / 32;
    const size_t per_half = (DATA ? cap * 8 : 0) + (WTS ? cap * 4 : 0) +
                            (size_t)kTilePix * Tile2Rec::STRIDE * 4;
    const size_t smem = per_half * 2 * nwarp;
    auto kern = scatter_tile2d_kernel<DATA, WTS>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const long long n_items = (long long)g.n_rec * g.n_pose;
    const long long ntiles = (long long)((g.Ho + 3) / 4) * ((g.Do + 3) / 4);
    const int splits = (int)item_splits(n_items, 3LL * sms, (ntiles + 2 * nwarp - 1) / (2 * nwarp));
    const long long n_work = n_items * splits;
    const long long cap_grid = 8LL * sms;
    const unsigned grid = (unsigned)(n_work < cap_grid ? n_work : cap_grid);
    kern<<<grid, kTile2Threads, smem, stream>>>(P, weights, rot, shift, VO, WO, g, splits, n_work);
}

template <bool DATA, bool WTS>
void launch_scatter_lane(const Geom& g, const float2* P, const float* weights, const float* rot,
                         const float* shift, float2* VO, float* WO, int sms, cudaStream_t stream)
{
    const size_t smem = lane_warp_bytes<DATA, WTS>() * (kThreads / 32);
    auto kern = scatter_lane_kernel<DATA, WTS>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const long long n_items = (long long)g.n_rec * g.n_pose;
    const long long ntiles = (long long)((g.Ho + 7) / 8) * ((g.Do + 3) / 4);
    const int splits = (int)item_splits(n_items, 3LL * sms, (ntiles + kThreads / 32 - 1) / (kThreads / 32));
    const long long n_work = n_items * splits;
    const long long cap = 8LL * sms;
    const unsigned grid = (unsigned)(n_work < cap ? n_work : cap);
    kern<<<grid, kThreads, smem, stream>>>(P, weights, rot, shift, VO, WO, g, splits, n_work);
}

template <int NDIM, int INTERP>
void launch_backproject_t(const Geom& g, const float2* P, const float* weights, const float* rot,
                          const float* shift, float2* VO, float* WO, int sms, cudaStream_t stream)
{
    if (g.Dv > kMaxScatterBox || g.Do > kMaxScatterBox) {
        const LaunchShape s = launch_shape(g, sms);
        backproject_kernel<NDIM, INTERP><<<s.grid, kThreads, 0, stream>>>(P, weights, rot, shift, VO,
                                                                           WO, g, s.splits, s.n_work);
        return;
    }
    if constexpr (NDIM == 3 && INTERP == kLinear) {
        if (VO && WO)
            launch_scatter_lane<true, true>(g, P, weights, rot, shift, VO, WO, sms, stream);
        else if (VO)
            launch_scatter_lane<true, false>(g, P, weights, rot, shift, VO, WO, sms, stream);
        else
            launch_scatter_lane<false, true>(g, P, weights, rot, shift, VO, WO, sms, stream);
    } else if constexpr (NDIM == 3) {
        if (VO && WO)
            launch_scatter_tile<INTERP, true, true>(g, P, weights, rot, shift, VO, WO, sms, stream);
        else if (VO)
            launch_scatter_tile<INTERP, true, false>(g, P, weights, rot, shift, VO, WO, sms, stream);
        else
            launch_scatter_tile<INTERP, false, true>(g, P, weights, rot, shift, VO, WO, sms, stream);
    } else {
        // 2D cubic with weights: the half-warp tile scatter (14.1 -> 10.4 ms for 8 192 images at
        // D = 256); the data alone ties with the owner-computes rows kernel (8.36 ms both),
        // which writes every voxel once, without atomics, and so keeps it
        if constexpr (INTERP == kCubic) {
            if (VO && WO) {
                launch_scatter_tile2d<true, true>(g, P, weights, rot, shift, VO, WO, sms, stream);
                return;
            }
        }
        if (VO && WO)
            launch_scatter_rows<NDIM, INTERP, true, true>(g, P, weights, rot, shift, VO, WO, sms, stream);
        else if (VO)
            launch_scatter_rows<NDIM, INTERP, true, false>(g, P, weights, rot, shift, VO, WO, sms, stream);
        else
            launch_scatter_rows<NDIM, INTERP, false, true>(g, P, weights, rot, shift, VO, WO, sms, stream);
    }
}

template <int NDIM, int INTERP>
void launch_weights_grad_t(const Geom& g, const float* gw, const float* weights, const float* rot,
                           float* gweights, float* grot, int sms, cudaStream_t stream)
{
    const LaunchShape s = launch_shape(g, sms);
    if (gweights && grot)
        weights_grad_kernel<NDIM, INTERP, true, true><<<s.grid, kThreads, 0, stream>>>(
            gw, weights, rot, gweights, grot, g, s.splits, s.n_work);
    else if (gweights)
        weights_grad_kernel<NDIM, INTERP, true, false><<<s.grid, kThreads, 0, stream>>>(
            gw, weights, rot, gweights, grot, g, s.splits, s.n_work);
    else if (grot)
        weights_grad_kernel<NDIM, INTERP, false, true><<<s.grid, kThreads, 0, stream>>>(
            gw, weights, rot, gweights, grot, g, s.splits, s.n_work);
}

}  // namespace

cudaError_t launch_weights_grad(int ndim, int interp, const Geom& g, const float* grad_wvol,
                                const float* weights, const float* rot, float* grad_weights,
                                float* grad_rot, int sms, cudaStream_t stream)
{
    if ((long long)g.n_rec * g.n_pose == 0 || (!grad_weights && !grad_rot)) return cudaSuccess;
    if (ndim == 3 && interp == kCubic)
        launch_weights_grad_t<3, kCubic>(g, grad_wvol, weights, rot, grad_weights, grad_rot, sms, stream);
    else if (ndim == 3)
        launch_weights_grad_t<3, kLinear>(g, grad_wvol, weights, rot, grad_weights, grad_rot, sms, stream);
    else if (interp == kCubic)
        launch_weights_grad_t<2, kCubic>(g, grad_wvol, weights, rot, grad_weights, grad_rot, sms, stream);
    else
        launch_weights_grad_t<2, kLinear>(g, grad_wvol, weights, rot, grad_weights, grad_rot, sms, stream);
    return cudaGetLastError();
}

cudaError_t launch_expand_groups(int interp, const Geom& g, const void* rec, void* grouped, int sms,
                                 cudaStream_t stream)
{
    const long long n_groups = (long long)g.n_rec * g.Dv * g.gplane;
    if (n_groups == 0) return cudaSuccess;
    const long long blocks = (n_groups + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(blocks < 64LL * sms ? blocks : 64LL * sms);
    auto V = static_cast<const float2*>(rec);
    auto Q = static_cast<float2*>(grouped);
    const bool narrow = n_groups < (1LL << 31);  // 32-bit index arithmetic
    if (interp == kCubic && narrow)
        expand_groups_kernel<4, unsigned><<<grid, kThreads, 0, stream>>>(
            V, Q, g.Dv, g.Hv, g.halfv, g.centered, g.grow, g.gplane, (unsigned)n_groups);
    else if (interp == kCubic)
        expand_groups_kernel<4, long long><<<grid, kThreads, 0, stream>>>(
            V, Q, g.Dv, g.Hv, g.halfv, g.centered, g.grow, g.gplane, n_groups);
    else if (narrow)
        expand_groups_kernel<2, unsigned><<<grid, kThreads, 0, stream>>>(
            V, Q, g.Dv, g.Hv, g.halfv, g.centered, g.grow, g.gplane, (unsigned)n_groups);
    else
        expand_groups_kernel<2, long long><<<grid, kThreads, 0, stream>>>(
            V, Q, g.Dv, g.Hv, g.halfv, g.centered, g.grow, g.gplane, n_groups);
    return cudaGetLastError();
}

cudaError_t launch_project(int ndim, int interp, const Geom& g, const void* rec,
                           const float* rot, const float* shift, void* out, int sms,
                           cudaStream_t stream, const void* grouped)
{
    if ((long long)g.n_rec * g.n_pose == 0) return cudaSuccess;
    auto R = static_cast<const float2*>(rec);
    auto Y = static_cast<float2*>(out);
    auto Q = static_cast<const float2*>(grouped);
    if (ndim == 3 && interp == kCubic)
        launch_project_t<3, kCubic>(g, R, rot, shift, Y, Q, sms, stream);
    else if (ndim == 3)
        launch_project_t<3, kLinear>(g, R, rot, shift, Y, Q, sms, stream);
    else if (interp == kCubic)
        launch_project_t<2, kCubic>(g, R, rot, shift, Y, nullptr, sms, stream);
    else
        launch_project_t<2, kLinear>(g, R, rot, shift, Y, nullptr, sms, stream);
    return cudaGetLastError();
}

cudaError_t launch_backward(int ndim, int interp, const Geom& g, const void* rec,
                            const float* rot, const float* shift, const void* grad_out,
                            void* grad_rec, float* grad_rot, float* grad_shift, int sms,
                            cudaStream_t stream, const void* grouped, bool fused)
{
    if ((long long)g.n_rec * g.n_pose == 0) return cudaSuccess;
    auto R = static_cast<const float2*>(rec);
    auto G = static_cast<const float2*>(grad_out);
    auto GR = static_cast<float2*>(grad_rec);
    auto Q = static_cast<const float2*>(grouped);
    const bool want_grad = grad_rot || (grad_shift && g.has_shift);
    if (fused && ndim == 3 && interp == kCubic && GR && want_grad) {
        // one pass: volume, rotation and shift gradients
        launch_scatter_tile_t<kCubic, true, false, true>(g, G, nullptr, rot, shift, GR, nullptr, sms,
                                                         stream, R, grad_rot, grad_shift);
        return cudaGetLastError();
    }
    if (want_grad) {
        if (ndim == 3 && interp == kCubic)
            launch_grad_t<3, kCubic>(g, R, rot, shift, G, grad_rot, grad_shift, Q, sms, stream);
        else if (ndim == 3)
            launch_grad_t<3, kLinear>(g, R, rot, shift, G, grad_rot, grad_shift, Q, sms, stream);
        else if (interp == kCubic)
            launch_grad_t<2, kCubic>(g, R, rot, shift, G, grad_rot, grad_shift, nullptr, sms, stream);
        else
            launch_grad_t<2, kLinear>(g, R, rot, shift, G, grad_rot, grad_shift, nullptr, sms, stream);
    }
    if (GR) {
        if (ndim == 3 && interp == kCubic)
            launch_backproject_t<3, kCubic>(g, G, nullptr, rot, shift, GR, nullptr, sms, stream);
        else if (ndim == 3)
            launch_backproject_t<3, kLinear>(g, G, nullptr, rot, shift, GR, nullptr, sms, stream);
        else if (interp == kCubic)
            launch_backproject_t<2, kCubic>(g, G, nullptr, rot, shift, GR, nullptr, sms, stream);
        else
            launch_backproject_t<2, kLinear>(g, G, nullptr, rot, shift, GR, nullptr, sms, stream);
    }
    return cudaGetLastError();
}

cudaError_t launch_backproject(int ndim, int interp, const Geom& g, const void* proj,
                               const float* weights, const float* rot, const float* shift,
                               void* vol_out, float* wvol_out, int sms, cudaStream_t stream)
{
    if ((long long)g.n_rec * g.n_pose == 0 || (!vol_out && !wvol_out)) return cudaSuccess;
    auto P = static_cast<const float2*>(proj);
    auto VO = static_cast<float2*>(vol_out);
    if (ndim == 3 && interp == kCubic)
        launch_backproject_t<3, kCubic>(g, P, weights, rot, shift, VO, wvol_out, sms, stream);
    else if (ndim == 3)
        launch_backproject_t<3, kLinear>(g, P, weights, rot, shift, VO, wvol_out, sms, stream);
    else if (interp == kCubic)
        launch_backproject_t<2, kCubic>(g, P, weights, rot, shift, VO, wvol_out, sms, stream);
    else
        launch_backproject_t<2, kLinear>(g, P, weights, rot, shift, VO, wvol_out, sms, stream);
    return cudaGetLastError();
}

}  // namespace tp
