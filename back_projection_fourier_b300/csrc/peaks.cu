// peaks.cu -- microbenchmarks of the on-chip units that bound the projection kernels.
//
// The projection kernels are bound by units inside the SM, not by HBM: the gathers by the
// L1 data pipe that serves their tap loads, the scatters by shared-memory read-modify-writes
// (and, for what leaves the SM, by L2 reductions).  Each microbenchmark here drives one of
// those units flat out on a buffer that stays resident in it, so that the caller can time it
// with CUDA events on the same device, in the same run, and divide a kernel's algorithmic
// work by the measured rate.  They compute nothing of the method.
//
// Every kernel keeps its result live by writing one value to `sink` under a condition the
// inputs never meet (an all-zero buffer never sums to a negative number), so the compiler
// cannot drop the work and nothing is stored in the timed loop.  All indices are masked into
// the buffers the host sized; no kernel waits on anything.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tp_peaks.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWindowBytes = 16384;   // per-CTA L1-resident window of the load kernels
constexpr int kWindows = 64;
constexpr size_t kRedBytes = 8u << 20;  // L2-resident target of the global reductions
constexpr int kRmwSlots = 512;          // float2 per warp of the read-modify-write kernels
constexpr size_t kSinkOffset = (size_t)kWindows * kWindowBytes + kRedBytes;
constexpr size_t kNeed = kSinkOffset + 256;

__device__ __forceinline__ uint32_t lcg(uint32_t x) { return x * 1664525u + 1013904223u; }

// Coalesced 16-byte loads from the CTA's window: the data pipe's best case (a warp reads
// 512 contiguous bytes per instruction).  Each round's offset depends on the values the
// previous round loaded (the window holds zeros, so it always advances by one round), which
// keeps the compiler from hoisting or merging loads whose addresses repeat every four rounds.
__global__ void __launch_bounds__(kThreads) l1_load_kernel(const float4* __restrict__ buf, int iters,
                                                           float* sink)
{
    const int n4 = kWindowBytes / 16;  // 1024 float4; one round reads 1024 of them
    const float4* w = buf + (size_t)(blockIdx.x % kWindows) * n4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t off = threadIdx.x;
    for (int it = 0; it < iters; ++it) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(w + ((off + u * kThreads) & (n4 - 1)));
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            acc.x += v[u].x;
            acc.y += v[u].y;
            acc.z += v[u].z;
            acc.w += v[u].w;
        }
        off += 4 * kThreads + (__float_as_uint(v[3].w) & 16u);
    }
    if (acc.x + acc.y + acc.z + acc.w < 0.f) sink[0] = acc.x;
}

// Loads of BYTES (8: one float2; 32: one aligned 32-byte row) at random positions of the
// CTA's window, every lane its own: the gathers' access pattern, L1-resident.
template <int BYTES>
__global__ void __launch_bounds__(kThreads) l1_gather_kernel(const float* __restrict__ buf, int iters,
                                                             float* sink)
{
    constexpr int NF = BYTES / 4;
    const int nslots = kWindowBytes / BYTES;
    const float* w = buf + (size_t)(blockIdx.x % kWindows) * (kWindowBytes / 4);
    uint32_t x = lcg(blockIdx.x * kThreads + threadIdx.x + 1);
    float acc = 0.f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            x = lcg(x);
            const float* p = w + (size_t)((x >> 9) & (nslots - 1)) * NF;
            if constexpr (NF == 2) {
                const float2 v = __ldg(reinterpret_cast<const float2*>(p));
                acc += v.x + v.y;
            } else {
                float e[8];
                asm volatile("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=f"(e[0]), "=f"(e[1]), "=f"(e[2]), "=f"(e[3]), "=f"(e[4]), "=f"(e[5]),
                               "=f"(e[6]), "=f"(e[7])
                             : "l"(p));
                acc += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
            }
        }
    }
    if (acc < 0.f) sink[0] = acc;
}

// Shared-memory float2 read-modify-writes.  CONFLICT_FREE: a warp touches 32 consecutive
// float2 (two wavefronts each way), the best case; otherwise every lane a random float2 of
// its warp's 512-entry region (distinct lanes may collide in banks, as random taps do).  The
// loads and stores are volatile, so each one reaches shared memory.
__device__ __forceinline__ float2 lds_v2(uint32_t a)
{
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ void sts_v2(uint32_t a, float2 v)
{
    asm volatile("st.shared.v2.f32 [%0], {%1,%2};" ::"r"(a), "f"(v.x), "f"(v.y) : "memory");
}

template <bool CONFLICT_FREE>
__global__ void __launch_bounds__(kThreads) smem_rmw_kernel(int iters, float* sink)
{
    __shared__ float2 box[kThreads / 32][kRmwSlots];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = lane; e < kRmwSlots; e += 32) box[warp][e] = make_float2(0.f, 0.f);
    __syncwarp();
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(&box[warp][0]);
    uint32_t x = lcg(threadIdx.x + 7);
    const float2 v = make_float2(1e-30f * (float)lane, 0.f);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int e;
            if constexpr (CONFLICT_FREE) {
                e = (((it * 4 + u) * 7) & (kRmwSlots / 32 - 1)) * 32 + lane;
            } else {
                x = lcg(x);
                e = (int)((x >> 9) & (kRmwSlots - 1));
            }
            const uint32_t a = base + 8u * (uint32_t)e;
            float2 c = lds_v2(a);
            c.x += v.x;
            c.y += v.y;
            sts_v2(a, c);
        }
    }
    __syncwarp();
    if (box[warp][lane].x < 0.f) sink[0] = box[warp][lane].y;
}

// Shared-memory float atomics (red.shared.add.f32) at random addresses of a 4 KB-per-warp
// region: the alternative to a plain read-modify-write when lanes may collide.
__global__ void __launch_bounds__(kThreads) smem_red_kernel(int iters, float* sink)
{
    __shared__ float box[kThreads / 32][1024];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = lane; e < 1024; e += 32) box[warp][e] = 0.f;
    __syncwarp();
    uint32_t x = lcg(threadIdx.x + 11);
    const float v = 1e-30f * (float)lane;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            x = lcg(x);
            atomicAdd(&box[warp][(x >> 9) & 1023], v);
        }
    }
    __syncwarp();
    if (box[warp][lane] < 0.f) sink[0] = box[warp][lane];
}

// Vector reductions red.global.add.v2.f32 at random 8-byte positions of an 8 MB buffer that
// stays in L2: the path by which a scatter's sums leave the SM.
__global__ void __launch_bounds__(kThreads) l2_red_kernel(float2* __restrict__ buf, int iters)
{
    const uint32_t n = (uint32_t)(kRedBytes / 8);
    uint32_t x = lcg(blockIdx.x * kThreads + threadIdx.x + 3);
    const float2 v = make_float2(1e-30f, 0.f);
    for (int it = 0; it < iters; ++it) {
        x = lcg(x);
        atomicAdd(buf + ((x >> 4) & (n - 1)), v);
    }
}

// Eight independent FMA chains per thread: the FP32 pipe's peak.
__global__ void __launch_bounds__(kThreads) fma_kernel(int iters, float* sink)
{
    float a[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = 1e-3f * (float)(threadIdx.x + k);
    const float m = 0.999f, c = 1e-7f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int k = 0; k < 8; ++k) a[k] = fmaf(a[k], m, c);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s += a[k];
    if (s < 0.f) sink[0] = s;
}

}  // namespace

extern "C" size_t tp_peak_scratch_bytes(void) { return kNeed; }

extern "C" int tp_peak_run(int kind, void* scratch, size_t scratch_bytes, int ctas, int iters,
                           void* stream, double* ops, double* bytes)
{
    if (!scratch || !ops || !bytes || scratch_bytes < kNeed || ctas < 1 || iters < 1 ||
        (reinterpret_cast<uintptr_t>(scratch) & 255))
        return 1;
    auto st = static_cast<cudaStream_t>(stream);
    auto* base = static_cast<unsigned char*>(scratch);
    float* sink = reinterpret_cast<float*>(base + kSinkOffset);
    const double threads = (double)ctas * kThreads;
    switch (kind) {
    case TP_PEAK_L1_LOAD:
        l1_load_kernel<<<ctas, kThreads, 0, st>>>(reinterpret_cast<const float4*>(base), iters, sink);
        *ops = threads * iters * 4;
        *bytes = *ops * 16;
        break;
    case TP_PEAK_L1_GATHER8:
        l1_gather_kernel<8><<<ctas, kThreads, 0, st>>>(reinterpret_cast<const float*>(base), iters, sink);
        *ops = threads * iters * 4;
        *bytes = *ops * 8;
        break;
    case TP_PEAK_L1_GATHER32:
        l1_gather_kernel<32><<<ctas, kThreads, 0, st>>>(reinterpret_cast<const float*>(base), iters, sink);
        *ops = threads * iters * 4;
        *bytes = *ops * 32;
        break;
    case TP_PEAK_SMEM_RMW:
        smem_rmw_kernel<true><<<ctas, kThreads, 0, st>>>(iters, sink);
        *ops = threads * iters * 4;
        *bytes = *ops * 16;
        break;
    case TP_PEAK_SMEM_RMW_RANDOM:
        smem_rmw_kernel<false><<<ctas, kThreads, 0, st>>>(iters, sink);
        *ops = threads * iters * 4;
        *bytes = *ops * 16;
        break;
    case TP_PEAK_SMEM_RED:
        smem_red_kernel<<<ctas, kThreads, 0, st>>>(iters, sink);
        *ops = threads * iters * 4;
        *bytes = *ops * 4;
        break;
    case TP_PEAK_L2_RED:
        l2_red_kernel<<<ctas, kThreads, 0, st>>>(
            reinterpret_cast<float2*>(base + (size_t)kWindows * kWindowBytes), iters);
        *ops = threads * iters;
        *bytes = *ops * 8;
        break;
    case TP_PEAK_FMA:
        fma_kernel<<<ctas, kThreads, 0, st>>>(iters, sink);
        *ops = threads * iters * 64 * 2;  // flops
        *bytes = 0;
        break;
    default:
        return 1;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
