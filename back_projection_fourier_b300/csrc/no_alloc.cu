// no_alloc.cu -- the 3D forward projection with the grouped-tap speed-up for callers that
// cannot allocate device memory.
//
// The workspace calls (tp_project_3d_to_2d_ws) need a buffer for the grouped copy of the
// volume, and the plain calls need none but are slower.  Some callers can neither
// allocate nor hand over a workspace: code whose device memory is owned entirely by
// another allocator (a framework's caching allocator or a fixed-budget memory pool that
// forbids allocations outside it), and code on a latency-critical path where cudaMalloc
// is not allowed because it can synchronise the device and take milliseconds.  This file
// gives them the grouped path with its scratch in a fixed array of device memory that the
// library itself holds, so the call allocates nothing.
#include <mutex>

#include "../../include/tp.h"
#include "tp_device.cuh"

namespace {

// The grouped copy of one D = 128 volume with cubic taps.
constexpr size_t kScratchBytes = (size_t)tp::grouped_volume_elems(128, 4) * 8;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device ordinal for
// the life of the process (a cudaDeviceReset would unload the array; the header tells
// callers not to use this entry point on a device they have reset).  In host code the name
// g_scratch is only a host-side stand-in, never a device address.
tp_status scratch_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return TP_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return TP_OK;
}

}  // namespace

extern "C" tp_status tp_project_3d_to_2d_noalloc(const void* vol, int n_rec, int Dv,
                                                 const float* rot, int n_rot, int n_pose,
                                                 const float* shift, int n_sh, void* out, int Do,
                                                 const tp_opts* opts, void* stream)
{
    const size_t need = tp_workspace_size(3, n_rec, Dv, opts);
    if (need > kScratchBytes) return TP_ERR_SHAPE;
    void* ws = nullptr;
    if (need > 0 && (long long)n_rec * n_pose > 0) {
        const tp_status st = scratch_address(&ws);
        if (st != TP_OK) return st;
    }
    // Every byte of the grouped copy that the gathers read is written first by this call,
    // so the previous call's contents never need clearing.
    return tp_project_3d_to_2d_ws(vol, n_rec, Dv, rot, n_rot, n_pose, shift, n_sh, out, Do, ws,
                                  ws ? kScratchBytes : 0, opts, stream);
}
