// kvc_compact_noalloc: the compaction with its scratch in a fixed device
// array owned by the library, for callers that cannot allocate device memory
// themselves.  Such callers include:
//   - engines whose allocator reserves the device's memory up front and
//     forbids any other allocation;
//   - code on latency-critical paths, where cudaMalloc / cudaFree may
//     synchronise the device and stall unrelated streams;
//   - plain C programs that have no device allocator at all.
//
// The scratch is one file-scope __device__ array of KVC_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Its
// device address is looked up once per device (the first call on that
// device, with the device current) and cached; that lookup allocates
// nothing.  The work itself is the same launch sequence as kvc_compact.
#include <mutex>

#include "common.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side handle, so the address must come from
// cudaGetSymbolAddress.
kvc_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVC_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KVC_OK;
}

}  // namespace

extern "C" kvc_status kvc_compact_noalloc(const kvc_problem* p, const kvc_params* prm, const void* Q_ref,
                                          const void* K, const void* V, const int32_t* budgets,
                                          const int32_t* offsets, int32_t* idx_out, void* C_k, float* beta,
                                          float* C_v, int32_t* head_status, kvc_stream_t stream) {
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    // stage timing would create CUDA events; this entry point creates nothing
    if (q.flags & KVC_FLAG_STAGE_TIMING) return KVC_ERR_INVALID_ARG;
    size_t need = 0;
    kvc_status s = kvc_workspace_size(p, &q, &need);
    if (s != KVC_OK) return s;
    if (need > (size_t)KVC_NOALLOC_SCRATCH_BYTES) return KVC_ERR_NOALLOC_LIMIT;
    void* scratch = nullptr;
    if ((s = scratch_for_current_device(&scratch)) != KVC_OK) return s;
    return kvc_compact(p, &q, Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status, scratch,
                       (size_t)KVC_NOALLOC_SCRATCH_BYTES, stream);
}
