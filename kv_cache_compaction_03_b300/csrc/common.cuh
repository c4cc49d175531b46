// Shared device helpers for the compaction kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Element loads that widen bf16/fp32 storage to fp32.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// A head whose status is already an error is skipped by every later kernel.
__device__ __forceinline__ bool head_ok(const int32_t* status, int h) {
    return status[h] == KVC_OK;
}

// Record the first error of a head (later errors do not overwrite it).
__device__ __forceinline__ void set_status(int32_t* status, int h, int32_t code) {
    atomicCAS(reinterpret_cast<int*>(status + h), KVC_OK, code);
}

// Index checks of the debug build (KVC_DEBUG): an index read from data (a
// kept position, a zero-set entry, a head's row range) is compared with the
// extent of the buffer it addresses; a bad one records KVC_ERR_DEBUG_BOUNDS
// for the head and the access is skipped (no trap).  In the normal build the
// check is compiled out and the index is trusted (the arguments were
// validated on entry).
#ifdef KVC_DEBUG
__device__ __forceinline__ bool debug_in_range(bool ok, const int32_t* status, int h) {
    if (!ok) set_status(const_cast<int32_t*>(status), h, KVC_ERR_DEBUG_BOUNDS);
    return ok;
}
#define KVC_IN_RANGE(cond, status, h) (::kvc::debug_in_range((cond), (status), (h)))
#else
#define KVC_IN_RANGE(cond, status, h) (true)
#endif

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Error-free transformations for double-float accumulation (Knuth TwoSum,
// FMA-based TwoProduct): (hi, lo) carries ~48 significant bits in fp32 units.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}
struct dfloat {
    float hi, lo;
};
__device__ __forceinline__ void df_add(dfloat& acc, float x) {
    float s, e;
    two_sum(acc.hi, x, s, e);
    e += acc.lo;
    acc.hi = s + e;
    acc.lo = e - (acc.hi - s);
}
__device__ __forceinline__ void df_fma(dfloat& acc, float a, float b) {
    float p = a * b;
    float pe = fmaf(a, b, -p);
    float s, e;
    two_sum(acc.hi, p, s, e);
    e += acc.lo + pe;
    acc.hi = s + e;
    acc.lo = e - (acc.hi - s);
}
__device__ __forceinline__ void df_add_df(dfloat& acc, dfloat x) {
    float s, e;
    two_sum(acc.hi, x.hi, s, e);
    e += acc.lo + x.lo;
    acc.hi = s + e;
    acc.lo = e - (acc.hi - s);
}
__device__ __forceinline__ dfloat warp_sum_df(dfloat v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        dfloat u;
        u.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        u.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        df_add_df(v, u);
    }
    return v;
}

__host__ __device__ constexpr int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Programmatic dependent launch.  The short kernels of the solver chains are
// launched with launch_dep: a launch may be set up while the previous one
// drains, and its CTAs call grid_dependency_wait() first, which returns once
// the previous launch has completed and its writes are visible (no kernel
// triggers its dependents early, so a waiting CTA never holds a slot that a
// CTA of the launch it waits for still needs).  Launched normally, the wait
// returns at once.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dep(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Per-head scalars kept in the workspace.
struct HeadScalars {
    float mu;        // NNLS ridge
    float lam;       // C_v ridge
    float trace;     // scratch
    int32_t nzero;   // |Z| at NNLS exit
    int32_t iters;   // NNLS pivoting iterations used
    int32_t pad[3];
};



}  // namespace kvc
