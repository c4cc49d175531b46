// Input preparation for the tensor-core attention pass ("Fast KV Compaction
// via Attention Matching", section 2, reference outputs O = softmax(S) V).
//
// Values: P enters P V as one fp16 term (11 significant bits; a single bf16
// term would leave O ~1e-3 off), and a tcgen05 product takes both operands
// in the same type, so V is rewritten in fp16 once per call:
// V16 = fp16(V * 2^-e_h).  e_h = 0 when 2^-3 <= max |V| < 2^15 for head h:
// the fp16 range ends at 65504, and every value down to max |V| 2^-11 is a
// normal fp16 number with its full 11 bits.  Outside that band e_h brings
// max |V| into [2^14, 2^15).  The scaling is exact; the attention epilogue
// multiplies O by 2^e_h again.  V
// is bf16 (a fresh cache) or fp32 (the refitted values of a compacted
// cache).  A head whose values hold a NaN or an infinity gets
// KVC_ERR_NONFINITE.
//
// Key biases (a compacted cache's beta, for periodic compaction): bias2 =
// bias * log2 e per key, in the padded layout [H][Tb] (Tb = T rounded up to
// 256, -inf beyond T) that the attention passes read in 128-key slices.  A
// NaN or +inf bias gets KVC_ERR_NONFINITE; -inf switches a key off.
#include <cuda_fp16.h>

#include "common.cuh"

namespace kvc {
namespace {

constexpr int kVecs = 8;           // 8-element groups per thread per CTA
constexpr int kGroup = 256 * kVecs * 8;     // elements per CTA

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// V16 = fp16(V) for every head, and the per-head max |V| as the bits of a
// non-negative float (those order like unsigned integers; +inf marks a
// non-finite value) into vmax, which must be zeroed.  One pass with the
// scale 1 (e_h = 0, the common case); k_v_fixup rewrites the heads whose
// max |V| falls outside [2^-3, 2^15).
// grid (ceil(per_head / kGroup), H), block 256.
template <typename TIn>
__global__ void __launch_bounds__(256) k_v_to_f16(const TIn* __restrict__ V, int64_t per_head, uint32_t* __restrict__ vmax,
                                                  __half* __restrict__ V16, const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const TIn* Vh = V + (int64_t)h * per_head;
    __half* Oh = V16 + (int64_t)h * per_head;
    float m = 0.f;
    bool bad = false;
    const int64_t base = (int64_t)blockIdx.x * kGroup;
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
        const int64_t e = base + ((int64_t)k * 256 + threadIdx.x) * 8;
        if (e < per_head) {
            float v[8];
            load8(Vh + e, v);
            __half2 o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = __floats2half2_rn(v[2 * q], v[2 * q + 1]);
            *reinterpret_cast<uint4*>(Oh + e) = *reinterpret_cast<const uint4*>(o);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float a = fabsf(v[q]);
                bad |= !(a <= 3.4028235e38f);
                m = fmaxf(m, a);
            }
        }
    }
    if (bad) m = __uint_as_float(0x7f800000u);
    m = warp_max(m);
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float x = red[0];
        for (int w = 1; w < 8; ++w) x = fmaxf(x, red[w]);
        atomicMax(vmax + h, __float_as_uint(x));
    }
}

// e_h to vexp[h]; heads with e_h != 0 are converted again as fp16(V 2^-e_h);
// a non-finite value gives KVC_ERR_NONFINITE.  Same grid as k_v_to_f16.
template <typename TIn>
__global__ void __launch_bounds__(256) k_v_fixup(const TIn* __restrict__ V, int64_t per_head,
                                                 const uint32_t* __restrict__ vmax, __half* __restrict__ V16,
                                                 int32_t* __restrict__ vexp, int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const float mx = __uint_as_float(vmax[h]);
    if (!(mx <= 3.4028235e38f)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, h, KVC_ERR_NONFINITE);
        return;
    }
    int E2 = 0;
    (void)frexpf(mx, &E2);                   // 2^(E2-1) <= mx < 2^E2 (E2 = 0 for mx = 0)
    // e = 0 for mx in [2^-3, 2^15), else mx 2^-e in [2^14, 2^15); the
    // clamp keeps 2^-e and 2^e normal fp32 numbers
    const int e = (E2 >= -2 && E2 <= 15) ? 0 : min(113, max(-100, E2 - 15));
    if (blockIdx.x == 0 && threadIdx.x == 0) vexp[h] = e;
    if (e == 0) return;
    const float sc = __uint_as_float((uint32_t)(127 - e) << 23);      // 2^-e
    const TIn* Vh = V + (int64_t)h * per_head;
    __half* Oh = V16 + (int64_t)h * per_head;
    const int64_t base = (int64_t)blockIdx.x * kGroup;
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
        const int64_t el = base + ((int64_t)k * 256 + threadIdx.x) * 8;
        if (el < per_head) {
            float v[8];
            load8(Vh + el, v);
            __half2 o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = __floats2half2_rn(v[2 * q] * sc, v[2 * q + 1] * sc);
            *reinterpret_cast<uint4*>(Oh + el) = *reinterpret_cast<const uint4*>(o);
        }
    }
}

// grid (Tb / 256, H), block 256.
__global__ void __launch_bounds__(256) k_bias_log2(const float* __restrict__ bias, int T, int Tb,
                                                   float* __restrict__ bias2, int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    const int j = blockIdx.x * 256 + threadIdx.x;
    float b = -INFINITY;
    if (j < T) {
        const float x = bias[(int64_t)h * T + j];
        if (x != x || x == INFINITY) set_status(status, h, KVC_ERR_NONFINITE);
        b = x * kLog2e;
    }
    bias2[(int64_t)h * Tb + j] = b;
}

template <typename TIn>
cudaError_t launch_v_to_f16_t(const void* V, int H, int64_t per_head, uint32_t* vmax, void* V16, int32_t* vexp,
                              int32_t* status, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(vmax, 0, sizeof(uint32_t) * H, st);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((per_head + kGroup - 1) / kGroup), H);
    k_v_to_f16<TIn><<<grid, 256, 0, st>>>((const TIn*)V, per_head, vmax, (__half*)V16, status);
    k_v_fixup<TIn><<<grid, 256, 0, st>>>((const TIn*)V, per_head, vmax, (__half*)V16, vexp, status);
    return cudaGetLastError();
}

}  // namespace

// V [H][per_head] (bf16, or fp32 with v_f32) -> V16 [H][per_head] fp16 with
// per-head exponents vexp [H]; vmax: H words of scratch.  per_head = T * d,
// a multiple of 8.
cudaError_t launch_v_to_f16(const void* V, bool v_f32, int H, int64_t per_head, uint32_t* vmax, void* V16,
                            int32_t* vexp, int32_t* status, cudaStream_t st) {
    return v_f32 ? launch_v_to_f16_t<float>(V, H, per_head, vmax, V16, vexp, status, st)
                 : launch_v_to_f16_t<__nv_bfloat16>(V, H, per_head, vmax, V16, vexp, status, st);
}

// bias [H][T] fp32 (natural units) -> bias2 [H][Tb] (log2 units, -inf padded);
// Tb = T rounded up to 256.
cudaError_t launch_bias_log2(const float* bias, int H, int T, float* bias2, int32_t* status, cudaStream_t st) {
    const int Tb = (int)round_up(T, 256);
    k_bias_log2<<<dim3(Tb / 256, H), 256, 0, st>>>(bias, T, Tb, bias2, status);
    return cudaGetLastError();
}

}  // namespace kvc
