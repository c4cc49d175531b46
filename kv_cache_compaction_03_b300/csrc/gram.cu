// Ridges and the biased softmax X of the two least-squares fits ("Fast KV
// Compaction via Attention Matching", section 2, fitting beta by NNLS and
// C_v by least squares through the normal equations; the Gram products
// themselves are in gram_tc.cu):
//   k_ridge_*      mu / lambda from the trace, added to the diagonal
//   k_xsoftmax     X_qi = softmax_i(l2_qi + log2 w_i), as bf16 hi / lo terms
// Matrices are per head, row-major with leading dimension ldA (a multiple
// of 64); only the lower triangle of G / M is read.
#include "tc.cuh"

namespace kvc {

constexpr int GT = 64;     // padding granule of the log-mass rows

// Trace of the lower-stored matrix diagonal, in double.  Block-wide.
__device__ double block_trace(const float* Gh, int t, int64_t ld, double* sred) {
    double s = 0.0;
    for (int i = threadIdx.x; i < t; i += blockDim.x) s += (double)Gh[(int64_t)i * ld + i];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) sred[threadIdx.x >> 5] = s;
    __syncthreads();
    double tot = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += sred[w];
    __syncthreads();
    return tot;
}

// Sum of a head's `count` trace parts in a fixed order (block-wide).
__device__ double block_parts(const double* p, int64_t count, double* sred) {
    double s = 0.0;
    for (int64_t k = threadIdx.x; k < count; k += blockDim.x) s += p[k];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) sred[threadIdx.x >> 5] = s;
    __syncthreads();
    double tot = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += sred[w];
    __syncthreads();
    return tot;
}

// NNLS ridge: mu = eps * tr(A'^T A')/t; G += mu I; f = b + mu.  The trace
// comes from the exact sums of squares of A' (sqpart, sq_count parts per
// head) when given, else from the diagonal of G.  grid H, block 256.
__global__ void k_ridge_g(float* __restrict__ G, const float* __restrict__ b, const int32_t* __restrict__ offsets,
                          int64_t ldA, float eps, const double* __restrict__ sqpart, int64_t sq_count,
                          float* __restrict__ f, HeadScalars* __restrict__ hs, int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    __shared__ double sred[32];
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    float* Gh = G + (int64_t)h * ldA * ldA;
    const double tr = sqpart ? block_parts(sqpart + (int64_t)h * sq_count, sq_count, sred)
                             : block_trace(Gh, t, ldA, sred);
    const float mu = (float)(eps * tr / t);
    if (!isfinite(tr) || !(tr > 0.0)) {
        if (threadIdx.x == 0) set_status(status, h, KVC_ERR_NONFINITE);
        return;
    }
    for (int i = threadIdx.x; i < t; i += blockDim.x) {
        Gh[(int64_t)i * ldA + i] += mu;
        f[off + i] = b[off + i] + mu;
    }
    if (threadIdx.x == 0) hs[h].mu = mu;
}

// C_v ridge: lam = eps * tr(M)/t; M += lam I; R += lam Vsel.
// k_ridge_m: grid (chunks, H), block 256: every CTA forms the trace (t
// entries) and updates its 4096-element slice of R; CTA 0 records lam.
// k_ridge_m_diag then adds lam to the diagonal (a separate launch, so that
// no CTA of the first one can read an already shifted diagonal).
constexpr int kRidgeChunk = 4096;

template <int D>
__global__ void k_ridge_m(float* __restrict__ M, float* __restrict__ R, const float* __restrict__ Vsel,
                          const int32_t* __restrict__ offsets, int64_t ldA, float eps, HeadScalars* __restrict__ hs,
                          int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    __shared__ double sred[32];
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int64_t e0 = (int64_t)blockIdx.x * kRidgeChunk;
    if (e0 >= (int64_t)t * D) return;
    float* Mh = M + (int64_t)h * ldA * ldA;
    const double tr = block_trace(Mh, t, ldA, sred);
    if (!isfinite(tr) || !(tr > 0.0)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, h, KVC_ERR_NONFINITE);
        return;
    }
    const float lam = (float)(eps * tr / t);
    const int64_t e1 = min((int64_t)t * D, e0 + kRidgeChunk);
    for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) R[(int64_t)off * D + e] += lam * Vsel[(int64_t)off * D + e];
    if (blockIdx.x == 0 && threadIdx.x == 0) hs[h].lam = lam;
}

// grid H, block 256.
__global__ void k_ridge_m_diag(float* __restrict__ M, const int32_t* __restrict__ offsets, int64_t ldA,
                               const HeadScalars* __restrict__ hs, const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    const int t = offsets[h + 1] - offsets[h];
    const float lam = hs[h].lam;
    float* Mh = M + (int64_t)h * ldA * ldA;
    for (int i = threadIdx.x; i < t; i += blockDim.x) Mh[(int64_t)i * ldA + i] += lam;
}

// X_qi = softmax_i(l2_qi + log2 w_i) over i < t, written as bf16 hi / lo
// terms (the Gram operand format, see gram_tc.cu); padding columns up to the
// next multiple of 64 are 0.  log2 w_i from the fitted weights (-inf where
// w = 0; the log-masses hold -inf past t as well).  grid (ceil(n/32), H),
// block 256: a warp per row, four rows per warp; the CTA's 32 rows share one
// staged copy of log2 w.  Each lane takes four adjacent columns per step
// (one 16-byte load, two 8-byte stores) in three passes over the row (the
// second and third read it from L1): the maximum, the sum of 2^(v - max),
// and the normalised terms.  The exponentials are the special-function
// unit's (ex2.approx, relative error ~2^-22), well inside the 2^-17 of the
// hi / lo split they feed.
__global__ void __launch_bounds__(256) k_xsoftmax(const float* __restrict__ L2, const float* __restrict__ wfit,
                                                  const int32_t* __restrict__ offsets, int n, int64_t ldA,
                                                  __nv_bfloat16* __restrict__ Xh, __nv_bfloat16* __restrict__ Xl,
                                                  const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    extern __shared__ float4 lw4[];
    float* lw = reinterpret_cast<float*>(lw4);
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int tp = (int)round_up(t, GT);
    // log2 of the fitted weights (not beta: on a biased cache the log-masses
    // already hold the kept keys' input biases, which beta also carries)
    for (int i = threadIdx.x; i < tp; i += blockDim.x) {
        const float w = i < t ? wfit[off + i] : 0.f;
        lw[i] = w > 0.f ? log2f(w) : -INFINITY;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    for (int rr = 0; rr < 4; ++rr) {
        const int q = blockIdx.x * 32 + (threadIdx.x >> 5) * 4 + rr;
        if (q >= n) break;
        const int64_t ro = ((int64_t)h * n + q) * ldA;
        const float4* row = reinterpret_cast<const float4*>(L2 + ro);
        float m = -INFINITY;
        for (int i = 4 * lane; i < tp; i += 128) {
            const float4 a = row[i >> 2], w = lw4[i >> 2];
            m = tc::fmax3(m, tc::fmax3(a.x + w.x, a.y + w.y, a.z + w.z), a.w + w.w);
        }
        const float mx = warp_max(m);
        const float nmx = mx > -INFINITY ? -mx : 0.f;
        const float2 nm2 = make_float2(nmx, nmx);
        float2 s2 = make_float2(0.f, 0.f);
        for (int i = 4 * lane; i < tp; i += 128) {
            const float4 a = row[i >> 2], w = lw4[i >> 2];
            const float2 v01 = tc::fadd2(tc::fadd2(make_float2(a.x, a.y), make_float2(w.x, w.y)), nm2);
            const float2 v23 = tc::fadd2(tc::fadd2(make_float2(a.z, a.w), make_float2(w.z, w.w)), nm2);
            const float2 e01 = make_float2(tc::ex2(v01.x), tc::ex2(v01.y));
            const float2 e23 = make_float2(tc::ex2(v23.x), tc::ex2(v23.y));
            s2 = tc::fadd2(s2, tc::fadd2(e01, e23));
        }
        const float s = warp_sum(s2.x + s2.y);
        const float inv = (s > 0.f && mx > -INFINITY) ? 1.f / s : 0.f;
        const float2 inv2 = make_float2(inv, inv);
        for (int i = 4 * lane; i < tp; i += 128) {
            const float4 a = row[i >> 2], w = lw4[i >> 2];
            const float2 v01 = tc::fadd2(tc::fadd2(make_float2(a.x, a.y), make_float2(w.x, w.y)), nm2);
            const float2 v23 = tc::fadd2(tc::fadd2(make_float2(a.z, a.w), make_float2(w.z, w.w)), nm2);
            float2 x01 = make_float2(tc::ex2(v01.x), tc::ex2(v01.y));
            float2 x23 = make_float2(tc::ex2(v23.x), tc::ex2(v23.y));
            x01.x *= inv2.x; x01.y *= inv2.y; x23.x *= inv2.x; x23.y *= inv2.y;
            uint2 hv, lv;
            hv.x = tc::pack_bf16(x01.x, x01.y);
            hv.y = tc::pack_bf16(x23.x, x23.y);
            lv.x = tc::pack_bf16(x01.x - tc::bf16_lo(hv.x), x01.y - tc::bf16_hi(hv.x));
            lv.y = tc::pack_bf16(x23.x - tc::bf16_lo(hv.y), x23.y - tc::bf16_hi(hv.y));
            *reinterpret_cast<uint2*>(Xh + ro + i) = hv;
            *reinterpret_cast<uint2*>(Xl + ro + i) = lv;
        }
    }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_ridge_g(float* G, const float* b, const int32_t* offsets, int H, int64_t ldA, float eps,
                           const double* sqpart, int64_t sq_count, float* f,
                           HeadScalars* hs, int32_t* status, cudaStream_t st) {
    {
        const cudaError_t le = launch_dep(k_ridge_g, dim3(H), dim3(256), 0, st, G, b, offsets, ldA, eps, sqpart,
                                          sq_count, f, hs, status);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}
cudaError_t launch_ridge_m(int d, float* M, float* R, const float* Vsel, const int32_t* offsets, int H, int64_t ldA,
                           float eps, HeadScalars* hs, int32_t* status, cudaStream_t st) {
    // launched before M is factored, after R is complete; the max_t bound is ldA
    const int chunks = (int)(((int64_t)ldA * d + kRidgeChunk - 1) / kRidgeChunk);
    if (d == 128)
        {
            const cudaError_t le = launch_dep(k_ridge_m<128>, dim3(dim3(chunks, H)), dim3(256), 0, st, M, R, Vsel,
                                              offsets, ldA, eps, hs, status);
            if (le != cudaSuccess) return le;
        }
    else
        {
            const cudaError_t le = launch_dep(k_ridge_m<64>, dim3(dim3(chunks, H)), dim3(256), 0, st, M, R, Vsel,
                                              offsets, ldA, eps, hs, status);
            if (le != cudaSuccess) return le;
        }
    {
        const cudaError_t le = launch_dep(k_ridge_m_diag, dim3(H), dim3(256), 0, st, M, offsets, ldA, hs, status);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}
// wfit: the fitted NNLS weights (clamped at 0), [sum t].
cudaError_t launch_xsoftmax(const float* L2, const float* wfit, const int32_t* offsets, int H, int n, int64_t ldA,
                            void* Xh, void* Xl, const int32_t* status, cudaStream_t st) {
    dim3 grid((n + 31) / 32, H);
    const size_t smem = (size_t)ldA * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_xsoftmax, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    {
        const cudaError_t le = launch_dep(k_xsoftmax, dim3(grid), dim3(256), smem, st, L2, wfit, offsets, n, ldA,
                                          (__nv_bfloat16*)Xh, (__nv_bfloat16*)Xl, status);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}

}  // namespace kvc
