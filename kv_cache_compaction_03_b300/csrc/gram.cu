// Gram matrices and the biased softmax X ("Fast KV Compaction via Attention
// Matching", section 2, fitting beta by NNLS and C_v by least squares through
// the normal equations):
//   k_gram<true>   G = A'^T A' with A' = exp2(l2) (l2 = log2 of the relative
//                  mass matrix), and b = A'^T 1
//   k_gram<false>  M = X^T X
//   k_xto          R = X^T O
//   k_ridge_*      mu / lambda from the trace, added to the diagonal
//   k_xsoftmax     X_qi = softmax_i(l2_qi + log2 w_i), in place over l2
// Matrices are per head, row-major with leading dimension ldA (a multiple
// of 64); only the lower triangle of G / M is written.
#include "common.cuh"

namespace kvc {

constexpr int GT = 64;     // Gram tile
constexpr int GQ = 32;     // rows of A per smem stage

__device__ __forceinline__ void tri_decode(int p, int& I, int& J) {
    int i = (int)((sqrtf(8.f * (float)p + 1.f) - 1.f) * 0.5f);
    while (i * (i + 1) / 2 > p) --i;
    while ((i + 1) * (i + 2) / 2 <= p) ++i;
    I = i;
    J = p - i * (i + 1) / 2;
}

// grid (ntiles*(ntiles+1)/2, H), block 256.
template <bool EXP>
__global__ void __launch_bounds__(256) k_gram(const float* __restrict__ A, const int32_t* __restrict__ offsets, int n,
                                              int64_t ldA, float* __restrict__ G, float* __restrict__ b,
                                              const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    int I, J;
    tri_decode(blockIdx.x, I, J);
    if (I * GT >= t) return;
    __shared__ float Ai[GQ][GT + 1];
    __shared__ float Aj[GQ][GT + 1];
    __shared__ double red[16][GT];
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const float* Ah = A + (int64_t)h * n * ldA;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
    float csum[4] = {0.f, 0.f, 0.f, 0.f};
    const bool diag = (I == J);
    for (int q0 = 0; q0 < n; q0 += GQ) {
        __syncthreads();
        for (int e = threadIdx.x; e < GQ * GT; e += 256) {
            const int r = e / GT, c = e % GT;
            const int q = q0 + r;
            float vi = 0.f, vj = 0.f;
            if (q < n) {
                vi = Ah[(int64_t)q * ldA + I * GT + c];
                vj = Ah[(int64_t)q * ldA + J * GT + c];
                if (EXP) {
                    vi = exp2f(vi);
                    vj = exp2f(vj);
                }
            }
            Ai[r][c] = vi;
            Aj[r][c] = vj;
        }
        __syncthreads();
#pragma unroll 8
        for (int r = 0; r < GQ; ++r) {
            float ai[4], aj[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) ai[a] = Ai[r][ty * 4 + a];
#pragma unroll
            for (int c = 0; c < 4; ++c) aj[c] = Aj[r][tx + 16 * c];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(ai[a], aj[c], acc[a][c]);
        }
        if (EXP && diag) {
#pragma unroll
            for (int c = 0; c < 4; ++c) csum[c] += Aj[ty][tx + 16 * c] + Aj[ty + 16][tx + 16 * c];
        }
    }
    float* Gh = G + (int64_t)h * ldA * ldA;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = I * GT + ty * 4 + a;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j = J * GT + tx + 16 * c;
            if (i < t && j < t && j <= i) Gh[(int64_t)i * ldA + j] = acc[a][c];
        }
    }
    if (EXP && diag) {
#pragma unroll
        for (int c = 0; c < 4; ++c) red[ty][tx + 16 * c] = (double)csum[c];
        __syncthreads();
        if (threadIdx.x < GT) {
            double s = 0.0;
            for (int r = 0; r < 16; ++r) s += red[r][threadIdx.x];
            const int j = I * GT + threadIdx.x;
            if (j < t) b[off + j] = (float)s;
        }
    }
}

// R[off+i][c] = sum_q X[h][q][i] O[h][q][c].  grid (ceil(max_t/64), H), block 256.
template <int D>
__global__ void __launch_bounds__(256) k_xto(const float* __restrict__ X, const float* __restrict__ O,
                                             const int32_t* __restrict__ offsets, int n, int64_t ldA,
                                             float* __restrict__ R, const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i0 = blockIdx.x * GT;
    if (i0 >= t) return;
    __shared__ float Xs[GQ][GT + 1];
    __shared__ float Os[GQ][D];
    constexpr int DC = D / 16;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    float acc[4][DC];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < DC; ++c) acc[a][c] = 0.f;
    const float* Xh = X + (int64_t)h * n * ldA;
    const float* Oh = O + (int64_t)h * n * D;
    for (int q0 = 0; q0 < n; q0 += GQ) {
        __syncthreads();
        for (int e = threadIdx.x; e < GQ * GT; e += 256) {
            const int r = e / GT, c = e % GT;
            Xs[r][c] = (q0 + r < n) ? Xh[(int64_t)(q0 + r) * ldA + i0 + c] : 0.f;
        }
        for (int e = threadIdx.x; e < GQ * D; e += 256) {
            const int r = e / D, c = e % D;
            Os[r][c] = (q0 + r < n) ? Oh[(int64_t)(q0 + r) * D + c] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < GQ; ++r) {
            float x[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) x[a] = Xs[r][ty * 4 + a];
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                const float o = Os[r][tx + 16 * c];
#pragma unroll
                for (int a = 0; a < 4; ++a) acc[a][c] = fmaf(x[a], o, acc[a][c]);
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = i0 + ty * 4 + a;
        if (i < t) {
#pragma unroll
            for (int c = 0; c < DC; ++c) R[((int64_t)off + i) * D + tx + 16 * c] = acc[a][c];
        }
    }
}

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

// NNLS ridge: mu = eps * tr(G)/t; G += mu I; f = b + mu.  grid H, block 256.
__global__ void k_ridge_g(float* __restrict__ G, const float* __restrict__ b, const int32_t* __restrict__ offsets,
                          int64_t ldA, float eps, float* __restrict__ f, HeadScalars* __restrict__ hs,
                          int32_t* __restrict__ status) {
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    __shared__ double sred[32];
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    float* Gh = G + (int64_t)h * ldA * ldA;
    const double tr = block_trace(Gh, t, ldA, sred);
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

// C_v ridge: lam = eps * tr(M)/t; M += lam I; R += lam Vsel.  grid H, block 256.
template <int D>
__global__ void k_ridge_m(float* __restrict__ M, float* __restrict__ R, const float* __restrict__ Vsel,
                          const int32_t* __restrict__ offsets, int64_t ldA, float eps, HeadScalars* __restrict__ hs,
                          int32_t* __restrict__ status) {
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    __shared__ double sred[32];
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    float* Mh = M + (int64_t)h * ldA * ldA;
    const double tr = block_trace(Mh, t, ldA, sred);
    if (!isfinite(tr) || !(tr > 0.0)) {
        if (threadIdx.x == 0) set_status(status, h, KVC_ERR_NONFINITE);
        return;
    }
    const float lam = (float)(eps * tr / t);
    for (int i = threadIdx.x; i < t; i += blockDim.x) Mh[(int64_t)i * ldA + i] += lam;
    for (int e = threadIdx.x; e < t * D; e += blockDim.x) R[(int64_t)off * D + e] += lam * Vsel[(int64_t)off * D + e];
    if (threadIdx.x == 0) hs[h].lam = lam;
}

// X_qi = softmax_i(l2_qi + log2 w_i) over i < t (padding columns set to 0),
// in place.  grid (ceil(n/8), H), block 256 (one warp per row).
__global__ void __launch_bounds__(256) k_xsoftmax(float* __restrict__ L2, const float* __restrict__ w,
                                                  const int32_t* __restrict__ offsets, int n, int64_t ldA,
                                                  const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int q = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (q >= n) return;
    float* row = L2 + ((int64_t)h * n + q) * ldA;
    float mx = -INFINITY;
    for (int i = lane; i < t; i += 32) mx = fmaxf(mx, row[i] + log2f(w[off + i]));
    mx = warp_max(mx);
    float s = 0.f;
    for (int i = lane; i < t; i += 32) s += exp2f(row[i] + log2f(w[off + i]) - mx);
    s = warp_sum(s);
    const float inv = (s > 0.f && mx > -INFINITY) ? 1.f / s : 0.f;
    const int tp = (int)round_up(t, GT);
    for (int i = lane; i < tp; i += 32) {
        float x = 0.f;
        if (i < t && inv > 0.f) x = exp2f(row[i] + log2f(w[off + i]) - mx) * inv;
        row[i] = x;
    }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_gram(bool exp_mode, const float* A, const int32_t* offsets, int H, int n, int max_t, int64_t ldA,
                        float* G, float* b, const int32_t* status, cudaStream_t st) {
    const int nt = (max_t + GT - 1) / GT;
    dim3 grid(nt * (nt + 1) / 2, H);
    if (exp_mode)
        k_gram<true><<<grid, 256, 0, st>>>(A, offsets, n, ldA, G, b, status);
    else
        k_gram<false><<<grid, 256, 0, st>>>(A, offsets, n, ldA, G, b, status);
    return cudaGetLastError();
}
cudaError_t launch_xto(int d, const float* X, const float* O, const int32_t* offsets, int H, int n, int max_t,
                       int64_t ldA, float* R, const int32_t* status, cudaStream_t st) {
    dim3 grid((max_t + GT - 1) / GT, H);
    if (d == 128)
        k_xto<128><<<grid, 256, 0, st>>>(X, O, offsets, n, ldA, R, status);
    else
        k_xto<64><<<grid, 256, 0, st>>>(X, O, offsets, n, ldA, R, status);
    return cudaGetLastError();
}
cudaError_t launch_ridge_g(float* G, const float* b, const int32_t* offsets, int H, int64_t ldA, float eps, float* f,
                           HeadScalars* hs, int32_t* status, cudaStream_t st) {
    k_ridge_g<<<H, 256, 0, st>>>(G, b, offsets, ldA, eps, f, hs, status);
    return cudaGetLastError();
}
cudaError_t launch_ridge_m(int d, float* M, float* R, const float* Vsel, const int32_t* offsets, int H, int64_t ldA,
                           float eps, HeadScalars* hs, int32_t* status, cudaStream_t st) {
    if (d == 128)
        k_ridge_m<128><<<H, 256, 0, st>>>(M, R, Vsel, offsets, ldA, eps, hs, status);
    else
        k_ridge_m<64><<<H, 256, 0, st>>>(M, R, Vsel, offsets, ldA, eps, hs, status);
    return cudaGetLastError();
}
cudaError_t launch_xsoftmax(float* L2, const float* w, const int32_t* offsets, int H, int n, int64_t ldA,
                            const int32_t* status, cudaStream_t st) {
    dim3 grid((n + 7) / 8, H);
    k_xsoftmax<<<grid, 256, 0, st>>>(L2, w, offsets, n, ldA, status);
    return cudaGetLastError();
}

}  // namespace kvc
