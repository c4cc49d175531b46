// CUDA-core (FFMA) kernels for the attention-shaped steps of the compaction
// ("Fast KV Compaction via Attention Matching", section 2):
//   k_attn_fwd     S = Q K^T * scale, lse per row, O = softmax(S) V
//   k_colscore     sum_q softmax(S)_qj^2 per key (the RMS key score)
//   k_masslogits   l_qi = S_q,idx_i * scale - lse_q (log of A'_qi) for kept keys
//   k_attend       softmax(Q C_k^T * scale + beta) C_v
// They serve every dtype and shape; the bf16 hot path also has tensor-core
// versions.  Logits are carried in log2 units (x * scale * log2 e) so that
// every kernel rounds them the same way; lse is stored in the same units.
// An optional per-key input bias (bias2, log2 units, [H][Tb] with Tb = T
// rounded up to 256; -inf switches a key off) is added to the logits: the cache of an earlier compaction, whose
// keys carry their fitted biases (periodic compaction).
#include "common.cuh"

namespace kvc {

constexpr int BM = 64;       // query rows per tile
constexpr int BN = 64;       // keys per tile
constexpr int NT = 256;      // threads per CTA (16 x 16)

// Load `rows` rows (row stride `ld` elements) of width D starting at `src`
// into smem tile dst[BM][D+1] as fp32; rows >= valid are zero.
template <typename TIn, int D>
__device__ __forceinline__ void load_tile(float* dst, const TIn* src, int valid, int64_t ld) {
    constexpr int P = D + 1;
    for (int e = threadIdx.x; e < BM * D; e += NT) {
        int r = e / D, c = e % D;
        dst[r * P + c] = (r < valid) ? to_f32(src[(int64_t)r * ld + c]) : 0.f;
    }
}
template <int D>
__device__ __forceinline__ void load_tile_f32_nopad(float* dst, const float* src, int valid, int64_t ld) {
    for (int e = threadIdx.x; e < BN * D; e += NT) {
        int r = e / D, c = e % D;
        dst[r * D + c] = (r < valid) ? src[(int64_t)r * ld + c] : 0.f;
    }
}
template <typename TIn, int D>
__device__ __forceinline__ void load_tile_nopad(float* dst, const TIn* src, int valid, int64_t ld) {
    for (int e = threadIdx.x; e < BN * D; e += NT) {
        int r = e / D, c = e % D;
        dst[r * D + c] = (r < valid) ? to_f32(src[(int64_t)r * ld + c]) : 0.f;
    }
}

// s[i][j] = sum_k A[ty*4+i][k] * B[tx+16j][k]  (A, B: smem tiles [64][D+1])
template <int D>
__device__ __forceinline__ void tile_dot(const float* A, const float* B, float s[4][4]) {
    constexpr int P = D + 1;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = A[(ty * 4 + i) * P + k];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = B[(tx + 16 * j) * P + k];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[i][j] = fmaf(a[i], b[j], s[i][j]);
    }
}

// ---------------------------------------------------------------- flash fwd
// grid (ceil(n/64), H), block 256.  O fp32 [H][n][D], lse2 [H][n] (log2 units).
template <typename TIn, int D>
__global__ void __launch_bounds__(NT) k_attn_fwd(const TIn* __restrict__ Q, const TIn* __restrict__ K,
                                                 const TIn* __restrict__ V, int n, int T, float c2,
                                                 float* __restrict__ O, float* __restrict__ lse2,
                                                 int32_t* __restrict__ status, int qdiv,
                                                 const float* __restrict__ bias2) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    extern __shared__ float sm[];
    constexpr int P = D + 1;
    float* Qs = sm;
    float* Ks = Qs + BM * P;
    float* Vs = Ks + BN * P;
    float* Ps = Vs + BN * D;          // [BM][BN+1]
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const int q0 = blockIdx.x * BM;
    const TIn* Qh = Q + ((int64_t)(h / qdiv) * n + q0) * D;
    const TIn* Kh = K + (int64_t)h * T * D;
    const TIn* Vh = V + (int64_t)h * T * D;
    load_tile<TIn, D>(Qs, Qh, min(BM, n - q0), D);

    constexpr int DC = D / 16;
    float o[4][DC];
    float m[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < DC; ++c) o[i][c] = 0.f;
    }
    for (int k0 = 0; k0 < T; k0 += BN) {
        const int kv = min(BN, T - k0);
        __syncthreads();
        load_tile<TIn, D>(Ks, Kh + (int64_t)k0 * D, kv, D);
        load_tile_nopad<TIn, D>(Vs, Vh + (int64_t)k0 * D, kv, D);
        __syncthreads();
        float s[4][4];
        tile_dot<D>(Qs, Ks, s);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float b = bias2 && tx + 16 * j < kv ? bias2[h * round_up(T, 256) + k0 + tx + 16 * j] : 0.f;
                s[i][j] = (tx + 16 * j < kv) ? fmaf(s[i][j], c2, b) : -INFINITY;
                mx = fmaxf(mx, s[i][j]);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float mnew = fmaxf(m[i], mx);
            const float corr = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - mnew);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // (mnew = -inf only while every key so far is switched off)
                float p = s[i][j] == -INFINITY ? 0.f : exp2f(s[i][j] - mnew);
                Ps[(ty * 4 + i) * (BN + 1) + tx + 16 * j] = p;
                rs += p;
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
            l[i] = l[i] * corr + rs;
            m[i] = mnew;
#pragma unroll
            for (int c = 0; c < DC; ++c) o[i][c] *= corr;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < BN; ++k) {
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = Ps[(ty * 4 + i) * (BN + 1) + k];
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                const float v = Vs[k * D + tx + 16 * c];
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i][c] = fmaf(p[i], v, o[i][c]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = q0 + ty * 4 + i;
        if (q < n) {
            const float inv = 1.f / l[i];
#pragma unroll
            for (int c = 0; c < DC; ++c) O[((int64_t)h * n + q) * D + tx + 16 * c] = o[i][c] * inv;
            if (tx == 0) lse2[(int64_t)h * n + q] = m[i] + log2f(l[i]);
            // every key switched off by its bias: no attention to match
            if (tx == 0 && !(l[i] > 0.f)) set_status(status, h, KVC_ERR_NONFINITE);
        }
    }
}

// ---------------------------------------------------------------- key score
// grid (ceil(T/64), H), block 256.  score [H][T] = sqrt(mean_q P_qj^2), or
// with MEAN the mean attention mean_q P_qj (the window importance of
// thought-aware compaction).
template <typename TIn, int D, bool MEAN = false>
__global__ void __launch_bounds__(NT) k_colscore(const TIn* __restrict__ Q, const TIn* __restrict__ K,
                                                 const float* __restrict__ lse2, int n, int T, float c2,
                                                 float* __restrict__ score, const int32_t* __restrict__ status,
                                                 int qdiv, const float* __restrict__ bias2) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    extern __shared__ float sm[];
    constexpr int P = D + 1;
    float* Ks = sm;
    float* Qs = Ks + BN * P;
    float* Ls = Qs + BM * P;          // [BM] lse of the q tile
    double* red = reinterpret_cast<double*>(Ls + BM);   // [16][BN]
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const int k0 = blockIdx.x * BN;
    const int kv = min(BN, T - k0);
    load_tile<TIn, D>(Ks, K + ((int64_t)h * T + k0) * D, kv, D);
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, cmp[4] = {0.f, 0.f, 0.f, 0.f};   // Kahan sums per key
    float kb[4];                                                          // the keys' input biases
#pragma unroll
    for (int j = 0; j < 4; ++j)
        kb[j] = bias2 && tx + 16 * j < kv ? bias2[h * round_up(T, 256) + k0 + tx + 16 * j] : 0.f;
    for (int q0 = 0; q0 < n; q0 += BM) {
        const int qv = min(BM, n - q0);
        __syncthreads();
        load_tile<TIn, D>(Qs, Q + ((int64_t)(h / qdiv) * n + q0) * D, qv, D);
        for (int e = threadIdx.x; e < BM; e += NT) Ls[e] = (e < qv) ? lse2[(int64_t)h * n + q0 + e] : INFINITY;
        __syncthreads();
        float s[4][4];
        tile_dot<D>(Qs, Ks, s);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x = fmaf(s[i][j], c2, kb[j]) - Ls[ty * 4 + i];   // log2 of P
                part += MEAN ? exp2f(x) : exp2f(x + x);          // P or P^2
            }
            const float y = part - cmp[j];
            const float tt = acc[j] + y;
            cmp[j] = (tt - acc[j]) - y;
            acc[j] = tt;
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) red[ty * BN + tx + 16 * j] = (double)acc[j] - (double)cmp[j];
    __syncthreads();
    if (threadIdx.x < BN && threadIdx.x < kv) {
        double sum = 0.0;
        for (int r = 0; r < 16; ++r) sum += red[r * BN + threadIdx.x];
        score[(int64_t)h * T + k0 + threadIdx.x] = MEAN ? (float)(sum / (double)n) : (float)sqrt(sum / (double)n);
    }
}

// ---------------------------------------------------------------- mass logits
// grid (ceil(max_t/64), ceil(n/64), H).  l2[h][q][i] = S c2 + bk_i - lse2_q
// for i < t_h, -inf for t_h <= i < round_up(t_h, 64).  C_k is the compacted
// key buffer; bk (optional, [sum t], log2 units) the kept keys' input biases.
template <typename TIn, int D>
__global__ void __launch_bounds__(NT) k_masslogits(const TIn* __restrict__ Q, const TIn* __restrict__ Ck,
                                                   const float* __restrict__ lse2, const int32_t* __restrict__ offsets,
                                                   int n, int64_t ldA, float c2, float* __restrict__ L2,
                                                   const int32_t* __restrict__ status, int qdiv,
                                                   const float* __restrict__ bk) {
    const int h = blockIdx.z;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int th = offsets[h + 1] - off;
    const int i0 = blockIdx.x * BN;
    if (i0 >= th) return;
    extern __shared__ float sm[];
    constexpr int P = D + 1;
    float* Qs = sm;
    float* Cs = Qs + BM * P;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const int q0 = blockIdx.y * BM;
    const int qv = min(BM, n - q0);
    load_tile<TIn, D>(Qs, Q + ((int64_t)(h / qdiv) * n + q0) * D, qv, D);
    load_tile<TIn, D>(Cs, Ck + ((int64_t)off + i0) * D, min(BN, th - i0), D);
    __syncthreads();
    float s[4][4];
    tile_dot<D>(Qs, Cs, s);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = q0 + ty * 4 + i;
        if (q >= n) continue;
        const float l = lse2[(int64_t)h * n + q];
        float* row = L2 + ((int64_t)h * n + q) * ldA;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = i0 + tx + 16 * j;
            row[c] = (c < th) ? fmaf(s[i][j], c2, bk ? bk[off + c] : 0.f) - l : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------- attend
// grid (ceil(nq/64), H).  O[h][q] = softmax_i(Q.C_k[i]*scale + beta_i) C_v[i].
template <typename TIn, int D>
__global__ void __launch_bounds__(NT) k_attend(const TIn* __restrict__ Q, int nq, const TIn* __restrict__ Ck,
                                               const float* __restrict__ beta, const float* __restrict__ Cv,
                                               const int32_t* __restrict__ offsets, float c2,
                                               float* __restrict__ O, int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    const int off = offsets[h];
    const int th = offsets[h + 1] - off;
    if (th <= 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, h, KVC_ERR_BAD_BUDGET);
        return;
    }
    extern __shared__ float sm[];
    constexpr int P = D + 1;
    float* Qs = sm;
    float* Ks = Qs + BM * P;
    float* Vs = Ks + BN * P;
    float* Ps = Vs + BN * D;
    float* Bs = Ps + BM * (BN + 1);   // [BN] bias in log2 units
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    const int q0 = blockIdx.x * BM;
    load_tile<TIn, D>(Qs, Q + ((int64_t)h * nq + q0) * D, min(BM, nq - q0), D);
    constexpr int DC = D / 16;
    float o[4][DC];
    float m[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < DC; ++c) o[i][c] = 0.f;
    }
    for (int k0 = 0; k0 < th; k0 += BN) {
        const int kv = min(BN, th - k0);
        __syncthreads();
        load_tile<TIn, D>(Ks, Ck + ((int64_t)off + k0) * D, kv, D);
        load_tile_f32_nopad<D>(Vs, Cv + ((int64_t)off + k0) * D, kv, D);
        for (int e = threadIdx.x; e < BN; e += NT) Bs[e] = (e < kv) ? beta[off + k0 + e] * kLog2e : -INFINITY;
        __syncthreads();
        float s[4][4];
        tile_dot<D>(Qs, Ks, s);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float b = Bs[tx + 16 * j];
                s[i][j] = (b == -INFINITY) ? -INFINITY : s[i][j] * c2 + b;
                mx = fmaxf(mx, s[i][j]);
            }
#pragma unroll
            for (int off2 = 8; off2 > 0; off2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off2));
            const float mnew = fmaxf(m[i], mx);
            const float mref = (mnew == -INFINITY) ? 0.f : mnew;
            const float corr = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - mref);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float p = exp2f(s[i][j] - mref);
                Ps[(ty * 4 + i) * (BN + 1) + tx + 16 * j] = p;
                rs += p;
            }
#pragma unroll
            for (int off2 = 8; off2 > 0; off2 >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off2);
            l[i] = l[i] * corr + rs;
            m[i] = mnew;
#pragma unroll
            for (int c = 0; c < DC; ++c) o[i][c] *= corr;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < BN; ++k) {
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = Ps[(ty * 4 + i) * (BN + 1) + k];
#pragma unroll
            for (int c = 0; c < DC; ++c) {
                const float v = Vs[k * D + tx + 16 * c];
#pragma unroll
                for (int i = 0; i < 4; ++i) o[i][c] = fmaf(p[i], v, o[i][c]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = q0 + ty * 4 + i;
        if (q < nq) {
            if (!(l[i] > 0.f)) {
                if (tx == 0) set_status(status, h, KVC_ERR_NONFINITE);
                continue;
            }
            const float inv = 1.f / l[i];
#pragma unroll
            for (int c = 0; c < DC; ++c) O[((int64_t)h * nq + q) * D + tx + 16 * c] = o[i][c] * inv;
        }
    }
}

// ---------------------------------------------------------------- launchers
template <typename TIn, int D>
static cudaError_t launch_attn_simt_t(const void* Q, const void* K, const void* V, int H, int n, int T, float c2,
                                      float* O, float* lse2, int32_t* status, int qdiv, const float* bias2,
                                      cudaStream_t st) {
    constexpr int P = D + 1;
    size_t smem = (size_t)(BM * P + BN * P + BN * D + BM * (BN + 1)) * sizeof(float);
    auto kern = k_attn_fwd<TIn, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((n + BM - 1) / BM, H);
    kern<<<grid, NT, smem, st>>>((const TIn*)Q, (const TIn*)K, (const TIn*)V, n, T, c2, O, lse2, status, qdiv, bias2);
    return cudaGetLastError();
}
template <typename TIn, int D>
static cudaError_t launch_colscore_simt_t(const void* Q, const void* K, const float* lse2, int H, int n, int T,
                                          float c2, float* score, const int32_t* status, int qdiv,
                                          const float* bias2, cudaStream_t st) {
    constexpr int P = D + 1;
    size_t smem = (size_t)(BN * P + BM * P + BM) * sizeof(float) + 16 * BN * sizeof(double) + 8;
    auto kern = k_colscore<TIn, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((T + BN - 1) / BN, H);
    kern<<<grid, NT, smem, st>>>((const TIn*)Q, (const TIn*)K, lse2, n, T, c2, score, status, qdiv, bias2);
    return cudaGetLastError();
}
template <typename TIn, int D>
static cudaError_t launch_colmean_simt_t(const void* Q, const void* K, const float* lse2, int H, int n, int T,
                                         float c2, float* out, const int32_t* status, cudaStream_t st) {
    constexpr int P = D + 1;
    size_t smem = (size_t)(BN * P + BM * P + BM) * sizeof(float) + 16 * BN * sizeof(double) + 8;
    auto kern = k_colscore<TIn, D, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((T + BN - 1) / BN, H);
    kern<<<grid, NT, smem, st>>>((const TIn*)Q, (const TIn*)K, lse2, n, T, c2, out, status, 1, nullptr);
    return cudaGetLastError();
}
template <typename TIn, int D>
static cudaError_t launch_masslogits_t(const void* Q, const void* Ck, const float* lse2, const int32_t* offsets,
                                       int H, int n, int max_t, int64_t ldA, float c2, float* L2,
                                       const int32_t* status, int qdiv, const float* bk, cudaStream_t st) {
    constexpr int P = D + 1;
    size_t smem = (size_t)(BM * P + BN * P) * sizeof(float);
    auto kern = k_masslogits<TIn, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((max_t + BN - 1) / BN, (n + BM - 1) / BM, H);
    kern<<<grid, NT, smem, st>>>((const TIn*)Q, (const TIn*)Ck, lse2, offsets, n, ldA, c2, L2, status, qdiv, bk);
    return cudaGetLastError();
}
template <typename TIn, int D>
static cudaError_t launch_attend_t(const void* Q, int nq, const void* Ck, const float* beta, const float* Cv,
                                   const int32_t* offsets, int H, float c2, float* O, int32_t* status,
                                   cudaStream_t st) {
    constexpr int P = D + 1;
    size_t smem = (size_t)(BM * P + BN * P + BN * D + BM * (BN + 1) + BN) * sizeof(float);
    auto kern = k_attend<TIn, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((nq + BM - 1) / BM, H);
    kern<<<grid, NT, smem, st>>>((const TIn*)Q, nq, (const TIn*)Ck, beta, Cv, offsets, c2, O, status);
    return cudaGetLastError();
}

#define KVC_DISPATCH(dtype, d, FN, ...)                                                      \
    ((dtype) == KVC_DTYPE_BF16                                                               \
         ? ((d) == 128 ? FN<__nv_bfloat16, 128>(__VA_ARGS__) : FN<__nv_bfloat16, 64>(__VA_ARGS__)) \
         : ((d) == 128 ? FN<float, 128>(__VA_ARGS__) : FN<float, 64>(__VA_ARGS__)))

// bias2 (optional): per-key input bias [H][round_up(T, 256)], log2 units.
cudaError_t launch_attn_fwd_simt(int dtype, int d, const void* Q, const void* K, const void* V, int H, int n, int T,
                                 float c2, float* O, float* lse2, int32_t* status, int qdiv, const float* bias2,
                                 cudaStream_t st) {
    return KVC_DISPATCH(dtype, d, launch_attn_simt_t, Q, K, V, H, n, T, c2, O, lse2, status, qdiv, bias2, st);
}
// mean_q softmax_j over queries Q (own lse2): out [H][T]
cudaError_t launch_colmean_simt(int dtype, int d, const void* Q, const void* K, const float* lse2, int H, int n, int T,
                                float c2, float* out, const int32_t* status, cudaStream_t st) {
    return KVC_DISPATCH(dtype, d, launch_colmean_simt_t, Q, K, lse2, H, n, T, c2, out, status, st);
}
cudaError_t launch_colscore_simt(int dtype, int d, const void* Q, const void* K, const float* lse2, int H, int n,
                                 int T, float c2, float* score, const int32_t* status, int qdiv, const float* bias2,
                                 cudaStream_t st) {
    return KVC_DISPATCH(dtype, d, launch_colscore_simt_t, Q, K, lse2, H, n, T, c2, score, status, qdiv, bias2, st);
}
cudaError_t launch_masslogits(int dtype, int d, const void* Q, const void* Ck, const float* lse2,
                              const int32_t* offsets, int H, int n, int max_t, int64_t ldA, float c2, float* L2,
                              const int32_t* status, int qdiv, const float* bk, cudaStream_t st) {
    return KVC_DISPATCH(dtype, d, launch_masslogits_t, Q, Ck, lse2, offsets, H, n, max_t, ldA, c2, L2, status, qdiv,
                        bk, st);
}
cudaError_t launch_attend(int dtype, int d, const void* Q, int nq, const void* Ck, const float* beta,
                          const float* Cv, const int32_t* offsets, int H, float c2, float* O, int32_t* status,
                          cudaStream_t st) {
    return KVC_DISPATCH(dtype, d, launch_attend_t, Q, nq, Ck, beta, Cv, offsets, H, c2, O, status, st);
}

}  // namespace kvc
