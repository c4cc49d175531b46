// Key selection by orthogonal matching pursuit ("Fast KV Compaction via
// Attention Matching", section 2 "Pipeline algorithmique": keys chosen
// greedily to best meet the attention-mass objective, then NNLS for the
// weights).  The dictionary is the columns p_j of the relative-mass matrix of
// all T keys, P_qj = exp(S_qj - lse_q), and the target is 1 per query.  With
// S the keys chosen so far and r = 1 - P_S w the residual of the least-
// squares fit of 1 on them, a step picks the key outside S with the largest
// <p_j, r> / ||p_j|| (ties to the lower position); forced positions are taken
// first, in ascending order.
//
// The residual is kept through an orthonormal basis of span(P_S): the new
// column is orthogonalised against the basis by two rounds of classical
// Gram-Schmidt, normalised and appended, and r loses its component along it.
// A column whose remainder is below 1e-5 of its norm adds no direction.
//
// bf16 inputs recompute the dictionary instead of storing it: ||p_j|| is
// sqrt(n) times the RMS key score, every step's <p_j, r> comes from the
// weighted form of the tensor-core key-score pass (S = K Q^T again,
// exp2(S c2 - lse2_q) weighted by r_q and summed; attn_tc.cu), and the
// picked key's column is recomputed from Q and K_j.  fp32 inputs keep P.
//
// Layout (all per head, fp32): P key-major [T][ldn] (fp32 inputs; a column is
// contiguous) or the correlations [T] (bf16 inputs), norms [T], residual r
// [ldn], basis [max_t][ldn], working column v [ldn].
// Kernels, all heads in parallel, one pursuit step per round of launches:
//   k_omp_probs     P = exp2(Q K^T c2 - lse2), written key-major (fp32)
//   k_omp_norms     ||p_j|| from P (fp32); k_omp_init from the RMS score (bf16)
//   k_omp_corr      <p_j, r> / ||p_j|| for the keys not chosen; CTA argmax
//                   (fp32: warp per key over P; bf16: k_omp_corr_pre, thread
//                   per key over the recomputed correlations)
//   k_omp_pick      the step's key (forced position or argmax); v = p_j
//                   (fp32: copied from P; bf16: k_omp_col recomputes it)
//   k_omp_proj      c_k = <basis_k, v>
//   k_omp_sub       v -= sum_k c_k basis_k
//   k_omp_finish    basis_s = v / ||v||, r -= <basis_s, r> basis_s
//   k_omp_idx       kept positions in ascending order
#include <algorithm>

#include "common.cuh"

namespace kvc {

namespace {

struct OmpArgs {
    float* P;                  // [H][T][ldn] (fp32 inputs; null for bf16)
    float* corr;               // [H][T] correlations, first the RMS scores (bf16 inputs)
    int32_t* pick;             // [H] the step's key
    float* norms;              // [H][T]
    uint8_t* chosen;           // [H][T]
    float* r;                  // [H][ldn]
    float* v;                  // [H][ldn]
    float* basis;              // [H][max_t][ldn]
    float* coef;               // [H][max_t]
    int32_t* nbasis;           // [H]
    float2* part;              // [H][ceil(T/8)]: (value, index as float bits)
    int32_t* order;            // [H][max_t]
    float* pnorm;              // [H]
    const int32_t* offsets;
    int n, T, max_t, ldn;
    int keep_first, keep_last;
    int32_t* status;
};

// forced positions of the cache (first keep_first, last keep_last), counted once
__device__ __forceinline__ int forced_count(int T, int kf, int kl) { return min(T, kf + kl); }
__device__ __forceinline__ int forced_at(int s, int T, int kf, int kl) {
    const int a = min(kf, T);
    return s < a ? s : max(a, T - kl) + (s - a);
}

// ---------------------------------------------------------------- P
// grid (ceil(T/64), ceil(n/64), H), block 256: a 64 x 64 tile of logits by
// FFMA over 32-wide slices of the head dimension, exponentiated and written
// key-major through shared memory.
template <typename TIn, int D>
__global__ void __launch_bounds__(256) k_omp_probs(const TIn* __restrict__ Q, const TIn* __restrict__ K,
                                                   const float* __restrict__ lse2, float c2, OmpArgs a) {
    const int h = blockIdx.z;
    if (!head_ok(a.status, h)) return;
    constexpr int DK = 32;
    __shared__ float Qs[64][DK + 1];
    __shared__ float Ks[64][DK + 1];
    __shared__ float Ls[64];
    __shared__ float Pt[64][65];          // [key][query]
    const int j0 = blockIdx.x * 64, q0 = blockIdx.y * 64;
    if (threadIdx.x < 64) Ls[threadIdx.x] = (q0 + threadIdx.x < a.n) ? lse2[(int64_t)h * a.n + q0 + threadIdx.x] : 0.f;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;   // queries 4 ty + i, keys tx + 16 jj
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) s[i][jj] = 0.f;
    for (int k0 = 0; k0 < D; k0 += DK) {
        __syncthreads();
        for (int e = threadIdx.x; e < 64 * DK; e += 256) {
            const int r = e / DK, c = e % DK;
            Qs[r][c] = (q0 + r < a.n) ? to_f32(Q[((int64_t)h * a.n + q0 + r) * D + k0 + c]) : 0.f;
            Ks[r][c] = (j0 + r < a.T) ? to_f32(K[((int64_t)h * a.T + j0 + r) * D + k0 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < DK; ++k) {
            float qa[4], kb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qa[i] = Qs[ty * 4 + i][k];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) kb[jj] = Ks[tx + 16 * jj][k];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) s[i][jj] = fmaf(qa[i], kb[jj], s[i][jj]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int q = ty * 4 + i;
            Pt[tx + 16 * jj][q] = (q0 + q < a.n) ? exp2f(s[i][jj] * c2 - Ls[q]) : 0.f;
        }
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int jr = e / 64, q = e % 64;
        if (j0 + jr < a.T && q0 + q < a.ldn) a.P[((int64_t)h * a.T + j0 + jr) * a.ldn + q0 + q] = Pt[jr][q];
    }
}

// grid (ceil(T/8), H), block 256: a warp per key.  Also resets the pursuit.
__global__ void __launch_bounds__(256) k_omp_norms(OmpArgs a) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    const int j = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (blockIdx.x == 0) {
        for (int q = threadIdx.x; q < a.ldn; q += 256) a.r[(int64_t)h * a.ldn + q] = q < a.n ? 1.f : 0.f;
        if (threadIdx.x == 0) a.nbasis[h] = 0;
    }
    if (j >= a.T) return;
    const float4* col = reinterpret_cast<const float4*>(a.P + ((int64_t)h * a.T + j) * a.ldn);
    float s = 0.f;
    for (int c = lane; c < a.ldn / 4; c += 32) {
        const float4 x = col[c];
        s = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, s))));
    }
    s = warp_sum(s);
    if (lane == 0) {
        a.norms[(int64_t)h * a.T + j] = sqrtf(s);
        a.chosen[(int64_t)h * a.T + j] = 0;
    }
}

// (value, position) with ties to the lower position
__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

// ---------------------------------------------------------------- one step
// grid (ceil(T/8), H), block 256: a warp per key; CTA argmax to part.
__global__ void __launch_bounds__(256) k_omp_corr(OmpArgs a, int s) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t || s < forced_count(a.T, a.keep_first, a.keep_last)) return;
    __shared__ float wv[8];
    __shared__ int wi[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + warp;
    float c = -INFINITY;
    if (j < a.T && !a.chosen[(int64_t)h * a.T + j]) {
        const float nj = a.norms[(int64_t)h * a.T + j];
        if (nj > 0.f) {
            const float4* col = reinterpret_cast<const float4*>(a.P + ((int64_t)h * a.T + j) * a.ldn);
            const float4* rr = reinterpret_cast<const float4*>(a.r + (int64_t)h * a.ldn);
            float d0 = 0.f, d1 = 0.f;
            int cc = lane;
            for (; cc + 32 < a.ldn / 4; cc += 64) {
                const float4 x = col[cc], y = rr[cc];
                const float4 x2 = col[cc + 32], y2 = rr[cc + 32];
                d0 = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, d0))));
                d1 = fmaf(x2.x, y2.x, fmaf(x2.y, y2.y, fmaf(x2.z, y2.z, fmaf(x2.w, y2.w, d1))));
            }
            if (cc < a.ldn / 4) {
                const float4 x = col[cc], y = rr[cc];
                d0 = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, d0))));
            }
            c = warp_sum(d0 + d1) / nj;
        }
    }
    if (lane == 0) {
        wv[warp] = c;
        wi[warp] = j;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float bv = -INFINITY;
        int bi = INT32_MAX;
        for (int w = 0; w < 8; ++w)
            if (wv[w] > -INFINITY) better(bv, bi, wv[w], wi[w]);
        a.part[(int64_t)h * gridDim.x + blockIdx.x] = make_float2(bv, __int_as_float(bi));
    }
}

// grid H, block 256: the step's key; v = its column.
__global__ void __launch_bounds__(256) k_omp_pick(OmpArgs a, int s, int nparts) {
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t) return;
    __shared__ float sv[256];
    __shared__ int si[256];
    __shared__ int pick;
    const int nf = forced_count(a.T, a.keep_first, a.keep_last);
    if (s < nf) {
        if (threadIdx.x == 0) pick = forced_at(s, a.T, a.keep_first, a.keep_last);
    } else {
        float bv = -INFINITY;
        int bi = INT32_MAX;
        for (int p = threadIdx.x; p < nparts; p += 256) {
            const float2 x = a.part[(int64_t)h * nparts + p];
            if (x.x > -INFINITY) better(bv, bi, x.x, __float_as_int(x.y));
        }
        sv[threadIdx.x] = bv;
        si[threadIdx.x] = bi;
        __syncthreads();
        for (int o = 128; o > 0; o >>= 1) {
            if (threadIdx.x < o && sv[threadIdx.x + o] > -INFINITY) {
                float v0 = sv[threadIdx.x];
                int i0 = si[threadIdx.x];
                better(v0, i0, sv[threadIdx.x + o], si[threadIdx.x + o]);
                sv[threadIdx.x] = v0;
                si[threadIdx.x] = i0;
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            int j = si[0];
            if (!(sv[0] > -INFINITY)) {
                // no candidate with a positive norm: the lowest position not chosen
                j = 0;
                while (j < a.T && a.chosen[(int64_t)h * a.T + j]) ++j;
            }
            pick = j;
        }
    }
    __syncthreads();
    const int j = pick;
    if (threadIdx.x == 0) {
        a.chosen[(int64_t)h * a.T + j] = 1;
        a.order[(int64_t)h * a.max_t + s] = j;
        a.pnorm[h] = a.norms[(int64_t)h * a.T + j];
    }
    if (threadIdx.x == 0) a.pick[h] = j;
    if (!a.P) return;                 // bf16: k_omp_col recomputes the column
    const float* col = a.P + ((int64_t)h * a.T + j) * a.ldn;
    for (int q = threadIdx.x; q < a.ldn; q += 256) a.v[(int64_t)h * a.ldn + q] = col[q];
}

// bf16 inputs: ||p_j|| = sqrt(n) * RMS score (the scores sit in corr), and the
// pursuit's reset.  grid (ceil(T/256), H), block 256.
__global__ void __launch_bounds__(256) k_omp_init(OmpArgs a) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    if (blockIdx.x == 0) {
        for (int q = threadIdx.x; q < a.ldn; q += 256) a.r[(int64_t)h * a.ldn + q] = q < a.n ? 1.f : 0.f;
        if (threadIdx.x == 0) a.nbasis[h] = 0;
    }
    const int j = blockIdx.x * 256 + threadIdx.x;
    if (j >= a.T) return;
    a.norms[(int64_t)h * a.T + j] = a.corr[(int64_t)h * a.T + j] * sqrtf((float)a.n);
    a.chosen[(int64_t)h * a.T + j] = 0;
}

// bf16 inputs: <p_j, r> / ||p_j|| from the recomputed correlations, a thread
// per key; CTA argmax to part.  grid (ceil(T/256), H), block 256.
__global__ void __launch_bounds__(256) k_omp_corr_pre(OmpArgs a, int s) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t || s < forced_count(a.T, a.keep_first, a.keep_last)) return;
    __shared__ float sv[256];
    __shared__ int si[256];
    const int j = blockIdx.x * 256 + threadIdx.x;
    float c = -INFINITY;
    if (j < a.T && !a.chosen[(int64_t)h * a.T + j]) {
        const float nj = a.norms[(int64_t)h * a.T + j];
        if (nj > 0.f) c = a.corr[(int64_t)h * a.T + j] / nj;
    }
    sv[threadIdx.x] = c;
    si[threadIdx.x] = c > -INFINITY ? j : INT32_MAX;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o && sv[threadIdx.x + o] > -INFINITY) {
            float v0 = sv[threadIdx.x];
            int i0 = si[threadIdx.x];
            better(v0, i0, sv[threadIdx.x + o], si[threadIdx.x + o]);
            sv[threadIdx.x] = v0;
            si[threadIdx.x] = i0;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) a.part[(int64_t)h * gridDim.x + blockIdx.x] = make_float2(sv[0], __int_as_float(si[0]));
}

// bf16 inputs: v = p_j for the picked key j, p_j[q] = exp2(q . K_j c2 -
// lse2_q) for q < n (0 up to ldn).  grid (ceil(ldn/64), H), block 256: a
// warp per 8 queries, lanes over the head dimension.
template <int D>
__global__ void __launch_bounds__(256) k_omp_col(OmpArgs a, int s, const __nv_bfloat16* __restrict__ Q,
                                                 const __nv_bfloat16* __restrict__ K, const float* __restrict__ lse2,
                                                 float c2) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t) return;
    const int j = a.pick[h];
    if (!KVC_IN_RANGE(j >= 0 && j < a.T, a.status, h)) return;
    constexpr int E = D / 32;                       // elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float kj[E];
#pragma unroll
    for (int e = 0; e < E; ++e) kj[e] = __bfloat162float(K[((int64_t)h * a.T + j) * D + lane * E + e]);
    for (int qq = 0; qq < 8; ++qq) {
        const int q = blockIdx.x * 64 + warp * 8 + qq;
        if (q >= a.ldn) break;
        float dot = 0.f;
        if (q < a.n) {
            const __nv_bfloat16* qr = Q + ((int64_t)h * a.n + q) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(__bfloat162float(qr[e]), kj[e], dot);
        }
        dot = warp_sum(dot);
        if (lane == 0) a.v[(int64_t)h * a.ldn + q] = q < a.n ? exp2f(fmaf(dot, c2, -lse2[(int64_t)h * a.n + q])) : 0.f;
    }
}

// grid (ceil(max_t/8), H), block 256: a warp per basis vector.
__global__ void __launch_bounds__(256) k_omp_proj(OmpArgs a, int s) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t) return;
    const int k = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (k >= a.nbasis[h]) return;
    const float4* b = reinterpret_cast<const float4*>(a.basis + ((int64_t)h * a.max_t + k) * a.ldn);
    const float4* v = reinterpret_cast<const float4*>(a.v + (int64_t)h * a.ldn);
    float d = 0.f;
    for (int c = lane; c < a.ldn / 4; c += 32) {
        const float4 x = b[c], y = v[c];
        d = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, d))));
    }
    d = warp_sum(d);
    if (lane == 0) a.coef[(int64_t)h * a.max_t + k] = d;
}

// grid (ceil(ldn/256), H), block 256: v[q] -= sum_k coef_k basis_k[q].
__global__ void __launch_bounds__(256) k_omp_sub(OmpArgs a, int s) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t) return;
    extern __shared__ float cf[];
    const int nb = a.nbasis[h];
    for (int k = threadIdx.x; k < nb; k += 256) cf[k] = a.coef[(int64_t)h * a.max_t + k];
    __syncthreads();
    const int q = blockIdx.x * 256 + threadIdx.x;
    if (q >= a.ldn) return;
    const float* b = a.basis + (int64_t)h * a.max_t * a.ldn + q;
    float acc0 = 0.f, acc1 = 0.f;
    int k = 0;
    for (; k + 1 < nb; k += 2) {
        acc0 = fmaf(cf[k], b[(int64_t)k * a.ldn], acc0);
        acc1 = fmaf(cf[k + 1], b[(int64_t)(k + 1) * a.ldn], acc1);
    }
    if (k < nb) acc0 = fmaf(cf[k], b[(int64_t)k * a.ldn], acc0);
    a.v[(int64_t)h * a.ldn + q] -= acc0 + acc1;
}

// grid H, block 256: append v / ||v|| to the basis and update the residual.
__global__ void __launch_bounds__(256) k_omp_finish(OmpArgs a, int s) {
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t) return;
    __shared__ float red[8];
    __shared__ float bc;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* v = a.v + (int64_t)h * a.ldn;
    float* r = a.r + (int64_t)h * a.ldn;
    auto block_sum = [&](float x) {
        x = warp_sum(x);
        if (lane == 0) red[warp] = x;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
            for (int w = 0; w < 8; ++w) tot += red[w];
            bc = tot;
        }
        __syncthreads();
        const float res = bc;
        __syncthreads();
        return res;
    };
    float ss = 0.f;
    for (int q = threadIdx.x; q < a.ldn; q += 256) ss = fmaf(v[q], v[q], ss);
    const float vn = sqrtf(block_sum(ss));
    const int nb = a.nbasis[h];
    if (!(vn > 1e-5f * a.pnorm[h]) || nb >= a.max_t) return;     // dependent column: no new direction
    const float inv = 1.f / vn;
    float* b = a.basis + ((int64_t)h * a.max_t + nb) * a.ldn;
    float dr = 0.f;
    for (int q = threadIdx.x; q < a.ldn; q += 256) {
        const float x = v[q] * inv;
        b[q] = x;
        dr = fmaf(x, r[q], dr);
    }
    const float alpha = block_sum(dr);
    for (int q = threadIdx.x; q < a.ldn; q += 256) r[q] = fmaf(-alpha, b[q], r[q]);
    if (threadIdx.x == 0) a.nbasis[h] = nb + 1;
}

// grid H, block 1024: kept positions (chosen flags) in ascending order.
__global__ void __launch_bounds__(1024) k_omp_idx(OmpArgs a, int32_t* __restrict__ idx_out) {
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return;
    __shared__ int wsum[32];
    __shared__ int base;
    if (threadIdx.x == 0) base = 0;
    __syncthreads();
    const int off = a.offsets[h];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j0 = 0; j0 < a.T; j0 += 1024) {
        const int j = j0 + threadIdx.x;
        const int f = (j < a.T && a.chosen[(int64_t)h * a.T + j]) ? 1 : 0;
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (lane == 0) wsum[warp] = __popc(m);
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        if (f) idx_out[off + base + before + __popc(m & ((1u << lane) - 1u))] = j;
        __syncthreads();
        if (threadIdx.x == 0) {
            int tot = 0;
            for (int w = 0; w < 32; ++w) tot += wsum[w];
            base += tot;
        }
        __syncthreads();
    }
}

template <typename TIn, int D>
cudaError_t launch_probs_t(const void* Q, const void* K, const float* lse2, float c2, const OmpArgs& a, int H,
                           cudaStream_t st) {
    dim3 grid((a.T + 63) / 64, (a.n + 63) / 64, H);
    k_omp_probs<TIn, D><<<grid, 256, 0, st>>>((const TIn*)Q, (const TIn*)K, lse2, c2, a);
    return cudaGetLastError();
}

}  // namespace

namespace {
// Bytes of the dictionary region: P for fp32 inputs, the correlations for bf16.
size_t omp_dict_bytes(int dtype, int H, int T, size_t ldn) {
    return dtype == KVC_DTYPE_F32 ? (size_t)H * T * ldn * 4 : (size_t)H * T * 4;
}
}  // namespace

// Workspace of the pursuit for a problem (bytes, 256-aligned pieces).
size_t omp_workspace_bytes(int dtype, int H, int n, int T, int max_t) {
    const size_t ldn = (size_t)round_up(n, 4);
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    return al(omp_dict_bytes(dtype, H, T, ldn)) + al((size_t)H * T * 4) + al((size_t)H * T) +
           2 * al((size_t)H * ldn * 4) + al((size_t)H * max_t * ldn * 4) + al((size_t)H * max_t * 4) +
           al((size_t)H * 4) + al((size_t)H * ((T + 7) / 8) * 8) + al((size_t)H * max_t * 4) + al((size_t)H * 4) +
           al((size_t)H * 4);
}

// Byte offset of the selection order [H][max_t] inside that workspace.
size_t omp_order_offset(int dtype, int H, int n, int T, int max_t) {
    const size_t ldn = (size_t)round_up(n, 4);
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    return al(omp_dict_bytes(dtype, H, T, ldn)) + al((size_t)H * T * 4) + al((size_t)H * T) +
           2 * al((size_t)H * ldn * 4) + al((size_t)H * max_t * ldn * 4) + al((size_t)H * max_t * 4) +
           al((size_t)H * 4) + al((size_t)H * ((T + 7) / 8) * 8);
}

int omp_launches(int dtype, int max_t) { return dtype == KVC_DTYPE_F32 ? 3 + 7 * max_t : 2 + 9 * max_t; }

cudaError_t launch_colscore_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T,
                               float c2, float* score, int32_t* status, int qdiv, long long wait_limit,
                               const float* bias2, cudaStream_t st);
cudaError_t launch_corr_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T, float c2,
                           const float* r, int64_t rstride, float* out, int32_t* status, long long wait_limit,
                           cudaStream_t st);

// The pursuit for every head: idx_out[off .. off + t) = chosen positions,
// ascending.  lse2 from the attention pass; forced positions first.
cudaError_t launch_omp_select(int dtype, int d, const void* Q, const void* K, const float* lse2, float c2, int H,
                              int n, int T, int max_t, const int32_t* offsets, int keep_first, int keep_last,
                              void* ws, int32_t* idx_out, int32_t* status, long long wait_limit, cudaStream_t st) {
    const int ldn = (int)round_up(n, 4);
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    const bool rec = dtype == KVC_DTYPE_BF16;          // recompute the dictionary on the tensor cores
    char* p = static_cast<char*>(ws);
    OmpArgs a{};
    a.P = rec ? nullptr : (float*)p;
    a.corr = rec ? (float*)p : nullptr;
    p += al(omp_dict_bytes(dtype, H, T, (size_t)ldn));
    a.norms = (float*)p;
    p += al((size_t)H * T * 4);
    a.chosen = (uint8_t*)p;
    p += al((size_t)H * T);
    a.r = (float*)p;
    p += al((size_t)H * ldn * 4);
    a.v = (float*)p;
    p += al((size_t)H * ldn * 4);
    a.basis = (float*)p;
    p += al((size_t)H * max_t * ldn * 4);
    a.coef = (float*)p;
    p += al((size_t)H * max_t * 4);
    a.nbasis = (int32_t*)p;
    p += al((size_t)H * 4);
    a.part = (float2*)p;
    p += al((size_t)H * ((T + 7) / 8) * 8);
    a.order = (int32_t*)p;
    p += al((size_t)H * max_t * 4);
    a.pnorm = (float*)p;
    p += al((size_t)H * 4);
    a.pick = (int32_t*)p;
    a.offsets = offsets;
    a.n = n;
    a.T = T;
    a.max_t = max_t;
    a.ldn = ldn;
    a.keep_first = keep_first;
    a.keep_last = keep_last;
    a.status = status;
    cudaError_t e;
    int nparts;
    if (rec) {
        // ||p_j|| from the RMS key score (into corr first)
        e = launch_colscore_tc(d, Q, K, lse2, H, n, T, c2, a.corr, status, 1, wait_limit, nullptr, st);
        if (e != cudaSuccess) return e;
        nparts = (T + 255) / 256;
        k_omp_init<<<dim3(nparts, H), 256, 0, st>>>(a);
    } else {
        e = d == 128 ? launch_probs_t<float, 128>(Q, K, lse2, c2, a, H, st)
                     : launch_probs_t<float, 64>(Q, K, lse2, c2, a, H, st);
        if (e != cudaSuccess) return e;
        nparts = (T + 7) / 8;
        k_omp_norms<<<dim3(nparts, H), 256, 0, st>>>(a);
    }
    const size_t sub_smem = (size_t)max_t * 4;
    if (sub_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(k_omp_sub, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sub_smem);
        if (e != cudaSuccess) return e;
    }
    const int nf = (int)std::min<int64_t>(T, (int64_t)keep_first + keep_last);   // forced steps need no correlations
    for (int s = 0; s < max_t; ++s) {
        if (rec) {
            if (s >= nf) {
                e = launch_corr_tc(d, Q, K, lse2, H, n, T, c2, a.r, ldn, a.corr, status, wait_limit, st);
                if (e != cudaSuccess) return e;
                k_omp_corr_pre<<<dim3(nparts, H), 256, 0, st>>>(a, s);
            }
        } else {
            k_omp_corr<<<dim3(nparts, H), 256, 0, st>>>(a, s);
        }
        k_omp_pick<<<H, 256, 0, st>>>(a, s, nparts);
        if (rec) {
            if (d == 128)
                k_omp_col<128><<<dim3((ldn + 63) / 64, H), 256, 0, st>>>(a, s, (const __nv_bfloat16*)Q,
                                                                       (const __nv_bfloat16*)K, lse2, c2);
            else
                k_omp_col<64><<<dim3((ldn + 63) / 64, H), 256, 0, st>>>(a, s, (const __nv_bfloat16*)Q,
                                                                      (const __nv_bfloat16*)K, lse2, c2);
        }
        for (int round = 0; round < 2; ++round) {
            k_omp_proj<<<dim3((max_t + 7) / 8, H), 256, 0, st>>>(a, s);
            k_omp_sub<<<dim3((ldn + 255) / 256, H), 256, sub_smem, st>>>(a, s);
        }
        k_omp_finish<<<H, 256, 0, st>>>(a, s);
    }
    k_omp_idx<<<H, 1024, 0, st>>>(a, idx_out);
    return cudaGetLastError();
}

}  // namespace kvc
