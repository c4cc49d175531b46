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
// Kernels, all heads in parallel:
//   k_omp_probs     P = exp2(Q K^T c2 - lse2), written key-major (fp32)
//   k_omp_norms     ||p_j|| from P (fp32); k_omp_init from the RMS score (bf16)
// one round of launches per pursuit step, fp32:
//   k_omp_corr      <p_j, r> / ||p_j|| for the keys not chosen (a warp per
//                   key over P); CTA argmax
//   k_omp_pick      the step's key (forced position or argmax); v = p_j
//   k_omp_proj      c_k = <basis_k, v>
//   k_omp_sub       v -= sum_k c_k basis_k
//   k_omp_finish    basis_s = v / ||v||, r -= <basis_s, r> basis_s
// two launches per step, bf16: the weighted key-score pass (the
// correlations), then k_omp_step, which does the pick, the column, the
// Gram-Schmidt rounds and the finish with a cluster of CTAs per head;
//   k_omp_idx       kept positions in ascending order
#include <algorithm>

#include <cooperative_groups.h>

#include "common.cuh"

namespace kvc {
namespace cg = cooperative_groups;

namespace {

struct OmpArgs {
    float* P;                  // [H][T][ldn] (fp32 inputs; null for bf16)
    float* corr;               // [H][T] the RMS key scores (bf16 inputs)
    float2* cpart;             // [nz][H][T] parts of the correlations <p_j, r>, fp32 pairs (bf16 inputs)
    int nz;
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


// One pursuit step of a head (bf16 inputs), fused into one launch: a cluster
// of CTAs per head splits the keys (the argmax), the queries (the recomputed
// column, the subtraction, the finish) and the basis vectors (the
// projections) between its CTAs, and meets at hardware cluster barriers;
// the partial results (argmax, squared norms, <q, r>) go through distributed
// shared memory and are combined in rank order, so every CTA takes the same
// decisions.  Steps: the key (forced position or argmax of <p_j, r> / ||p_j||
// over keys not chosen, ties to the lower position), v = p_j recomputed from
// Q and K_j, classical Gram-Schmidt against the basis (a second round when
// the first removed more than half of ||p_j||^2), and the finish (basis_nb =
// v / ||v||, r -= <basis_nb, r> basis_nb).  A column that keeps less than
// 1e-5 of its norm adds no direction.  The basis is streamed from L2 with
// many 16-byte loads in flight per SM (1024 threads, several loads each).
// grid (CL, H) in clusters of (CL, 1, 1) (16, or 8 where a cluster of 16
// cannot be placed), block 1024; dynamic shared memory: max_t + ldn floats
// (the projection coefficients and a copy of v).
constexpr int kStepThreads = 1024;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kStepKg = kStepThreads / 64;             // k-groups of the subtraction

size_t omp_step_smem(int max_t, int ldn) { return (size_t)(max_t + ldn) * 4; }

template <int D>
__global__ void __launch_bounds__(kStepThreads, 1)
    k_omp_step(OmpArgs a, int s, const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
               const float* __restrict__ lse2, float c2) {
    cg::cluster_group cluster = cg::this_cluster();
    grid_dependency_wait();                            // launched dependent on the correlation pass
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;                 // the same for every CTA of the cluster
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t) return;
    extern __shared__ float4 dyn4[];
    float* vs = reinterpret_cast<float*>(dyn4);        // [ldn] copy of v
    float* cf = vs + a.ldn;                            // [max_t] coefficients
    __shared__ float red_v[kStepThreads];
    __shared__ int red_i[kStepThreads];
    __shared__ float4 red4[kStepKg][64];               // the subtraction's k-group partials
    __shared__ float part_v;                           // this CTA's partials (read by the cluster)
    __shared__ int part_i;
    __shared__ float part_s;
    const int rank = (int)cluster.block_rank();
    const int CL = (int)cluster.num_blocks();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = a.nbasis[h];
    const int nf = forced_count(a.T, a.keep_first, a.keep_last);
    // this CTA's slice of the queries (a multiple of 4 long)
    const int qsz = (int)round_up((a.ldn + CL - 1) / CL, 4);
    const int q0 = min(a.ldn, rank * qsz), q1 = min(a.ldn, q0 + qsz);
    float* v = a.v + (int64_t)h * a.ldn;
    float* r = a.r + (int64_t)h * a.ldn;
    const float* basis = a.basis + (int64_t)h * a.max_t * a.ldn;
    const int n4 = a.ldn / 4;

    // block sum of one float per thread (every thread gets it)
    auto block_sum = [&](float x) {
        x = warp_sum(x);
        __syncthreads();
        if (lane == 0) red_v[warp] = x;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kStepWarps; ++w) tot += red_v[w];
        return tot;
    };
    // sum over the cluster of one float per CTA: lane c of every warp reads
    // rank c's value (the remote loads overlap), then a fixed shuffle tree
    // adds them, the same tree in every CTA
    auto cluster_sum = [&](float mine) {
        if (tid == 0) part_s = mine;
        cluster.sync();
        float x = lane < CL ? *cluster.map_shared_rank(&part_s, lane) : 0.f;
        x = warp_sum(x);
        cluster.sync();                                // part_s may be rewritten after this
        return x;
    };

    // ---- the key
    int j;
    if (s < nf) {
        j = forced_at(s, a.T, a.keep_first, a.keep_last);
    } else {
        const int ksz = (a.T + CL - 1) / CL;
        const int k0 = min(a.T, rank * ksz), k1 = min(a.T, k0 + ksz);
        float bv = -INFINITY;
        int bi = INT32_MAX;
        for (int k = k0 + tid; k < k1; k += kStepThreads) {
            if (a.chosen[(int64_t)h * a.T + k]) continue;
            const float nk = a.norms[(int64_t)h * a.T + k];
            if (nk > 0.f) {
                float c = 0.f;                         // the correlation: its parts, in order
                for (int z = 0; z < a.nz; ++z) {
                    const float2 pz = a.cpart[((int64_t)z * gridDim.y + h) * a.T + k];
                    c += pz.x + pz.y;
                }
                better(bv, bi, c / nk, k);
            }
        }
        red_v[tid] = bv;
        red_i[tid] = bi;
        __syncthreads();
        for (int o = kStepThreads / 2; o > 0; o >>= 1) {
            if (tid < o && red_v[tid + o] > -INFINITY) {
                float v0 = red_v[tid];
                int i0 = red_i[tid];
                better(v0, i0, red_v[tid + o], red_i[tid + o]);
                red_v[tid] = v0;
                red_i[tid] = i0;
            }
            __syncthreads();
        }
        if (tid == 0) {
            part_v = red_v[0];
            part_i = red_i[0];
        }
        cluster.sync();
        // lane c reads rank c's candidate; the (largest, then lowest position)
        // rule does not depend on the order the candidates meet in
        float gv = -INFINITY;
        int gi = INT32_MAX;
        if (lane < CL) {
            gv = *cluster.map_shared_rank(&part_v, lane);
            gi = *cluster.map_shared_rank(&part_i, lane);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, gv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, gi, o);
            if (ov > -INFINITY) better(gv, gi, ov, oi);
        }
        if (!(gv > -INFINITY)) {
            // no candidate with a positive norm: the lowest position not chosen
            gi = 0;
            while (gi < a.T && a.chosen[(int64_t)h * a.T + gi]) ++gi;
        }
        j = gi;
        cluster.sync();                                // the partials are read; red_* may be reused
    }
    if (!KVC_IN_RANGE(j >= 0 && j < a.T, a.status, h)) return;
    const float pn = a.norms[(int64_t)h * a.T + j];
    if (rank == 0 && tid == 0) {
        a.chosen[(int64_t)h * a.T + j] = 1;
        a.order[(int64_t)h * a.max_t + s] = j;
        a.pnorm[h] = pn;
        a.pick[h] = j;
    }

    // ---- v = p_j on this CTA's queries: exp2(q . K_j c2 - lse2_q), 0 past n;
    // a warp takes 8 queries, and their rows are loaded before any is used
    {
        constexpr int E = D / 32;
        float kj[E];
#pragma unroll
        for (int e = 0; e < E; ++e) kj[e] = __bfloat162float(K[((int64_t)h * a.T + j) * D + lane * E + e]);
        for (int qb = q0 + warp * 8; qb < q1; qb += kStepWarps * 8) {
            float x[8][E];
            float lq[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = qb + u;
                const bool in = q < q1 && q < a.n;
                const __nv_bfloat16* qr = Q + ((int64_t)h * a.n + (in ? q : 0)) * D + lane * E;
#pragma unroll
                for (int e = 0; e < E; ++e) x[u][e] = in ? __bfloat162float(qr[e]) : 0.f;
                lq[u] = in ? lse2[(int64_t)h * a.n + q] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = qb + u;
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) dot = fmaf(x[u][e], kj[e], dot);
                dot = warp_sum(dot);
                if (lane == 0 && q < q1) v[q] = q < a.n ? exp2f(fmaf(dot, c2, -lq[u])) : 0.f;
            }
        }
    }
    cluster.sync();                                    // v complete

    // ---- classical Gram-Schmidt against the nb basis vectors
    float vv = 0.f;                                    // ||v||^2 after the last round
    for (int round = 0; round < 2; ++round) {
        // the whole of v in shared memory for the projections
        for (int c = tid; c < n4; c += kStepThreads) dyn4[c] = reinterpret_cast<const float4*>(v)[c];
        __syncthreads();
        // projections: warp (rank, warp) takes basis vectors rank * 32 + warp, step 32 CL;
        // eight 16-byte loads in flight per lane
        for (int k = rank * kStepWarps + warp; k < nb; k += kStepWarps * CL) {
            const float4* b4 = reinterpret_cast<const float4*>(basis + (int64_t)k * a.ldn);
            float d[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int c = lane; c < n4; c += 256) {
                float4 x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c + 32 * u < n4) x[u] = b4[c + 32 * u];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c + 32 * u < n4) {
                        const float4 y = dyn4[c + 32 * u];
                        d[u] = fmaf(x[u].x, y.x, fmaf(x[u].y, y.y, fmaf(x[u].z, y.z, fmaf(x[u].w, y.w, d[u]))));
                    }
            }
            const float dd = warp_sum(((d[0] + d[1]) + (d[2] + d[3])) + ((d[4] + d[5]) + (d[6] + d[7])));
            if (lane == 0) a.coef[(int64_t)h * a.max_t + k] = dd;
        }
        cluster.sync();                                // every coefficient written
        for (int k = tid; k < nb; k += kStepThreads) cf[k] = a.coef[(int64_t)h * a.max_t + k];
        __syncthreads();
        // subtraction on this CTA's queries: thread (kg, c) sums basis vectors
        // k = kg (mod 16) over query group c (four queries, one 16-byte load per
        // vector), and the sixteen k-groups meet in shared memory
        float ss = 0.f;
        const int kg = tid >> 6, c4l = tid & 63;
        const int nq4 = (q1 - q0) / 4;
        for (int base = 0; base < nq4; base += 64) {
            const int c4 = base + c4l;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c4 < nq4) {
                const float4* b4 = reinterpret_cast<const float4*>(basis + q0) + c4;
                int k = kg;
                for (; k + 7 * kStepKg < nb; k += 8 * kStepKg) {
                    float4 x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) x[u] = b4[(int64_t)(k + kStepKg * u) * n4];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float f = cf[k + kStepKg * u];
                        acc.x = fmaf(f, x[u].x, acc.x);
                        acc.y = fmaf(f, x[u].y, acc.y);
                        acc.z = fmaf(f, x[u].z, acc.z);
                        acc.w = fmaf(f, x[u].w, acc.w);
                    }
                }
                for (; k < nb; k += kStepKg) {
                    const float4 x = b4[(int64_t)k * n4];
                    const float f = cf[k];
                    acc.x = fmaf(f, x.x, acc.x);
                    acc.y = fmaf(f, x.y, acc.y);
                    acc.z = fmaf(f, x.z, acc.z);
                    acc.w = fmaf(f, x.w, acc.w);
                }
            }
            red4[kg][c4l] = acc;
            __syncthreads();
            if (kg == 0 && c4 < nq4) {
                float4 tot = red4[0][c4l];
#pragma unroll
                for (int g = 1; g < kStepKg; ++g) {
                    const float4 y = red4[g][c4l];
                    tot.x += y.x;
                    tot.y += y.y;
                    tot.z += y.z;
                    tot.w += y.w;
                }
                float4* vq = reinterpret_cast<float4*>(v + q0) + c4;
                float4 x = *vq;
                x.x -= tot.x;
                x.y -= tot.y;
                x.z -= tot.z;
                x.w -= tot.w;
                *vq = x;
                ss = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, ss))));
            }
            __syncthreads();
        }
        // the cluster sum orders the subtraction before the next round's reads of v
        vv = cluster_sum(block_sum(ss));
        // a second round only when the first removed more than half of
        // ||p_j||^2 (one round is then exact to rounding: "twice is enough")
        if (vv > 0.5f * pn * pn) break;
    }

    // ---- finish: a new basis vector unless v is (numerically) in the span
    const float vn = sqrtf(vv);
    if (!(vn > 1e-5f * pn) || nb >= a.max_t) return;  // the same decision in every CTA
    const float inv = 1.f / vn;
    float* bn = a.basis + ((int64_t)h * a.max_t + nb) * a.ldn;
    float dr = 0.f;
    for (int q = q0 + tid; q < q1; q += kStepThreads) {
        const float x = v[q] * inv;
        bn[q] = x;
        dr = fmaf(x, r[q], dr);
    }
    const float alpha = cluster_sum(block_sum(dr));
    for (int q = q0 + tid; q < q1; q += kStepThreads) r[q] = fmaf(-alpha, bn[q], r[q]);
    if (rank == 0 && tid == 0) a.nbasis[h] = nb + 1;
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
// v -= sum_k c_k basis_k: a thread per query, the basis vectors in groups of
// eight independent loads.  grid (ceil(ldn / 128), H), block 128.
__global__ void __launch_bounds__(128) k_omp_sub(OmpArgs a, int s) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    const int t = a.offsets[h + 1] - a.offsets[h];
    if (s >= t) return;
    extern __shared__ float cf[];
    const int nb = a.nbasis[h];
    for (int k = threadIdx.x; k < nb; k += 128) cf[k] = a.coef[(int64_t)h * a.max_t + k];
    __syncthreads();
    const int q = blockIdx.x * 128 + threadIdx.x;
    if (q >= a.ldn) return;
    const float* b = a.basis + (int64_t)h * a.max_t * a.ldn + q;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int k = 0;
    for (; k + 8 <= nb; k += 8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = b[(int64_t)(k + u) * a.ldn];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u & 3] = fmaf(cf[k + u], x[u], acc[u & 3]);
    }
    for (; k < nb; ++k) acc[0] = fmaf(cf[k], b[(int64_t)k * a.ldn], acc[0]);
    a.v[(int64_t)h * a.ldn + q] -= (acc[0] + acc[1]) + (acc[2] + acc[3]);
}
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
// Parts the queries of a correlation pass are split into: only a pass with
// fewer CTAs than the GPU's 148 SMs is split (at most 8 parts, at most one
// per 256-query block); a split pass repeats each CTA's set-up and the
// parts' sum, which costs more than a partly filled second wave.
int omp_corr_split(int H, int n, int T) {
    const int ctas = (T + 255) / 256 * H;
    if (ctas >= 148) return 1;
    const int want = (148 + ctas - 1) / ctas;
    return std::max(1, std::min(std::min(8, want), (n + 255) / 256));
}
size_t al256(size_t b) { return (b + 255) / 256 * 256; }
// Bytes of the dictionary region: P for fp32 inputs; for bf16 the key scores
// and the parts of the correlations.
size_t omp_dict_bytes(int dtype, int H, int n, int T, size_t ldn) {
    return dtype == KVC_DTYPE_F32 ? (size_t)H * T * ldn * 4
                                  : al256((size_t)H * T * 4) + (size_t)omp_corr_split(H, n, T) * H * T * 8;
}
}  // namespace

// Workspace of the pursuit for a problem (bytes, 256-aligned pieces).
size_t omp_workspace_bytes(int dtype, int H, int n, int T, int max_t) {
    const size_t ldn = (size_t)round_up(n, 4);
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    return al(omp_dict_bytes(dtype, H, n, T, ldn)) + al((size_t)H * T * 4) + al((size_t)H * T) +
           2 * al((size_t)H * ldn * 4) + al((size_t)H * max_t * ldn * 4) + al((size_t)H * max_t * 4) +
           al((size_t)H * 4) + al((size_t)H * ((T + 7) / 8) * 8) + al((size_t)H * max_t * 4) + al((size_t)H * 4) +
           al((size_t)H * 4);
}

// Byte offset of the selection order [H][max_t] inside that workspace.
size_t omp_order_offset(int dtype, int H, int n, int T, int max_t) {
    const size_t ldn = (size_t)round_up(n, 4);
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    return al(omp_dict_bytes(dtype, H, n, T, ldn)) + al((size_t)H * T * 4) + al((size_t)H * T) +
           2 * al((size_t)H * ldn * 4) + al((size_t)H * max_t * ldn * 4) + al((size_t)H * max_t * 4) +
           al((size_t)H * 4) + al((size_t)H * ((T + 7) / 8) * 8);
}

// Launches of launch_omp_select; nf forced positions need no correlations.
int omp_launches(int dtype, int max_t, int nf) {
    return dtype == KVC_DTYPE_F32 ? 3 + 7 * max_t : 3 + max_t + std::max(0, max_t - nf);
}

cudaError_t launch_colscore_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T,
                               float c2, float* score, int32_t* status, int qdiv, long long wait_limit,
                               const float* bias2, cudaStream_t st);
cudaError_t launch_corr_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T, float c2,
                           const float* r, int64_t rstride, float2* part, int nz, int32_t* status,
                           long long wait_limit, cudaStream_t st);

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
    a.nz = rec ? omp_corr_split(H, n, T) : 0;
    a.cpart = rec ? (float2*)(p + al((size_t)H * T * 4)) : nullptr;
    p += al(omp_dict_bytes(dtype, H, n, T, (size_t)ldn));
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
    if (rec) {
        // bf16: per step the correlations on the tensor cores, then one fused
        // launch (a cluster per head) for the rest of the step
        auto step = d == 128 ? k_omp_step<128> : k_omp_step<64>;
        const size_t step_smem = omp_step_smem(max_t, ldn);
        if (step_smem > 16 * 1024) {
            e = cudaFuncSetAttribute(step, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)step_smem);
            if (e != cudaSuccess) return e;
        }
        e = cudaFuncSetAttribute(step, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.blockDim = dim3(kStepThreads);
        cfg.dynamicSmemBytes = step_smem;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;                                  // the occupancy query sees the cluster alone
        // a cluster of 16 CTAs per head where one can be placed, else 8
        int cl = 16, nclusters = 0;
        attr[0].val.clusterDim.x = cl;
        cfg.gridDim = dim3(cl, H);
        if (cudaOccupancyMaxActiveClusters(&nclusters, step, &cfg) != cudaSuccess || nclusters < 1) {
            (void)cudaGetLastError();
            cl = 8;
            attr[0].val.clusterDim.x = cl;
            cfg.gridDim = dim3(cl, H);
        }
        cfg.numAttrs = 2;                                  // steps launched dependent on their predecessor
        const __nv_bfloat16* Qb = (const __nv_bfloat16*)Q;
        const __nv_bfloat16* Kb = (const __nv_bfloat16*)K;
        for (int s = 0; s < max_t; ++s) {
            if (s >= nf) {
                e = launch_corr_tc(d, Q, K, lse2, H, n, T, c2, a.r, ldn, a.cpart, a.nz, status, wait_limit, st);
                if (e != cudaSuccess) return e;
            }
            e = cudaLaunchKernelEx(&cfg, step, a, s, Qb, Kb, lse2, c2);
            if (e != cudaSuccess) return e;
        }
        k_omp_idx<<<H, 1024, 0, st>>>(a, idx_out);
        return cudaGetLastError();
    }
    for (int s = 0; s < max_t; ++s) {
        k_omp_corr<<<dim3(nparts, H), 256, 0, st>>>(a, s);
        k_omp_pick<<<H, 256, 0, st>>>(a, s, nparts);
        for (int round = 0; round < 2; ++round) {
            // the basis holds at most s vectors before step s
            k_omp_proj<<<dim3(std::max(1, (s + 7) / 8), H), 256, 0, st>>>(a, s);
            k_omp_sub<<<dim3((ldn + 127) / 128, H), 128, sub_smem, st>>>(a, s);
        }
        k_omp_finish<<<H, 256, 0, st>>>(a, s);
    }
    k_omp_idx<<<H, 1024, 0, st>>>(a, idx_out);
    return cudaGetLastError();
}

}  // namespace kvc
