// Thought-aware compaction on top of the Attention Matching pipeline
// ("Thought-Aware KV Cache Compaction" explainer, section 2: B adaptive
// budget allocation, C pivot-token protection):
//   k_tam_plan      per head: alpha_j (the mean attention key j receives from
//                   the window queries) against delta = c * mean alpha marks
//                   the pivots; segment i gets t_i ~ sqrt(w_i) n_i of the
//                   budget left after the pivots (w_i = sum of alpha over the
//                   segment, n_i its non-pivot count), capped at n_i with the
//                   excess re-shared, made integral by largest remainder
//                   (ties to the lower segment); all in double
//   k_tam_kept      which kept rows are pivots
//   k_tam_rhs_g / k_tam_rhs_m   move the pivots' contribution to the right-
//                   hand sides: f_i -= sum_p G_ip (w_p = 1), R_i -= sum_p
//                   M_ip V_p (C_v,p = V_p); pivot rows get f_p = 1, R_p = V_p
//   k_tam_pin       pivot rows and columns of G / M become the identity, so
//                   the solves return w_p = 1 (beta = 0) and C_v,p = V_p exactly
// The ridges keep their definitions over all t kept keys (they are added
// before the fix).  Segment boundaries are shared by every head.
#include "common.cuh"

namespace kvc {

namespace {

constexpr int kMaxSeg = 1024;

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block sums in a fixed order (1024 threads): every thread gets the total.
__device__ double block_sum_d(double v, double* red) {
    v = warp_sum_d(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    double tot = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    __syncthreads();
    return tot;
}
__device__ int block_sum_i(int v, int* red) {
    v = warp_sum_i(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    __syncthreads();
    return tot;
}

// grid H, block 1024.
__global__ void __launch_bounds__(1024) k_tam_plan(const float* __restrict__ alpha, int T,
                                                   const int32_t* __restrict__ bounds, int S, double c,
                                                   const int32_t* __restrict__ offsets, uint8_t* __restrict__ pivot,
                                                   int32_t* __restrict__ seg_bud, int32_t* __restrict__ seg_keep,
                                                   int32_t* __restrict__ seg_off, int32_t* __restrict__ status) {
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    __shared__ double w[kMaxSeg], x[kMaxSeg], sh[kMaxSeg];
    __shared__ int pc[kMaxSeg], nz[kMaxSeg], base[kMaxSeg];
    __shared__ uint8_t capped[kMaxSeg], inc[kMaxSeg];
    __shared__ double redd[32];
    __shared__ int redi[32];
    __shared__ int s_any;
    const int t = offsets[h + 1] - offsets[h];
    const float* al = alpha + (int64_t)h * T;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the bounds index every later access: 0 = b_0 < b_1 < ... < b_S = T
    int bad = 0;
    for (int i = threadIdx.x; i < S; i += blockDim.x) bad |= !(bounds[i] < bounds[i + 1]);
    if (threadIdx.x == 0) bad |= (bounds[0] != 0) | (bounds[S] != T);
    if (block_sum_i(bad, redi) != 0) {
        if (threadIdx.x == 0) set_status(status, h, KVC_ERR_BAD_BUDGET);
        return;
    }
    // threshold
    double s = 0.0;
    for (int j = threadIdx.x; j < T; j += blockDim.x) s += (double)al[j];
    const double delta = c * (block_sum_d(s, redd) / (double)T);
    // pivots and per-segment statistics, a warp per segment (fixed order)
    for (int i = warp; i < S; i += 32) {
        const int lo = bounds[i], hi = bounds[i + 1];
        double ws = 0.0;
        int p = 0;
        for (int j = lo + lane; j < hi; j += 32) {
            const float a = al[j];
            const bool pv = (double)a > delta;
            pivot[(int64_t)h * T + j] = pv ? 1 : 0;
            p += pv;
            ws += (double)a;
        }
        ws = warp_sum_d(ws);
        p = warp_sum_i(p);
        if (lane == 0) {
            w[i] = ws;
            pc[i] = p;
            nz[i] = (hi - lo) - p;
        }
    }
    __syncthreads();
    int np = 0;
    for (int i = threadIdx.x; i < S; i += blockDim.x) np += pc[i];
    const int npiv = block_sum_i(np, redi);
    if (npiv > t) {
        if (threadIdx.x == 0) set_status(status, h, KVC_ERR_BAD_BUDGET);
        return;
    }
    const int left = t - npiv;
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        sh[i] = sqrt(fmax(w[i], 0.0)) * (double)nz[i];
        capped[i] = 0;
        x[i] = 0.0;
    }
    __syncthreads();
    // water-filling: shares of what the capped segments leave
    for (int iter = 0; iter <= S; ++iter) {
        double tot = 0.0, capsum = 0.0;
        for (int i = threadIdx.x; i < S; i += blockDim.x) {
            if (capped[i]) capsum += (double)nz[i];
            else if (sh[i] > 0.0) tot += sh[i];
        }
        tot = block_sum_d(tot, redd);
        const double rem = (double)left - block_sum_d(capsum, redd);
        if (threadIdx.x == 0) s_any = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < S; i += blockDim.x)
            if (!capped[i] && sh[i] > 0.0) {
                x[i] = tot > 0.0 ? rem * sh[i] / tot : 0.0;
                if (x[i] > (double)nz[i]) s_any = 1;
            }
        __syncthreads();
        if (!s_any) break;
        for (int i = threadIdx.x; i < S; i += blockDim.x)
            if (!capped[i] && sh[i] > 0.0 && x[i] > (double)nz[i]) {
                x[i] = (double)nz[i];
                capped[i] = 1;
            }
        __syncthreads();
    }
    // integral: floors, then the largest remainders (ties to the lower segment)
    int bs = 0;
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        base[i] = min((int)floor(x[i] + 1e-12), nz[i]);
        bs += base[i];
    }
    const int shortage = left - block_sum_i(bs, redi);
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        inc[i] = 0;
        if (base[i] >= nz[i]) continue;
        const double fi = x[i] - (double)base[i];
        int rank = 0;
        for (int k = 0; k < S; ++k) {
            if (k == i || base[k] >= nz[k]) continue;
            const double fk = x[k] - (double)base[k];
            rank += (fk > fi) || (fk == fi && k < i);
        }
        if (rank < shortage) inc[i] = 1;         // applied once every rank is known
    }
    __syncthreads();
    for (int i = threadIdx.x; i < S; i += blockDim.x) base[i] += inc[i];
    __syncthreads();
    if (threadIdx.x == 0) {
        int tot = 0;
        for (int i = 0; i < S; ++i) tot += base[i];
        int rest = left - tot;                   // only when every share was 0: fill in order
        for (int i = 0; i < S && rest > 0; ++i) {
            const int add = min(rest, nz[i] - base[i]);
            base[i] += add;
            rest -= add;
        }
        int o = 0;
        for (int i = 0; i < S; ++i) {
            seg_bud[(int64_t)h * S + i] = base[i];
            seg_keep[(int64_t)h * S + i] = base[i] + pc[i];
            seg_off[(int64_t)h * S + i] = o;
            o += base[i] + pc[i];
        }
    }
}

// grid H, block 1024: kp[off + i] = pivot[h][idx[off + i]], and the kept
// rows that are pivots listed in ascending order: plist[off ..], count npk[h].
__global__ void __launch_bounds__(1024) k_tam_kept(const uint8_t* __restrict__ pivot, int T,
                                                   const int32_t* __restrict__ idx,
                                                   const int32_t* __restrict__ offsets, uint8_t* __restrict__ kp,
                                                   int32_t* __restrict__ plist, int32_t* __restrict__ npk,
                                                   const int32_t* __restrict__ status) {
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    __shared__ int wsum[32];
    __shared__ int base;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) base = 0;
    __syncthreads();
    for (int i0 = 0; i0 < t; i0 += 1024) {
        const int i = i0 + threadIdx.x;
        const int f = (i < t) ? pivot[(int64_t)h * T + idx[off + i]] : 0;
        if (i < t) kp[off + i] = (uint8_t)f;
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (lane == 0) wsum[warp] = __popc(m);
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        if (f) plist[off + base + before + __popc(m & ((1u << lane) - 1u))] = i;
        __syncthreads();
        if (threadIdx.x == 0) {
            int tot = 0;
            for (int w = 0; w < 32; ++w) tot += wsum[w];
            base += tot;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) npk[h] = base;
}

// grid (ceil(max_t/256), H), block 256: f_i -= sum_p G_ip over the kept pivots p; f_p = 1.
__global__ void k_tam_rhs_g(const float* __restrict__ G, int64_t ldA, float* __restrict__ f,
                            const uint8_t* __restrict__ kp, const int32_t* __restrict__ plist,
                            const int32_t* __restrict__ npk, const int32_t* __restrict__ offsets,
                            const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= t) return;
    if (kp[off + i]) {
        f[off + i] = 1.f;
        return;
    }
    const float* row = G + ((int64_t)h * ldA + i) * ldA;
    double acc = 0.0;
    for (int k = 0; k < npk[h]; ++k) acc += (double)row[plist[off + k]];
    f[off + i] -= (float)acc;
}

// grid (max_t, H), block d: row i of R: pivot rows R_p = V_p, others
// R_i -= sum_p M_ip V_p over the kept pivots p.
__global__ void k_tam_rhs_m(const float* __restrict__ M, int64_t ldA, float* __restrict__ R,
                            const float* __restrict__ Vsel, int d, const uint8_t* __restrict__ kp,
                            const int32_t* __restrict__ plist, const int32_t* __restrict__ npk,
                            const int32_t* __restrict__ offsets, const int32_t* __restrict__ status) {
    const int h = blockIdx.y, i = blockIdx.x;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    if (i >= t) return;
    const int c = threadIdx.x;
    if (kp[off + i]) {
        R[((int64_t)off + i) * d + c] = Vsel[((int64_t)off + i) * d + c];
        return;
    }
    const float* row = M + ((int64_t)h * ldA + i) * ldA;
    float acc = 0.f;
    for (int k = 0; k < npk[h]; ++k) {
        const int p = plist[off + k];
        acc = fmaf(row[p], Vsel[((int64_t)off + p) * d + c], acc);
    }
    R[((int64_t)off + i) * d + c] -= acc;
}

// grid (ceil(max_t/256), H), block 256: pivot rows and columns -> identity.
__global__ void k_tam_pin(float* __restrict__ A, int64_t ldA, const uint8_t* __restrict__ kp,
                          const int32_t* __restrict__ plist, const int32_t* __restrict__ npk,
                          const int32_t* __restrict__ offsets, const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= t) return;
    float* row = A + ((int64_t)h * ldA + i) * ldA;
    if (kp[off + i]) {
        for (int j = 0; j < t; ++j) row[j] = (j == i) ? 1.f : 0.f;
    } else {
        for (int k = 0; k < npk[h]; ++k) row[plist[off + k]] = 0.f;
    }
}

}  // namespace

int tam_max_segments() { return kMaxSeg; }

cudaError_t launch_tam_plan(const float* alpha, int H, int T, const int32_t* bounds, int S, double c,
                            const int32_t* offsets, uint8_t* pivot, int32_t* seg_bud, int32_t* seg_keep,
                            int32_t* seg_off, int32_t* status, cudaStream_t st) {
    k_tam_plan<<<H, 1024, 0, st>>>(alpha, T, bounds, S, c, offsets, pivot, seg_bud, seg_keep, seg_off, status);
    return cudaGetLastError();
}
// kp: uint8 [sum t]; plist: int32 [sum t] then npk: int32 [H] (one scratch block)
cudaError_t launch_tam_kept(const uint8_t* pivot, int H, int T, int max_t, const int32_t* idx,
                            const int32_t* offsets, uint8_t* kp, int32_t* plist, int32_t* npk,
                            const int32_t* status, cudaStream_t st) {
    (void)max_t;
    k_tam_kept<<<H, 1024, 0, st>>>(pivot, T, idx, offsets, kp, plist, npk, status);
    return cudaGetLastError();
}
// G, f after the ridge: pivots held at w = 1
cudaError_t launch_tam_fix_g(float* G, int64_t ldA, float* f, const uint8_t* kp, const int32_t* plist,
                             const int32_t* npk, const int32_t* offsets, int H, int max_t, const int32_t* status,
                             cudaStream_t st) {
    dim3 grid((max_t + 255) / 256, H);
    k_tam_rhs_g<<<grid, 256, 0, st>>>(G, ldA, f, kp, plist, npk, offsets, status);
    k_tam_pin<<<grid, 256, 0, st>>>(G, ldA, kp, plist, npk, offsets, status);
    return cudaGetLastError();
}
// M, R after the ridge: pivot rows of C_v held at V
cudaError_t launch_tam_fix_m(float* M, int64_t ldA, float* R, const float* Vsel, int d, const uint8_t* kp,
                             const int32_t* plist, const int32_t* npk, const int32_t* offsets, int H, int max_t,
                             const int32_t* status, cudaStream_t st) {
    k_tam_rhs_m<<<dim3(max_t, H), d, 0, st>>>(M, ldA, R, Vsel, d, kp, plist, npk, offsets, status);
    k_tam_pin<<<dim3((max_t + 255) / 256, H), 256, 0, st>>>(M, ldA, kp, plist, npk, offsets, status);
    return cudaGetLastError();
}

}  // namespace kvc
