// Budget validation, per-head top-t selection by radix select, and the gather
// of the kept keys/values ("Fast KV Compaction via Attention Matching",
// section 2, key selection: the original keys with the highest attention
// over the reference queries; kept entries are stored contiguously in
// ascending position order).
#include "common.cuh"

namespace kvc {

// Forced positions of head h.  When a KV head's cache is split into `chunks`
// contiguous chunks of T positions each (heads h = head * chunks + c), the
// caller's keep_first / keep_last count positions of the whole cache: chunk c
// keeps [0, kf) and [T - kl, T) with kf, kl the parts of those ranges that
// fall inside it.  chunks = 1 is the unchunked cache.
struct ForcedRange {
    int kf, kl;
};
__device__ __forceinline__ ForcedRange forced_range(int h, int T, int chunks, int keep_first, int keep_last) {
    const int c = h % chunks;
    const int64_t kf = (int64_t)keep_first - (int64_t)c * T;
    const int64_t kl = (int64_t)keep_last - (int64_t)(chunks - 1 - c) * T;
    return ForcedRange{(int)max((int64_t)0, min((int64_t)T, kf)), (int)max((int64_t)0, min((int64_t)T, kl))};
}

// ---------------------------------------------------------------- validate
// grid ceil(H/256), block 256.  head_status[h] = OK or BAD_BUDGET.
__global__ void k_validate(const int32_t* __restrict__ budgets, const int32_t* __restrict__ offsets, int H, int T,
                           int max_t, int chunks, int keep_first, int keep_last, int32_t* __restrict__ status,
                           HeadScalars* __restrict__ hs) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    const ForcedRange fr = forced_range(h, T, chunks, keep_first, keep_last);
    const int forced = min(T, fr.kf + fr.kl);
    const int t = budgets[h];
    bool ok = t >= 1 && t <= T && t <= max_t && t >= forced;
    ok = ok && offsets[h + 1] - offsets[h] == t;
    // per-head workspace rows are indexed by offsets: keep them inside H*max_t
    ok = ok && offsets[h] >= 0 && (int64_t)offsets[h + 1] <= (int64_t)H * max_t;
    if (h == 0) ok = ok && offsets[0] == 0;
    status[h] = ok ? KVC_OK : KVC_ERR_BAD_BUDGET;
    hs[h] = HeadScalars{};
}

// ---------------------------------------------------------------- block scan
// Exclusive scan of one int per thread over a 1024-thread block; returns the
// exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* sbuf, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sbuf[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? sbuf[lane] : 0;
        int z = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, z, o);
            if (lane >= o) z += y;
        }
        sbuf[lane] = z - w;          // exclusive warp offsets
        if (lane == 31) sbuf[32] = z;
    }
    __syncthreads();
    int res = sbuf[wid] + x - v;
    *total = sbuf[32];
    __syncthreads();
    return res;
}

// Monotone uint32 key of a non-negative float score; +inf marks a forced key.
__device__ __forceinline__ uint32_t score_bits(float v) { return __float_as_uint(v) & 0x7fffffffu; }
constexpr uint32_t kForcedKey = 0x7f800000u;

// The `keep` largest keys of positions [lo, hi) (key(j) as above), written
// ascending to out[0 .. keep).  The keep-th largest key is found by four 8-bit
// radix passes over the key bits; ties at the threshold go to the lowest
// positions.  Block-wide (1024 threads); returns false if a key is NaN.
template <typename KeyFn>
__device__ bool radix_select_range(KeyFn key, int lo, int hi, int keep, int32_t* __restrict__ out, int* hist,
                                   int* sbuf) {
    __shared__ uint32_t s_digit;
    __shared__ int s_krem, s_nan;
    if (threadIdx.x == 0) {
        s_krem = keep;
        s_nan = 0;
    }
    uint32_t prefix = 0, pmask = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int j = lo + threadIdx.x; j < hi; j += blockDim.x) {
            const uint32_t k = key(j);
            if (shift == 24 && k > kForcedKey) s_nan = 1;
            if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // the highest digit whose keys (with all higher ones) reach s_krem:
            // lane l sums bins 255 - 8 l .. 248 - 8 l, a warp scan finds the
            // lane, and that lane walks its eight bins
            const int lane = threadIdx.x;
            const int kr = s_krem;
            int c[8], sum = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                c[u] = hist[255 - (lane * 8 + u)];
                sum += c[u];
            }
            int inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, inc >= kr);
            const int L = hit ? __ffs(hit) - 1 : -1;
            if (lane == L) {
                int cum = inc - sum;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (cum + c[u] >= kr) {
                        s_digit = (uint32_t)(255 - (lane * 8 + u));
                        s_krem = kr - cum;
                        break;
                    }
                    cum += c[u];
                }
            } else if (L < 0 && lane == 0) {
                s_digit = 0;                     // unreachable for a valid budget
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        pmask |= 255u << shift;
    }
    if (s_nan) return false;
    const uint32_t tau = prefix;
    const int krem = s_krem;                 // keys equal to tau still to take
    const int len = hi - lo;
    const int chunk = (len + blockDim.x - 1) / blockDim.x;
    const int j0 = lo + min(len, (int)threadIdx.x * chunk), j1 = min(hi, j0 + chunk);
    int gt = 0, eq = 0;
    for (int j = j0; j < j1; ++j) {
        const uint32_t k = key(j);
        gt += k > tau;
        eq += k == tau;
    }
    int tot;
    const int eq_before = block_exclusive_scan(eq, sbuf, &tot);
    const int take_eq = max(0, min(eq, krem - eq_before));
    const int pos0 = block_exclusive_scan(gt + take_eq, sbuf, &tot);
    int pos = pos0, er = eq_before;
    for (int j = j0; j < j1; ++j) {
        const uint32_t k = key(j);
        bool take = k > tau;
        if (k == tau) {
            take = er < krem;
            ++er;
        }
        if (take) out[pos++] = j;
    }
    return true;
}

// ---------------------------------------------------------------- select
// grid H, block 1024.  idx_out[off .. off+t) = kept positions, ascending.
__global__ void __launch_bounds__(1024) k_select(const float* __restrict__ score, int T, const int32_t* __restrict__ offsets,
                                                 int chunks, int keep_first, int keep_last,
                                                 int32_t* __restrict__ idx_out, int32_t* __restrict__ status) {
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    const ForcedRange fr = forced_range(h, T, chunks, keep_first, keep_last);
    __shared__ int hist[256];
    __shared__ int sbuf[33];
    const float* sc = score + (int64_t)h * T;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    auto key = [&](int j) -> uint32_t {
        return (j < fr.kf || j >= T - fr.kl) ? kForcedKey : score_bits(sc[j]);
    };
    if (!radix_select_range(key, 0, T, t, idx_out + off, hist, sbuf) && threadIdx.x == 0)
        set_status(status, h, KVC_ERR_NONFINITE);
}

// grid (segments, H), block 1024.  Segment i = positions [bounds[i],
// bounds[i+1]) keeps its pivots (pivot[h][j] != 0) and its seg_keep[h][i] -
// pivots highest-scoring other keys, written ascending at
// idx_out[off + seg_off[h][i] ..]; segments are contiguous, so the head's
// list is ascending.
__global__ void __launch_bounds__(1024) k_select_seg(const float* __restrict__ score, int T,
                                                     const int32_t* __restrict__ offsets,
                                                     const int32_t* __restrict__ bounds, int nseg,
                                                     const uint8_t* __restrict__ pivot,
                                                     const int32_t* __restrict__ seg_keep,
                                                     const int32_t* __restrict__ seg_off,
                                                     int32_t* __restrict__ idx_out, int32_t* __restrict__ status) {
    const int h = blockIdx.y, i = blockIdx.x;
    if (!head_ok(status, h)) return;
    __shared__ int hist[256];
    __shared__ int sbuf[33];
    const float* sc = score + (int64_t)h * T;
    const uint8_t* pv = pivot + (int64_t)h * T;
    const int keep = seg_keep[(int64_t)h * nseg + i];
    if (keep == 0) return;
    auto key = [&](int j) -> uint32_t { return pv[j] ? kForcedKey : score_bits(sc[j]); };
    if (!radix_select_range(key, bounds[i], bounds[i + 1], keep, idx_out + offsets[h] + seg_off[(int64_t)h * nseg + i],
                            hist, sbuf) &&
        threadIdx.x == 0)
        set_status(status, h, KVC_ERR_NONFINITE);
}

// ---------------------------------------------------------------- gather
// grid (ceil(max_t/8), H), block 256 (one warp per kept row).
// C_k[off+i] = K[h][idx[off+i]] (storage dtype, 16-byte vectors) and
// Vsel[off+i] = fp32(V[h][idx[off+i]]) (V in the storage dtype, or fp32 for
// the values of a compacted cache).  When Ckw is given, the kept keys are
// also copied to Ckw[h][i] (rows padded per head to ldw), the layout the
// tensor-core mass pass reads through TMA.  When bias2 is given (keys with
// input biases, [H][Tb] log2 units), bk[off+i] = bias2[h][idx[off+i]].
template <typename TIn, typename TV, int D>
__global__ void __launch_bounds__(256) k_gather(const TIn* __restrict__ K, const TV* __restrict__ V, int T,
                                                const int32_t* __restrict__ offsets, const int32_t* __restrict__ idx,
                                                TIn* __restrict__ Ck, float* __restrict__ Vsel,
                                                TIn* __restrict__ Ckw, int64_t ldw,
                                                const int32_t* __restrict__ status, const float* __restrict__ bias2,
                                                int64_t Tb, float* __restrict__ bk) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (i >= t) return;
    const int j = idx[off + i];
    if (!KVC_IN_RANGE(j >= 0 && j < T, status, h)) return;
    constexpr int VEC = 16 / sizeof(TIn);          // elements per 16-byte vector
    constexpr int NV = D / VEC;
    const uint4* src = reinterpret_cast<const uint4*>(K + ((int64_t)h * T + j) * D);
    uint4* dst = reinterpret_cast<uint4*>(Ck + ((int64_t)off + i) * D);
    uint4* dw = Ckw ? reinterpret_cast<uint4*>(Ckw + ((int64_t)h * ldw + i) * D) : nullptr;
    for (int v = lane; v < NV; v += 32) {
        const uint4 x = src[v];
        dst[v] = x;
        if (dw) dw[v] = x;
    }
    const TV* vr = V + ((int64_t)h * T + j) * D;
    float* vo = Vsel + ((int64_t)off + i) * D;
    for (int c = lane; c < D; c += 32) vo[c] = to_f32(vr[c]);
    if (bias2 && lane == 0) bk[off + i] = bias2[(int64_t)h * Tb + j];
}

// ---------------------------------------------------------------- chunk shift
// grid (ceil(max_t/256), H), block 256.  Chunk c = h % chunks of a cache
// split into chunks of T positions: idx[off .. off+t) += c * T, turning
// positions inside the chunk into positions in the whole cache.
__global__ void k_shift_idx(int32_t* __restrict__ idx, const int32_t* __restrict__ offsets, int T, int chunks,
                            const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < t) idx[off + i] += (h % chunks) * T;
}

cudaError_t launch_validate(const int32_t* budgets, const int32_t* offsets, int H, int T, int max_t, int chunks,
                            int keep_first, int keep_last, int32_t* status, HeadScalars* hs, cudaStream_t st) {
    k_validate<<<(H + 255) / 256, 256, 0, st>>>(budgets, offsets, H, T, max_t, chunks, keep_first, keep_last, status,
                                                hs);
    return cudaGetLastError();
}
cudaError_t launch_select(const float* score, int H, int T, const int32_t* offsets, int chunks, int keep_first,
                          int keep_last, int32_t* idx_out, int32_t* status, cudaStream_t st) {
    k_select<<<H, 1024, 0, st>>>(score, T, offsets, chunks, keep_first, keep_last, idx_out, status);
    return cudaGetLastError();
}
cudaError_t launch_select_seg(const float* score, int H, int T, const int32_t* offsets, const int32_t* bounds,
                              int nseg, const uint8_t* pivot, const int32_t* seg_keep, const int32_t* seg_off,
                              int32_t* idx_out, int32_t* status, cudaStream_t st) {
    k_select_seg<<<dim3(nseg, H), 1024, 0, st>>>(score, T, offsets, bounds, nseg, pivot, seg_keep, seg_off, idx_out,
                                                 status);
    return cudaGetLastError();
}
cudaError_t launch_shift_idx(int32_t* idx, const int32_t* offsets, int H, int T, int max_t, int chunks,
                             const int32_t* status, cudaStream_t st) {
    k_shift_idx<<<dim3((max_t + 255) / 256, H), 256, 0, st>>>(idx, offsets, T, chunks, status);
    return cudaGetLastError();
}
template <typename TIn, typename TV, int D>
static cudaError_t launch_gather_t(const void* K, const void* V, int H, int T, int max_t, const int32_t* offsets,
                                   const int32_t* idx, void* Ck, float* Vsel, void* Ckw, int64_t ldw,
                                   const int32_t* status, const float* bias2, int64_t Tb, float* bk,
                                   cudaStream_t st) {
    dim3 grid((max_t + 7) / 8, H);
    k_gather<TIn, TV, D><<<grid, 256, 0, st>>>((const TIn*)K, (const TV*)V, T, offsets, idx, (TIn*)Ck, Vsel,
                                               (TIn*)Ckw, ldw, status, bias2, Tb, bk);
    return cudaGetLastError();
}
template <typename TIn>
static cudaError_t launch_gather_k(int d, bool v_f32, const void* K, const void* V, int H, int T, int max_t,
                                   const int32_t* offsets, const int32_t* idx, void* Ck, float* Vsel, void* Ckw,
                                   int64_t ldw, const int32_t* status, const float* bias2, int64_t Tb, float* bk,
                                   cudaStream_t st) {
    if (v_f32)
        return d == 128 ? launch_gather_t<TIn, float, 128>(K, V, H, T, max_t, offsets, idx, Ck, Vsel, Ckw, ldw, status,
                                                           bias2, Tb, bk, st)
                        : launch_gather_t<TIn, float, 64>(K, V, H, T, max_t, offsets, idx, Ck, Vsel, Ckw, ldw, status,
                                                          bias2, Tb, bk, st);
    return d == 128 ? launch_gather_t<TIn, TIn, 128>(K, V, H, T, max_t, offsets, idx, Ck, Vsel, Ckw, ldw, status,
                                                     bias2, Tb, bk, st)
                    : launch_gather_t<TIn, TIn, 64>(K, V, H, T, max_t, offsets, idx, Ck, Vsel, Ckw, ldw, status,
                                                    bias2, Tb, bk, st);
}
// v_f32: V is fp32 whatever the keys' dtype; bias2 / bk: optional key biases.
cudaError_t launch_gather(int dtype, int d, const void* K, const void* V, bool v_f32, int H, int T, int max_t,
                          const int32_t* offsets, const int32_t* idx, void* Ck, float* Vsel, void* Ckw, int64_t ldw,
                          const int32_t* status, const float* bias2, int64_t Tb, float* bk, cudaStream_t st) {
    if (dtype == KVC_DTYPE_BF16)
        return launch_gather_k<__nv_bfloat16>(d, v_f32, K, V, H, T, max_t, offsets, idx, Ck, Vsel, Ckw, ldw, status,
                                              bias2, Tb, bk, st);
    return launch_gather_k<float>(d, true, K, V, H, T, max_t, offsets, idx, Ck, Vsel, nullptr, 0, status, bias2, Tb,
                                  bk, st);
}

}  // namespace kvc
