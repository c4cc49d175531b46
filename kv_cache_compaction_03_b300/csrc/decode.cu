// Decode-time read of a compacted cache ("Fast KV Compaction via Attention
// Matching", section 2 objective, and section 5 on serving a compacted cache
// with standard attention kernels: the per-key bias beta is added to the
// logits):
//   O[h][q] = softmax_i(Q[h][q] . C_k[i] * scale + beta[i]) C_v[i]
// over head h's rows [offsets[h], offsets[h+1]), for a few queries per head
// (decode: one new token per query head of a GQA group).
//
// With few queries the work of a head is a stream over its keys, so a head
// gets a cluster of CTAs that split its keys into contiguous ranges: 8 when
// there are fewer heads than SMs, 4 otherwise (with many heads the grid is
// already several waves deep, and fewer, longer ranges per head pipeline
// better and merge less: 80 against 102 us for 256 heads of 655 keys).
// Every CTA streams its range in tiles of 32 keys (cp.async, two stages:
// the shared memory stays small enough for three CTAs per SM, whose
// interleaving hides more latency than deeper stages of one CTA would),
// keeps an online softmax per query, and leaves its partial (max, sum,
// unnormalised output) in shared memory; rank 0 of the cluster merges the
// partials through distributed shared memory and writes O.  Nothing goes
// through global scratch.
//   k_attend_decode   grid (CL, H) in clusters of (CL, 1, 1), block 128
// Logits are in log2 units (Q pre-scaled by scale * log2 e; beta * log2 e).
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace kvc {

namespace {

constexpr int kDecThreads = 128;
constexpr int kDecQ = 16;           // most queries per head this kernel takes
constexpr int kDecKT = 32;          // keys per tile
constexpr int kDecNS = 2;           // pipeline stages (tiles in flight: kDecNS - 1)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename TIn, int D>
struct DecSmem {
    static constexpr int KP = D + 16 / (int)sizeof(TIn);    // key row padded by 16 bytes
    float q[kDecQ][D];                   // queries x scale x log2 e
    TIn k[kDecNS][kDecKT][KP];
    float v[kDecNS][kDecKT][D];
    float b[kDecNS][kDecKT];             // bias x log2 e
    float s[kDecQ][kDecKT];              // logits, then probabilities
    float m[kDecQ], l[kDecQ], corr[kDecQ];
    float o[kDecQ][D];                   // this CTA's unnormalised partial output
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename TIn, int D, int kDecCluster>
__global__ void __launch_bounds__(kDecThreads, 3)
    k_attend_decode(const TIn* __restrict__ Q, int nq, const TIn* __restrict__ Ck, const float* __restrict__ beta,
                    const float* __restrict__ Cv, const int32_t* __restrict__ offsets, float c2,
                    float* __restrict__ O, int32_t* __restrict__ status) {
    using S = DecSmem<TIn, D>;
    extern __shared__ __align__(16) uint8_t dec_raw[];
    S& sm = *reinterpret_cast<S*>(dec_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int h = blockIdx.y;
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int off = offsets[h];
    const int th = offsets[h + 1] - off;
    // this CTA's keys [k_beg, k_end)
    const int kc = th > 0 ? (th + kDecCluster - 1) / kDecCluster : 0;
    const int k_beg = min(th > 0 ? th : 0, rank * kc), k_end = min(th > 0 ? th : 0, k_beg + kc);
    const int ntile = (k_end - k_beg + kDecKT - 1) / kDecKT;

    for (int e = tid; e < kDecQ * D; e += kDecThreads) {
        const int q = e / D, c = e % D;
        sm.q[q][c] = q < nq ? to_f(Q[((int64_t)h * nq + q) * D + c]) * c2 : 0.f;
    }
    if (tid < kDecQ) {
        sm.m[tid] = -INFINITY;
        sm.l[tid] = 0.f;
    }
    // one tile of keys / values / biases into stage `st`
    auto load_tile = [&](int it, int st) {
        const int k0 = k_beg + it * kDecKT;
        const int kv = min(kDecKT, k_end - k0);
        constexpr int KCH = D * (int)sizeof(TIn) / 16;      // 16-byte chunks per key row
        for (int e = tid; e < kDecKT * KCH; e += kDecThreads) {
            const int r = e / KCH, c = e % KCH;
            if (r < kv)
                cp_async16(reinterpret_cast<uint8_t*>(&sm.k[st][r][0]) + 16 * c,
                           reinterpret_cast<const uint8_t*>(Ck + ((int64_t)off + k0 + r) * D) + 16 * c);
        }
        constexpr int VCH = D / 4;
        for (int e = tid; e < kDecKT * VCH; e += kDecThreads) {
            const int r = e / VCH, c = e % VCH;
            if (r < kv) cp_async16(&sm.v[st][r][4 * c], Cv + ((int64_t)off + k0 + r) * D + 4 * c);
        }
        if (tid < kDecKT) sm.b[st][tid] = tid < kv ? beta[off + k0 + tid] * kLog2e : -INFINITY;
        cp_async_commit();
    };

    // output ownership: dims 4 dg .. 4 dg + 3 of queries qg + QG i
    constexpr int DG = D / 4;
    constexpr int QG = kDecThreads / DG;
    constexpr int QPT = kDecQ / QG;
    const int dg = tid % DG, qg = tid / DG;
    float acc[QPT][4];
#pragma unroll
    for (int i = 0; i < QPT; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;

    // prologue: tiles 0 .. NS-2 in flight (an empty group stands for a missing tile)
#pragma unroll
    for (int p = 0; p < kDecNS - 1; ++p) {
        if (p < ntile) load_tile(p, p);
        else cp_async_commit();
    }
    for (int it = 0; it < ntile; ++it) {
        const int st = it % kDecNS;
        const int kv = min(kDecKT, k_end - (k_beg + it * kDecKT));
        // refill the stage consumed in the previous iteration
        if (it + kDecNS - 1 < ntile) load_tile(it + kDecNS - 1, (it + kDecNS - 1) % kDecNS);
        else cp_async_commit();
        cp_async_wait<kDecNS - 1>();     // tile it has landed
        __syncthreads();
        // logits: key lane, queries warp + 4 i (element-wise key reads
        // measured faster here than 16-byte chunks unpacked per query)
        {
            const int k = lane;
#pragma unroll
            for (int i = 0; i < kDecQ / 4; ++i) {
                const int q = warp + 4 * i;
                if (q < nq) {
                    float dot = 0.f;
                    if (k < kv) {
#pragma unroll 8
                        for (int c = 0; c < D; c += 4) {
                            const float4 qq = *reinterpret_cast<const float4*>(&sm.q[q][c]);
                            dot = fmaf(qq.x, to_f(sm.k[st][k][c]), dot);
                            dot = fmaf(qq.y, to_f(sm.k[st][k][c + 1]), dot);
                            dot = fmaf(qq.z, to_f(sm.k[st][k][c + 2]), dot);
                            dot = fmaf(qq.w, to_f(sm.k[st][k][c + 3]), dot);
                        }
                    }
                    const float bb = sm.b[st][k];
                    sm.s[q][k] = (k < kv && bb != -INFINITY) ? dot + bb : -INFINITY;
                }
            }
        }
        __syncwarp();
        // online softmax: warp w owns queries w + 4 i (its own logits above)
#pragma unroll
        for (int i = 0; i < kDecQ / 4; ++i) {
            const int q = warp + 4 * i;
            if (q < nq) {
                const float x = sm.s[q][lane];
                const float mt = warp_max(x);
                const float mold = sm.m[q];
                const float mnew = fmaxf(mold, mt);
                const float mref = mnew == -INFINITY ? 0.f : mnew;
                const float p = x == -INFINITY ? 0.f : exp2f(x - mref);
                sm.s[q][lane] = p;
                const float ps = warp_sum(p);
                if (lane == 0) {
                    const float cr = mold == -INFINITY ? 0.f : exp2f(mold - mref);
                    sm.corr[q] = cr;
                    sm.l[q] = sm.l[q] * cr + ps;
                    sm.m[q] = mnew;
                }
            }
        }
        __syncthreads();
        // acc = acc * corr + P V (full tiles fully unrolled; even and odd keys
        // accumulate separately so that the FMA chains are independent)
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            const int q = qg + QG * i;
            if (q < nq) {
                const float cr = sm.corr[q];
                float a[2][4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    a[0][c] = acc[i][c] * cr;
                    a[1][c] = 0.f;
                }
                if (kv == kDecKT) {
#pragma unroll
                    for (int k = 0; k < kDecKT; ++k) {
                        const float p = sm.s[q][k];
                        const float4 vv = *reinterpret_cast<const float4*>(&sm.v[st][k][4 * dg]);
                        a[k & 1][0] = fmaf(p, vv.x, a[k & 1][0]);
                        a[k & 1][1] = fmaf(p, vv.y, a[k & 1][1]);
                        a[k & 1][2] = fmaf(p, vv.z, a[k & 1][2]);
                        a[k & 1][3] = fmaf(p, vv.w, a[k & 1][3]);
                    }
                } else {
                    for (int k = 0; k < kv; ++k) {
                        const float p = sm.s[q][k];
                        const float4 vv = *reinterpret_cast<const float4*>(&sm.v[st][k][4 * dg]);
                        a[0][0] = fmaf(p, vv.x, a[0][0]);
                        a[0][1] = fmaf(p, vv.y, a[0][1]);
                        a[0][2] = fmaf(p, vv.z, a[0][2]);
                        a[0][3] = fmaf(p, vv.w, a[0][3]);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[i][c] = a[0][c] + a[1][c];
            }
        }
        __syncthreads();     // stage st is refilled by a later iteration
    }
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
        const int q = qg + QG * i;
        *reinterpret_cast<float4*>(&sm.o[q][4 * dg]) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
    // every CTA of the cluster has its partial in shared memory
    cluster.sync();
    if (rank == 0) {
        if (th <= 0) {
            if (tid == 0) set_status(status, h, KVC_ERR_BAD_BUDGET);
        } else {
            for (int e = tid; e < nq * D; e += kDecThreads) {
                const int q = e / D, c = e % D;
                float mr[kDecCluster];
                float M = -INFINITY;
#pragma unroll
                for (int r = 0; r < kDecCluster; ++r) {
                    const S* rs = cluster.map_shared_rank(&sm, r);
                    mr[r] = rs->m[q];
                    M = fmaxf(M, mr[r]);
                }
                float L = 0.f, acc_o = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int r = 0; r < kDecCluster; ++r) {
                        const S* rs = cluster.map_shared_rank(&sm, r);
                        const float w = mr[r] == -INFINITY ? 0.f : exp2f(mr[r] - M);
                        L = fmaf(rs->l[q], w, L);
                        acc_o = fmaf(rs->o[q][c], w, acc_o);
                    }
                }
                if (!(L > 0.f)) {
                    if (c == 0) set_status(status, h, KVC_ERR_NONFINITE);
                    continue;
                }
                O[((int64_t)h * nq + q) * D + c] = acc_o / L;
            }
        }
    }
    // keep every CTA's shared memory alive until rank 0 has read it
    cluster.sync();
}

template <typename TIn, int D, int CL>
cudaError_t launch_decode_cl(const void* Q, int nq, const void* Ck, const float* beta, const float* Cv,
                             const int32_t* offsets, int H, float c2, float* O, int32_t* status, cudaStream_t st) {
    auto kern = k_attend_decode<TIn, D, CL>;
    constexpr int smem = (int)sizeof(DecSmem<TIn, D>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(CL, H);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, (const TIn*)Q, nq, (const TIn*)Ck, beta, Cv, offsets, c2, O, status);
}
template <typename TIn, int D>
cudaError_t launch_decode_t(const void* Q, int nq, const void* Ck, const float* beta, const float* Cv,
                            const int32_t* offsets, int H, float c2, float* O, int32_t* status, cudaStream_t st) {
    return H >= 148 ? launch_decode_cl<TIn, D, 4>(Q, nq, Ck, beta, Cv, offsets, H, c2, O, status, st)
                    : launch_decode_cl<TIn, D, 8>(Q, nq, Ck, beta, Cv, offsets, H, c2, O, status, st);
}

}  // namespace

int attend_decode_max_queries() { return kDecQ; }

cudaError_t launch_attend_decode(int dtype, int d, const void* Q, int nq, const void* Ck, const float* beta,
                                 const float* Cv, const int32_t* offsets, int H, float c2, float* O, int32_t* status,
                                 cudaStream_t st) {
    if (dtype == KVC_DTYPE_BF16)
        return d == 128 ? launch_decode_t<__nv_bfloat16, 128>(Q, nq, Ck, beta, Cv, offsets, H, c2, O, status, st)
                        : launch_decode_t<__nv_bfloat16, 64>(Q, nq, Ck, beta, Cv, offsets, H, c2, O, status, st);
    return d == 128 ? launch_decode_t<float, 128>(Q, nq, Ck, beta, Cv, offsets, H, c2, O, status, st)
                    : launch_decode_t<float, 64>(Q, nq, Ck, beta, Cv, offsets, H, c2, O, status, st);
}

}  // namespace kvc
