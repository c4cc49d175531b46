// Tensor-core (tcgen05 + TMEM + TMA) kernels for the two attention passes of
// the compaction ("Fast KV Compaction via Attention Matching", section 2):
//
//   k_attn_fwd_tc   Q-major flash pass: S = Q K^T * scale on the tensor cores,
//                   online softmax in registers, P written back into tensor
//                   memory as two bf16 terms (P = P_hi + P_lo, ~16 significant
//                   bits), O += P_hi V + P_lo V on the tensor cores; outputs
//                   the reference outputs O = softmax(S) V (fp32) and the
//                   log-mass lse_q (log2 units).  A single bf16 term would
//                   leave O with ~1e-3 relative error, which the least-squares
//                   fit of C_v amplifies past its tolerance.
//   k_colscore_tc   K-major pass: S^T = K Q^T per key tile, then every key
//                   row sums exp(2 (S - lse)) over all queries: the RMS
//                   attention score of each key (key selection aggregated
//                   by RMS).
//
// bf16 inputs, fp32 accumulation.  One CTA = 6 warps:
//   warp 0       TMA producer (one elected thread)
//   warp 1       tcgen05.mma issuer (one elected thread); owns the TMEM
//                allocation
//   warps 2..5   consumers, one tile row (query or key) per thread; warp w
//                reads TMEM lanes 32*(w%4) .. 32*(w%4)+31
// Operand tiles are [128 rows][64 bf16] TMA boxes with 128-byte swizzle; a
// d = 128 row is two boxes.  Every wait is bounded: a wait that runs out
// raises a CTA-wide abort flag, writes KVC_ERR_TIMEOUT for the head, lets
// the issued copies and MMAs finish and frees the tensor memory.
#include "tc.cuh"

namespace kvc {
using namespace tc;

namespace {

constexpr int TB = 128;                 // tile rows (queries or keys) and keys per tile
constexpr int kBox = 128 * 128;         // bytes of one [128][64] bf16 box
constexpr int kThreads = 192;
constexpr int kConsumer0 = 2;           // first consumer warp

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait for our own issued copies / MMAs at teardown: bounded, but it does
// not give up early on the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    int never = 0;
    (void)mbar_wait(bar, parity, &never);
}

// K-major operand descriptor for k-step kk (16 bf16 along K) of a [128][D]
// tile stored as D/64 swizzled boxes.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_addr, int kk) {
    return sdesc_sw128(tile_addr + (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32), 16, 1024);
}

// ------------------------------------------------------------ attention forward
template <int D, int NS>
struct FwdLayout {
    static constexpr int kTile = (D / 64) * kBox;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTile;
    static constexpr int kV = kK + NS * kTile;
    static constexpr int kBar = kV + NS * kTile;
    static constexpr int kBytes = kBar + 256 + 1024;     // + alignment slack
};

template <int D, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_fwd_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                  const __grid_constant__ CUtensorMap mV, int n, int T, float c2, float* __restrict__ O,
                  float* __restrict__ lse2, int32_t* __restrict__ status) {
    using L = FwdLayout<D, NS>;
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* v_full = k_full + NS;
    uint64_t* kv_empty = v_full + NS;
    uint64_t* s_full = kv_empty + NS;     // [2]
    uint64_t* p_full = s_full + 2;        // [2]
    uint64_t* o_done = p_full + 2;        // one phase per P V product
    uint64_t* o_final = o_done + 1;       // the last P V product
    uint64_t* mma_done = o_final + 1;     // everything the MMA thread issued
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(v_full + s, 1);
            mbar_init(kv_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + b, 1);
            mbar_init(p_full + b, 128);
        }
        mbar_init(o_done, 1);
        mbar_init(o_final, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_O = tmem + 256;
    const int nt = (T + TB - 1) / TB;
    const int q0 = blockIdx.x * TB;
    constexpr uint32_t kTileBytes = (uint32_t)L::kTile;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&mQ);
            prefetch_tmap(&mK);
            prefetch_tmap(&mV);
            mbar_expect_tx(q_full, kTileBytes);
            for (int c = 0; c < D / 64; ++c) tma_load_3d(sm + L::kQ + c * kBox, &mQ, q_full, c * 64, q0, h);
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait(kv_empty + s, (uint32_t)((j / NS) - 1) & 1u, abort_flag)) break;
                mbar_expect_tx(k_full + s, kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm + L::kK + s * L::kTile + c * kBox, &mK, k_full + s, c * 64, j * TB, h);
                mbar_expect_tx(v_full + s, kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm + L::kV + s * L::kTile + c * kBox, &mV, v_full + s, c * 64, j * TB, h);
                issued = j + 1;
            }
            // our copies must land before the CTA exits
            drain_wait(q_full, 0);
            for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j) {
                drain_wait(k_full + j % NS, (uint32_t)(j / NS) & 1u);
                drain_wait(v_full + j % NS, (uint32_t)(j / NS) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
            const uint32_t aQ = smem_addr(sm + L::kQ);
            bool ok = mbar_wait(q_full, 0, abort_flag);
            for (int j = 0; ok && j <= nt; ++j) {
                if (j < nt) {
                    const int s = j % NS;
                    if (!mbar_wait(k_full + s, (uint32_t)(j / NS) & 1u, abort_flag)) break;
                    fence_after_sync();
                    const uint32_t aK = smem_addr(sm + L::kK + s * L::kTile);
                    const uint32_t dS = tmem + (uint32_t)(j & 1) * 128;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(dS, kmajor_desc(aQ, kk), kmajor_desc(aK, kk), idesc_qk, kk > 0);
                    mma_commit(s_full + (j & 1));
                }
                if (j >= 1) {
                    const int jp = j - 1, sp = jp % NS;
                    if (!mbar_wait(p_full + (jp & 1), (uint32_t)(jp >> 1) & 1u, abort_flag)) break;
                    if (!mbar_wait(v_full + sp, (uint32_t)(jp / NS) & 1u, abort_flag)) break;
                    fence_after_sync();
                    const uint32_t aV = smem_addr(sm + L::kV + sp * L::kTile);
                    const uint32_t aP = tmem + (uint32_t)(jp & 1) * 128;
#pragma unroll
                    for (int kk = 0; kk < TB / 16; ++kk) {
                        const uint64_t bV = sdesc_sw128(aV + kk * 2048, kBox, 1024);
                        mma_ts(tmem_O, aP + kk * 8, bV, idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
                        mma_ts(tmem_O, aP + 64 + kk * 8, bV, idesc_pv, 1u);
                    }
                    mma_commit(o_done);
                    if (jp == nt - 1) mma_commit(o_final);
                    mma_commit(kv_empty + sp);
                }
            }
            mma_commit(mma_done);
            drain_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // consumers: one query row per thread
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(s_full + (j & 1), (uint32_t)(j >> 1) & 1u, abort_flag));
            if (!ok) break;
            fence_after_sync();
            const uint32_t sbase = tmem + lane_off + (uint32_t)(j & 1) * 128;
            float s[128];
            {
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    tmem_ld32(sbase + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
                }
            }
            const int kv = T - j * TB;          // valid keys in this tile (>= 1)
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                const float v = (c < kv) ? s[c] * c2 : -INFINITY;
                s[c] = v;
                mx = fmaxf(mx, v);
            }
            // Conditional rescaling: the reference maximum only moves when a
            // row's maximum grows by more than 2^8, so P stays <= 256.
            const bool need = mx > m_used + 8.f;
            const bool any = __any_sync(0xffffffffu, need);
            float corr = 1.f;
            if (need) {
                corr = ex2(m_used - mx);
                m_used = mx;
            }
            // P_hi overwrites columns 0..63 of this S buffer, P_lo columns 64..127
            float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const int k = cc * 32 + c;
                    const float p0 = ex2(s[k] - m_used), p1 = ex2(s[k + 1] - m_used);
                    const float p2 = ex2(s[k + 2] - m_used), p3 = ex2(s[k + 3] - m_used);
                    ps0 += p0;
                    ps1 += p1;
                    ps2 += p2;
                    ps3 += p3;
                    const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
                    hi[c / 2] = h01;
                    hi[c / 2 + 1] = h23;
                    lo[c / 2] = pack_bf16(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
                    lo[c / 2 + 1] = pack_bf16(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
                }
                tmem_st16(sbase + cc * 16, hi);
                tmem_st16(sbase + 64 + cc * 16, lo);
            }
            l = l * corr + ((ps0 + ps1) + (ps2 + ps3));
            tmem_st_wait();
            if (any && j > 0) {
                // O must hold every earlier P V product before it is rescaled
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (uint32_t)(j - 1) & 1u, abort_flag));
                if (!ok) break;
                fence_after_sync();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tmem_O + lane_off + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                    tmem_st32(tmem_O + lane_off + c * 32, r);
                }
                tmem_st_wait();
            }
            fence_before_sync();
            mbar_arrive(p_full + (j & 1));
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final, 0, abort_flag));
        if (ok) {
            fence_after_sync();
            const int q = q0 + row;
            const float inv = 1.f / l;
            float* orow = O + ((int64_t)h * n + q) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem_O + lane_off + c * 32, r);
                tmem_ld_wait();
                if (q < n) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        float4 v = make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                               __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
                        *reinterpret_cast<float4*>(orow + c * 32 + i) = v;
                    }
                }
            }
            if (q < n) lse2[(int64_t)h * n + q] = m_used + log2f(l);
        }
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ key scores
constexpr int kLseChunk = 8192;     // queries whose lse sits in shared memory at once

template <int D, int NS>
struct ColLayout {
    static constexpr int kTile = (D / 64) * kBox;
    static constexpr int kK = 0;
    static constexpr int kQ = kK + kTile;
    static constexpr int kLse = kQ + NS * kTile;
    static constexpr int kBar = kLse + kLseChunk * 4;
    static constexpr int kBytes = kBar + 256 + 1024;
};

template <int D, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    k_colscore_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
                  const float* __restrict__ lse2, int n, int T, float c2, float* __restrict__ score,
                  int32_t* __restrict__ status) {
    using L = ColLayout<D, NS>;
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* lse_s = reinterpret_cast<float*>(sm + L::kLse);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
    uint64_t* k_full = bars;
    uint64_t* q_full = bars + 1;          // [NS]
    uint64_t* q_empty = q_full + NS;      // [NS]
    uint64_t* s_full = q_empty + NS;      // [2]
    uint64_t* s_empty = s_full + 2;       // [2]
    uint64_t* mma_done = s_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    if (threadIdx.x == 0) {
        mbar_init(k_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(q_full + s, 1);
            mbar_init(q_empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + b, 1);
            mbar_init(s_empty + b, 128);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 256);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nq = (n + TB - 1) / TB;
    const int k0 = blockIdx.x * TB;
    constexpr uint32_t kTileBytes = (uint32_t)L::kTile;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&mK);
            prefetch_tmap(&mQ);
            mbar_expect_tx(k_full, kTileBytes);
            for (int c = 0; c < D / 64; ++c) tma_load_3d(sm + L::kK + c * kBox, &mK, k_full, c * 64, k0, h);
            int issued = 0;
            for (int i = 0; i < nq; ++i) {
                const int s = i % NS;
                if (i >= NS && !mbar_wait(q_empty + s, (uint32_t)((i / NS) - 1) & 1u, abort_flag)) break;
                mbar_expect_tx(q_full + s, kTileBytes);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm + L::kQ + s * L::kTile + c * kBox, &mQ, q_full + s, c * 64, i * TB, h);
                issued = i + 1;
            }
            drain_wait(k_full, 0);
            for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
                drain_wait(q_full + i % NS, (uint32_t)(i / NS) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
            const uint32_t aK = smem_addr(sm + L::kK);
            bool ok = mbar_wait(k_full, 0, abort_flag);
            for (int i = 0; ok && i < nq; ++i) {
                const int s = i % NS;
                if (!mbar_wait(q_full + s, (uint32_t)(i / NS) & 1u, abort_flag)) break;
                if (i >= 2 && !mbar_wait(s_empty + (i & 1), (uint32_t)((i >> 1) - 1) & 1u, abort_flag)) break;
                fence_after_sync();
                const uint32_t aQ = smem_addr(sm + L::kQ + s * L::kTile);
                const uint32_t dS = tmem + (uint32_t)(i & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(dS, kmajor_desc(aK, kk), kmajor_desc(aQ, kk), idesc, kk > 0);
                mma_commit(s_full + (i & 1));
                mma_commit(q_empty + s);
            }
            mma_commit(mma_done);
            drain_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // consumers: one key row per thread
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int ct = threadIdx.x - kConsumer0 * 32;       // 0..127
        double acc = 0.0;
        bool ok = true;
        // Every consumer warp runs all iterations (after an abort it only
        // skips the work) so that the named barrier around the log-mass
        // reload is always reached by all four warps.
        for (int i = 0; i < nq; ++i) {
            const int qb = i * TB;
            if (qb % kLseChunk == 0) {
                // log-masses of the next chunk of queries; +inf past n zeroes those columns
                asm volatile("bar.sync 1, 128;" ::: "memory");
                for (int e = ct; e < kLseChunk; e += 128) {
                    const int q = qb + e;
                    lse_s[e] = (q < n) ? lse2[(int64_t)h * n + q] : INFINITY;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
            }
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(s_full + (i & 1), (uint32_t)(i >> 1) & 1u, abort_flag));
            if (!ok) continue;
            fence_after_sync();
            const uint32_t sbase = tmem + lane_off + (uint32_t)(i & 1) * 128;
            float s[128];
            {
                uint32_t r[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    tmem_ld32(sbase + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) s[c * 32 + k] = __uint_as_float(r[k]);
                }
            }
            fence_before_sync();
            mbar_arrive(s_empty + (i & 1));
            const float* ls = lse_s + (qb % kLseChunk);
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int c = 0; c < 128; c += 4) {
                const float x0 = fmaf(s[c], c2, -ls[c]);
                const float x1 = fmaf(s[c + 1], c2, -ls[c + 1]);
                const float x2 = fmaf(s[c + 2], c2, -ls[c + 2]);
                const float x3 = fmaf(s[c + 3], c2, -ls[c + 3]);
                a0 += ex2(x0 + x0);
                a1 += ex2(x1 + x1);
                a2 += ex2(x2 + x2);
                a3 += ex2(x3 + x3);
            }
            acc += (double)((a0 + a1) + (a2 + a3));
        }
        const int key = k0 + row;
        if (ok && key < T) score[(int64_t)h * T + key] = (float)sqrt(acc / (double)n);
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// [H][rows][d] bf16 viewed as a 3-D tensor (d, rows, H); boxes of
// [128 rows][64 elements] with 128-byte swizzle; rows past the end of a head
// read as zero.
bool make_map(CUtensorMap* m, const void* base, int d, int rows, int H) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int NS>
cudaError_t launch_fwd_t(const void* Q, const void* K, const void* V, int H, int n, int T, float c2, float* O,
                         float* lse2, int32_t* status, cudaStream_t st) {
    CUtensorMap mQ, mK, mV;
    if (!make_map(&mQ, Q, D, n, H) || !make_map(&mK, K, D, T, H) || !make_map(&mV, V, D, T, H))
        return cudaErrorInvalidValue;
    constexpr int smem = FwdLayout<D, NS>::kBytes;
    auto kern = k_attn_fwd_tc<D, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((n + TB - 1) / TB, H);
    kern<<<grid, kThreads, smem, st>>>(mQ, mK, mV, n, T, c2, O, lse2, status);
    return cudaGetLastError();
}

template <int D, int NS>
cudaError_t launch_col_t(const void* Q, const void* K, const float* lse2, int H, int n, int T, float c2,
                         float* score, int32_t* status, cudaStream_t st) {
    CUtensorMap mK, mQ;
    if (!make_map(&mK, K, D, T, H) || !make_map(&mQ, Q, D, n, H)) return cudaErrorInvalidValue;
    constexpr int smem = ColLayout<D, NS>::kBytes;
    auto kern = k_colscore_tc<D, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((T + TB - 1) / TB, H);
    kern<<<grid, kThreads, smem, st>>>(mK, mQ, lse2, n, T, c2, score, status);
    return cudaGetLastError();
}

}  // namespace

bool tc_maps_available() { return encode_fn() != nullptr; }

cudaError_t launch_attn_fwd_tc(int d, const void* Q, const void* K, const void* V, int H, int n, int T, float c2,
                               float* O, float* lse2, int32_t* status, cudaStream_t st) {
    return d == 128 ? launch_fwd_t<128, 2>(Q, K, V, H, n, T, c2, O, lse2, status, st)
                    : launch_fwd_t<64, 4>(Q, K, V, H, n, T, c2, O, lse2, status, st);
}

cudaError_t launch_colscore_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T,
                               float c2, float* score, int32_t* status, cudaStream_t st) {
    return d == 128 ? launch_col_t<128, 4>(Q, K, lse2, H, n, T, c2, score, status, st)
                    : launch_col_t<64, 6>(Q, K, lse2, H, n, T, c2, score, status, st);
}

}  // namespace kvc
