// Tensor-core (tcgen05 + TMEM + TMA) kernels for the two attention passes of
// the compaction ("Fast KV Compaction via Attention Matching", section 2):
//
//   k_attn_fwd_tc   Q-major flash pass: S = Q K^T * scale on the tensor cores
//                   (bf16), online softmax in registers, P written back into
//                   tensor memory as fp16 (11 significant bits), O += P V16
//                   on the tensor cores with V16 the values in fp16 under a
//                   per-head power-of-two scale (vconv.cu); outputs the
//                   reference outputs O = softmax(S) V (fp32) and the
//                   log-mass lse_q (log2 units).  A bf16 P (8 bits) would
//                   leave O with ~1e-3 relative error, which the
//                   least-squares fit of C_v carries past its tolerance; fp16
//                   leaves ~5e-5.
//   k_masslogits_tc log2 of the relative mass matrix A' for the kept keys,
//                   S = Q C_k^T on the tensor cores; the epilogue also
//                   writes A' as bf16 hi / lo terms (the Gram operand),
//                   per-tile column sums of A' (partials of b = A'^T 1) and
//                   per-tile sums of A'^2 (partials of tr(A'^T A'), the
//                   scale of the NNLS ridge).
//   k_colscore_tc   K-major pass: S^T = K Q^T per key tile, then every key
//                   row sums exp(2 (S - lse)) over all queries: the RMS
//                   attention score of each key (key selection aggregated
//                   by RMS).  Its WEIGHTED form sums exp(S - lse_q) r_q
//                   instead, <p_j, r> for every key j: the correlations of a
//                   step of key selection by matching pursuit (omp.cu).
//
// Q heads: head h reads reference queries of head h / qdiv (qdiv > 1 when
// several chunks of one cache share its queries).
//
// With BIAS the keys carry an input bias (the cache of an earlier
// compaction: periodic compaction), bias2 [H][Tb] fp32 in log2 units with Tb
// = T rounded up to 256 and -inf padding; it is added to every logit.  The
// forward pass brings each tile's 128 biases into shared memory with the K
// tile (one 512-byte bulk copy on the same barrier); the key-score pass
// holds its row's bias in a register; the mass pass reads the kept keys'
// biases bk [sum t] (log2 units).
//
// bf16 inputs, fp32 accumulation.  One CTA = 10 warps and two 128-row
// tiles (query tiles for the forward pass, key tiles for the scores):
//   warp 0       TMA producer (one elected thread)
//   warp 1       tcgen05.mma issuer (one elected thread); owns the TMEM
//                allocation (all 512 columns)
//   warps 2..9   two consumer warpgroups, one per tile, one tile row per
//                thread; warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31
// Operand tiles are [128 rows][64 bf16] TMA boxes with 128-byte swizzle; a
// d = 128 row is two boxes.  Every wait is bounded: a wait that runs out
// raises a CTA-wide abort flag, writes KVC_ERR_TIMEOUT for the head, lets
// the issued copies and MMAs finish and frees the tensor memory.
#include "tc.cuh"

namespace kvc {
using namespace tc;

bool make_map(CUtensorMap* m, const void* base, int d, int rows, int H);   // tmap.cu
bool make_map_f32(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H);             // tmap.cu
bool make_map_bf16_rows32(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H);     // tmap.cu
bool make_map_rows256(CUtensorMap* m, const void* base, int d, int rows, int H);                         // tmap.cu

namespace {

constexpr int TB = 128;                 // tile rows (queries or keys) and keys per tile
constexpr int kBox = 128 * 128;         // bytes of one [128][64] bf16 box

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
template <int D, int NS, bool BIAS>
struct FwdLayout {
    static constexpr int kTile = (D / 64) * kBox;
    static constexpr int kQ = 0;                  // two query tiles
    static constexpr int kK = kQ + 2 * kTile;
    static constexpr int kV = kK + NS * kTile;
    static constexpr int kBias = kV + NS * kTile; // [NS][128] fp32 key biases (BIAS)
    static constexpr int kBar = kBias + (BIAS ? NS * TB * 4 : 0);
    static constexpr int kBytes = kBar + 256 + 1024;     // + alignment slack
};
constexpr int kFwdThreads = 320;          // TMA warp, MMA warp, two softmax warpgroups

// One CTA = two query tiles g = 0, 1 of 128 rows (rows q0 + 128 g ..).  TMEM
// columns: tile g owns S_g at 256 g (128 columns; after the softmax the fp16
// P sits in its first 64 columns) and O_g at 256 g + 128.  The MMA thread interleaves the tiles so that one tile's
// softmax overlaps the other tile's products:
//   QK_0[j], PV_1[j-1], QK_1[j], PV_0[j], QK_0[j+1], PV_1[j], ...
// tcgen05 operations of one thread complete in issue order, so when S_g[j]
// is complete every earlier P V product of tile g is too: the softmax may
// rescale O_g in place without another wait, and QK_g[j+1] may overwrite
// the P_g[j] that PV_g[j] read.
template <int D, int NS, bool BIAS>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_attn_fwd_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                  const __grid_constant__ CUtensorMap mV, int n, int T, float c2, float* __restrict__ O,
                  float* __restrict__ lse2, const int32_t* __restrict__ vexp, int32_t* __restrict__ status,
                  int qdiv, long long wait_limit, const float* __restrict__ bias2, int Tb) {
    using L = FwdLayout<D, NS, BIAS>;
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
    uint64_t* s_full = kv_empty + NS;     // [2] one per query tile
    uint64_t* p_full = s_full + 2;        // [2]
    uint64_t* o_final = p_full + 2;       // [2]
    uint64_t* mma_done = o_final + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(v_full + s, 1);
            mbar_init(kv_empty + s, 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(s_full + g, 1);
            mbar_init(p_full + g, 128);
            mbar_init(o_final + g, 1);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nt = (T + TB - 1) / TB;
    const int q0 = blockIdx.x * 2 * TB;
    constexpr uint32_t kTileBytes = (uint32_t)L::kTile;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&mQ);
            prefetch_tmap(&mK);
            prefetch_tmap(&mV);
            mbar_expect_tx(q_full, 2 * kTileBytes);
            for (int g = 0; g < 2; ++g)
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm + L::kQ + g * L::kTile + c * kBox, &mQ, q_full, c * 64, q0 + g * TB, h / qdiv);
            int issued = 0;
            for (int j = 0; j < nt; ++j) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait(kv_empty + s, (uint32_t)((j / NS) - 1) & 1u, abort_flag, wait_limit)) break;
                mbar_expect_tx(k_full + s, kTileBytes + (BIAS ? TB * 4u : 0u));
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm + L::kK + s * L::kTile + c * kBox, &mK, k_full + s, c * 64, j * TB, h);
                if (BIAS) bulk_load(sm + L::kBias + s * TB * 4, bias2 + (int64_t)h * Tb + (int64_t)j * TB, TB * 4u,
                                    k_full + s);
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
            constexpr uint32_t idesc_pv = idesc_f16(128, D, false, true);
            const uint32_t aQ0 = smem_addr(sm + L::kQ);
            auto qk = [&](int g, int j) {
                const uint32_t aQ = aQ0 + (uint32_t)(g * L::kTile);
                const uint32_t aK = smem_addr(sm + L::kK + (j % NS) * L::kTile);
                const uint32_t dS = tmem + (uint32_t)g * 256;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss(dS, kmajor_desc(aQ, kk), kmajor_desc(aK, kk), idesc_qk, kk > 0);
                mma_commit(s_full + g);
            };
            auto pv = [&](int g, int j) {
                const uint32_t aV = smem_addr(sm + L::kV + (j % NS) * L::kTile);
                const uint32_t aP = tmem + (uint32_t)g * 256;
                const uint32_t dO = aP + 128;
#pragma unroll
                for (int kk = 0; kk < TB / 16; ++kk) {
                    const uint64_t bV = sdesc_sw128(aV + kk * 2048, kBox, 1024);
                    mma_ts(dO, aP + kk * 8, bV, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (j == nt - 1) mma_commit(o_final + g);
            };
            bool ok = mbar_wait(q_full, 0, abort_flag, wait_limit);
            for (int j = 0; ok && j <= nt; ++j) {
                if (j < nt) {
                    if (!mbar_wait(k_full + j % NS, (uint32_t)(j / NS) & 1u, abort_flag, wait_limit)) break;
                    fence_after_sync();
                    qk(0, j);
                }
                if (j >= 1) {
                    const int jp = j - 1;
                    if (!mbar_wait(p_full + 1, (uint32_t)jp & 1u, abort_flag, wait_limit)) break;
                    if (!mbar_wait(v_full + jp % NS, (uint32_t)(jp / NS) & 1u, abort_flag, wait_limit)) break;
                    fence_after_sync();
                    pv(1, jp);
                    mma_commit(kv_empty + jp % NS);      // both tiles are done with K, V [jp]
                }
                if (j < nt) {
                    qk(1, j);
                    if (!mbar_wait(p_full + 0, (uint32_t)j & 1u, abort_flag, wait_limit)) break;
                    if (!mbar_wait(v_full + j % NS, (uint32_t)(j / NS) & 1u, abort_flag, wait_limit)) break;
                    fence_after_sync();
                    pv(0, j);
                }
            }
            mma_commit(mma_done);
            drain_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // softmax warpgroup g: one query row per thread
        const int g = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)g * 256;
        const uint32_t tO = tS + 128;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(s_full + g, (uint32_t)j & 1u, abort_flag, wait_limit));
            // the tile's key biases came with K (complete by now; the wait
            // makes the bulk copy's shared-memory writes visible here)
            if (BIAS && ok)
                ok = __all_sync(0xffffffffu, mbar_wait(k_full + j % NS, (uint32_t)(j / NS) & 1u, abort_flag, wait_limit));
            if (!ok) break;
            fence_after_sync();
            float s[128];
            tmem_ld128_wait(tS, s);             // the whole row in one load
            const int kv = T - j * TB;          // valid keys in this tile (>= 1)
            if (kv < TB) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= kv) s[c] = -INFINITY;
            }
            if (BIAS) {
                // logits in log2 units with the key biases (-inf for switched-off keys)
                const float4* b4 = reinterpret_cast<const float4*>(sm + L::kBias + (j % NS) * TB * 4);
                const float2 cc2 = make_float2(c2, c2);
#pragma unroll
                for (int c = 0; c < 128; c += 4) {
                    const float4 b = b4[c / 4];
                    const float2 x01 = ffma2(make_float2(s[c], s[c + 1]), cc2, make_float2(b.x, b.y));
                    const float2 x23 = ffma2(make_float2(s[c + 2], s[c + 3]), cc2, make_float2(b.z, b.w));
                    s[c] = x01.x;
                    s[c + 1] = x01.y;
                    s[c + 2] = x23.x;
                    s[c + 3] = x23.y;
                }
            }
            float m0 = s[0], m1 = s[1];
#pragma unroll
            for (int c = 2; c < 126; c += 4) {
                m0 = fmax3(m0, s[c], s[c + 1]);
                m1 = fmax3(m1, s[c + 2], s[c + 3]);
            }
            float mx = fmax3(m0, m1, fmaxf(s[126], s[127]));
            if (!BIAS) mx *= c2;                // c2 > 0: the maximum commutes with the scale
            // Conditional rescaling: the reference maximum only moves when a
            // row's maximum grows by more than 2^8, so P stays <= 256.
            const bool need = mx > m_used + 8.f;
            const bool any = __any_sync(0xffffffffu, need);
            float corr = 1.f;
            if (need) {
                corr = ex2(m_used - mx);
                m_used = mx;
            }
            // (with biases the reference stays -inf while every key so far is
            // switched off; those keys' P is then ex2(-inf) = 0)
            const float nm = (BIAS && m_used == -INFINITY) ? 0.f : -m_used;
            const float cs = BIAS ? 1.f : c2;   // scale still to apply to s
            // the fp16 P overwrites columns 0..63 of S (P <= 256)
            const float2 cs2 = make_float2(cs, cs), nm2 = make_float2(nm, nm);
            float2 ps01 = make_float2(0.f, 0.f), ps23 = make_float2(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pw[16];
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const int k = cc * 32 + c;
                    const float2 x01 = ffma2(make_float2(s[k], s[k + 1]), cs2, nm2);
                    const float2 x23 = ffma2(make_float2(s[k + 2], s[k + 3]), cs2, nm2);
                    const float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
                    const float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
                    ps01 = fadd2(ps01, p01);
                    ps23 = fadd2(ps23, p23);
                    pw[c / 2] = pack_f16(p01.x, p01.y);
                    pw[c / 2 + 1] = pack_f16(p23.x, p23.y);
                }
                tmem_st16(tS + cc * 16, pw);
            }
            l = l * corr + ((ps01.x + ps01.y) + (ps23.x + ps23.y));
            if (any && j > 0) {
                // S_g[j] complete => every earlier P V product of this tile is too
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tO + c * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                    tmem_st32(tO + c * 32, r);
                }
            }
            tmem_st_wait();
            fence_before_sync();
            mbar_arrive(p_full + g);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final + g, 0, abort_flag, wait_limit));
        if (ok) {
            fence_after_sync();
            const int q = q0 + g * TB + row;
            // undo the values' scale 2^-e (vconv.cu)
            const float inv = __uint_as_float((uint32_t)(127 + vexp[h]) << 23) / l;
            float* orow = O + ((int64_t)h * n + q) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + c * 32, r);
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
            // every key switched off by its bias: nothing to match
            if (BIAS && q < n && !(l > 0.f)) set_status(status, h, KVC_ERR_NONFINITE);
        }
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ key scores
constexpr int kLseChunk = 4096;     // queries whose lse sits in shared memory at once
constexpr int QB = 256;             // queries per block: the N of every key-score product
constexpr int kColThreads = 576;    // TMA warp, MMA warp, four consumer warpgroups

template <int D, int NS>
struct ColLayout {
    static constexpr int kTileK = (D / 64) * kBox;          // [128 keys][D]
    static constexpr int kBoxQ = QB * 128;                  // [256 rows][64 bf16]
    static constexpr int kTileQ = (D / 64) * kBoxQ;         // [256 queries][D]
    static constexpr int kK = 0;                            // two key tiles
    static constexpr int kQ = kK + 2 * kTileK;
    static constexpr int kLse = kQ + NS * kTileQ;
    static constexpr int kRed = kLse + kLseChunk * 4;       // [2 key tiles][128 rows] (hi, lo) fp32
    static constexpr int kBar = kRed + 2 * 128 * 8;
    static constexpr int kBytes = kBar + 256 + 1024;
};

// One CTA = two key tiles g = 0, 1 of 128 keys; the queries stream through in
// blocks of 256.  For every block i the MMA thread computes S^T_g = K_g Q_i^T
// (M = 128 keys, N = 256 queries: an N = 256 product runs the tensor pipe
// about 1.7 times faster per flop on this part than two of N = 128) into
// TMEM buffer g (columns 256 g .. 256 g + 255); the two buffers alternate, so
// the product of one key tile overlaps the exponentials of the other.  Two
// consumer warpgroups share each key tile: both take the same rows (one key
// per thread), warpgroup half takes the queries 128 half .. 128 half + 127
// of the block in two loads of 64 columns and frees the buffer after the
// second.  Each adds exp2(2 (S c2 - lse2_q)) over its queries; the two
// halves' sums meet in shared memory at the end.  The log-masses are kept
// doubled and negated in shared memory so that one FFMA (two, paired, per
// instruction) forms the exponent.
template <int D, int NS, bool BIAS, bool WEIGHTED>
__global__ void __launch_bounds__(kColThreads, 1)
    k_colscore_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mQ,
                  const float* __restrict__ lse2, int n, int T, float c2, float* __restrict__ score,
                  int32_t* __restrict__ status, int qdiv, long long wait_limit, const float* __restrict__ bias2,
                  int Tb, const float* __restrict__ rw, int64_t rstride, float2* __restrict__ part) {
    // WEIGHTED: the shared log-mass chunk holds half the queries, followed by
    // their weights r_q
    constexpr int kChunk = WEIGHTED ? kLseChunk / 2 : kLseChunk;
    static_assert(kChunk % QB == 0, "a log-mass chunk holds whole query blocks");
    using L = ColLayout<D, NS>;
    grid_dependency_wait();   // launched dependent on the previous kernel (launch_dep)
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
    uint64_t* s_full = q_empty + NS;      // [2 key tiles]
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
        for (int g = 0; g < 2; ++g) {
            mbar_init(s_full + g, 1);
            mbar_init(s_empty + g, 256);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // this CTA's query blocks: the gridDim.z parts of the n queries
    // (WEIGHTED only; the key scores take all queries in one CTA)
    const int nq_all = (n + QB - 1) / QB;
    const int per = WEIGHTED ? (nq_all + (int)gridDim.z - 1) / (int)gridDim.z : nq_all;
    const int ib = WEIGHTED ? min(nq_all, (int)blockIdx.z * per) : 0;
    const int nq = min(nq_all, ib + per) - ib;
    const int k0 = blockIdx.x * 2 * TB;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&mK);
            prefetch_tmap(&mQ);
            mbar_expect_tx(k_full, 2 * (uint32_t)L::kTileK);
            for (int g = 0; g < 2; ++g)
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm + L::kK + g * L::kTileK + c * kBox, &mK, k_full, c * 64, k0 + g * TB, h);
            int issued = 0;
            for (int i = 0; i < nq; ++i) {
                const int s = i % NS;
                if (i >= NS && !mbar_wait(q_empty + s, (uint32_t)((i / NS) - 1) & 1u, abort_flag, wait_limit)) break;
                mbar_expect_tx(q_full + s, (uint32_t)L::kTileQ);
                for (int c = 0; c < D / 64; ++c)
                    tma_load_3d(sm + L::kQ + s * L::kTileQ + c * L::kBoxQ, &mQ, q_full + s, c * 64, (ib + i) * QB,
                                h / qdiv);
                issued = i + 1;
            }
            drain_wait(k_full, 0);
            for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
                drain_wait(q_full + i % NS, (uint32_t)(i / NS) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, QB, false, false);
            const uint32_t aK0 = smem_addr(sm + L::kK);
            bool ok = mbar_wait(k_full, 0, abort_flag, wait_limit);
            for (int i = 0; ok && i < nq; ++i) {
                const int s = i % NS;
                if (!mbar_wait(q_full + s, (uint32_t)(i / NS) & 1u, abort_flag, wait_limit)) break;
                const uint32_t aQ = smem_addr(sm + L::kQ + s * L::kTileQ);
                for (int g = 0; g < 2; ++g) {
                    // buffer g is free once both warpgroups loaded block i - 1 from it
                    if (i >= 1 && !mbar_wait(s_empty + g, (uint32_t)(i - 1) & 1u, abort_flag, wait_limit)) {
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t aK = aK0 + (uint32_t)(g * L::kTileK);
                    const uint32_t dS = tmem + (uint32_t)(g * QB);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(dS, kmajor_desc(aK, kk),
                               sdesc_sw128(aQ + (uint32_t)((kk >> 2) * L::kBoxQ + (kk & 3) * 32), 16, 1024), idesc,
                               kk > 0);
                    mma_commit(s_full + g);
                }
                if (!ok) break;
                mma_commit(q_empty + s);
            }
            mma_commit(mma_done);
            drain_wait(mma_done, 0);
        }
        __syncwarp();
    } else {
        // consumer warpgroup (g, half): one key row per thread, half the queries
        const int cw = (warp - 2) >> 2;
        const int g = cw >> 1, half = cw & 1;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int ct = threadIdx.x - 64;            // 0..511 over the four warpgroups
        const float c2x = 2.f * c2;
        // this row's key bias, doubled like the logit (the grid covers Tb keys)
        const float kb2 = BIAS ? 2.f * bias2[(int64_t)h * Tb + k0 + g * TB + row] : 0.f;
        // fp32 pairs (hi, lo) carry the sum over the queries: the fp64 pipe
        // of this part is far too slow for a per-block double add
        dfloat acc{0.f, 0.f};
        bool ok = true;
        // Every consumer warp runs all blocks (after an abort it only skips
        // the work) so that the named barriers around the log-mass reload
        // and the final combine are always reached by all sixteen.
        int cbase = 0;                              // first query of the log-mass chunk in shared memory
        for (int i = 0; i < nq; ++i) {
            const int qb = (ib + i) * QB;
            if (WEIGHTED ? (i == 0 || qb - cbase >= kChunk) : (qb % kChunk == 0)) {
                cbase = qb;
                // the next chunk's log-masses, negated (doubled for P^2); -inf
                // past n zeroes those columns; WEIGHTED: and the weights
                const int cnt = min(kChunk, ((n - qb + QB - 1) / QB) * QB);
                asm volatile("bar.sync 1, 512;" ::: "memory");
                for (int e = ct; e < cnt; e += 512) {
                    const int q = qb + e;
                    lse_s[e] = (q < n) ? (WEIGHTED ? -1.f : -2.f) * lse2[(int64_t)h * n + q] : -INFINITY;
                    if (WEIGHTED) lse_s[kChunk + e] = (q < n) ? rw[(int64_t)h * rstride + q] : 0.f;
                }
                asm volatile("bar.sync 1, 512;" ::: "memory");
            }
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(s_full + g, (uint32_t)i & 1u, abort_flag, wait_limit));
            if (!ok) continue;
            fence_after_sync();
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
                const int col = half * 128 + part * 64;          // query column within the block
                float s[64];
                tmem_ld64_wait(tmem + lane_off + (uint32_t)(g * QB + col), s);
                if (part == 1) {
                    fence_before_sync();
                    mbar_arrive(s_empty + g);
                }
                const int c0 = (WEIGHTED ? qb - cbase : qb % kChunk) + col;
                const float4* ls = reinterpret_cast<const float4*>(lse_s + c0);
                float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
                if (WEIGHTED) {
                    const float4* rs = reinterpret_cast<const float4*>(lse_s + kChunk + c0);
                    const float2 cc2 = make_float2(c2, c2);
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        const float4 l4 = ls[c / 4], r4 = rs[c / 4];     // -lse2 and r of four queries
                        const float2 x01 = ffma2(make_float2(s[c], s[c + 1]), cc2, make_float2(l4.x, l4.y));
                        const float2 x23 = ffma2(make_float2(s[c + 2], s[c + 3]), cc2, make_float2(l4.z, l4.w));
                        a01 = ffma2(make_float2(ex2(x01.x), ex2(x01.y)), make_float2(r4.x, r4.y), a01);
                        a23 = ffma2(make_float2(ex2(x23.x), ex2(x23.y)), make_float2(r4.z, r4.w), a23);
                    }
                } else {
                    const float2 cx2 = make_float2(c2x, c2x), kb = make_float2(kb2, kb2);
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        const float4 l4 = ls[c / 4];    // -2 lse2 of four queries
                        float2 n01 = make_float2(l4.x, l4.y), n23 = make_float2(l4.z, l4.w);
                        if (BIAS) {
                            n01 = fadd2(n01, kb);
                            n23 = fadd2(n23, kb);
                        }
                        const float2 x01 = ffma2(make_float2(s[c], s[c + 1]), cx2, n01);
                        const float2 x23 = ffma2(make_float2(s[c + 2], s[c + 3]), cx2, n23);
                        a01 = fadd2(a01, make_float2(ex2(x01.x), ex2(x01.y)));
                        a23 = fadd2(a23, make_float2(ex2(x23.x), ex2(x23.y)));
                    }
                }
                df_add(acc, (a01.x + a01.y) + (a23.x + a23.y));
            }
        }
        // the second half's sum joins the first's (a fixed order)
        float2* red = reinterpret_cast<float2*>(sm + L::kRed);
        if (half == 1) red[g * 128 + row] = ok ? make_float2(acc.hi, acc.lo) : make_float2(NAN, 0.f);
        asm volatile("bar.sync 1, 512;" ::: "memory");
        if (half == 0) {
            const float2 o = red[g * 128 + row];
            df_add_df(acc, dfloat{o.x, o.y});
            const double tot = (double)acc.hi + (double)acc.lo;
            const int key = k0 + g * TB + row;
            if (ok && key < T) {
                if (part)
                    part[((int64_t)blockIdx.z * gridDim.y + h) * T + key] = make_float2(acc.hi, acc.lo);
                else
                    score[(int64_t)h * T + key] = WEIGHTED ? (float)tot : (float)sqrt(tot / (double)n);
            }
        }
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ mass logits
// l2[h][q][i] = S_q,idx_i c2 - lse2_q (log2 of A'_qi) for i < t_h and -inf
// for t_h <= i < roundup(t_h, 64): one 128 x 128 tile per CTA, S = Q C_k^T on
// the tensor cores.  The kept keys come from their per-head copy Ckw
// [H][ldA][d] (bf16) that the gather writes.
// Epilogue staging (after the product is done it reuses the operand tiles):
// per epilogue warp one [32 rows][32 columns] fp32 box of log-masses and one
// [32 rows][64 columns] bf16 box for each of A'_hi, A'_lo, all in the
// 128-byte swizzled layout of the TMA store maps; then the column-sum
// exchange, [4 chunks][4 warps][32] fp32.
template <int D>
struct MassLayout {
    static constexpr int kTile = (D / 64) * kBox;
    static constexpr int kQ = 0;
    static constexpr int kC = kTile;
    static constexpr int kWarpStage = 12 * 1024;          // L2 box 4 KB + A'_hi box 4 KB + A'_lo box 4 KB
    static constexpr int kStage = 0;
    static constexpr int kRed = kStage + 4 * kWarpStage;
    static constexpr int kRedSq = kRed + 4 * 4 * 32 * 4;      // [4 warps] double
    static constexpr int kEnd = kRedSq + 4 * 8;
    static constexpr int kBar = (2 * kTile > kEnd) ? 2 * kTile : kEnd;
    static constexpr int kBytes = kBar + 256 + 1024;
};
constexpr int kMassThreads = 192;

// Byte offset of 16-byte chunk j of row r in a box whose rows are 128 bytes,
// with the 128-byte swizzle (chunk index XOR row mod 8; box base 1024-aligned).
__device__ __forceinline__ uint32_t sw128_off(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

// Per-column sums of a warp's 32 x 32 block (lane = row, v[k] = column k):
// a butterfly that halves the columns each lane keeps at every step; lane l
// ends with the sum of column l in v[0].  Fixed order, so deterministic.
template <int W>
__device__ __forceinline__ void colsum_step(float (&v)[32], int lane) {
    const bool up = (lane & W) != 0;
#pragma unroll
    for (int k = 0; k < W; ++k) {
        const float send = up ? v[k] : v[k + W];
        const float keep = up ? v[k + W] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, W);
    }
}

// One CTA = 128 queries x 128 kept keys of one head; the product S = Q C_k^T
// in one shot (K = d).  Epilogue per thread = one query row, in four chunks
// of 32 keys: l2 = S * c2 - lse2 (the log2 relative mass, -inf past t_h),
// A' = exp2(l2) as bf16 hi / lo terms (the Gram operand; 0 past t_h and for
// rows past n), and the CTA's column sums of A' (one partial of b = A'^T 1
// per 128-query tile, added in a fixed order by the total kernel).  The
// three arrays leave through TMA stores of swizzled boxes (rows past n are
// clipped by the maps); columns are written up to t_h rounded up to 64.
// The CTA's sum of A'^2 (fp32 over each thread's 32-column chunk, double
// from there on) goes to sqpart[h][blockIdx.y][blockIdx.x], zeroed by the
// caller: the NNLS
// ridge mu = eps tr(A'^T A') / t is formed from these exact squares of the
// fp32 A' rather than from the bf16-term Gram, whose diagonal misses the
// lo * lo products (~2^-18 of each square, always the same sign) and would
// shift mu, and so the solution of the refinement, by ~1e-5.
template <int D>
__global__ void __launch_bounds__(kMassThreads, 3)
    k_masslogits_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mC,
                    const __grid_constant__ CUtensorMap mL2, const __grid_constant__ CUtensorMap mAh,
                    const __grid_constant__ CUtensorMap mAl, const float* __restrict__ lse2,
                    const int32_t* __restrict__ offsets, int n, float c2, float* __restrict__ colpart,
                    int64_t part_stride, double* __restrict__ sqpart, int32_t* __restrict__ status, int qdiv,
                    long long wait_limit, const float* __restrict__ bk) {
    using L = MassLayout<D>;
    const int h = blockIdx.z;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int th = offsets[h + 1] - off;
    const int i0 = blockIdx.x * TB;
    const int q0 = blockIdx.y * TB;
    const int tpad = (int)round_up(th, 64);
    if (i0 >= tpad) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
    uint64_t* full = bars;
    uint64_t* done = bars + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&mL2);
            prefetch_tmap(&mAh);
            prefetch_tmap(&mAl);
            mbar_expect_tx(full, 2u * L::kTile);
            for (int c = 0; c < D / 64; ++c) {
                tma_load_3d(sm + L::kQ + c * kBox, &mQ, full, c * 64, q0, h / qdiv);
                tma_load_3d(sm + L::kC + c * kBox, &mC, full, c * 64, i0, h);
            }
            drain_wait(full, 0);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            if (mbar_wait(full, 0, abort_flag, wait_limit)) {
                fence_after_sync();
                constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
                const uint32_t aQ = smem_addr(sm + L::kQ), aC = smem_addr(sm + L::kC);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem, kmajor_desc(aQ, kk), kmajor_desc(aC, kk), idesc, kk > 0);
            }
            mma_commit(done);
            drain_wait(done, 0);
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3;             // TMEM lanes 32 * quarter .. (the warp's rows)
        const int row = quarter * 32 + lane;
        const int qw = q0 + quarter * 32;         // the warp's first query
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0, abort_flag, wait_limit));
        const int q = q0 + row;
        const float lq = (ok && q < n) ? lse2[(int64_t)h * n + q] : 0.f;
        uint8_t* bL = sm + L::kStage + quarter * L::kWarpStage;
        uint8_t* bH = bL + 4096;
        uint8_t* bO = bL + 8192;
        float* red = reinterpret_cast<float*>(sm + L::kRed);      // [chunk][warp][32]
        const bool store = ok && qw < n;
        double sq = 0.0;
        if (ok) fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            const int ib = i0 + c * 32;
            float x[32];
            if (ok) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + c * 32, r);
                tmem_ld_wait();
                // the kept keys' input biases (lane k holds column ib + k)
                const float bl = (bk && ib + lane < th) ? bk[off + ib + lane] : 0.f;
                float sqc = 0.f;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float bkk = bk ? __shfl_sync(0xffffffffu, bl, k) : 0.f;
                    const float v = (ib + k < th) ? fmaf(__uint_as_float(r[k]), c2, bkk - lq) : -INFINITY;
                    // the special-function unit's 2^v (relative error ~2^-22), far
                    // inside the 2^-17 of the hi / lo terms it feeds
                    x[k] = (q < n && ib + k < th) ? ex2(v) : 0.f;
                    r[k] = __float_as_uint(v);
                    sqc = fmaf(x[k], x[k], sqc);
                }
                sq += (double)sqc;
                if (store && ib < tpad) {
                    // the previous chunk's boxes must have been read out before we overwrite them
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4*>(bL + sw128_off(lane, j)) =
                            make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        __align__(16) __nv_bfloat16 hv[8], lv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            hv[e] = __float2bfloat16_rn(x[8 * j + e]);
                            lv[e] = __float2bfloat16_rn(x[8 * j + e] - __bfloat162float(hv[e]));
                        }
                        const uint32_t o = sw128_off(lane, (c & 1) * 4 + j);
                        *reinterpret_cast<uint4*>(bH + o) = *reinterpret_cast<const uint4*>(hv);
                        *reinterpret_cast<uint4*>(bO + o) = *reinterpret_cast<const uint4*>(lv);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&mL2, bL, ib, qw, h);
                        if (c & 1) {
                            tma_store_3d(&mAh, bH, ib - 32, qw, h);
                            tma_store_3d(&mAl, bO, ib - 32, qw, h);
                        }
                        bulk_commit();
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) x[k] = 0.f;
            }
            colsum_step<16>(x, lane);
            colsum_step<8>(x, lane);
            colsum_step<4>(x, lane);
            colsum_step<2>(x, lane);
            colsum_step<1>(x, lane);
            red[(c * 4 + quarter) * 32 + lane] = x[0];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        double* redsq = reinterpret_cast<double*>(sm + L::kRedSq);
        if (lane == 0) redsq[quarter] = sq;
        // every epilogue warp reaches the barrier, whatever `ok` was
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (ok && quarter == 0 && lane == 0)
            sqpart[((int64_t)h * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x] =
                (redsq[0] + redsq[1]) + (redsq[2] + redsq[3]);
        const int cc = quarter;                   // warp `quarter` totals chunk `quarter`
        const int col = i0 + cc * 32 + lane;
        if (ok && col < th) {
            const float* rc = red + cc * 4 * 32 + lane;
            colpart[(int64_t)blockIdx.y * part_stride + off + col] = (rc[0] + rc[32]) + (rc[64] + rc[96]);
        }
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 128);
}

// ------------------------------------------------------------ host side
template <int D, int NS, bool BIAS>
cudaError_t launch_fwd_t(const void* Q, const void* K, const void* V, int H, int n, int T, float c2, float* O,
                         float* lse2, const int32_t* vexp, int32_t* status, int qdiv, long long wait_limit,
                         const float* bias2, cudaStream_t st) {
    CUtensorMap mQ, mK, mV;
    if (!make_map(&mQ, Q, D, n, H / qdiv) || !make_map(&mK, K, D, T, H) || !make_map(&mV, V, D, T, H))
        return cudaErrorInvalidValue;
    constexpr int smem = FwdLayout<D, NS, BIAS>::kBytes;
    auto kern = k_attn_fwd_tc<D, NS, BIAS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((n + 2 * TB - 1) / (2 * TB), H);
    kern<<<grid, kFwdThreads, smem, st>>>(mQ, mK, mV, n, T, c2, O, lse2, vexp, status, qdiv, wait_limit, bias2,
                                          (int)round_up(T, 256));
    return cudaGetLastError();
}

template <int D, int NS, bool BIAS, bool WEIGHTED = false>
cudaError_t launch_col_t(const void* Q, const void* K, const float* lse2, int H, int n, int T, float c2,
                         float* score, int32_t* status, int qdiv, long long wait_limit, const float* bias2,
                         cudaStream_t st, const float* rw = nullptr, int64_t rstride = 0, float2* part = nullptr,
                         int nz = 1) {
    CUtensorMap mK, mQ;
    if (!make_map(&mK, K, D, T, H) || !make_map_rows256(&mQ, Q, D, n, H / qdiv)) return cudaErrorInvalidValue;
    constexpr int smem = ColLayout<D, NS>::kBytes;
    static_assert(smem <= 227 * 1024, "key-score shared memory");
    auto kern = k_colscore_tc<D, NS, BIAS, WEIGHTED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: in the matching pursuit this pass
    // alternates with the step kernel, hundreds of times per call
    return launch_dep(kern, dim3((T + 2 * TB - 1) / (2 * TB), H, nz), dim3(kColThreads), smem, st, mK, mQ, lse2, n,
                      T, c2, score, status, qdiv, wait_limit, bias2, (int)round_up(T, 256), rw, rstride, part);
}

template <int D>
cudaError_t launch_mass_t(const void* Q, const void* Ck, const float* lse2, const int32_t* offsets, int H, int n,
                          int max_t, int64_t ldA, float c2, float* L2, void* Ah, void* Al, float* colpart,
                          int64_t part_stride, double* sqpart, int32_t* status, int qdiv, long long wait_limit,
                          const float* bk, cudaStream_t st) {
    CUtensorMap mQ, mC, mL2, mAh, mAl;
    if (!make_map(&mQ, Q, D, n, H / qdiv) || !make_map(&mC, Ck, D, (int)ldA, H) ||
        !make_map_f32(&mL2, L2, (int)ldA, ldA, n, H) || !make_map_bf16_rows32(&mAh, Ah, (int)ldA, ldA, n, H) ||
        !make_map_bf16_rows32(&mAl, Al, (int)ldA, ldA, n, H))
        return cudaErrorInvalidValue;
    constexpr int smem = MassLayout<D>::kBytes;
    auto kern = k_masslogits_tc<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((max_t + TB - 1) / TB, (n + TB - 1) / TB, H);
    kern<<<grid, kMassThreads, smem, st>>>(mQ, mC, mL2, mAh, mAl, lse2, offsets, n, c2, colpart, part_stride, sqpart,
                                           status, qdiv, wait_limit, bk);
    return cudaGetLastError();
}

}  // namespace

// L2: fp32 [H][n][ldA] log2 A'; Ah / Al: A' as bf16 hi / lo terms, same
// layout; colpart: column sums of A' per 128-query tile, [tile][part_stride]
// (entry off_h + i); sqpart: sums of A'^2 per CTA, double
// [H][ceil(n/128)][ceil(max_t/128)], zeroed here first.  All required but
// bk: the kept keys' input biases [sum t] (log2 units), or null.
cudaError_t launch_masslogits_tc(int d, const void* Q, const void* Ck, const float* lse2, const int32_t* offsets,
                                 int H, int n, int max_t, int64_t ldA, float c2, float* L2, void* Ah, void* Al,
                                 float* colpart, int64_t part_stride, double* sqpart, int32_t* status, int qdiv,
                                 long long wait_limit, const float* bk, cudaStream_t st) {
    const size_t nsq = (size_t)H * ((n + TB - 1) / TB) * ((max_t + TB - 1) / TB);
    cudaError_t e = cudaMemsetAsync(sqpart, 0, nsq * sizeof(double), st);
    if (e != cudaSuccess) return e;
    return d == 128 ? launch_mass_t<128>(Q, Ck, lse2, offsets, H, n, max_t, ldA, c2, L2, Ah, Al, colpart, part_stride,
                                         sqpart, status, qdiv, wait_limit, bk, st)
                    : launch_mass_t<64>(Q, Ck, lse2, offsets, H, n, max_t, ldA, c2, L2, Ah, Al, colpart, part_stride,
                                        sqpart, status, qdiv, wait_limit, bk, st);
}

// V16: the values in fp16 with per-head exponents vexp (launch_v_to_f16).
// bias2 (optional): key biases [H][round_up(T, 256)], log2 units, -inf padded.
cudaError_t launch_attn_fwd_tc(int d, const void* Q, const void* K, const void* V16, const int32_t* vexp, int H,
                               int n, int T, float c2, float* O, float* lse2, int32_t* status, int qdiv,
                               long long wait_limit, const float* bias2, cudaStream_t st) {
    if (bias2)
        return d == 128 ? launch_fwd_t<128, 2, true>(Q, K, V16, H, n, T, c2, O, lse2, vexp, status, qdiv, wait_limit,
                                                     bias2, st)
                        : launch_fwd_t<64, 3, true>(Q, K, V16, H, n, T, c2, O, lse2, vexp, status, qdiv, wait_limit,
                                                    bias2, st);
    return d == 128 ? launch_fwd_t<128, 2, false>(Q, K, V16, H, n, T, c2, O, lse2, vexp, status, qdiv, wait_limit,
                                                  nullptr, st)
                    : launch_fwd_t<64, 3, false>(Q, K, V16, H, n, T, c2, O, lse2, vexp, status, qdiv, wait_limit,
                                                 nullptr, st);
}

cudaError_t launch_colscore_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T,
                               float c2, float* score, int32_t* status, int qdiv, long long wait_limit,
                               const float* bias2, cudaStream_t st) {
    if (bias2)
        return d == 128 ? launch_col_t<128, 2, true>(Q, K, lse2, H, n, T, c2, score, status, qdiv, wait_limit, bias2,
                                                     st)
                        : launch_col_t<64, 4, true>(Q, K, lse2, H, n, T, c2, score, status, qdiv, wait_limit, bias2,
                                                    st);
    return d == 128 ? launch_col_t<128, 2, false>(Q, K, lse2, H, n, T, c2, score, status, qdiv, wait_limit, nullptr,
                                                  st)
                    : launch_col_t<64, 4, false>(Q, K, lse2, H, n, T, c2, score, status, qdiv, wait_limit, nullptr,
                                                 st);
}

// part[z][h][j] = the z-th of nz parts (query blocks split evenly) of
// sum_q exp2(S_qj c2 - lse2_q) r[h][q] for every key j, as an fp32 pair
// (hi, lo) (bf16 inputs, tensor cores): the matching-pursuit correlations
// <p_j, r> are the parts' sum.  Splitting the queries gives small problems
// more CTAs.  r has row stride rstride.
cudaError_t launch_corr_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T, float c2,
                           const float* r, int64_t rstride, float2* part, int nz, int32_t* status,
                           long long wait_limit, cudaStream_t st) {
    return d == 128 ? launch_col_t<128, 2, false, true>(Q, K, lse2, H, n, T, c2, nullptr, status, 1, wait_limit,
                                                        nullptr, st, r, rstride, part, nz)
                    : launch_col_t<64, 4, false, true>(Q, K, lse2, H, n, T, c2, nullptr, status, 1, wait_limit,
                                                       nullptr, st, r, rstride, part, nz);
}

}  // namespace kvc
