// Tensor-core Gram products of the two least-squares fits ("Fast KV
// Compaction via Attention Matching", section 2, fitting beta by NNLS and
// C_v by least squares through the normal equations):
//
//   G = A'^T A'   (mass matrix, t x t; lower tiles computed, mirrored)
//   M = X^T X     (biased softmax, t x t; lower tiles computed, mirrored)
//   R = X^T O     (t x d)
//
// C[i][j] = sum_q A[q][i] B[q][j] over the n reference queries.  Every fp32
// operand value x is stored as two bf16 terms, hi = bf16(x) and
// lo = bf16(x - hi) (round to nearest), in separate [H][n][ld] arrays
// written once by the pass that produces the operand (the tensor-core mass
// logits' epilogue for A' with bf16 inputs, k_split_hilo below for A' with
// fp32 inputs and for O, the biased softmax for X).  The products run on the tcgen05
// tensor cores in bf16: C accumulates A_hi B_hi + A_hi B_lo + A_lo B_hi in
// fp32.  The split carries ~2^-17 of each value and the dropped A_lo B_lo
// term is ~2^-18 relative; both errors have random sign, so a sum over the
// queries keeps close to fp32 accuracy.  (Both operands are MN-major: the
// queries are the contraction and the outer dimension of the stored arrays.)
//
// One CTA per output tile (x head).  The symmetric products pair the lower
// 128 x 128 blocks of a block row: a CTA computes blocks (I, J) and (I, J + 1)
// as one M = 128, N = 256 product (an N = 256 product runs the tensor pipe
// about 1.4 times faster per flop on this part than two of N = 128, and
// reads A_I once); a row with an odd block count ends in a single N = 128
// tile.  The rectangular product has one 128 x NB tile per row block.
// Warp roles:
//   warp 0       TMA producer: [64 queries][64 columns] bf16 boxes with
//                128-byte swizzle (the MN-major operand layout)
//   warp 1       MMA issuer; owns the TMEM accumulator (256 columns)
//   warps 2..5   epilogue (TMEM -> global)
#include "tc.cuh"

namespace kvc {
using namespace tc;

namespace {

constexpr int GB = 128;                 // output tile
constexpr int GK = 64;                  // queries per pipeline stage
constexpr int kGBox = GK * 128;         // one [64 queries][64 columns] bf16 box: 8 KB
constexpr int kGThreads = 192;

// Pipeline stages: a symmetric stage holds A_I and up to 256 columns of B
// (96 KB), a rectangular one A_I and NB columns of B (64 KB at most).
template <bool SYM>
__host__ __device__ constexpr int gram_stages() { return SYM ? 2 : 3; }

__device__ __forceinline__ uint8_t* align1024g(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
    int never = 0;
    (void)mbar_wait(bar, parity, &never);
}

// Paired lower tiles: block row I holds I / 2 + 1 tiles, so the rows before
// I hold m (m + 1) tiles for I = 2m and (m + 1)^2 for I = 2m + 1.  Tile p ->
// block row I, first block column J, width 1 or 2 blocks.
__host__ __device__ inline int paired_before(int I) {
    const int m = I / 2;
    return (I & 1) ? (m + 1) * (m + 1) : m * (m + 1);
}
__device__ __forceinline__ void paired_tile(int p, int& I, int& J, int& width) {
    int i = max(0, 2 * (int)sqrtf((float)p) - 2);    // paired_before(i) <= p for this start
    while (i > 0 && paired_before(i) > p) --i;
    while (paired_before(i + 1) <= p) ++i;
    I = i;
    J = 2 * (p - paired_before(i));
    width = (J + 1 <= I) ? 2 : 1;
}

struct GramArgs {
    float* C;                    // [H][ldc][ldc] (symmetric) or off-indexed [sum t][ldc] (rect)
    const int32_t* offsets;
    int64_t ldc;
    int n;
    int nb;                      // B operand columns (rect mode: d)
    int32_t* status;
    long long wait_limit;        // bounded-wait limit, SM clock cycles
};

// grid (tiles, H), block 192.  SYM: the paired lower tiles of the t x t
// product of A with itself (B maps = A maps), written to C[h] with leading
// dimension ldc and mirrored into the upper triangle (NB = 256, the widest
// tile).  RECT: tiles (I, 0) of A^T B with B [n][nb], written to C[off +
// i][j].  Maps: bf16 hi / lo arrays.
template <bool SYM, int NB>
__global__ void __launch_bounds__(kGThreads, 1)
    k_gram_tc(const __grid_constant__ CUtensorMap mAh, const __grid_constant__ CUtensorMap mAl,
              const __grid_constant__ CUtensorMap mBh, const __grid_constant__ CUtensorMap mBl, GramArgs g) {
    const long long wait_limit = g.wait_limit;
    const int h = blockIdx.y;
    if (!head_ok(g.status, h)) return;
    const int off = g.offsets[h];
    const int t = g.offsets[h + 1] - off;
    int I, J, width = 1;
    if (SYM) paired_tile(blockIdx.x, I, J, width);
    else {
        I = blockIdx.x;
        J = 0;
    }
    if (I * GB >= t) return;
    constexpr int kStages = gram_stages<SYM>();
    const int nbw = SYM ? width * GB : NB;        // this tile's B columns (the MMA's N)
    constexpr int kA = 2 * kGBox;                 // one 128-column operand term
    constexpr int kB = (NB / 64) * kGBox;
    constexpr int kAH = 0, kAL = kA, kBH = 2 * kA, kBL = 2 * kA + kB;
    constexpr int kStage = 2 * kA + 2 * kB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024g(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kStages * kStage);
    uint64_t* full = bars;                  // [kStages] TMA landed
    uint64_t* empty = full + kStages;       // [kStages] MMAs done reading
    uint64_t* acc_full = empty + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 256);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nk = (g.n + GK - 1) / GK;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&mAh);
            prefetch_tmap(&mAl);
            prefetch_tmap(&mBh);
            prefetch_tmap(&mBl);
            int issued = 0;
            for (int k = 0; k < nk; ++k) {
                const int s = k % kStages;
                if (k >= kStages && !mbar_wait(empty + s, (uint32_t)((k / kStages) - 1) & 1u, abort_flag, wait_limit)) break;
                uint8_t* st = sm + s * kStage;
                mbar_expect_tx(full + s, (uint32_t)(2 * kA + 2 * (nbw / 64) * kGBox));
                for (int b = 0; b < 2; ++b) {
                    tma_load_3d(st + kAH + b * kGBox, &mAh, full + s, I * GB + 64 * b, k * GK, h);
                    tma_load_3d(st + kAL + b * kGBox, &mAl, full + s, I * GB + 64 * b, k * GK, h);
                }
                for (int b = 0; b < nbw / 64; ++b) {
                    tma_load_3d(st + kBH + b * kGBox, &mBh, full + s, J * GB + 64 * b, k * GK, h);
                    tma_load_3d(st + kBL + b * kGBox, &mBl, full + s, J * GB + 64 * b, k * GK, h);
                }
                issued = k + 1;
            }
            for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
                drain(full + k % kStages, (uint32_t)(k / kStages) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, nbw, true, true);
            for (int k = 0; k < nk; ++k) {
                const int s = k % kStages;
                if (!mbar_wait(full + s, (uint32_t)(k / kStages) & 1u, abort_flag, wait_limit)) break;
                fence_after_sync();
                const uint32_t st = smem_addr(sm + s * kStage);
#pragma unroll
                for (int kk = 0; kk < GK / 16; ++kk) {
                    // 16 queries = two 8-row groups; 64-column blocks kGBox apart
                    const uint32_t o = (uint32_t)kk * 2048;
                    const uint64_t dAH = sdesc_sw128(st + kAH + o, kGBox, 1024);
                    const uint64_t dAL = sdesc_sw128(st + kAL + o, kGBox, 1024);
                    const uint64_t dBH = sdesc_sw128(st + kBH + o, kGBox, 1024);
                    const uint64_t dBL = sdesc_sw128(st + kBL + o, kGBox, 1024);
                    mma_ss(tmem, dAH, dBH, idesc, (k > 0 || kk > 0) ? 1u : 0u);
                    mma_ss(tmem, dAH, dBL, idesc, 1u);
                    mma_ss(tmem, dAL, dBH, idesc, 1u);
                }
                mma_commit(empty + s);
            }
            mma_commit(acc_full);
            drain(acc_full, 0);
        }
        __syncwarp();
    } else {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, wait_limit));
        if (ok) {
            fence_after_sync();
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const int i = I * GB + row;
            const int jmax = SYM ? t : g.nb;
#pragma unroll 1
            for (int c = 0; c < nbw / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + c * 32, r);
                tmem_ld_wait();
                const int jb = J + c / 4;             // block column of these 32 (SYM)
                if (i < t) {
                    float* dst = SYM ? g.C + ((int64_t)h * g.ldc + i) * g.ldc + J * GB + c * 32
                                     : g.C + ((int64_t)off + i) * g.ldc + c * 32;
                    const int j0 = J * GB + c * 32;
                    if (j0 + 32 <= jmax) {
#pragma unroll
                        for (int q = 0; q < 32; q += 4)
                            *reinterpret_cast<float4*>(dst + q) =
                                make_float4(__uint_as_float(r[q]), __uint_as_float(r[q + 1]),
                                            __uint_as_float(r[q + 2]), __uint_as_float(r[q + 3]));
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (j0 + q < jmax) dst[q] = __uint_as_float(r[q]);
                    }
                    if (SYM && I != jb) {
                        // mirror into the upper triangle (the sweep inverse reads
                        // both); for a fixed column a warp writes 32 consecutive rows
                        float* dT = g.C + ((int64_t)h * g.ldc + j0) * g.ldc + i;
#pragma unroll 4
                        for (int q = 0; q < 32; ++q)
                            if (j0 + q < jmax) dT[(int64_t)q * g.ldc] = __uint_as_float(r[q]);
                    }
                }
            }
        }
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(g.status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

template <bool SYM, int NB>
constexpr int gram_smem() {
    return gram_stages<SYM>() * (4 * kGBox + 2 * (NB / 64) * kGBox) + 256 + 1024;
}

// fp32 [H][rows][ld] (first `cols` columns) -> bf16 hi / lo arrays of the same
// shape; EXP: the stored values are log2 x.  Columns in [cols, cpad) are
// written as 0.  When colsum is given, the CTA's 128-row column sums of x go
// to colsum[rowtile][off + c] (fp32), to be added in a fixed order; when
// sqpart is given, the CTA's sum of x^2 (double-float per thread) goes to
// sqpart[h][blockIdx.y][blockIdx.x] (the exact trace of x^T x, by parts).
// grid (ceil(cpad / 64), ceil(rows / 128), H), block 256 (64 columns x 4 row groups).
template <bool EXP>
__global__ void __launch_bounds__(256) k_split_hilo(const float* __restrict__ X, int rows, int64_t ld,
                                                    const int32_t* __restrict__ offsets, int fixed_cols,
                                                    __nv_bfloat16* __restrict__ Xh, __nv_bfloat16* __restrict__ Xl,
                                                    float* __restrict__ colsum, int64_t colsum_stride,
                                                    double* __restrict__ sqpart, const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.z;
    if (!head_ok(status, h)) return;
    const int off = offsets ? offsets[h] : 0;
    const int cols = offsets ? offsets[h + 1] - off : fixed_cols;
    const int cpad = (int)round_up(cols, 64);
    const int c = blockIdx.x * 64 + (threadIdx.x & 63);
    if (blockIdx.x * 64 >= cpad) return;
    const int rg = threadIdx.x >> 6;
    const int q0 = blockIdx.y * 128;
    float s = 0.f;
    dfloat sq{0.f, 0.f};
    for (int q = q0 + rg; q < min(rows, q0 + 128); q += 4) {
        const int64_t e = ((int64_t)h * rows + q) * ld + c;
        float x = 0.f;
        if (c < cols) x = EXP ? exp2f(X[e]) : X[e];
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        Xh[e] = hi;
        Xl[e] = __float2bfloat16_rn(x - __bfloat162float(hi));
        s += x;
        df_fma(sq, x, x);
    }
    if (sqpart) {
        __shared__ double wsq[8];
        sq = warp_sum_df(sq);
        if ((threadIdx.x & 31) == 0) wsq[threadIdx.x >> 5] = (double)sq.hi + (double)sq.lo;
        __syncthreads();
        if (threadIdx.x == 0) {
            double tot = 0.0;
            for (int w = 0; w < 8; ++w) tot += wsq[w];
            sqpart[((int64_t)h * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x] = tot;
        }
    }
    if (colsum) {
        __shared__ float red[4][64];
        red[rg][threadIdx.x & 63] = s;
        __syncthreads();
        if (rg == 0 && c < cols)
            colsum[(int64_t)blockIdx.y * colsum_stride + off + c] =
                (red[0][threadIdx.x] + red[1][threadIdx.x]) + (red[2][threadIdx.x] + red[3][threadIdx.x]);
    }
}

// b[off + c] = sum over row tiles of colsum (double, fixed order).  grid (ceil(max_t / 256), H).
__global__ void k_colsum_total(const float* __restrict__ colsum, int ntiles, int64_t stride,
                               const int32_t* __restrict__ offsets, float* __restrict__ b,
                               const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int c = blockIdx.x * 256 + threadIdx.x;
    if (c >= t) return;
    double v = 0.0;
    for (int k = 0; k < ntiles; ++k) v += (double)colsum[(int64_t)k * stride + off + c];
    b[off + c] = (float)v;
}

// ---------------------------------------------------------------- C_v = M^{-1} R
// The least-squares values from the explicit inverse of M (symmetric, so
// C[i][c] = sum_p Minv[p][i] R[p][c]), on the tensor cores with both operands
// as three exact bf16 terms (hi + mid + lo = the fp32 value) and the six
// products hi.hi, hi.mid, mid.hi, hi.lo, lo.hi, mid.mid: the dropped products
// are below 2^-25 of |m||r|, under fp32 rounding, which an inverse with a
// large condition number needs.  The contraction runs over each head's own
// t_h rows (64 per stage, two stages); rows past t_h are zero in the split
// arrays.

__device__ __forceinline__ void split3(float x, __nv_bfloat16& hi, __nv_bfloat16& mid, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);
    mid = __float2bfloat16_rn(r1);
    lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
}

// grid (ceil(ldA/256), ldA, H): Minv rows/columns < t_h -> [3][H][ldA][ldA], 0 elsewhere.
__global__ void k_split3_square(const float* __restrict__ Minv, int64_t ldA, const int32_t* __restrict__ offsets,
                                __nv_bfloat16* __restrict__ out, int64_t ts, const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.z;
    if (!head_ok(status, h)) return;
    const int t = offsets[h + 1] - offsets[h];
    const int r = blockIdx.y, c = blockIdx.x * 256 + threadIdx.x;
    if (c >= ldA) return;
    const int64_t e = ((int64_t)h * ldA + r) * ldA + c;
    const float x = (r < t && c < t) ? Minv[e] : 0.f;
    __nv_bfloat16 a, b, d;
    split3(x, a, b, d);
    out[e] = a;
    out[ts + e] = b;
    out[2 * ts + e] = d;
}

// grid (ldA, H), block d: R [sum t][d] -> [3][H][ldA][d], rows past t_h zero.
__global__ void k_split3_rows(const float* __restrict__ R, int d, int64_t ldA, const int32_t* __restrict__ offsets,
                              __nv_bfloat16* __restrict__ out, int64_t ts, const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.y, r = blockIdx.x, c = threadIdx.x;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const float x = r < t ? R[((int64_t)off + r) * d + c] : 0.f;
    const int64_t e = ((int64_t)h * ldA + r) * d + c;
    __nv_bfloat16 a, b, dd;
    split3(x, a, b, dd);
    out[e] = a;
    out[ts + e] = b;
    out[2 * ts + e] = dd;
}

constexpr int kApStages = 2;

template <int NB>
__host__ __device__ constexpr int apply3_stage() {
    return 3 * 2 * kGBox + 3 * (NB / 64) * kGBox;
}
template <int NB>
__host__ __device__ constexpr int apply3_smem() {
    return kApStages * apply3_stage<NB>() + 256 + 1024;
}

// grid (ceil(max_t/128), H), block 192: rows 128 I .. of C_v for head h.
// Warp 0 TMA, warp 1 MMA and TMEM owner, warps 2..5 epilogue (lane = row).
template <int NB>
__global__ void __launch_bounds__(kGThreads, 1)
    k_apply3_tc(const __grid_constant__ CUtensorMap mM0, const __grid_constant__ CUtensorMap mM1,
                const __grid_constant__ CUtensorMap mM2, const __grid_constant__ CUtensorMap mR0,
                const __grid_constant__ CUtensorMap mR1, const __grid_constant__ CUtensorMap mR2,
                const int32_t* __restrict__ offsets, float* __restrict__ C, int32_t* __restrict__ status,
                long long wait_limit) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int I = blockIdx.x;
    if (I * GB >= t) return;
    constexpr int kA = 2 * kGBox;                 // one 128-column term of Minv
    constexpr int kB = (NB / 64) * kGBox;         // one term of R
    constexpr int kStage = apply3_stage<NB>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024g(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kApStages * kStage);
    uint64_t* full = bars;
    uint64_t* empty = full + kApStages;
    uint64_t* acc_full = empty + kApStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kApStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, NB < 32 ? 32 : NB);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nk = (t + GK - 1) / GK;

    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap* mm[3] = {&mM0, &mM1, &mM2};
            const CUtensorMap* mr[3] = {&mR0, &mR1, &mR2};
            int issued = 0;
            for (int k = 0; k < nk; ++k) {
                const int s = k % kApStages;
                if (k >= kApStages && !mbar_wait(empty + s, (uint32_t)((k / kApStages) - 1) & 1u, abort_flag, wait_limit)) break;
                uint8_t* st = sm + s * kStage;
                mbar_expect_tx(full + s, (uint32_t)kStage);
#pragma unroll
                for (int q = 0; q < 3; ++q) {
#pragma unroll
                    for (int b = 0; b < 2; ++b)
                        tma_load_3d(st + q * kA + b * kGBox, mm[q], full + s, I * GB + 64 * b, k * GK, h);
#pragma unroll
                    for (int b = 0; b < NB / 64; ++b)
                        tma_load_3d(st + 3 * kA + q * kB + b * kGBox, mr[q], full + s, 64 * b, k * GK, h);
                }
                issued = k + 1;
            }
            for (int k = (issued > kApStages ? issued - kApStages : 0); k < issued; ++k)
                drain(full + k % kApStages, (uint32_t)(k / kApStages) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, NB, true, true);
            // (Minv term, R term) pairs, smallest products first
            constexpr int pa[6] = {2, 0, 1, 1, 0, 0};
            constexpr int pb[6] = {0, 2, 1, 0, 1, 0};
            for (int k = 0; k < nk; ++k) {
                const int s = k % kApStages;
                if (!mbar_wait(full + s, (uint32_t)(k / kApStages) & 1u, abort_flag, wait_limit)) break;
                fence_after_sync();
                const uint32_t st = smem_addr(sm + s * kStage);
#pragma unroll
                for (int kk = 0; kk < GK / 16; ++kk) {
                    const uint32_t o = (uint32_t)kk * 2048;
#pragma unroll
                    for (int m = 0; m < 6; ++m) {
                        const uint64_t da = sdesc_sw128(st + pa[m] * kA + o, kGBox, 1024);
                        const uint64_t db = sdesc_sw128(st + 3 * kA + pb[m] * kB + o, kGBox, 1024);
                        mma_ss(tmem, da, db, idesc, (k > 0 || kk > 0 || m > 0) ? 1u : 0u);
                    }
                }
                mma_commit(empty + s);
            }
            mma_commit(acc_full);
            drain(acc_full, 0);
        }
        __syncwarp();
    } else {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, wait_limit));
        if (ok) {
            fence_after_sync();
            const int quarter = warp & 3;
            const int i = I * GB + quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
#pragma unroll 1
            for (int c = 0; c < NB / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + c * 32, r);
                tmem_ld_wait();
                if (i < t) {
                    float* dst = C + ((int64_t)off + i) * NB + c * 32;
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4*>(dst + q) =
                            make_float4(__uint_as_float(r[q]), __uint_as_float(r[q + 1]), __uint_as_float(r[q + 2]),
                                        __uint_as_float(r[q + 3]));
                }
            }
        }
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, NB < 32 ? 32 : NB);
}

}  // namespace

bool make_map_bf16(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H);   // tmap.cu

// C = A^T A (lower tiles, mirrored) from the hi / lo arrays of A
// ([H][n][ld] bf16), t_h columns per head.
cudaError_t launch_gram_sym_tc(const void* Ah, const void* Al, const int32_t* offsets, int H, int n, int max_t,
                               int64_t ld, float* C, int64_t ldc, int32_t* status, long long wait_limit,
                               cudaStream_t st) {
    CUtensorMap mh, ml;
    if (!make_map_bf16(&mh, Ah, (int)ld, ld, n, H) || !make_map_bf16(&ml, Al, (int)ld, ld, n, H))
        return cudaErrorInvalidValue;
    constexpr int smem = gram_smem<true, 256>();
    static_assert(smem <= 227 * 1024, "Gram shared memory");
    cudaError_t e = cudaFuncSetAttribute(k_gram_tc<true, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nt = (max_t + GB - 1) / GB;
    GramArgs g{C, offsets, ldc, n, 0, status, wait_limit};
    k_gram_tc<true, 256><<<dim3(paired_before(nt), H), kGThreads, smem, st>>>(mh, ml, mh, ml, g);
    return cudaGetLastError();
}

// C[off + i][j] = sum_q A[q][i] B[q][j] from hi / lo arrays: A [H][n][ld], B [H][n][d].
cudaError_t launch_gram_rect_tc(int d, const void* Ah, const void* Al, const void* Bh, const void* Bl,
                                const int32_t* offsets, int H, int n, int max_t, int64_t ld, float* C,
                                int32_t* status, long long wait_limit, cudaStream_t st) {
    CUtensorMap mah, mal, mbh, mbl;
    if (!make_map_bf16(&mah, Ah, (int)ld, ld, n, H) || !make_map_bf16(&mal, Al, (int)ld, ld, n, H) ||
        !make_map_bf16(&mbh, Bh, d, d, n, H) || !make_map_bf16(&mbl, Bl, d, d, n, H))
        return cudaErrorInvalidValue;
    GramArgs g{C, offsets, d, n, d, status, wait_limit};
    dim3 grid((max_t + GB - 1) / GB, H);
    if (d == 128) {
        constexpr int smem = gram_smem<false, 128>();
        cudaError_t e = cudaFuncSetAttribute(k_gram_tc<false, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_gram_tc<false, 128><<<grid, kGThreads, smem, st>>>(mah, mal, mbh, mbl, g);
    } else {
        constexpr int smem = gram_smem<false, 64>();
        cudaError_t e = cudaFuncSetAttribute(k_gram_tc<false, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_gram_tc<false, 64><<<grid, kGThreads, smem, st>>>(mah, mal, mbh, mbl, g);
    }
    return cudaGetLastError();
}

// b[off + c] = sum over the row-tile partials (fixed order).
cudaError_t launch_colsum_total(const float* part, int ntiles, int64_t stride, const int32_t* offsets, float* b,
                                int H, int max_cols, const int32_t* status, cudaStream_t st) {
    {
        const cudaError_t le = launch_dep(k_colsum_total, dim3(dim3((max_cols + 255) / 256, H)), dim3(256), 0, st,
                                          part, ntiles, stride, offsets, b, status);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}

// fp32 [H][rows][ld] -> bf16 hi / lo.  offsets given: t_h addressed columns
// per head (padded to 64 with zeros); else `cols` for every head.  exp_mode:
// stored values are log2.  colsum (optional): b = column sums, through the
// per-row-tile partials in `part` ([ceil(rows/128)][H * max_t]).
cudaError_t launch_split_hilo(bool exp_mode, const float* X, int H, int rows, int64_t ld, const int32_t* offsets,
                              int cols, int max_cols, void* Xh, void* Xl, float* part, float* colsum, double* sqpart,
                              const int32_t* status, cudaStream_t st) {
    const int rt = (rows + 127) / 128;
    const int64_t stride = (int64_t)H * max_cols;
    dim3 grid((unsigned)((round_up(max_cols, 64) + 63) / 64), rt, H);
    if (sqpart) {
        cudaError_t e = cudaMemsetAsync(sqpart, 0, sizeof(double) * grid.x * grid.y * H, st);
        if (e != cudaSuccess) return e;
    }
    if (exp_mode)
        {
            const cudaError_t le = launch_dep(k_split_hilo<true>, dim3(grid), dim3(256), 0, st, X, rows, ld, offsets,
                                              cols, (__nv_bfloat16*)Xh, (__nv_bfloat16*)Xl, colsum ? part : nullptr,
                                              stride, sqpart, status);
            if (le != cudaSuccess) return le;
        }
    else
        {
            const cudaError_t le = launch_dep(k_split_hilo<false>, dim3(grid), dim3(256), 0, st, X, rows, ld, offsets,
                                              cols, (__nv_bfloat16*)Xh, (__nv_bfloat16*)Xl, colsum ? part : nullptr,
                                              stride, sqpart, status);
            if (le != cudaSuccess) return le;
        }
    if (colsum && offsets)
        {
            const cudaError_t le = launch_dep(k_colsum_total, dim3(dim3((max_cols + 255) / 256, H)), dim3(256), 0, st,
                                              part, rt, stride, offsets, colsum, status);
            if (le != cudaSuccess) return le;
        }
    return cudaGetLastError();
}

// C [sum t][d] = M^{-1} R on the tensor cores.  Minv: fp32 [H][ldA][ldA]
// (rows / columns < t_h valid); R: fp32 [sum t][d]; split: scratch of
// 6 * H * ldA * (ldA + d) bytes (the bf16 terms of both operands).
size_t apply_inverse_tc_scratch(int H, int64_t ldA, int d) { return (size_t)6 * H * ldA * (ldA + d); }

cudaError_t launch_apply_inverse_tc(int d, const float* Minv, const float* R, const int32_t* offsets, int H,
                                    int max_t, int64_t ldA, void* split, float* C, int32_t* status,
                                    long long wait_limit, cudaStream_t st) {
    __nv_bfloat16* Ms = static_cast<__nv_bfloat16*>(split);
    const int64_t tsm = (int64_t)H * ldA * ldA;
    __nv_bfloat16* Rs = Ms + 3 * tsm;
    const int64_t tsr = (int64_t)H * ldA * d;
    {
        const cudaError_t le = launch_dep(k_split3_square, dim3(dim3((unsigned)((ldA + 255) / 256), (unsigned)ldA,
                                          H)), dim3(256), 0, st, Minv, ldA, offsets, Ms, tsm, status);
        if (le != cudaSuccess) return le;
    }
    {
        const cudaError_t le = launch_dep(k_split3_rows, dim3(dim3((unsigned)ldA, H)), dim3(d), 0, st, R, d, ldA,
                                          offsets, Rs, tsr, status);
        if (le != cudaSuccess) return le;
    }
    CUtensorMap mm[3], mr[3];
    for (int q = 0; q < 3; ++q)
        if (!make_map_bf16(&mm[q], Ms + q * tsm, (int)ldA, ldA, (int)ldA, H) ||
            !make_map_bf16(&mr[q], Rs + q * tsr, d, d, (int)ldA, H))
            return cudaErrorInvalidValue;
    dim3 grid((max_t + GB - 1) / GB, H);
    if (d == 128) {
        constexpr int smem = apply3_smem<128>();
        cudaError_t e = cudaFuncSetAttribute(k_apply3_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_apply3_tc<128><<<grid, kGThreads, smem, st>>>(mm[0], mm[1], mm[2], mr[0], mr[1], mr[2], offsets, C, status,
                                                        wait_limit);
    } else {
        constexpr int smem = apply3_smem<64>();
        cudaError_t e = cudaFuncSetAttribute(k_apply3_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_apply3_tc<64><<<grid, kGThreads, smem, st>>>(mm[0], mm[1], mm[2], mr[0], mr[1], mr[2], offsets, C, status,
                                                        wait_limit);
    }
    return cudaGetLastError();
}

}  // namespace kvc

