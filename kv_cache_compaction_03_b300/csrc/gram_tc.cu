// Tensor-core Gram products of the two least-squares fits ("Fast KV
// Compaction via Attention Matching", section 2, fitting beta by NNLS and
// C_v by least squares through the normal equations):
//
//   G = A'^T A'   (mass matrix, t x t, lower tiles)
//   M = X^T X     (biased softmax, t x t, lower tiles)
//   R = X^T O     (t x d)
//
// C[i][j] = sum_q A[q][i] B[q][j] over the n reference queries, with A and B
// fp32 row-major [n][ld].  The products run on the tcgen05 tensor cores in
// bf16 with three terms per product: every operand is split as x = hi + lo
// with hi = bf16(x) and lo = bf16(x - hi) (round to nearest), and C
// accumulates A_hi B_hi + A_hi B_lo + A_lo B_hi in fp32.  The split carries
// ~2^-17 of each value and the dropped A_lo B_lo term is ~2^-18 relative;
// both errors have random sign, so a sum over the queries keeps close to fp32
// accuracy.  (Both operands are MN-major here: the queries are the
// contraction and the outer dimension of the stored matrices.)
//
// For G the stored operand is log2 A' (as the mass-logit pass writes it) and
// the split stage applies exp2 first; the CTAs of the first column tile also
// sum A' over the queries, b = A'^T 1, per column, in double, in a fixed
// order.
//
// One CTA per 128 x 128 output tile (x head).  Warp roles:
//   warp 0       TMA producer: raw fp32 tiles [32 queries][32 columns] with
//                128-byte swizzle, four per 128-column operand tile
//   warp 1       MMA issuer; owns the TMEM accumulator (128 columns)
//   warps 2..5   split every landed fp32 element into bf16 (hi, lo) and write
//                them into the MN-major 128-byte-swizzled operand layout
//                ([32 queries][64 columns] blocks), then run the epilogue
//                (TMEM -> global)
#include "tc.cuh"

namespace kvc {
using namespace tc;

namespace {

constexpr int GB = 128;                 // output tile
constexpr int GK = 32;                  // queries per pipeline stage
constexpr int kGBox = GK * 128;         // one [32][32] fp32 box, or one [32][64] bf16 block: 4 KB
constexpr int kOpBytes = 4 * kGBox;     // one 128-column fp32 operand tile: 16 KB
constexpr int kStages = 3;
constexpr int kGThreads = 192;

__device__ __forceinline__ uint8_t* align1024g(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
    int never = 0;
    (void)mbar_wait(bar, parity, &never);
}

__device__ __forceinline__ void tri_tile(int p, int& I, int& J) {
    int i = (int)((sqrtf(8.f * (float)p + 1.f) - 1.f) * 0.5f);
    while (i * (i + 1) / 2 > p) --i;
    while ((i + 1) * (i + 2) / 2 <= p) ++i;
    I = i;
    J = p - i * (i + 1) / 2;
}

struct GramArgs {
    float* C;                    // [H][ldc_rows][ldc] (symmetric) or off-indexed [sum t][ldc] (rect)
    float* colsum;               // EXP mode: b[off + i] = sum_q A'[q][i]
    const int32_t* offsets;
    int64_t ldc;
    int n;
    int nb;                      // B operand columns (rect mode: d)
    int32_t* status;
};

// One float4 of a landed raw tile (4 consecutive columns of one query row)
// -> bf16 (hi, lo) pairs.  EXP applies exp2 first and zeroes rows past the
// last query (the TMA fill value 0 would become 1).  Returns the fp32 values
// (for the column sums).
template <bool EXP>
__device__ __forceinline__ float4 split4(float4 x, uint2& hi, uint2& lo, bool row_valid) {
    if (EXP) {
        x.x = row_valid ? exp2f(x.x) : 0.f;
        x.y = row_valid ? exp2f(x.y) : 0.f;
        x.z = row_valid ? exp2f(x.z) : 0.f;
        x.w = row_valid ? exp2f(x.w) : 0.f;
    }
    hi.x = pack_bf16(x.x, x.y);
    hi.y = pack_bf16(x.z, x.w);
    lo.x = pack_bf16(x.x - bf16_lo(hi.x), x.y - bf16_hi(hi.x));
    lo.y = pack_bf16(x.z - bf16_lo(hi.y), x.w - bf16_hi(hi.y));
    return x;
}

// grid (tiles, H), block 192.  SYM: lower tiles of the t x t product of A with
// itself (B map = A map), written to C[h] with leading dimension ldc.  RECT:
// tiles (I, 0) of A^T B with B [n][nb], written to C[off + i][j].
template <bool SYM, int NB, bool EXP>
__global__ void __launch_bounds__(kGThreads, 1)
    k_gram_tc(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB, GramArgs g) {
    const int h = blockIdx.y;
    if (!head_ok(g.status, h)) return;
    const int off = g.offsets[h];
    const int t = g.offsets[h + 1] - off;
    int I, J;
    if (SYM) tri_tile(blockIdx.x, I, J);
    else {
        I = blockIdx.x;
        J = 0;
    }
    if (I * GB >= t) return;
    constexpr int kBBytes = (NB / 32) * kGBox;               // raw fp32 B tile
    // stage: raw A | raw B | A hi | A lo | B hi | B lo (bf16 tiles are half size)
    constexpr int kAHi = kOpBytes + kBBytes;
    constexpr int kALo = kAHi + kOpBytes / 2;
    constexpr int kBHi = kALo + kOpBytes / 2;
    constexpr int kBLo = kBHi + kBBytes / 2;
    constexpr int kStage = kBLo + kBBytes / 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024g(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kStages * kStage);
    uint64_t* full = bars;                  // [kStages] TMA landed
    uint64_t* conv = full + kStages;        // [kStages] split done (128 arrivals)
    uint64_t* empty = conv + kStages;       // [kStages] MMAs done reading
    uint64_t* acc_full = empty + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(conv + s, 128);
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nk = (g.n + GK - 1) / GK;
    auto stage_ptr = [&](int s) { return sm + s * kStage; };

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&mA);
            prefetch_tmap(&mB);
            int issued = 0;
            for (int k = 0; k < nk; ++k) {
                const int s = k % kStages;
                if (k >= kStages && !mbar_wait(empty + s, (uint32_t)((k / kStages) - 1) & 1u, abort_flag)) break;
                uint8_t* st = stage_ptr(s);
                mbar_expect_tx(full + s, (uint32_t)(kOpBytes + kBBytes));
                for (int b = 0; b < 4; ++b) tma_load_3d(st + b * kGBox, &mA, full + s, I * GB + 32 * b, k * GK, h);
                for (int b = 0; b < NB / 32; ++b)
                    tma_load_3d(st + kOpBytes + b * kGBox, &mB, full + s, J * GB + 32 * b, k * GK, h);
                issued = k + 1;
            }
            for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
                drain(full + k % kStages, (uint32_t)(k / kStages) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, NB, true, true);
            for (int k = 0; k < nk; ++k) {
                const int s = k % kStages;
                if (!mbar_wait(conv + s, (uint32_t)(k / kStages) & 1u, abort_flag)) break;
                fence_after_sync();
                const uint32_t st = smem_addr(stage_ptr(s));
#pragma unroll
                for (int kk = 0; kk < GK / 16; ++kk) {
                    // 16 queries = two 8-row groups; 64-column blocks kGBox apart
                    const uint32_t o = (uint32_t)kk * 2048;
                    const uint64_t dAH = sdesc_sw128(st + kAHi + o, kGBox, 1024);
                    const uint64_t dAL = sdesc_sw128(st + kALo + o, kGBox, 1024);
                    const uint64_t dBH = sdesc_sw128(st + kBHi + o, kGBox, 1024);
                    const uint64_t dBL = sdesc_sw128(st + kBLo + o, kGBox, 1024);
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
        const int ct = threadIdx.x - 64;            // 0..127
        // Column sums (EXP mode, first column tile): float4 e = ct + 128 m of
        // the A tile lies in box m/2, row (ct/8) + 16 (m%2), and its 16-byte
        // chunk is the logical chunk (ct%8) ^ ((ct/8)%8) under the 128-byte
        // swizzle, so each thread always sees the same 16 columns.
        const bool do_b = EXP && J == 0;
        double bsum[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) bsum[q] = 0.0;
        bool ok = true;
        for (int k = 0; k < nk; ++k) {
            const int s = k % kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(full + s, (uint32_t)(k / kStages) & 1u, abort_flag));
            if (!ok) break;
            uint8_t* st = stage_ptr(s);
            // float4 e = ct + 128 m of a raw tile: box m / 2, query row
            // (ct / 8) + 16 (m % 2), physical 16-byte chunk ct % 8, logical
            // chunk lc = (ct % 8) ^ (row % 8) -> columns 32 (m / 2) + 4 lc ..+3.
            // Its bf16 image goes to 64-column block m / 4, logical chunk
            // ((m / 2) % 2) * 4 + lc / 2, half lc % 2, swizzled by row % 8.
            const int r0 = k * GK + (ct >> 3);
            const int lc = (ct & 7) ^ ((ct >> 3) & 7);
            const float4* raw = reinterpret_cast<const float4*>(st);
#pragma unroll
            for (int m = 0; m < kOpBytes / 16 / 128; ++m) {
                const int q = (ct >> 3) + 16 * (m & 1);
                uint2 hi, lo;
                const float4 v = split4<EXP>(raw[ct + 128 * m], hi, lo, r0 + 16 * (m & 1) < g.n);
                if (do_b) {
                    bsum[(m >> 1) * 4 + 0] += (double)v.x;
                    bsum[(m >> 1) * 4 + 1] += (double)v.y;
                    bsum[(m >> 1) * 4 + 2] += (double)v.z;
                    bsum[(m >> 1) * 4 + 3] += (double)v.w;
                }
                const int lc2 = ((m >> 1) & 1) * 4 + (lc >> 1);
                const int byte = (m >> 2) * kGBox + q * 128 + ((lc2 ^ (q & 7)) << 4) + (lc & 1) * 8;
                *reinterpret_cast<uint2*>(st + kAHi + byte) = hi;
                *reinterpret_cast<uint2*>(st + kALo + byte) = lo;
            }
            const float4* rawb = reinterpret_cast<const float4*>(st + kOpBytes);
#pragma unroll
            for (int m = 0; m < kBBytes / 16 / 128; ++m) {
                const int q = (ct >> 3) + 16 * (m & 1);
                uint2 hi, lo;
                (void)split4<EXP>(rawb[ct + 128 * m], hi, lo, r0 + 16 * (m & 1) < g.n);
                const int lc2 = ((m >> 1) & 1) * 4 + (lc >> 1);
                const int byte = (m >> 2) * kGBox + q * 128 + ((lc2 ^ (q & 7)) << 4) + (lc & 1) * 8;
                *reinterpret_cast<uint2*>(st + kBHi + byte) = hi;
                *reinterpret_cast<uint2*>(st + kBLo + byte) = lo;
            }
            fence_proxy_async();
            mbar_arrive(conv + s);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag));
        if (do_b) {
            // every MMA is done, so stage 0 can hold the [16][128] partial sums
            double* red = reinterpret_cast<double*>(sm);
            const int grp = ct >> 3, chunk = (ct & 7) ^ ((ct >> 3) & 7);
            if (ok) {
#pragma unroll
                for (int q = 0; q < 16; ++q) red[grp * 128 + (q >> 2) * 32 + chunk * 4 + (q & 3)] = bsum[q];
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int i = I * GB + ct;
            if (ok && i < t) {
                double v = 0.0;
                for (int r = 0; r < 16; ++r) v += red[r * 128 + ct];
                g.colsum[off + i] = (float)v;
            }
        }
        if (ok) {
            fence_after_sync();
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const int i = I * GB + row;
            const int jmax = SYM ? t : g.nb;
#pragma unroll 1
            for (int c = 0; c < NB / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + c * 32, r);
                tmem_ld_wait();
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
                }
            }
        }
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(g.status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 128);
}

template <int NB>
constexpr int gram_smem() {
    // per stage: raw fp32 A and B, plus bf16 hi and lo images of both (same total bytes)
    return kStages * 2 * (kOpBytes + (NB / 32) * kGBox) + 256 + 1024;
}

}  // namespace

bool make_map_f32(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H);   // tmap.cu

// C = A^T A (lower tiles) for A fp32 [H][n][ld] with t_h columns per head.
// exp_mode: the stored values are log2 A (C = exp2(.)^T exp2(.)), and the
// column sums of exp2(A) go to colsum (off-indexed).
cudaError_t launch_gram_sym_tc(bool exp_mode, const float* A, const int32_t* offsets, int H, int n, int max_t,
                               int64_t ld, float* C, int64_t ldc, float* colsum, int32_t* status, cudaStream_t st) {
    CUtensorMap mA;
    if (!make_map_f32(&mA, A, (int)ld, ld, n, H)) return cudaErrorInvalidValue;
    constexpr int smem = gram_smem<128>();
    const int nt = (max_t + GB - 1) / GB;
    GramArgs g{C, colsum, offsets, ldc, n, 0, status};
    dim3 grid(nt * (nt + 1) / 2, H);
    if (exp_mode) {
        cudaError_t e = cudaFuncSetAttribute(k_gram_tc<true, 128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_gram_tc<true, 128, true><<<grid, kGThreads, smem, st>>>(mA, mA, g);
    } else {
        cudaError_t e = cudaFuncSetAttribute(k_gram_tc<true, 128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_gram_tc<true, 128, false><<<grid, kGThreads, smem, st>>>(mA, mA, g);
    }
    return cudaGetLastError();
}

// C[off + i][j] = sum_q A[q][i] B[q][j] for A fp32 [H][n][ld], B fp32 [H][n][d].
cudaError_t launch_gram_rect_tc(int d, const float* A, const float* B, const int32_t* offsets, int H, int n,
                                int max_t, int64_t ld, float* C, int32_t* status, cudaStream_t st) {
    CUtensorMap mA, mB;
    if (!make_map_f32(&mA, A, (int)ld, ld, n, H) || !make_map_f32(&mB, B, d, d, n, H)) return cudaErrorInvalidValue;
    GramArgs g{C, nullptr, offsets, d, n, d, status};
    dim3 grid((max_t + GB - 1) / GB, H);
    if (d == 128) {
        constexpr int smem = gram_smem<128>();
        cudaError_t e = cudaFuncSetAttribute(k_gram_tc<false, 128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_gram_tc<false, 128, false><<<grid, kGThreads, smem, st>>>(mA, mB, g);
    } else {
        constexpr int smem = gram_smem<64>();
        cudaError_t e = cudaFuncSetAttribute(k_gram_tc<false, 64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_gram_tc<false, 64, false><<<grid, kGThreads, smem, st>>>(mA, mB, g);
    }
    return cudaGetLastError();
}

}  // namespace kvc
