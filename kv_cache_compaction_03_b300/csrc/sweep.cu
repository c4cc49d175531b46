// Explicit inverse of the normal-equation matrices ("Fast KV Compaction via
// Attention Matching", section 2, fitting beta by NNLS and C_v by least
// squares): the block-principal-pivoting NNLS works entirely with H^{-1}
// (its columns for the zero set, the unconstrained solution H^{-1} f and
// refinement steps), and C_v = M^{-1} R, so one inverse per matrix replaces
// every triangular solve.
//
// The inverse is formed in place by the symmetric sweep operator, 64 x 64
// block by block.  With P = A_kk^{-1}, a sweep on block k maps
//   A_ij -> A_ij - A_ik P A_kj,  A_ik -> A_ik P,  A_kj -> P A_kj,  A_kk -> -P
// (i, j != k); after every block has been swept the matrix holds -H^{-1}.
// For a symmetric positive definite H every pivot block is a Schur
// complement and stays positive definite, so no pivoting is needed.  Rows
// and columns past t act as an identity block.
//
//   k_sweep_pivot   grid (blocks, H): every CTA takes the inverse P of the
//                   64 x 64 pivot block (the first block's it forms itself,
//                   by 16 four-pivot sweeps in registers), then computes
//                   U_i = A_ik P for its row block i (stored transposed) and
//                   copies V_i = A_ki; the CTA of row block k + 1 also copies
//                   the next pivot block's inputs
//   k_sweep_update_tc  grid (1 + lower 128 x 128 tiles, H): A_ij -= U_i V_j on
//                   the tcgen05 tensor cores (operands as three exact bf16
//                   terms, six products), with the pivot row / column copies
//                   in the epilogue; on a head's last block the stored result
//                   is negated, so the matrix ends as +H^{-1}.  CTA 0 of each
//                   head meanwhile forms the next pivot block as this step
//                   leaves it and inverts it (look-ahead), so the dependent
//                   chain of step k + 1 overlaps the update of step k
//   k_sweep_mirror  copies the lower triangle into the upper one
//   k_symv          y = H^{-1} v for every head (one warp per row)
// The sweep keeps the symmetric matrix in its lower triangle (row-major,
// leading dimension ldA); an entry above the diagonal is read from its
// mirror image.  The finished inverse is stored in full.
#include "tc.cuh"

namespace kvc {
using namespace tc;

namespace {
constexpr int SB = 64;     // sweep block


struct SweepArgs {
    float* A;                 // [H][ldA][ldA]
    float* U;                 // [H][64][ldA]  U^T: U[p][r] = (A_ik P)[r][p]
    __nv_bfloat16* Us;        // [3][H][64][ldA]  U^T as three bf16 terms
    __nv_bfloat16* Vs;        // [3][H][64][ldA]  V[p][r] = A_kr[p][r], three bf16 terms
    float* P;                 // [H][64][64]  P = A_kk^{-1} of this step
    float* Xnext;             // [H][2][64][64]  A_{k,k+1} and the stored A_{k+1,k+1} before this step's update
    float* Pnext;             // [H][64][64]  P of the next step, formed while this step's update runs
    const int32_t* offsets;
    int64_t ldA;
    int64_t ts;               // elements between the terms of Us / Vs (H * 64 * ldA)
    int k0;                   // first row of the pivot block
    int32_t* status;
    int have_p;               // P of this step was formed by the previous update launch
    long long wait_limit;     // bounded-wait limit of the tensor-core update, SM clock cycles
};

// x = hi + mid + lo exactly (three bf16 terms of 8 significant bits each;
// the subtractions are exact), for fp32 x away from the underflow range.
__device__ __forceinline__ void split3(float x, __nv_bfloat16& hi, __nv_bfloat16& mid, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);
    mid = __float2bfloat16_rn(r1);
    lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
}


constexpr int kPS = SB + 4;      // padded smem row, 16-byte aligned
constexpr int kPivThreads = 128;
constexpr int kCR = 4;           // chain tile rows per thread (columns: 8)

// The 64 x 64 pivot block's inverse in place: Dn holds the block (its lower
// triangle is what is read; rows / columns past t act as identity) and ends
// holding P = D^{-1}.  Run by 128 threads (tid 0..127) that synchronise on
// named barrier 1.
//
// The inversion is a dependent chain, so its cost is the latency of one
// step times the number of steps.  It sweeps four pivots per step (16 steps
// instead of 64 scalar ones): the owner threads publish the group's four
// rows through shared memory, one barrier, then every thread forms the
// group's 4 x 4 inverse in registers and applies it to its own entries.
// Each thread holds a 4 x 8 register tile (rows 4 ty .., columns 8 tx ..);
// the group loop runs as 8 x 2 with the inner 2 unrolled, so the group's
// columns have static register indices.  A non-positive or non-finite
// pivot sets *bad.
__device__ __forceinline__ void sync128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void chain_invert(float (*Dn)[kPS], float (*grp)[4][SB], int* bad_p, int tid, int k0,
                                             int t) {
    constexpr int R = kCR;
    volatile int& bad = *bad_p;
    const int tx = tid & 7, ty = tid >> 3;
    float a[R][8];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = R * ty + i, c = 8 * tx + j;
            const bool in = (k0 + r < t) && (k0 + c < t);    // rows / columns past t: identity
            a[i][j] = in ? ((c <= r) ? Dn[r][c] : Dn[c][r]) : (r == c ? 1.f : 0.f);
        }
    // 16 block steps, each sweeping four pivots at once (rows / columns
    // 4g .. 4g + 3).  With D the group's 4 x 4 block, Qn = -D^{-1}:
    //   a_ij += (a_ig Qn) a_gj,  a_ig <- -(a_ig Qn),  a_gj <- -(Qn a_gj),
    //   a_gg <- Qn,
    // which is exactly four scalar sweeps applied together.  The threads that
    // own the group's rows (ty == g) publish them; after one barrier every
    // thread reads D, the group rows over its own columns and (by symmetry)
    // the group columns over its own rows, forms Qn by four scalar sweeps of
    // D in registers, and updates its tile.
#pragma unroll 1
    for (int gp = 0; gp < 8; ++gp) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int g = 2 * gp + h2;
            float(*Rg)[SB] = grp[h2];
            if (ty == g) {
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    *reinterpret_cast<float4*>(&Rg[i][8 * tx]) = make_float4(a[i][0], a[i][1], a[i][2], a[i][3]);
                    *reinterpret_cast<float4*>(&Rg[i][8 * tx + 4]) = make_float4(a[i][4], a[i][5], a[i][6], a[i][7]);
                }
            }
            sync128();
            float q[4][4], cg[4][4], rg[4][8];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 d4 = *reinterpret_cast<const float4*>(&Rg[m][4 * g]);
                const float4 c4 = *reinterpret_cast<const float4*>(&Rg[m][R * ty]);
                const float4 x0 = *reinterpret_cast<const float4*>(&Rg[m][8 * tx]);
                const float4 x1 = *reinterpret_cast<const float4*>(&Rg[m][8 * tx + 4]);
                q[m][0] = d4.x; q[m][1] = d4.y; q[m][2] = d4.z; q[m][3] = d4.w;
                cg[m][0] = c4.x; cg[m][1] = c4.y; cg[m][2] = c4.z; cg[m][3] = c4.w;
                rg[m][0] = x0.x; rg[m][1] = x0.y; rg[m][2] = x0.z; rg[m][3] = x0.w;
                rg[m][4] = x1.x; rg[m][5] = x1.y; rg[m][6] = x1.z; rg[m][7] = x1.w;
            }
            // q <- -D^{-1} by four scalar sweeps
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                float d = q[p][p];
                if (!(d > 0.f) || !isfinite(d)) {
                    bad = 1;
                    d = 1.f;
                }
                // reciprocal: hardware approximation plus one Newton step (~1 ulp)
                float inv;
                asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(d));
                inv = inv * fmaf(-d, inv, 2.f);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i == p) continue;
                    const float f = q[i][p] * inv;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j != p) q[i][j] = fmaf(-f, q[p][j], q[i][j]);
                    q[i][p] = f;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j != p) q[p][j] *= inv;
                q[p][p] = -inv;
            }
            // one update for every row, so no warp runs two paths: for the
            // group's own rows w = -Qn[i][:] and the old entry is dropped
            // (a_gj <- -(Qn a_gj)); for the others w = a_ig Qn (a_ig = a_gi
            // by symmetry) and a_ij += w a_gj; the group's columns then
            // become -w (a_ig <- -(a_ig Qn), a_gg <- Qn)
            const bool grow = (ty == g);
#pragma unroll
            for (int i = 0; i < R; ++i) {
                float w[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float v = 0.f;
#pragma unroll
                    for (int l = 0; l < 4; ++l) v = fmaf(cg[l][i], q[l][m], v);
                    w[m] = grow ? -q[i][m] : v;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float v = grow ? 0.f : a[i][j];
#pragma unroll
                    for (int m = 0; m < 4; ++m) v = fmaf(w[m], rg[m][j], v);
                    a[i][j] = v;
                }
                if (tx == gp) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) a[i][4 * h2 + jj] = -w[jj];
                }
            }
        }
    }
    // the block now holds -P: store P
    sync128();
#pragma unroll
    for (int i = 0; i < R; ++i) {
        *reinterpret_cast<float4*>(&Dn[R * ty + i][8 * tx]) = make_float4(-a[i][0], -a[i][1], -a[i][2], -a[i][3]);
        *reinterpret_cast<float4*>(&Dn[R * ty + i][8 * tx + 4]) = make_float4(-a[i][4], -a[i][5], -a[i][6], -a[i][7]);
    }
    sync128();
}

// grid (blocks, H), block 128.  Every CTA takes the pivot block's inverse P
// (formed here for the first block, else by the previous update launch),
// then (row blocks i != k) forms U_i = A_ik P.  The CTA of row block k + 1
// also copies A_{k,k+1} and A_{k+1,k+1} for the update launch, whose first
// CTA forms the next pivot block D' = A_{k+1,k+1} - U_{k+1} A_{k,k+1} from
// them (the other CTAs rewrite A meanwhile) and inverts it.
__global__ void __launch_bounds__(kPivThreads) k_sweep_pivot(SweepArgs s) {
    constexpr int NT = kPivThreads;
    grid_dependency_wait();
    const int h = blockIdx.y;
    if (!head_ok(s.status, h)) return;
    const int t = s.offsets[h + 1] - s.offsets[h];
    const int k0 = s.k0;
    if (k0 >= t) return;
    const int r0 = blockIdx.x * SB;
    if (r0 >= t) return;
    __shared__ __align__(16) float Dn[SB][kPS];     // pivot block, then P
    __shared__ __align__(16) float At[SB][kPS];     // At[p][r] = A_ik[r][p]
    __shared__ __align__(16) float grp[2][4][SB];    // a pivot group's rows, double-buffered
    __shared__ int bad;
    const float* A = s.A + (int64_t)h * s.ldA * s.ldA;
    const int tid = threadIdx.x;
    const bool diag = (r0 == k0);
    const bool nextblk = (r0 == k0 + SB);      // row block k + 1: hands the next pivot block's inputs on
    // stage the pivot block (its stored lower triangle is what gets used) or
    // its inverse when that is already formed, and A_ik (rows below the
    // pivot: stored directly; above: the transpose of the stored tile
    // (k, i)); every load is issued before the first store
    {
        const float* Pn = s.Pnext + (int64_t)h * SB * SB;
        float4 dv[8], av[8], xv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + NT * q, r = e >> 4, c4 = (e & 15) * 4;
            dv[q] = s.have_p ? *reinterpret_cast<const float4*>(Pn + r * SB + c4)
                             : *reinterpret_cast<const float4*>(A + (int64_t)(k0 + r) * s.ldA + k0 + c4);
            if (nextblk) xv[q] = *reinterpret_cast<const float4*>(A + (int64_t)(r0 + r) * s.ldA + r0 + c4);
            if (!diag) {
                if (r0 > k0) av[q] = *reinterpret_cast<const float4*>(A + (int64_t)(r0 + r) * s.ldA + k0 + c4);
                else av[q] = *reinterpret_cast<const float4*>(A + (int64_t)(k0 + r) * s.ldA + r0 + c4);
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + NT * q, r = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(&Dn[r][c4]) = dv[q];
            if (nextblk) *reinterpret_cast<float4*>(s.Xnext + ((int64_t)h * 2 + 1) * SB * SB + r * SB + c4) = xv[q];
            if (!diag) {
                const float x[4] = {av[q].x, av[q].y, av[q].z, av[q].w};
                if (r0 > k0) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) At[c4 + j][r] = (r0 + r < t && k0 + c4 + j < t) ? x[j] : 0.f;
                } else {
                    // stored row k0 + r, columns r0 + c4 + j: A_ik[c4 + j][r]
                    *reinterpret_cast<float4*>(&At[r][c4]) = make_float4(
                        (k0 + r < t && r0 + c4 < t) ? x[0] : 0.f, (k0 + r < t && r0 + c4 + 1 < t) ? x[1] : 0.f,
                        (k0 + r < t && r0 + c4 + 2 < t) ? x[2] : 0.f, (k0 + r < t && r0 + c4 + 3 < t) ? x[3] : 0.f);
                }
            }
        }
    }
    __syncthreads();
    if (nextblk) {
        // the next pivot block is D' = A_{k+1,k+1} - U_{k+1} A_{k,k+1}; the
        // update launch forms it (with U_{k+1} from U) and inverts it, from
        // copies of A_{k,k+1} and of A_{k+1,k+1}, which that launch rewrites
        float* X = s.Xnext + (int64_t)h * 2 * SB * SB;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + NT * q, r = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(X + r * SB + c4) = *reinterpret_cast<const float4*>(&At[r][c4]);
        }
    }
    // the first pivot block is inverted here; later ones by the previous
    // update launch (look-ahead)
    if (!s.have_p) {
        if (tid == 0) bad = 0;
        __syncthreads();
        chain_invert(Dn, grp, &bad, tid, k0, t);
        __syncthreads();
        if (bad) {
            if (blockIdx.x == 0 && tid == 0) set_status(s.status, h, KVC_ERR_NOT_SPD);
            return;
        }
    }
    __syncthreads();
    if (diag) {
        float* Ph = s.P + (int64_t)h * SB * SB;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + NT * q, r = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(Ph + r * SB + c4) = *reinterpret_cast<const float4*>(&Dn[r][c4]);
        }
        return;
    }
    // U_i = A_ik P: thread (uy, ux) forms rows 8 uy .. 8 uy + 7, columns 4 ux .. 4 ux + 3
    const int ux = tid & 15, uy = tid >> 4;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int p = 0; p < SB; ++p) {
        const float4 a0 = *reinterpret_cast<const float4*>(&At[p][8 * uy]);
        const float4 a1 = *reinterpret_cast<const float4*>(&At[p][8 * uy + 4]);
        const float4 pv = *reinterpret_cast<const float4*>(&Dn[p][4 * ux]);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float bv[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    // U^T[c][r0 + r] = U[r][c]: for each column c, 8 consecutive rows, in
    // fp32 (the pivot row / column copies) and as three bf16 terms (the
    // tensor-core update's operand)
    const int64_t hb = (int64_t)h * SB * s.ldA + r0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t o = hb + (int64_t)(4 * ux + j) * s.ldA + 8 * uy;
        *reinterpret_cast<float4*>(s.U + o) = make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
        *reinterpret_cast<float4*>(s.U + o + 4) = make_float4(acc[4][j], acc[5][j], acc[6][j], acc[7][j]);
        __align__(16) __nv_bfloat16 th[8], tm[8], tl[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) split3(acc[i][j], th[i], tm[i], tl[i]);
        *reinterpret_cast<uint4*>(s.Us + o) = *reinterpret_cast<const uint4*>(th);
        *reinterpret_cast<uint4*>(s.Us + s.ts + o) = *reinterpret_cast<const uint4*>(tm);
        *reinterpret_cast<uint4*>(s.Us + 2 * s.ts + o) = *reinterpret_cast<const uint4*>(tl);
    }
    // V_i = A_ki = A_ik^T: V[c][r0 + r] = A_ik[r][c] = At[c][r], as three bf16 terms
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int e = tid + NT * q, c = e >> 4, r4 = (e & 15) * 4;
        const float4 v = *reinterpret_cast<const float4*>(&At[c][r4]);
        const float x[4] = {v.x, v.y, v.z, v.w};
        __align__(8) __nv_bfloat16 th[4], tm[4], tl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split3(x[i], th[i], tm[i], tl[i]);
        const int64_t o = hb + (int64_t)c * s.ldA + r4;
        *reinterpret_cast<uint2*>(s.Vs + o) = *reinterpret_cast<const uint2*>(th);
        *reinterpret_cast<uint2*>(s.Vs + s.ts + o) = *reinterpret_cast<const uint2*>(tm);
        *reinterpret_cast<uint2*>(s.Vs + 2 * s.ts + o) = *reinterpret_cast<const uint2*>(tl);
    }
}

__device__ __forceinline__ void tri_tile(int p, int& I, int& J) {
    int i = (int)((sqrtf(8.f * (float)p + 1.f) - 1.f) * 0.5f);
    while (i * (i + 1) / 2 > p) --i;
    while ((i + 1) * (i + 2) / 2 <= p) ++i;
    I = i;
    J = p - i * (i + 1) / 2;
}

// ---------------------------------------------------------------- update
// A_ij -= U_i V_j for every 128 x 128 tile (I >= J) of the lower triangle,
// on the tcgen05 tensor cores: C[i][j] = sum_p U^T[p][i] V[p][j] with K = 64
// (one pivot block).  Both operands are stored [64][ldA] (p rows, the tile
// dimension contiguous): the MN-major layout, loaded by TMA as [64][64]
// bf16 boxes with 128-byte swizzle.  Each fp32 operand is three exact bf16
// terms; the six products hi.hi, hi.mid, mid.hi, hi.lo, lo.hi, mid.mid are
// accumulated in fp32 in tensor memory (smallest first).  The three dropped
// products are below 2^-25 of |u||v|, under fp32 rounding, so the update
// keeps the accuracy of an fp32 FMA product.
// Rows / columns of the pivot block take the sweep's copies instead:
// A_ik <- U_i, A_kj <- U_j^T, A_kk <- -P.  On a head's last pivot block the
// stored result is negated, so the matrix ends as +H^{-1}.
// The fp32 tile of A comes in by TMA too ([32][32] boxes, 128-byte
// swizzle), into the operand space once the products are done (so that two
// CTAs fit on an SM); the epilogue subtracts in shared memory and writes the
// boxes back with TMA stores.  Entries past t inside a box are
// rewritten with sg times their old value minus a zero product (rows and
// columns past t of U and V are zero); nothing reads them.
// Warp roles: warp 0 TMA, warp 1 MMA issuer and TMEM owner (128 columns),
// warps 2..5 epilogue (32 tile rows each).
constexpr int UB = 128;                    // update tile
constexpr int kUBox = 64 * 128;            // [64 p][64 columns] bf16 box: 8 KB
constexpr int kABox = 32 * 128;            // [32 rows][32 columns] fp32 box: 4 KB
constexpr int kUOps = 12 * kUBox;          // operand boxes
constexpr int kUThreads = 192;
constexpr int kUSmem = kUOps + 1024 + 64;
static_assert(16 * kABox <= kUOps, "the A tile reuses the operand space");

__global__ void __launch_bounds__(kUThreads, 2)
    k_sweep_update_tc(const __grid_constant__ CUtensorMap mU0, const __grid_constant__ CUtensorMap mU1,
                      const __grid_constant__ CUtensorMap mU2, const __grid_constant__ CUtensorMap mV0,
                      const __grid_constant__ CUtensorMap mV1, const __grid_constant__ CUtensorMap mV2,
                      const __grid_constant__ CUtensorMap mA, SweepArgs s) {
    grid_dependency_wait();
    const long long wait_limit = s.wait_limit;
    const int h = blockIdx.y;
    if (!head_ok(s.status, h)) return;
    const int t = s.offsets[h + 1] - s.offsets[h];
    const int k0 = s.k0;
    if (k0 >= t) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (blockIdx.x == 0) {
        // look-ahead, while the other CTAs update the tiles: the next pivot
        // block D' = A_{k+1,k+1} - U_{k+1} A_{k,k+1} from the copies the pivot
        // launch took and its U_{k+1}, then its inverse, for the next pivot
        // launch.  The arrays are addressed from a shared-memory symbol (no
        // integer round trip), so the compiler emits shared loads.
        const int tid = threadIdx.x;
        const int r1 = k0 + SB;
        if (r1 >= t || tid >= kPivThreads) return;
        float(*Dn)[kPS] = reinterpret_cast<float(*)[kPS]>(smem_raw);                        // D', then P
        float(*Ut)[kPS] = reinterpret_cast<float(*)[kPS]>(smem_raw + SB * kPS * 4);         // Ut[p][r] = U_{k+1}[r][p]
        float(*Vt)[kPS] = reinterpret_cast<float(*)[kPS]>(smem_raw + 2 * SB * kPS * 4);     // Vt[p][c] = A_{k,k+1}[p][c]
        float(*grp)[4][SB] = reinterpret_cast<float(*)[4][SB]>(smem_raw + 3 * SB * kPS * 4);
        int* bad = reinterpret_cast<int*>(smem_raw + 3 * SB * kPS * 4 + 2 * 4 * SB * 4);
        const float* X = s.Xnext + (int64_t)h * 2 * SB * SB;
        const float* Uh = s.U + (int64_t)h * SB * s.ldA + r1;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + kPivThreads * q, r = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(&Vt[r][c4]) = *reinterpret_cast<const float4*>(X + r * SB + c4);
            *reinterpret_cast<float4*>(&Dn[r][c4]) = *reinterpret_cast<const float4*>(X + SB * SB + r * SB + c4);
            *reinterpret_cast<float4*>(&Ut[r][c4]) = *reinterpret_cast<const float4*>(Uh + r * s.ldA + c4);
        }
        sync128();
        // D'[r][c] for the stored (lower) entries; thread (uy, ux): rows
        // 8 uy .., columns 4 ux ..; each thread rewrites only its own entries
        const int ux = tid & 15, uy = tid >> 4;
        float dn[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 d4 = *reinterpret_cast<const float4*>(&Dn[8 * uy + i][4 * ux]);
            dn[i][0] = d4.x; dn[i][1] = d4.y; dn[i][2] = d4.z; dn[i][3] = d4.w;
        }
#pragma unroll 4
        for (int p = 0; p < SB; ++p) {
            const float4 u0 = *reinterpret_cast<const float4*>(&Ut[p][8 * uy]);
            const float4 u1 = *reinterpret_cast<const float4*>(&Ut[p][8 * uy + 4]);
            const float4 v4 = *reinterpret_cast<const float4*>(&Vt[p][4 * ux]);
            const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) dn[i][j] = fmaf(-uv[i], vv[j], dn[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(&Dn[8 * uy + i][4 * ux]) = make_float4(dn[i][0], dn[i][1], dn[i][2], dn[i][3]);
        if (tid == 0) *bad = 0;
        sync128();
        chain_invert(Dn, grp, bad, tid, r1, t);
        if (*reinterpret_cast<volatile int*>(bad)) {
            if (tid == 0) set_status(s.status, h, KVC_ERR_NOT_SPD);
            return;
        }
        float* Ph = s.Pnext + (int64_t)h * SB * SB;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + kPivThreads * q, r = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(Ph + r * SB + c4) = *reinterpret_cast<const float4*>(&Dn[r][c4]);
        }
        return;
    }
    int I, J;
    tri_tile(blockIdx.x - 1, I, J);
    if (I * UB >= t) return;
    const float sg = (k0 + SB >= t) ? -1.f : 1.f;
    uint8_t* smA = sm;                       // A boxes (after the MMAs): (row quarter q, chunk c) at (4 q + c) * kABox
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kUOps);
    uint64_t* fullA = full + 1;
    uint64_t* acc_full = full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(fullA, 1);
        mbar_init(acc_full, 1);
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
            const CUtensorMap* mu[3] = {&mU0, &mU1, &mU2};
            const CUtensorMap* mv[3] = {&mV0, &mV1, &mV2};
            prefetch_tmap(&mA);
            mbar_expect_tx(full, (uint32_t)kUOps);
#pragma unroll
            for (int q = 0; q < 3; ++q)
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    tma_load_3d(sm + (2 * q + b) * kUBox, mu[q], full, I * UB + 64 * b, 0, h);
                    tma_load_3d(sm + (6 + 2 * q + b) * kUBox, mv[q], full, J * UB + 64 * b, 0, h);
                }
            // the A tile goes where the operands were, once the MMAs have read them
            if (mbar_wait(acc_full, 0, abort_flag, wait_limit)) {
                mbar_expect_tx(fullA, 16u * kABox);
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tma_load_3d(smA + (4 * q + c) * kABox, &mA, fullA, J * UB + 32 * c, I * UB + 32 * q, h);
                int never = 0;
                (void)mbar_wait(fullA, 0, &never);
            } else {
                // given up: the operand copies issued above must still land
                // before the CTA leaves
                int never = 0;
                (void)mbar_wait(full, 0, &never);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            if (mbar_wait(full, 0, abort_flag, wait_limit)) {
                fence_after_sync();
                constexpr uint32_t idesc = idesc_bf16(128, 128, true, true);
                const uint32_t base = smem_addr(sm);
                // (U term, V term) pairs, smallest products first
                constexpr int pu[6] = {2, 0, 1, 1, 0, 0};
                constexpr int pv[6] = {0, 2, 1, 0, 1, 0};
#pragma unroll
                for (int kk = 0; kk < SB / 16; ++kk) {
                    const uint32_t o = (uint32_t)kk * 2048;     // 16 rows of p: two 8-row groups
#pragma unroll
                    for (int m = 0; m < 6; ++m) {
                        const uint64_t da = sdesc_sw128(base + 2 * pu[m] * kUBox + o, kUBox, 1024);
                        const uint64_t db = sdesc_sw128(base + (6 + 2 * pv[m]) * kUBox + o, kUBox, 1024);
                        mma_ss(tmem, da, db, idesc, (kk > 0 || m > 0) ? 1u : 0u);
                    }
                }
            }
            mma_commit(acc_full);
            int never = 0;
            (void)mbar_wait(acc_full, 0, &never);
        }
        __syncwarp();
    } else {
        // lane = tile row i (TMEM lane quarter); the 32 rows lie all inside or
        // all outside the pivot block, and so do a chunk's 32 columns
        const int quarter = warp & 3;
        const int i0 = I * UB + quarter * 32;
        const int i = i0 + lane;
        const int64_t ld = s.ldA;
        const bool rowK = i0 >= k0 && i0 < k0 + SB;
        const float* Uh = s.U + (int64_t)h * SB * ld;
        const float* Ph = s.P + (int64_t)h * SB * SB;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, wait_limit) && mbar_wait(fullA, 0, abort_flag, wait_limit));
        if (ok) {
            fence_after_sync();
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
#pragma unroll 1
            for (int c = 0; c < UB / 32; ++c) {
                const int j0 = J * UB + c * 32;
                const bool colK = j0 >= k0 && j0 < k0 + SB;
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + c * 32, r);
                tmem_ld_wait();
                // row `lane` of the swizzled box: 16-byte chunk x sits at x ^ (lane & 7)
                uint8_t* rowp = smA + (4 * quarter + c) * kABox + lane * 128;
                if (!rowK && !colK) {
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        float4* p4 = reinterpret_cast<float4*>(rowp + ((x ^ (lane & 7)) << 4));
                        float4 v = *p4;
                        v.x = sg * (v.x - __uint_as_float(r[4 * x]));
                        v.y = sg * (v.y - __uint_as_float(r[4 * x + 1]));
                        v.z = sg * (v.z - __uint_as_float(r[4 * x + 2]));
                        v.w = sg * (v.w - __uint_as_float(r[4 * x + 3]));
                        *p4 = v;
                    }
                } else if (i < t) {
                    // copies: A_kk <- -P, A_ik <- U_i, A_kj <- U_j^T (the chunk
                    // ends inside the row: j0 < t <= ldA, both multiples of 32)
                    float v[32];
                    if (colK && !rowK) {
#pragma unroll
                        for (int q = 0; q < 32; ++q) v[q] = Uh[(int64_t)(j0 - k0 + q) * ld + i];
                    } else {
                        const float* src = colK ? Ph + (i - k0) * SB + (j0 - k0) : Uh + (int64_t)(i - k0) * ld + j0;
#pragma unroll
                        for (int q = 0; q < 32; q += 4) {
                            const float4 x = *reinterpret_cast<const float4*>(src + q);
                            v[q] = colK ? -x.x : x.x;
                            v[q + 1] = colK ? -x.y : x.y;
                            v[q + 2] = colK ? -x.z : x.z;
                            v[q + 3] = colK ? -x.w : x.w;
                        }
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        *reinterpret_cast<float4*>(rowp + ((x ^ (lane & 7)) << 4)) =
                            make_float4(sg * v[4 * x], sg * v[4 * x + 1], sg * v[4 * x + 2], sg * v[4 * x + 3]);
                }
            }
            // this warp's four boxes back to A (boxes starting past t hold nothing needed)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (i0 < t) {
#pragma unroll 1
                    for (int c = 0; c < UB / 32; ++c)
                        if (J * UB + 32 * c < t)
                            tma_store_3d(&mA, smA + (4 * quarter + c) * kABox, J * UB + 32 * c, i0, h);
                }
                bulk_commit();
                bulk_wait_read_all();
            }
            __syncwarp();
        }
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(s.status, h, KVC_ERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, 128);
}

// Upper triangle <- lower triangle.  grid (blocks * (blocks - 1) / 2 + blocks, H), block 256.
__global__ void __launch_bounds__(256) k_sweep_mirror(float* __restrict__ Am, const int32_t* __restrict__ offsets,
                                                      int64_t ldA, const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int t = offsets[h + 1] - offsets[h];
    int bi, bj;
    tri_tile(blockIdx.x, bi, bj);
    const int ri = bi * SB, rj = bj * SB;
    if (ri >= t) return;
    float* A = Am + (int64_t)h * ldA * ldA;
    __shared__ float tile[SB][SB + 1];
    for (int e = threadIdx.x; e < SB * SB; e += 256) {
        const int r = e / SB, c = e % SB;
        if (ri + r < t && rj + c < t) tile[r][c] = A[(int64_t)(ri + r) * ldA + rj + c];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < SB * SB; e += 256) {
        const int c = e / SB, r = e % SB;       // write row rj + c, column ri + r
        if (ri + r < t && rj + c < t && ri + r > rj + c) A[(int64_t)(rj + c) * ldA + ri + r] = tile[r][c];
    }
}

// y[off + r] = sum_c Hinv[r][c] v[off + c]; grid (ceil(max_t / 8), H), block 256 (a warp per row).
__global__ void __launch_bounds__(256) k_symv(const float* __restrict__ Hinv, const float* __restrict__ v,
                                              const int32_t* __restrict__ offsets, int64_t ldA,
                                              float* __restrict__ y, const int32_t* __restrict__ done,
                                              int done_stride, const int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    if (done && done[(int64_t)h * done_stride]) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= t) return;
    const float* row = Hinv + ((int64_t)h * ldA + r) * ldA;
    const float* vh = v + off;
    float a0 = 0.f, a1 = 0.f;
    int c = lane;
    for (; c + 32 < t; c += 64) {
        a0 = fmaf(row[c], vh[c], a0);
        a1 = fmaf(row[c + 32], vh[c + 32], a1);
    }
    if (c < t) a0 = fmaf(row[c], vh[c], a0);
    const float s = warp_sum(a0 + a1);
    if (lane == 0) y[off + r] = s;
}

}  // namespace

int sweep_launches(int max_t) { return 2 * ((max_t + SB - 1) / SB) + 1; }

bool make_map_bf16(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H);   // tmap.cu
bool make_map_f32(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H);    // tmap.cu

// H^{-1} in place for every head (max_t bounds t_h).  U: fp32 [H][64][ldA];
// split: bf16 [6][H][64][ldA] (U^T and V as three terms each); P: fp32
// [4][H][64][64] (the step's pivot inverse, the next pivot block's two inputs,
// its inverse).
cudaError_t launch_sweep_inverse(float* A, const int32_t* offsets, int H, int max_t, int64_t ldA, float* U,
                                 void* split, float* P, int32_t* status, long long wait_limit, cudaStream_t st) {
    const int nb = (max_t + SB - 1) / SB;
    const int ntri = nb * (nb + 1) / 2;
    const int nu = (max_t + UB - 1) / UB;
    const int64_t ts = (int64_t)H * SB * ldA;
    __nv_bfloat16* Us = static_cast<__nv_bfloat16*>(split);
    __nv_bfloat16* Vs = Us + 3 * ts;
    CUtensorMap mu[3], mv[3], ma;
    for (int q = 0; q < 3; ++q)
        if (!make_map_bf16(&mu[q], Us + q * ts, (int)ldA, ldA, SB, H) ||
            !make_map_bf16(&mv[q], Vs + q * ts, (int)ldA, ldA, SB, H))
            return cudaErrorInvalidValue;
    if (!make_map_f32(&ma, A, (int)ldA, ldA, (int)ldA, H)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_sweep_update_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kUSmem);
    if (e != cudaSuccess) return e;
    float* Xn = P + (int64_t)H * SB * SB;
    float* Pn = P + 3 * (int64_t)H * SB * SB;
    for (int k = 0; k < nb; ++k) {
        SweepArgs s{A, U, Us, Vs, P, Xn, Pn, offsets, ldA, ts, k * SB, status, k > 0, wait_limit};
        // pivot and update launches follow one another with programmatic
        // dependent launch (common.cuh)
        e = launch_dep(k_sweep_pivot, dim3(nb, H), dim3(kPivThreads), 0, st, s);
        if (e != cudaSuccess) return e;
        // CTA 0 of each head forms and inverts the next pivot block
        e = launch_dep(k_sweep_update_tc, dim3(nu * (nu + 1) / 2 + 1, H), dim3(kUThreads), kUSmem, st, mu[0], mu[1],
                       mu[2], mv[0], mv[1], mv[2], ma, s);
        if (e != cudaSuccess) return e;
    }
    {
        const cudaError_t le = launch_dep(k_sweep_mirror, dim3(dim3(ntri, H)), dim3(256), 0, st, A, offsets, ldA,
                                          status);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}

cudaError_t launch_symv(const float* Hinv, const float* v, const int32_t* offsets, int H, int max_t, int64_t ldA,
                        float* y, const int32_t* done, int done_stride, const int32_t* status, cudaStream_t st) {
    {
        const cudaError_t le = launch_dep(k_symv, dim3(dim3((max_t + 7) / 8, H)), dim3(256), 0, st, Hinv, v, offsets,
                                          ldA, y, done, done_stride, status);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}

}  // namespace kvc
