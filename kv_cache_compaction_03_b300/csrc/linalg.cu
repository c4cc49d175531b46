// Batched dense solvers for the two fits of the compaction ("Fast KV
// Compaction via Attention Matching", section 2, "Ajustement du biais et des
// valeurs": beta by non-negative least squares, C_v by least squares).
//
//   k_chol_panel / k_chol_update
//       blocked right-looking Cholesky of every head's t x t matrix, one
//       launch pair per 64-wide panel: the diagonal block is factored and
//       inverted in registers, the panel is a product with that inverse, and
//       the trailing update is spread over 64 x 64 tiles so that a handful of
//       heads still fills the GPU
//   k_solve_cols
//       (L L^T) x = b for many right-hand sides, one CTA per group of
//       columns, blocked with the stored inverses of the diagonal blocks
//       (the C_v columns)
//   k_bpp_solve
//       block principal pivoting for min_{w>=0} 1/2 w'Hw - f'w, all steps of
//       a head in one CTA; each step forms the
//       free-set solution through the Schur complement (H^{-1})_ZZ of the
//       explicit inverse (sweep.cu), the feasibility / optimality check and
//       the exchange of violators
//   k_refine_resid / k_colresid_sum / k_refine_apply
//       iterative refinement of w with the residual A'^T(1 - A'w) + mu(1 - w)
//       taken from A' itself (not from the rounded Gram), one pass over the
//       log-masses per step
//   k_beta_out
//       beta = log w
// Matrices are row-major fp32 with leading dimension ldA; only the lower
// triangle of a symmetric matrix is read.
#include "tc.cuh"

namespace kvc {

constexpr int CB = 64;     // Cholesky panel / tile width

// ------------------------------------------------------------ helpers
// Unblocked Cholesky of the kb x kb lower block D (smem, stride CB+1) by one
// warp.  Returns false if a pivot is not positive / finite (warp-uniform).
__device__ bool warp_chol_block(float* D, int kb) {
    const int lane = threadIdx.x & 31;
    for (int j = 0; j < kb; ++j) {
        const float djj = D[j * (CB + 1) + j];
        if (!(djj > 0.f) || !isfinite(djj)) return false;
        const float r = sqrtf(djj);
        __syncwarp();
        if (lane == 0) D[j * (CB + 1) + j] = r;
        for (int i = j + 1 + lane; i < kb; i += 32) D[i * (CB + 1) + j] /= r;
        __syncwarp();
        for (int i = j + 1 + lane; i < kb; i += 32) {
            const float lij = D[i * (CB + 1) + j];
            for (int k = j + 1; k <= i; ++k) D[i * (CB + 1) + k] -= lij * D[k * (CB + 1) + j];
        }
        __syncwarp();
    }
    return true;
}

// In-place lower Cholesky of a small n x n matrix (n <= zmax) by one CTA,
// right-looking with CB panels; smem: CB*(CB+1) + n*(CB+1) floats.
__device__ bool cta_chol_small(float* A, int n, int64_t lda, float* smem, int* sflag) {
    float* D = smem;
    float* Pn = smem + CB * (CB + 1);
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int k0 = 0; k0 < n; k0 += CB) {
        const int kb = min(CB, n - k0);
        __syncthreads();
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            D[i * (CB + 1) + j] = (j <= i) ? A[(int64_t)(k0 + i) * lda + k0 + j] : 0.f;
        }
        if (tid == 0) *sflag = 0;
        __syncthreads();
        if (tid < 32) {
            const bool ok = warp_chol_block(D, kb);
            if (!ok && tid == 0) *sflag = 1;
        }
        __syncthreads();
        if (*sflag) return false;
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            if (j <= i) A[(int64_t)(k0 + i) * lda + k0 + j] = D[i * (CB + 1) + j];
        }
        const int m = n - k0 - kb;
        for (int r = tid; r < m; r += nt) {
            float* row = A + (int64_t)(k0 + kb + r) * lda + k0;
            for (int j = 0; j < kb; ++j) {
                float v = row[j];
                for (int p = 0; p < j; ++p) v -= Pn[r * (CB + 1) + p] * D[j * (CB + 1) + p];
                v /= D[j * (CB + 1) + j];
                Pn[r * (CB + 1) + j] = v;
                row[j] = v;
            }
        }
        __syncthreads();
        for (int e = tid; e < m * m; e += nt) {
            const int i = e / m, j = e % m;
            if (j > i) continue;
            float acc = 0.f;
            for (int p = 0; p < kb; ++p) acc += Pn[i * (CB + 1) + p] * Pn[j * (CB + 1) + p];
            A[(int64_t)(k0 + kb + i) * lda + k0 + kb + j] -= acc;
        }
    }
    __syncthreads();
    return true;
}

__device__ float block_max_abs(const float* v, int n, float* sred) {
    float m = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, fabsf(v[i]));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) sred[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, sred[w]);
    __syncthreads();
    return r;
}

// ------------------------------------------------------------ Cholesky
// Panel k0 of the blocked right-looking factorisation.  Every CTA factors
// the 64 x 64 diagonal block A_kk in registers (one row per 4 threads, 16
// columns each) and forms its inverse L_kk^{-1}; CTA 0 stores that inverse in
// dinv[h][k0/64] for the solves, CTA rb >= 1 computes its 64 rows of the
// panel, L_ik = A_ik L_kk^{-T}, as a small matrix product.  The diagonal
// blocks of L are never stored in the matrix (only their inverses are used),
// so no CTA writes what a sibling reads.  Rows past t are padded with the
// identity.  grid (1 + row blocks, H), block 256.
__global__ void __launch_bounds__(256) k_chol_panel(float* __restrict__ mats, const int32_t* __restrict__ offsets,
                                                    int64_t ldA, int k0, float* __restrict__ dinv,
                                                    int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int t = offsets[h + 1] - offsets[h];
    if (k0 >= t) return;
    const int rb = blockIdx.x;
    const int r0 = k0 + CB * rb;
    if (rb > 0 && r0 >= t) return;
    __shared__ float colb[2][CB];
    __shared__ float sdiag[CB];
    __shared__ float Ls[CB][CB + 1];     // L_kk, then L_kk^{-1}
    __shared__ float Ps[CB][CB + 1];     // panel rows (rb >= 1)
    __shared__ int bad;
    float* A = mats + (int64_t)h * ldA * ldA;
    const int kb = min(CB, t - k0);
    const int tid = threadIdx.x;
    const int i = tid >> 2, cq = tid & 3;   // row i, columns cq + 4m
    float a[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int c = cq + 4 * m;
        a[m] = (c <= i && i < kb) ? A[(int64_t)(k0 + i) * ldA + k0 + c] : (c == i ? 1.f : 0.f);
    }
    if (tid == 0) bad = 0;
    if (rb > 0) {
        const int nr = min(CB, t - r0);
        for (int e = tid; e < CB * CB; e += 256) {
            const int rr = e / CB, c = e % CB;
            Ps[rr][c] = (rr < nr && c < kb) ? A[(int64_t)(r0 + rr) * ldA + k0 + c] : 0.f;
        }
    }
    // right-looking elimination on unscaled columns: after step j the
    // trailing entries hold A - sum_{p<=j} u_p u_p^T / d_p (fully unrolled so
    // that the register row is indexed statically)
#pragma unroll
    for (int j = 0; j < CB; ++j) {
        float* cb = colb[j & 1];
        if (cq == (j & 3)) cb[i] = a[j >> 2];
        __syncthreads();
        float d = cb[j];
        if (!(d > 0.f) || !isfinite(d)) {
            if (tid == 0) bad = 1;
            d = 1.f;
        }
        const float li = cb[i] / d;
        // columns c = cq + 4m; those <= j are final.  m is static, so whole
        // groups are skipped at compile time.  Entries above the diagonal
        // (c > i) are never read back.
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            if (4 * m + 3 <= j) continue;
            const int c = cq + 4 * m;
            if (4 * m > j || c > j) a[m] = fmaf(-li, cb[c], a[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < 16; ++m)
        if (cq + 4 * m == i) sdiag[i] = a[m];
    __syncthreads();
    if (bad) {
        if (rb == 0 && tid == 0) set_status(status, h, KVC_ERR_NOT_SPD);
        return;
    }
    // L = u_ic / sqrt(d_c) below the diagonal, sqrt(d_c) on it
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int c = cq + 4 * m;
        Ls[i][c] = (c < i) ? a[m] / sqrtf(sdiag[c]) : (c == i ? sqrtf(sdiag[c]) : 0.f);
    }
    __syncthreads();
    // L X = I by forward substitution on the rows: after step j, row j of X is final
    float x[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) x[m] = (cq + 4 * m == i) ? 1.f : 0.f;
    // row j of X = L^{-1} has no entries right of column j, so step j only
    // touches column groups m <= j / 4 (static after unrolling)
#pragma unroll
    for (int j = 0; j < CB; ++j) {
        float* rbuf = colb[j & 1];
        if (i == j) {
            const float inv = 1.f / Ls[j][j];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                if (4 * m > j) continue;
                x[m] *= inv;
                rbuf[cq + 4 * m] = x[m];
            }
        }
        __syncthreads();
        if (i > j) {
            const float lij = Ls[i][j];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                if (4 * m > j) continue;
                x[m] = fmaf(-lij, rbuf[cq + 4 * m], x[m]);
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 16; ++m) Ls[i][cq + 4 * m] = x[m];
    __syncthreads();
    if (rb == 0) {
        float* Dh = dinv + ((int64_t)h * ldA + k0) * CB;
        for (int e = tid; e < CB * CB; e += 256) Dh[e] = Ls[e / CB][e % CB];
        return;
    }
    // L_ik = P L_kk^{-T}: out[rr][c] = sum_{m <= c} P[rr][m] Linv[c][m]
    const int nr = min(CB, t - r0);
    float acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m] = 0.f;
    for (int p = 0; p < CB; ++p) {
        const float pv = Ps[i][p];
#pragma unroll
        for (int m = 0; m < 16; ++m) acc[m] = fmaf(pv, Ls[cq + 4 * m][p], acc[m]);
    }
    if (i < nr) {
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int c = cq + 4 * m;
            if (c < kb) A[(int64_t)(r0 + i) * ldA + k0 + c] = acc[m];
        }
    }
}

__device__ __forceinline__ void tri_decode_u(int p, int& I, int& J) {
    int i = (int)((sqrtf(8.f * (float)p + 1.f) - 1.f) * 0.5f);
    while (i * (i + 1) / 2 > p) --i;
    while ((i + 1) * (i + 2) / 2 <= p) ++i;
    I = i;
    J = p - i * (i + 1) / 2;
}

// Trailing update after panel k0: A_IJ -= L_I L_J^T for the lower 64 x 64
// tiles of rows/cols >= k0 + 64.  grid (ntiles*(ntiles+1)/2, H), block 256.
__global__ void __launch_bounds__(256) k_chol_update(float* __restrict__ mats, const int32_t* __restrict__ offsets,
                                                     int64_t ldA, int k0, const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int t = offsets[h + 1] - offsets[h];
    const int k1 = k0 + CB;
    if (k1 >= t) return;
    int I, J;
    tri_decode_u(blockIdx.x, I, J);
    const int ri = k1 + CB * I, rj = k1 + CB * J;
    if (ri >= t) return;
    __shared__ float Li[CB * (CB + 1)];
    __shared__ float Lj[CB * (CB + 1)];
    float* A = mats + (int64_t)h * ldA * ldA;
    for (int e = threadIdx.x; e < CB * CB; e += 256) {
        const int i = e / CB, p = e % CB;
        Li[i * (CB + 1) + p] = (ri + i < t) ? A[(int64_t)(ri + i) * ldA + k0 + p] : 0.f;
        Lj[i * (CB + 1) + p] = (rj + i < t) ? A[(int64_t)(rj + i) * ldA + k0 + p] : 0.f;
    }
    __syncthreads();
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 8
    for (int p = 0; p < CB; ++p) {
        float li[4], lj[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) li[a] = Li[(ty * 4 + a) * (CB + 1) + p];
#pragma unroll
        for (int c = 0; c < 4; ++c) lj[c] = Lj[(tx + 16 * c) * (CB + 1) + p];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(li[a], lj[c], acc[a][c]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int r = ri + ty * 4 + a;
        if (r >= t) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int col = rj + tx + 16 * c;
            if (col < t && col <= r) A[(int64_t)r * ldA + col] -= acc[a][c];
        }
    }
}

// ------------------------------------------------------------ column solves
enum SolveMode : int { SOLVE_VEC = 0, SOLVE_UNIT_Z = 1, SOLVE_RHS_D = 2 };

struct SolveArgs {
    const float* L;            // [H][ldA][ldA] factors (off-diagonal blocks)
    const float* dinv;         // [H][ldA/64][64][64] inverses of the diagonal blocks
    const int32_t* offsets;
    int64_t ldA;
    int mode;
    const float* vin;          // SOLVE_VEC: off-indexed rhs
    float* vout;               // SOLVE_VEC: off-indexed solution
    const int32_t* zlist;      // SOLVE_UNIT_Z: [H][zmax]
    const int32_t* nz;         // SOLVE_UNIT_Z: [H]
    float* W;                  // SOLVE_UNIT_Z: [H][zmax][ldA]
    int zmax;
    const float* R;            // SOLVE_RHS_D: [sum t][d] rhs
    float* X;                  // SOLVE_RHS_D: [sum t][d] solution
    int d;
    const int32_t* done;       // optional per-head flag (done[h * done_stride]): skip finished heads
    int done_stride;
    const int32_t* status;
};

// (L L^T) X = B for a group of CG right-hand sides per CTA, blocked by 64
// rows with the stored inverses of the diagonal blocks: forward
// y_k = L_kk^{-1} (b_k - sum_{m<k} L_km y_m), then backward
// x_k = L_kk^{-T} (y_k - sum_{m>k} L_mk^T x_m), both right-looking so every
// block step is a dense product spread over the CTA.  The CTA keeps its
// columns of the whole vector in shared memory.  In the forward update the
// L panel below the diagonal block is staged through shared memory 256 rows
// at a time with coalesced 16-byte loads; in the backward update consecutive
// threads read consecutive columns of L rows directly.
// grid (ceil(columns / CG), H), block 256;
// smem: ldA*CG + 64*65 + 256*65 floats.
constexpr int kSolveRows = 256;

template <int CG>
__global__ void __launch_bounds__(256) k_solve_cols(SolveArgs a) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    if (a.done && a.done[(int64_t)h * a.done_stride]) return;
    const int off = a.offsets[h];
    const int t = a.offsets[h + 1] - off;
    int ncol = 1;
    if (a.mode == SOLVE_UNIT_Z) ncol = a.nz[h];
    if (a.mode == SOLVE_RHS_D) ncol = a.d;
    const int c0 = blockIdx.x * CG;
    if (c0 >= ncol) return;
    extern __shared__ float sm[];
    float* Y = sm;                                   // [rows][CG]
    float* Ds = sm + a.ldA * CG;                     // [64][65]
    float* Lc = Ds + CB * (CB + 1);                  // [256][65]
    const int tid = threadIdx.x;
    const int nb = (t + CB - 1) / CB;
    const int rows = nb * CB;
    const float* L = a.L + (int64_t)h * a.ldA * a.ldA;
    const float* Dh = a.dinv + (int64_t)h * a.ldA * CB;
    for (int e = tid; e < rows * CG; e += 256) {
        const int r = e / CG, cc = e % CG, c = c0 + cc;
        float v = 0.f;
        if (r < t && c < ncol) {
            if (a.mode == SOLVE_VEC) v = a.vin[off + r];
            else if (a.mode == SOLVE_UNIT_Z) v = (r == a.zlist[(int64_t)h * a.zmax + c]) ? 1.f : 0.f;
            else v = a.R[((int64_t)off + r) * a.d + c];
        }
        Y[e] = v;
    }
    // y_k <- D_k y_k (TRANS: D_k^T), D_k the stored 64 x 64 inverse
    auto diag = [&](int k64, bool trans) {
        __syncthreads();
        for (int e = tid; e < CB * CB; e += 256) Ds[(e / CB) * (CB + 1) + e % CB] = Dh[(int64_t)k64 * CB + e];
        __syncthreads();
        constexpr int NV = (CB * CG + 255) / 256;
        float v[NV];
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int e = tid + 256 * u;
            float acc = 0.f;
            if (e < CB * CG) {
                const int i = e / CG, cc = e % CG;
                if (!trans)
                    for (int m = 0; m <= i; ++m) acc = fmaf(Ds[i * (CB + 1) + m], Y[(k64 + m) * CG + cc], acc);
                else
                    for (int m = i; m < CB; ++m) acc = fmaf(Ds[m * (CB + 1) + i], Y[(k64 + m) * CG + cc], acc);
            }
            v[u] = acc;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int e = tid + 256 * u;
            if (e < CB * CG) Y[k64 * CG + e] = v[u];
        }
        __syncthreads();
    };
    // ---- forward
    for (int k = 0; k < nb; ++k) {
        const int k64 = k * CB;
        diag(k64, false);
        const int kb = min(CB, t - k64);
        for (int r0 = k64 + CB; r0 < t; r0 += kSolveRows) {
            const int nr = min(kSolveRows, t - r0);
            // stage rows r0 .. r0+nr-1, columns k64 .. k64+63 of L (16 float4 per row)
            for (int idx = tid; idx < nr * (CB / 4); idx += 256) {
                const int rr = idx >> 4, c4 = idx & 15;
                const float4 q = *reinterpret_cast<const float4*>(L + (int64_t)(r0 + rr) * a.ldA + k64 + 4 * c4);
                float* dst = Lc + rr * (CB + 1) + 4 * c4;
                dst[0] = q.x;
                dst[1] = q.y;
                dst[2] = q.z;
                dst[3] = q.w;
            }
            __syncthreads();
            if (tid < nr) {
                float acc[CG];
#pragma unroll
                for (int cc = 0; cc < CG; ++cc) acc[cc] = 0.f;
                const float* lr = Lc + tid * (CB + 1);
                for (int m = 0; m < kb; ++m) {
                    const float l = lr[m];
#pragma unroll
                    for (int cc = 0; cc < CG; ++cc) acc[cc] = fmaf(l, Y[(k64 + m) * CG + cc], acc[cc]);
                }
#pragma unroll
                for (int cc = 0; cc < CG; ++cc) Y[(r0 + tid) * CG + cc] -= acc[cc];
            }
            __syncthreads();
        }
    }
    // ---- backward
    for (int k = nb - 1; k >= 0; --k) {
        const int k64 = k * CB;
        diag(k64, true);
        const int kb = min(CB, t - k64);
        for (int r = tid; r < k64; r += 256) {
            float acc[CG];
#pragma unroll
            for (int cc = 0; cc < CG; ++cc) acc[cc] = 0.f;
            for (int m = 0; m < kb; ++m) {
                const float l = L[(int64_t)(k64 + m) * a.ldA + r];
#pragma unroll
                for (int cc = 0; cc < CG; ++cc) acc[cc] = fmaf(l, Y[(k64 + m) * CG + cc], acc[cc]);
            }
#pragma unroll
            for (int cc = 0; cc < CG; ++cc) Y[r * CG + cc] -= acc[cc];
        }
    }
    __syncthreads();
    for (int e = tid; e < t * CG; e += 256) {
        const int r = e / CG, cc = e % CG, c = c0 + cc;
        if (c >= ncol) continue;
        if (a.mode == SOLVE_VEC) a.vout[off + r] = Y[e];
        else if (a.mode == SOLVE_UNIT_Z) a.W[((int64_t)h * a.zmax + c) * a.ldA + r] = Y[e];
        else a.X[((int64_t)off + r) * a.d + c] = Y[e];
    }
}

// ------------------------------------------------------------ NNLS
// Per-head pivoting state lives in the workspace:
//   zflag[off+i]  1 if w_i is held at zero
//   zlist[h][k]   ascending indices of the zero set, nz[h] = |Z|
//   Hinv[h]       H^{-1} in full (k_sweep_*): row z is H^{-1} e_z
//   S[h]          Cholesky factor of (H^{-1})_ZZ
//   x0            H^{-1} f;  x  current iterate
//   piv[h]        {done, best, budget, iterations}
struct BppArgs {
    const float* x0;
    float* x;
    int8_t* zflag;
    int32_t* zlist;
    int32_t* nz;
    const float* Hinv;         // [H][ldA][ldA]
    float* S;
    int32_t* piv;              // [H][4]
    const int32_t* offsets;
    const float* f;
    int64_t ldA;
    int zmax;
    HeadScalars* hs;
    int32_t* status;
};

// Rebuild the ascending zero-set list from the flags; returns |Z|.
__device__ int build_zlist(const int8_t* zf, int t, int* zl, int zmax, int* sbuf) {
    const int chunk = (t + blockDim.x - 1) / blockDim.x;
    const int j0 = min(t, (int)threadIdx.x * chunk), j1 = min(t, j0 + chunk);
    int c = 0;
    for (int j = j0; j < j1; ++j) c += zf[j] != 0;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = c;
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sbuf[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? sbuf[lane] : 0;
        int z = w;
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, z, o);
            if (lane >= o) z += y;
        }
        sbuf[lane] = z - w;
        if (lane == 31) sbuf[32] = z;
    }
    __syncthreads();
    int pos = sbuf[wid] + x - c;
    const int total = sbuf[32];
    if (total <= zmax)
        for (int j = j0; j < j1; ++j)
            if (zf[j]) zl[pos++] = j;
    __syncthreads();
    return total;
}

// Free-set solution for the current Z: x = x0 + W nu with (H^{-1})_ZZ nu = -x0_Z.
// sx: [t] smem (out), snu: [nz] smem (out: nu = gradient on Z).  Factors S when
// `factor` is set.  Returns false if (H^{-1})_ZZ is not numerically SPD.
// A zero set of at most CB indices (the usual case: a few dozen weights at
// zero) is factored and solved in shared memory (the Cholesky scratch, row
// stride CB + 1); the factor also goes to S for later calls without
// `factor`, which bring it back into shared memory.  Larger zero sets work
// on S in global memory.
__device__ bool schur_solution(const BppArgs& a, int h, int off, int t, int nz, const int* zl, bool factor,
                               const float* src, float* sx, float* snu, float* sm_chol, int* sflag) {
    const float* Hi = a.Hinv + (int64_t)h * a.ldA * a.ldA;    // row z = H^{-1} e_z (symmetric)
    float* S = a.S + (int64_t)h * a.zmax * a.zmax;
    if (nz > 0) {
        const float* Ls = S;
        int64_t lds = a.zmax;
        if (nz <= CB) {
            float* D = sm_chol;
            if (factor) {
                for (int e = threadIdx.x; e < nz * nz; e += blockDim.x) {
                    const int r = e / nz, c = e % nz;
                    D[r * (CB + 1) + c] = c <= r ? Hi[(int64_t)zl[c] * a.ldA + zl[r]] : 0.f;
                }
                if (threadIdx.x == 0) *sflag = 0;
                __syncthreads();
                if (threadIdx.x < 32) {
                    const bool ok = warp_chol_block(D, nz);
                    if (!ok && threadIdx.x == 0) *sflag = 1;
                }
                __syncthreads();
                if (*sflag) return false;
                for (int e = threadIdx.x; e < nz * nz; e += blockDim.x) {
                    const int r = e / nz, c = e % nz;
                    if (c <= r) S[(int64_t)r * a.zmax + c] = D[r * (CB + 1) + c];
                }
            } else {
                for (int e = threadIdx.x; e < nz * nz; e += blockDim.x) {
                    const int r = e / nz, c = e % nz;
                    D[r * (CB + 1) + c] = c <= r ? S[(int64_t)r * a.zmax + c] : 0.f;
                }
            }
            Ls = D;
            lds = CB + 1;
        } else if (factor) {
            for (int e = threadIdx.x; e < nz * nz; e += blockDim.x) {
                const int r = e / nz, c = e % nz;
                S[(int64_t)r * a.zmax + c] = Hi[(int64_t)zl[c] * a.ldA + zl[r]];
            }
            __syncthreads();
            if (!cta_chol_small(S, nz, a.zmax, sm_chol, sflag)) return false;
        }
        for (int k = threadIdx.x; k < nz; k += blockDim.x) snu[k] = -src[zl[k]];
        __syncthreads();
        if (threadIdx.x < 32) {
            // (L L^T) nu = rhs for the small system, one warp
            const int lane = threadIdx.x;
            if (nz <= 32) {
                // lane i holds entry i; column by column: the pivot lane
                // divides, the lanes below (forward) or above (backward)
                // take its value off their own entries
                float y = lane < nz ? snu[lane] : 0.f;
                for (int j = 0; j < nz; ++j) {
                    const float yj = __shfl_sync(0xffffffffu, y / Ls[(int64_t)j * lds + j], j);
                    if (lane == j) y = yj;
                    else if (lane > j && lane < nz) y = fmaf(-Ls[(int64_t)lane * lds + j], yj, y);
                }
                for (int j = nz - 1; j >= 0; --j) {
                    const float xj = __shfl_sync(0xffffffffu, y / Ls[(int64_t)j * lds + j], j);
                    if (lane == j) y = xj;
                    else if (lane < j) y = fmaf(-Ls[(int64_t)j * lds + lane], xj, y);
                }
                if (lane < nz) snu[lane] = y;
            } else {
                // dot products by lanes
                for (int i = 0; i < nz; ++i) {
                    float acc = 0.f;
                    for (int p = lane; p < i; p += 32) acc += Ls[(int64_t)i * lds + p] * snu[p];
                    acc = warp_sum(acc);
                    if (lane == 0) snu[i] = (snu[i] - acc) / Ls[(int64_t)i * lds + i];
                    __syncwarp();
                }
                for (int i = nz - 1; i >= 0; --i) {
                    float acc = 0.f;
                    for (int p = i + 1 + lane; p < nz; p += 32) acc += Ls[(int64_t)p * lds + i] * snu[p];
                    acc = warp_sum(acc);
                    if (lane == 0) snu[i] = (snu[i] - acc) / Ls[(int64_t)i * lds + i];
                    __syncwarp();
                }
            }
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < t; i += blockDim.x) {
        float v = src[i];
#pragma unroll 4
        for (int k = 0; k < nz; ++k) v = fmaf(Hi[(int64_t)zl[k] * a.ldA + i], snu[k], v);
        sx[i] = v;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < nz; k += blockDim.x) sx[zl[k]] = 0.f;
    __syncthreads();
    return true;
}

// grid H, block 512.  smem: 2*ldA floats + zmax floats + zmax ints + chol scratch.
__device__ bool bpp_step_body(const BppArgs& a) {
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return true;
    int32_t* piv = a.piv + 4 * h;
    if (piv[0]) return true;                          // converged
    extern __shared__ float sm[];
    const int off = a.offsets[h];
    const int t = a.offsets[h + 1] - off;
    float* sx = sm;
    float* ssrc = sx + a.ldA;
    float* snu = ssrc + a.ldA;
    int* zl = reinterpret_cast<int*>(snu + a.zmax);
    float* sm_chol = reinterpret_cast<float*>(zl + a.zmax);
    __shared__ int sbuf[33];
    __shared__ int sflag, s_nbad, s_maxbad, s_full;
    __shared__ float sred[32];
    const int nz = a.nz[h];
    if (!KVC_IN_RANGE(nz >= 0 && nz <= a.zmax, a.status, h)) return true;
    for (int k = threadIdx.x; k < nz; k += blockDim.x) {
        const int z = a.zlist[(int64_t)h * a.zmax + k];
        zl[k] = KVC_IN_RANGE(z >= 0 && z < t, a.status, h) ? z : 0;
    }
    for (int i = threadIdx.x; i < t; i += blockDim.x) ssrc[i] = a.x0[off + i];
    __syncthreads();
    if (!schur_solution(a, h, off, t, nz, zl, true, ssrc, sx, snu, sm_chol, &sflag)) {
        if (threadIdx.x == 0) set_status(a.status, h, KVC_ERR_NOT_SPD);
        return true;
    }
    int8_t* zf = a.zflag + off;
    // gradient on Z: y_{z_k} = nu_k
    const float xmax = block_max_abs(sx, t, sred);
    const float fmax = block_max_abs(a.f + off, t, sred);
    const float tolx = 1e-6f * xmax, toly = 1e-6f * fmax;
    if (threadIdx.x == 0) {
        s_nbad = 0;
        s_maxbad = -1;
    }
    __syncthreads();
    // map nu back to indices: violators on Z have nu < -toly
    int nb = 0, mb = -1;
    for (int k = threadIdx.x; k < nz; k += blockDim.x)
        if (snu[k] < -toly) {
            ++nb;
            mb = max(mb, zl[k]);
        }
    for (int i = threadIdx.x; i < t; i += blockDim.x)
        if (!zf[i] && sx[i] < -tolx) {
            ++nb;
            mb = max(mb, i);
        }
    if (nb) {
        atomicAdd(&s_nbad, nb);
        atomicMax(&s_maxbad, mb);
    }
    __syncthreads();
    const int nbad = s_nbad;
    if (nbad == 0) {
        for (int i = threadIdx.x; i < t; i += blockDim.x) a.x[off + i] = zf[i] ? 0.f : sx[i];
        if (threadIdx.x == 0) {
            piv[0] = 1;
            a.hs[h].nzero = nz;
            a.hs[h].iters = piv[3] + 1;
        }
        return true;
    }
    if (threadIdx.x == 0) {
        int best = piv[1], budget = piv[2];
        int full = 0;
        if (nbad < best) {
            best = nbad;
            budget = 3;
            full = 1;
        } else if (budget > 0) {
            --budget;
            full = 1;
        }
        piv[1] = best;
        piv[2] = budget;
        piv[3] += 1;
        s_full = full;
    }
    __syncthreads();
    const int maxbad = s_maxbad;
    // exchange violators (all, or only the largest index under the backup rule)
    for (int k = threadIdx.x; k < nz; k += blockDim.x)
        if (snu[k] < -toly && (s_full || zl[k] == maxbad)) zf[zl[k]] = 2;    // leaves Z
    __syncthreads();
    for (int i = threadIdx.x; i < t; i += blockDim.x) {
        if (zf[i] == 2) zf[i] = 0;
        else if (!zf[i] && sx[i] < -tolx && (s_full || i == maxbad)) zf[i] = 1;
    }
    __syncthreads();
    const int nz2 = build_zlist(zf, t, zl, a.zmax, sbuf);
    if (nz2 > a.zmax) {
        if (threadIdx.x == 0) {
            set_status(a.status, h, KVC_ERR_NNLS_MAXITER);
            piv[0] = 1;
        }
        return true;
    }
    for (int k = threadIdx.x; k < nz2; k += blockDim.x) a.zlist[(int64_t)h * a.zmax + k] = zl[k];
    for (int i = threadIdx.x; i < t; i += blockDim.x) a.x[off + i] = zf[i] ? 0.f : fmaxf(sx[i], 0.f);
    if (threadIdx.x == 0) a.nz[h] = nz2;
    return false;
}

// All pivoting steps of a head in one CTA: the state (zero set, iterate,
// counters) lives in global memory between steps and is re-read after a
// block barrier.  grid H, block 512.
__global__ void __launch_bounds__(512) k_bpp_solve(BppArgs a, int max_iter) {
    grid_dependency_wait();
    for (int it = 0; it < max_iter; ++it) {
        if (bpp_step_body(a)) break;
        __syncthreads();
    }
}

// Reset the pivoting state (grid ceil(sum/256) x H); also zero the zero set.
__global__ void k_bpp_init(BppArgs a) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    const int off = a.offsets[h];
    const int t = a.offsets[h + 1] - off;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (!head_ok(a.status, h)) return;
    if (i < t) a.zflag[off + i] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        int32_t* piv = a.piv + 4 * h;
        piv[0] = 0;
        piv[1] = t + 1;
        piv[2] = 3;
        piv[3] = 0;
        a.nz[h] = 0;
    }
}

// Heads still pivoting after the last step hit the iteration cap.
__global__ void k_bpp_finish(BppArgs a, int H) {
    grid_dependency_wait();
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H || !head_ok(a.status, h)) return;
    if (!a.piv[4 * h]) set_status(a.status, h, KVC_ERR_NNLS_MAXITER);
}

// df_fma on two independent accumulators (hi, lo) at once, with paired fp32
// instructions: the same error-free product and sum in the same order, each
// difference x - y written as fma(y, -1, x).  Being inline assembly, none of
// it can be fused by the compiler.
__device__ __forceinline__ void df_fma2(float2& hi, float2& lo, float2 a, float2 b) {
    const float2 m1 = make_float2(-1.f, -1.f), z = make_float2(0.f, 0.f);
    const float2 p = tc::ffma2(a, b, z);
    const float2 pe = tc::ffma2(a, b, tc::ffma2(p, m1, z));
    const float2 s = tc::fadd2(hi, p);
    const float2 bb = tc::ffma2(hi, m1, s);                                   // s - hi
    const float2 e0 = tc::fadd2(tc::ffma2(tc::ffma2(bb, m1, s), m1, hi),      // hi - (s - bb)
                                tc::ffma2(bb, m1, p));                        // p - bb
    const float2 e = tc::fadd2(e0, tc::fadd2(lo, pe));
    hi = tc::fadd2(s, e);
    lo = tc::ffma2(tc::ffma2(s, m1, hi), m1, e);                              // e - (hi - s)
}

// The residual of the refinement, r_i = sum_q A'_qi u_q + mu (1 - x_i) with
// u_q = 1 - sum_i A'_qi x_i, in one pass over the log-masses: a CTA takes
// `qb` query rows of one head, brings them into shared memory with one bulk
// copy per row (the copy engine keeps the whole block in flight), turns them
// into A' = 2^l2, forms each row's u_q (a warp per row, double-float), then
// adds its rows' share of every column, sum over its rows of A'_qi u_q (a
// thread per column, double-float, from shared memory), and writes that
// partial to part[block][off + i].  k_colresid_sum then adds the blocks'
// partials in a fixed order, so the result does not depend on scheduling.
// The copy wait is bounded; a CTA that gives up reports TIMEOUT for the head
// after its copies have landed.
// grid (ceil(n/qb), H), block 256, dynamic smem (qb * ldA + qb) floats + 16.
__global__ void __launch_bounds__(256) k_refine_resid(const float* __restrict__ L2, const float* __restrict__ x,
                                                      const int32_t* __restrict__ offsets, int n, int64_t ldA,
                                                      int qb, int64_t part_stride, dfloat* __restrict__ part,
                                                      int32_t* __restrict__ status) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    extern __shared__ __align__(16) float sa[];    // [qb][ldA] A', then [qb] u, then the barrier
    float* su = sa + (int64_t)qb * ldA;
    uint64_t* bar = reinterpret_cast<uint64_t*>(su + round_up(qb, 4));
    __shared__ int abort_flag;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int q0 = blockIdx.x * qb;
    const int rows = min(qb, n - q0);
    const uint32_t rowbytes = (uint32_t)round_up(t, 4) * 4u;   // columns t.. of a row hold -inf
    if (threadIdx.x == 0) {
        tc::mbar_init(bar, 1);
        abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tc::mbar_expect_tx(bar, (uint32_t)rows * rowbytes);
        for (int r = 0; r < rows; ++r)
            tc::bulk_load(sa + (int64_t)r * ldA, L2 + ((int64_t)h * n + q0 + r) * ldA, rowbytes, bar);
    }
    if (!tc::mbar_wait(bar, 0, &abort_flag)) {
        int never = 0;
        (void)tc::mbar_wait(bar, 0, &never);          // the copies must land before the CTA leaves
        if (threadIdx.x == 0) set_status(status, h, KVC_ERR_TIMEOUT);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int rr = warp; rr < qb; rr += 8) {
        float* arow = sa + (int64_t)rr * ldA;
        // a lane takes pairs of adjacent columns (paired arithmetic); with t
        // odd the pair's second column, t, is set to 0 (ldA > t then)
        float2 hi = make_float2(0.f, 0.f), lo = make_float2(0.f, 0.f);
        if (rr < rows) {
            for (int i = 2 * lane; i < t; i += 64) {
                const bool two = i + 1 < t;
                const float2 l = *reinterpret_cast<const float2*>(arow + i);
                const float2 a = make_float2(exp2f(l.x), two ? exp2f(l.y) : 0.f);
                *reinterpret_cast<float2*>(arow + i) = a;
                df_fma2(hi, lo, a, make_float2(x[off + i], two ? x[off + i + 1] : 0.f));
            }
        } else {
            for (int i = lane; i < t; i += 32) arow[i] = 0.f;
        }
        dfloat acc{hi.x, lo.x};
        df_add_df(acc, dfloat{hi.y, lo.y});
        acc = warp_sum_df(acc);
        if (lane == 0) su[rr] = rr < rows ? (1.f - acc.hi) - acc.lo : 0.f;
    }
    __syncthreads();
    // a thread per pair of adjacent columns, paired arithmetic
    const int npair = (t + 1) >> 1;
    for (int cp = threadIdx.x; cp < npair; cp += 256) {
        const int c = 2 * cp;
        float2 hi = make_float2(0.f, 0.f), lo = make_float2(0.f, 0.f);
        for (int rr = 0; rr < qb; ++rr) {
            const float u = su[rr];
            df_fma2(hi, lo, *reinterpret_cast<const float2*>(sa + (int64_t)rr * ldA + c), make_float2(u, u));
        }
        dfloat* pp = part + (int64_t)blockIdx.x * part_stride + off + c;
        pp[0] = dfloat{hi.x, lo.x};
        if (c + 1 < t) pp[1] = dfloat{hi.y, lo.y};
    }
}

// Query rows per CTA of k_refine_resid: a multiple of the 8 warps, as many
// as keep its shared-memory tile (rows x ldA floats) within 72 KB, so that
// three CTAs share an SM and one's copies overlap the others' arithmetic
// (ldA up to 2304; beyond that 8 rows, up to 128 KB at the largest budget).
int refine_rows(int64_t ldA) {
    const int64_t r = 2304 / ldA;
    return 8 * (int)(r < 1 ? 1 : (r > 8 ? 8 : r));
}
// Bytes of the per-block partial sums of k_refine_resid.
size_t refine_part_bytes(int H, int n, int max_t, int64_t ldA) {
    const int qb = refine_rows(ldA);
    return (size_t)((n + qb - 1) / qb) * H * max_t * sizeof(dfloat);
}

// grid (ceil(max_t/256), H), block 256.
__global__ void __launch_bounds__(256) k_colresid_sum(const dfloat* __restrict__ part, int64_t part_stride,
                                                      int nblk, const float* __restrict__ x,
                                                      const int8_t* __restrict__ zflag,
                                                      const int32_t* __restrict__ offsets,
                                                      const HeadScalars* __restrict__ hs, float* __restrict__ r,
                                                      const uint8_t* __restrict__ fixed,
                                                      const int32_t* __restrict__ status) {
    grid_dependency_wait();
    // thread (g, cl): column blockIdx.x * 32 + cl, partials [g nb8, (g + 1) nb8);
    // the eight group sums then meet in group order (a fixed order)
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    __shared__ dfloat gs[8][32];
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int cl = threadIdx.x & 31, g = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + cl;
    const int nb8 = (nblk + 7) / 8;
    const int s0 = min(nblk, g * nb8), s1 = min(nblk, s0 + nb8);
    dfloat acc{0.f, 0.f};
    if (c < t)
        for (int sp = s0; sp < s1; ++sp) df_add_df(acc, part[(int64_t)sp * part_stride + off + c]);
    gs[g][cl] = acc;
    __syncthreads();
    if (g != 0 || c >= t) return;
    for (int k = 1; k < 8; ++k) df_add_df(acc, gs[k][cl]);
    df_fma(acc, hs[h].mu, 1.f - x[off + c]);
    // weights held fixed (thought-aware pivots) take no refinement step
    r[off + c] = (zflag[off + c] || (fixed && fixed[off + c])) ? 0.f : acc.hi + acc.lo;
}

// x += H_FF^{-1} r_F: d0 = H^{-1} r is in `d0`; apply the Schur correction
// with the stored factor of (H^{-1})_ZZ.  grid H, block 512.
__global__ void __launch_bounds__(512) k_refine_apply(BppArgs a, const float* __restrict__ d0) {
    grid_dependency_wait();
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return;
    extern __shared__ float sm[];
    const int off = a.offsets[h];
    const int t = a.offsets[h + 1] - off;
    float* sx = sm;
    float* ssrc = sx + a.ldA;
    float* snu = ssrc + a.ldA;
    int* zl = reinterpret_cast<int*>(snu + a.zmax);
    float* sm_chol = reinterpret_cast<float*>(zl + a.zmax);
    __shared__ int sflag;
    const int nz = a.nz[h];
    if (!KVC_IN_RANGE(nz >= 0 && nz <= a.zmax, a.status, h)) return;
    for (int k = threadIdx.x; k < nz; k += blockDim.x) {
        const int z = a.zlist[(int64_t)h * a.zmax + k];
        zl[k] = KVC_IN_RANGE(z >= 0 && z < t, a.status, h) ? z : 0;
    }
    for (int i = threadIdx.x; i < t; i += blockDim.x) ssrc[i] = d0[off + i];
    __syncthreads();
    schur_solution(a, h, off, t, nz, zl, false, ssrc, sx, snu, sm_chol, &sflag);
    for (int i = threadIdx.x; i < t; i += blockDim.x)
        if (!a.zflag[off + i]) a.x[off + i] += sx[i];
}

// beta = log w (w clamped at 0; -inf where w = 0), plus the kept key's input
// bias when the keys carry one (bias_in [H][T] natural units, positions
// idx).  grid (ceil(max_t/256), H).
__global__ void k_beta_out(float* __restrict__ x, const int32_t* __restrict__ offsets, float* __restrict__ beta,
                           const int32_t* __restrict__ status, const float* __restrict__ bias_in,
                           const int32_t* __restrict__ idx, int T) {
    grid_dependency_wait();
    const int h = blockIdx.y;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= t || !head_ok(status, h)) return;
    const float w = fmaxf(x[off + i], 0.f);
    x[off + i] = w;
    float b0 = 0.f;
    if (bias_in) {
        const int j = idx[off + i];
        if (!KVC_IN_RANGE(j >= 0 && j < T, status, h)) return;
        b0 = bias_in[(int64_t)h * T + j];
    }
    beta[off + i] = (w > 0.f) ? b0 + logf(w) : -INFINITY;
}

// ------------------------------------------------------------ launchers
cudaError_t launch_chol(float* mats, const int32_t* offsets, int H, int max_t, int64_t ldA, float* dinv,
                        int32_t* status, cudaStream_t st) {
    for (int k0 = 0; k0 < max_t; k0 += CB) {
        const int rows_below = max(0, max_t - k0 - CB);
        const int nrb = (rows_below + CB - 1) / CB;
        k_chol_panel<<<dim3(1 + nrb, H), 256, 0, st>>>(mats, offsets, ldA, k0, dinv, status);
        if (nrb > 0) {
            k_chol_update<<<dim3(nrb * (nrb + 1) / 2, H), 256, 0, st>>>(mats, offsets, ldA, k0, status);
        }
    }
    return cudaGetLastError();
}

int chol_launches(int max_t) {
    int c = 0;
    for (int k0 = 0; k0 < max_t; k0 += CB) c += (max_t - k0 - CB > 0) ? 2 : 1;
    return c;
}

// Solve for every column of the mode with CG columns per CTA.
template <int CG>
static cudaError_t launch_solve_t(const SolveArgs& a, int ncols, int H, cudaStream_t st) {
    const size_t smem = (size_t)(a.ldA * CG + CB * (CB + 1) + kSolveRows * (CB + 1)) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_solve_cols<CG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_solve_cols<CG><<<dim3((ncols + CG - 1) / CG, H), 256, smem, st>>>(a);
    return cudaGetLastError();
}
// Columns per CTA: one for a single right-hand side; otherwise as many as
// keep about two CTAs per SM busy (more columns per CTA = fewer reads of L),
// within the shared-memory budget.
static cudaError_t launch_solve(const SolveArgs& a, int ncols, int H, cudaStream_t st) {
    if (ncols <= 1) return launch_solve_t<1>(a, ncols, H, st);
    const int64_t work = (int64_t)ncols * H;
    const bool fits16 = (a.ldA * 16 + CB * (CB + 1) + kSolveRows * (CB + 1)) * 4 <= 200 * 1024;
    if (fits16 && work >= 16 * 2 * 148) return launch_solve_t<16>(a, ncols, H, st);
    if (work >= 8 * 2 * 148) return launch_solve_t<8>(a, ncols, H, st);
    return launch_solve_t<4>(a, ncols, H, st);
}

cudaError_t launch_cholsolve(int d, const float* L, const float* dinv, const float* R, const int32_t* offsets, int H,
                             int64_t ldA, float* Cv, const int32_t* status, cudaStream_t st) {
    SolveArgs a{};
    a.L = L;
    a.dinv = dinv;
    a.offsets = offsets;
    a.ldA = ldA;
    a.mode = SOLVE_RHS_D;
    a.R = R;
    a.X = Cv;
    a.d = d;
    a.status = status;
    return launch_solve(a, d, H, st);
}

static size_t bpp_smem(int64_t ldA, int zmax) {
    return (size_t)(2 * ldA + zmax) * sizeof(float) + (size_t)zmax * sizeof(int) +
           (size_t)(CB * (CB + 1) + (size_t)zmax * (CB + 1)) * sizeof(float);
}

cudaError_t launch_symv(const float* Hinv, const float* v, const int32_t* offsets, int H, int max_t, int64_t ldA,
                        float* y, const int32_t* done, int done_stride, const int32_t* status, cudaStream_t st);

// The whole NNLS from the explicit inverse: x0 = H^{-1} f, `max_iter`
// pivoting steps (each reads the zero-set rows of H^{-1}), refinement.
cudaError_t launch_nnls_all(const float* Hinv, const float* f, const int32_t* offsets, int H, int n, int max_t,
                            int64_t ldA, const float* L2, float* x, float* x0, int8_t* zflag, int32_t* zlist,
                            int32_t* nz, float* S, int32_t* piv, float* r, float* d0, HeadScalars* hs,
                            int zmax, int max_iter, int refine_iters, void* rpart_ws, const uint8_t* fixed,
                            int32_t* status, cudaStream_t st, int* launches) {
    dfloat* rpart = static_cast<dfloat*>(rpart_ws);
    const int64_t part_stride = (int64_t)H * max_t;
    BppArgs b{x0, x, zflag, zlist, nz, Hinv, S, piv, offsets, f, ldA, zmax, hs, status};
    int nl = 0;
    {
        const cudaError_t le = launch_dep(k_bpp_init, dim3(dim3((max_t + 255) / 256, H)), dim3(256), 0, st, b);
        if (le != cudaSuccess) return le;
    }
    cudaError_t e = launch_symv(Hinv, f, offsets, H, max_t, ldA, x0, nullptr, 0, status, st);
    if (e != cudaSuccess) return e;
    nl += 2;
    const size_t smem = bpp_smem(ldA, zmax);
    e = cudaFuncSetAttribute(k_bpp_solve, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_refine_apply, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    {
        const cudaError_t le = launch_dep(k_bpp_solve, dim3(H), dim3(512), smem, st, b, max_iter);
        if (le != cudaSuccess) return le;
    }
    ++nl;
    {
        const cudaError_t le = launch_dep(k_bpp_finish, dim3((H + 127) / 128), dim3(128), 0, st, b, H);
        if (le != cudaSuccess) return le;
    }
    ++nl;
    const int qb = refine_rows(ldA);
    const int nblk = (n + qb - 1) / qb;
    const size_t rsmem = (size_t)(qb * ldA + round_up(qb, 4)) * sizeof(float) + 16;
    e = cudaFuncSetAttribute(k_refine_resid, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rsmem);
    if (e != cudaSuccess) return e;
    for (int it = 0; it < refine_iters; ++it) {
        {
            const cudaError_t le = launch_dep(k_refine_resid, dim3(dim3(nblk, H)), dim3(256), rsmem, st, L2, x,
                                              offsets, n, ldA, qb, part_stride, rpart, status);
            if (le != cudaSuccess) return le;
        }
        {
            const cudaError_t le = launch_dep(k_colresid_sum, dim3(dim3((max_t + 31) / 32, H)), dim3(256), 0, st,
                                              rpart, part_stride, nblk, x, zflag, offsets, hs, r, fixed, status);
            if (le != cudaSuccess) return le;
        }
        e = launch_symv(Hinv, r, offsets, H, max_t, ldA, d0, nullptr, 0, status, st);
        if (e != cudaSuccess) return e;
        {
            const cudaError_t le = launch_dep(k_refine_apply, dim3(H), dim3(512), smem, st, b, d0);
            if (le != cudaSuccess) return le;
        }
        nl += 4;
    }
    if (launches) *launches = nl;
    return cudaGetLastError();
}

cudaError_t launch_beta_out(float* x, const int32_t* offsets, int H, int max_t, float* beta, const int32_t* status,
                            const float* bias_in, const int32_t* idx, int T, cudaStream_t st) {
    dim3 grid((max_t + 255) / 256, H);
    {
        const cudaError_t le = launch_dep(k_beta_out, dim3(grid), dim3(256), 0, st, x, offsets, beta, status, bias_in,
                                          idx, T);
        if (le != cudaSuccess) return le;
    }
    return cudaGetLastError();
}

}  // namespace kvc
