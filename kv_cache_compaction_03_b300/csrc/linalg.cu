// Batched dense solvers for the two fits of the compaction ("Fast KV
// Compaction via Attention Matching", section 2, "Ajustement du biais et des
// valeurs": beta by non-negative least squares, C_v by least squares).
//
//   k_chol_panel / k_chol_update
//       blocked right-looking Cholesky of every head's t x t matrix, one
//       launch pair per 64-wide panel; the trailing update is spread over
//       64 x 64 tiles so that a handful of heads still fills the GPU
//   k_trsv_cols
//       (L L^T) x = b for many right-hand sides, one CTA per column group:
//       x0 = H^{-1} f, the zero-set columns H^{-1} e_z, refinement steps and
//       the C_v columns
//   k_bpp_step
//       one block-principal-pivoting step of min_{w>=0} 1/2 w'Hw - f'w: the
//       free-set solution through the Schur complement (H^{-1})_ZZ, the
//       feasibility / optimality check and the exchange of violators
//   k_rowmass / k_colresid / k_refine_apply
//       iterative refinement of w with the residual A'^T(1 - A'w) + mu(1 - w)
//       taken from A' itself (not from the rounded Gram)
//   k_beta_out
//       beta = log w
// Matrices are row-major fp32 with leading dimension ldA; only the lower
// triangle of a symmetric matrix is read.
#include "common.cuh"

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

// (L L^T) x = x in place for a vector in smem (length n), L in global.
// Block-wide; Ds: CB*(CB+1) floats of scratch.
__device__ void cta_cholsolve_vec(const float* L, int n, int64_t lda, float* xs, float* Ds) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
    // forward: L y = b
    for (int k0 = 0; k0 < n; k0 += CB) {
        const int kb = min(CB, n - k0);
        __syncthreads();
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            Ds[i * (CB + 1) + j] = (j <= i) ? L[(int64_t)(k0 + i) * lda + k0 + j] : 0.f;
        }
        __syncthreads();
        if (tid < 32) {
            for (int j = 0; j < kb; ++j) {
                const float y = xs[k0 + j] / Ds[j * (CB + 1) + j];
                __syncwarp();
                if (lane == 0) xs[k0 + j] = y;
                for (int i = j + 1 + lane; i < kb; i += 32) xs[k0 + i] -= Ds[i * (CB + 1) + j] * y;
                __syncwarp();
            }
        }
        __syncthreads();
        for (int r = k0 + kb + tid; r < n; r += nt) {
            const float* lr = L + (int64_t)r * lda + k0;
            float v = xs[r];
            if (kb == CB) {
                const float4* l4 = reinterpret_cast<const float4*>(lr);
#pragma unroll 4
                for (int p = 0; p < CB / 4; ++p) {
                    const float4 q = l4[p];
                    v -= q.x * xs[k0 + 4 * p] + q.y * xs[k0 + 4 * p + 1] + q.z * xs[k0 + 4 * p + 2] +
                         q.w * xs[k0 + 4 * p + 3];
                }
            } else {
                for (int p = 0; p < kb; ++p) v -= lr[p] * xs[k0 + p];
            }
            xs[r] = v;
        }
    }
    // backward: L^T x = y
    for (int k0 = ((n - 1) / CB) * CB; k0 >= 0; k0 -= CB) {
        const int kb = min(CB, n - k0);
        __syncthreads();
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            Ds[i * (CB + 1) + j] = (j <= i) ? L[(int64_t)(k0 + i) * lda + k0 + j] : 0.f;
        }
        __syncthreads();
        if (tid < 32) {
            for (int j = kb - 1; j >= 0; --j) {
                const float x = xs[k0 + j] / Ds[j * (CB + 1) + j];
                __syncwarp();
                if (lane == 0) xs[k0 + j] = x;
                for (int i = lane; i < j; i += 32) xs[k0 + i] -= Ds[j * (CB + 1) + i] * x;
                __syncwarp();
            }
        }
        __syncthreads();
        for (int r = tid; r < k0; r += nt) {
            float v = xs[r];
            for (int p = 0; p < kb; ++p) v -= L[(int64_t)(k0 + p) * lda + r] * xs[k0 + p];
            xs[r] = v;
        }
    }
    __syncthreads();
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
// Panel k0: CTA 0 factors the diagonal block; CTA rb >= 1 factors its own
// copy of the diagonal block (cheaper than another launch) and solves the
// 64 rows [k0 + 64 rb, ...) of the panel.  grid (1 + row blocks, H), block 128.
// The factored diagonal block cannot be stored into the matrix by this
// launch (sibling CTAs read the unfactored block), so CTA 0 parks it in
// dscr[h] and the next panel launch's CTA 0 copies it into place; the last
// block of a head has no siblings and is stored directly.
__global__ void __launch_bounds__(128) k_chol_panel(float* __restrict__ mats, const int32_t* __restrict__ offsets,
                                                    int64_t ldA, int k0, float* __restrict__ dscr,
                                                    int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int t = offsets[h + 1] - offsets[h];
    if (k0 >= t) return;
    const int rb = blockIdx.x;
    const int r0 = k0 + CB * rb;
    if (rb > 0 && r0 >= t) return;
    __shared__ float D[CB * (CB + 1)];
    __shared__ float P[CB * (CB + 1)];
    __shared__ int bad;
    float* A = mats + (int64_t)h * ldA * ldA;
    float* Dh = dscr + (int64_t)h * CB * CB;
    const int kb = min(CB, t - k0);
    if (rb == 0 && k0 > 0) {
        // the previous block (k0 - 64) was not this head's last: store its factor
        for (int e = threadIdx.x; e < CB * CB; e += blockDim.x) {
            const int i = e / CB, j = e % CB;
            if (j <= i) A[(int64_t)(k0 - CB + i) * ldA + k0 - CB + j] = Dh[e];
        }
    }
    for (int e = threadIdx.x; e < kb * kb; e += blockDim.x) {
        const int i = e / kb, j = e % kb;
        D[i * (CB + 1) + j] = (j <= i) ? A[(int64_t)(k0 + i) * ldA + k0 + j] : 0.f;
    }
    const int nr = (rb > 0) ? min(CB, t - r0) : 0;
    for (int e = threadIdx.x; e < nr * kb; e += blockDim.x) {
        const int i = e / kb, j = e % kb;
        P[i * (CB + 1) + j] = A[(int64_t)(r0 + i) * ldA + k0 + j];
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const bool ok = warp_chol_block(D, kb);
        if (threadIdx.x == 0) bad = ok ? 0 : 1;
    }
    __syncthreads();
    if (bad) {
        if (rb == 0 && threadIdx.x == 0) set_status(status, h, KVC_ERR_NOT_SPD);
        return;
    }
    if (rb == 0) {
        const bool last = (k0 + kb >= t);
        for (int e = threadIdx.x; e < kb * kb; e += blockDim.x) {
            const int i = e / kb, j = e % kb;
            if (j > i) continue;
            if (last)
                A[(int64_t)(k0 + i) * ldA + k0 + j] = D[i * (CB + 1) + j];
            else
                Dh[i * CB + j] = D[i * (CB + 1) + j];
        }
        return;
    }
    // X D^T = P, row by row (forward substitution along the columns)
    if (threadIdx.x < nr) {
        const int i = threadIdx.x;
        for (int j = 0; j < kb; ++j) {
            float v = P[i * (CB + 1) + j];
            for (int p = 0; p < j; ++p) v -= P[i * (CB + 1) + p] * D[j * (CB + 1) + p];
            P[i * (CB + 1) + j] = v / D[j * (CB + 1) + j];
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nr * kb; e += blockDim.x) {
        const int i = e / kb, j = e % kb;
        A[(int64_t)(r0 + i) * ldA + k0 + j] = P[i * (CB + 1) + j];
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
    const float* L;            // [H][ldA][ldA] factors
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

// grid (column CTAs, H), block 256; smem: ldA + CB*(CB+1) floats.
__global__ void __launch_bounds__(256) k_trsv_cols(SolveArgs a) {
    const int h = blockIdx.y;
    if (!head_ok(a.status, h)) return;
    if (a.done && a.done[(int64_t)h * a.done_stride]) return;
    extern __shared__ float sm[];
    float* xs = sm;
    float* Ds = sm + a.ldA;
    const int off = a.offsets[h];
    const int t = a.offsets[h + 1] - off;
    const float* L = a.L + (int64_t)h * a.ldA * a.ldA;
    int ncol = 1;
    if (a.mode == SOLVE_UNIT_Z) ncol = a.nz[h];
    if (a.mode == SOLVE_RHS_D) ncol = a.d;
    for (int c = blockIdx.x; c < ncol; c += gridDim.x) {
        __syncthreads();
        if (a.mode == SOLVE_VEC) {
            for (int i = threadIdx.x; i < t; i += blockDim.x) xs[i] = a.vin[off + i];
        } else if (a.mode == SOLVE_UNIT_Z) {
            const int z = a.zlist[(int64_t)h * a.zmax + c];
            for (int i = threadIdx.x; i < t; i += blockDim.x) xs[i] = (i == z) ? 1.f : 0.f;
        } else {
            for (int i = threadIdx.x; i < t; i += blockDim.x) xs[i] = a.R[((int64_t)off + i) * a.d + c];
        }
        cta_cholsolve_vec(L, t, a.ldA, xs, Ds);
        if (a.mode == SOLVE_VEC) {
            for (int i = threadIdx.x; i < t; i += blockDim.x) a.vout[off + i] = xs[i];
        } else if (a.mode == SOLVE_UNIT_Z) {
            float* wc = a.W + ((int64_t)h * a.zmax + c) * a.ldA;
            for (int i = threadIdx.x; i < t; i += blockDim.x) wc[i] = xs[i];
        } else {
            for (int i = threadIdx.x; i < t; i += blockDim.x) a.X[((int64_t)off + i) * a.d + c] = xs[i];
        }
    }
}

// ------------------------------------------------------------ NNLS
// Per-head pivoting state lives in the workspace:
//   zflag[off+i]  1 if w_i is held at zero
//   zlist[h][k]   ascending indices of the zero set, nz[h] = |Z|
//   W[h][k][:]    H^{-1} e_{zlist[k]} (computed by k_trsv_cols before each step)
//   S[h]          Cholesky factor of (H^{-1})_ZZ
//   x0            H^{-1} f;  x  current iterate
//   piv[h]        {done, best, budget, iterations}
struct BppArgs {
    const float* x0;
    float* x;
    int8_t* zflag;
    int32_t* zlist;
    int32_t* nz;
    const float* W;
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
__device__ bool schur_solution(const BppArgs& a, int h, int off, int t, int nz, const int* zl, bool factor,
                               const float* src, float* sx, float* snu, float* sm_chol, int* sflag) {
    const float* W = a.W + (int64_t)h * a.zmax * a.ldA;
    float* S = a.S + (int64_t)h * a.zmax * a.zmax;
    if (nz > 0) {
        if (factor) {
            for (int e = threadIdx.x; e < nz * nz; e += blockDim.x) {
                const int r = e / nz, c = e % nz;
                S[(int64_t)r * a.zmax + c] = W[(int64_t)c * a.ldA + zl[r]];
            }
            __syncthreads();
            if (!cta_chol_small(S, nz, a.zmax, sm_chol, sflag)) return false;
        }
        for (int k = threadIdx.x; k < nz; k += blockDim.x) snu[k] = -src[zl[k]];
        __syncthreads();
        if (threadIdx.x < 32) {
            // (L L^T) nu = rhs for the small system, one warp (dot products by lanes)
            const int lane = threadIdx.x;
            for (int i = 0; i < nz; ++i) {
                float acc = 0.f;
                for (int p = lane; p < i; p += 32) acc += S[(int64_t)i * a.zmax + p] * snu[p];
                acc = warp_sum(acc);
                if (lane == 0) snu[i] = (snu[i] - acc) / S[(int64_t)i * a.zmax + i];
                __syncwarp();
            }
            for (int i = nz - 1; i >= 0; --i) {
                float acc = 0.f;
                for (int p = i + 1 + lane; p < nz; p += 32) acc += S[(int64_t)p * a.zmax + i] * snu[p];
                acc = warp_sum(acc);
                if (lane == 0) snu[i] = (snu[i] - acc) / S[(int64_t)i * a.zmax + i];
                __syncwarp();
            }
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < t; i += blockDim.x) {
        float v = src[i];
        for (int k = 0; k < nz; ++k) v = fmaf(W[(int64_t)k * a.ldA + i], snu[k], v);
        sx[i] = v;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < nz; k += blockDim.x) sx[zl[k]] = 0.f;
    __syncthreads();
    return true;
}

// grid H, block 512.  smem: 2*ldA floats + zmax floats + zmax ints + chol scratch.
__global__ void __launch_bounds__(512) k_bpp_step(BppArgs a) {
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return;
    int32_t* piv = a.piv + 4 * h;
    if (piv[0]) return;                               // converged
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
    for (int k = threadIdx.x; k < nz; k += blockDim.x) zl[k] = a.zlist[(int64_t)h * a.zmax + k];
    for (int i = threadIdx.x; i < t; i += blockDim.x) ssrc[i] = a.x0[off + i];
    __syncthreads();
    if (!schur_solution(a, h, off, t, nz, zl, true, ssrc, sx, snu, sm_chol, &sflag)) {
        if (threadIdx.x == 0) set_status(a.status, h, KVC_ERR_NOT_SPD);
        return;
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
        return;
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
        return;
    }
    for (int k = threadIdx.x; k < nz2; k += blockDim.x) a.zlist[(int64_t)h * a.zmax + k] = zl[k];
    for (int i = threadIdx.x; i < t; i += blockDim.x) a.x[off + i] = zf[i] ? 0.f : fmaxf(sx[i], 0.f);
    if (threadIdx.x == 0) a.nz[h] = nz2;
}

// Reset the pivoting state (grid ceil(sum/256) x H); also zero the zero set.
__global__ void k_bpp_init(BppArgs a) {
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
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H || !head_ok(a.status, h)) return;
    if (!a.piv[4 * h]) set_status(a.status, h, KVC_ERR_NNLS_MAXITER);
}

// v_q = sum_i A'_qi x_i (double-float), u_q = 1 - v_q.  grid (ceil(n/8), H), block 256.
__global__ void __launch_bounds__(256) k_rowmass(const float* __restrict__ L2, const float* __restrict__ x,
                                                 const int32_t* __restrict__ offsets, int n, int64_t ldA,
                                                 float* __restrict__ u, const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int q = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (q >= n) return;
    const float* row = L2 + ((int64_t)h * n + q) * ldA;
    dfloat acc{0.f, 0.f};
    for (int i = lane; i < t; i += 32) df_fma(acc, exp2f(row[i]), x[off + i]);
    acc = warp_sum_df(acc);
    if (lane == 0) u[(int64_t)h * n + q] = (1.f - acc.hi) - acc.lo;
}

// r_i = sum_q A'_qi u_q + mu (1 - x_i) on the free set, 0 on the zero set.
// grid (ceil(max_t/64), H), block 256 (4 row groups x 64 columns).
__global__ void __launch_bounds__(256) k_colresid(const float* __restrict__ L2, const float* __restrict__ u,
                                                  const float* __restrict__ x, const int8_t* __restrict__ zflag,
                                                  const int32_t* __restrict__ offsets, int n, int64_t ldA,
                                                  const HeadScalars* __restrict__ hs, float* __restrict__ r,
                                                  const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int c = blockIdx.x * 64 + (threadIdx.x & 63);
    const int rg = threadIdx.x >> 6;
    __shared__ dfloat red[4][64];
    dfloat acc{0.f, 0.f};
    if (c < t) {
        const float* col = L2 + (int64_t)h * n * ldA + c;
        const float* uh = u + (int64_t)h * n;
        for (int q = rg; q < n; q += 4) df_fma(acc, exp2f(col[(int64_t)q * ldA]), uh[q]);
    }
    red[rg][threadIdx.x & 63] = acc;
    __syncthreads();
    if (rg == 0 && c < t) {
        for (int g = 1; g < 4; ++g) df_add_df(acc, red[g][threadIdx.x]);
        const float mu = hs[h].mu;
        df_fma(acc, mu, 1.f - x[off + c]);
        r[off + c] = zflag[off + c] ? 0.f : acc.hi + acc.lo;
    }
}

// x += H_FF^{-1} r_F: d0 = H^{-1} r is in `d0`; apply the Schur correction
// with the stored factor of (H^{-1})_ZZ.  grid H, block 512.
__global__ void __launch_bounds__(512) k_refine_apply(BppArgs a, const float* __restrict__ d0) {
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
    for (int k = threadIdx.x; k < nz; k += blockDim.x) zl[k] = a.zlist[(int64_t)h * a.zmax + k];
    for (int i = threadIdx.x; i < t; i += blockDim.x) ssrc[i] = d0[off + i];
    __syncthreads();
    schur_solution(a, h, off, t, nz, zl, false, ssrc, sx, snu, sm_chol, &sflag);
    for (int i = threadIdx.x; i < t; i += blockDim.x)
        if (!a.zflag[off + i]) a.x[off + i] += sx[i];
}

// beta = log w (w clamped at 0; -inf where w = 0).  grid (ceil(max_t/256), H).
__global__ void k_beta_out(float* __restrict__ x, const int32_t* __restrict__ offsets, float* __restrict__ beta,
                           const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= t || !head_ok(status, h)) return;
    const float w = fmaxf(x[off + i], 0.f);
    x[off + i] = w;
    beta[off + i] = (w > 0.f) ? logf(w) : -INFINITY;
}

// ------------------------------------------------------------ launchers
cudaError_t launch_chol(float* mats, const int32_t* offsets, int H, int max_t, int64_t ldA, float* dscr,
                        int32_t* status, cudaStream_t st) {
    for (int k0 = 0; k0 < max_t; k0 += CB) {
        const int rows_below = max(0, max_t - k0 - CB);
        const int nrb = (rows_below + CB - 1) / CB;
        k_chol_panel<<<dim3(1 + nrb, H), 128, 0, st>>>(mats, offsets, ldA, k0, dscr, status);
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

static cudaError_t launch_trsv(const SolveArgs& a, int ncta, int H, cudaStream_t st) {
    const size_t smem = (size_t)(a.ldA + CB * (CB + 1)) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_trsv_cols, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_trsv_cols<<<dim3(ncta, H), 256, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_cholsolve(int d, const float* L, const float* R, const int32_t* offsets, int H, int64_t ldA,
                             float* Cv, const int32_t* status, cudaStream_t st) {
    SolveArgs a{};
    a.L = L;
    a.offsets = offsets;
    a.ldA = ldA;
    a.mode = SOLVE_RHS_D;
    a.R = R;
    a.X = Cv;
    a.d = d;
    a.status = status;
    return launch_trsv(a, d, H, st);
}

static size_t bpp_smem(int64_t ldA, int zmax) {
    return (size_t)(2 * ldA + zmax) * sizeof(float) + (size_t)zmax * sizeof(int) +
           (size_t)(CB * (CB + 1) + (size_t)zmax * (CB + 1)) * sizeof(float);
}

// The whole NNLS: x0 = H^{-1} f, `max_iter` pivoting steps, refinement.
cudaError_t launch_nnls_all(const float* L, const float* f, const int32_t* offsets, int H, int n, int max_t,
                            int64_t ldA, const float* L2, float* x, float* x0, int8_t* zflag, int32_t* zlist,
                            int32_t* nz, float* W, float* S, int32_t* piv, float* u, float* r, float* d0,
                            HeadScalars* hs, int zmax, int max_iter, int refine_iters, int32_t* status,
                            cudaStream_t st, int* launches) {
    BppArgs b{x0, x, zflag, zlist, nz, W, S, piv, offsets, f, ldA, zmax, hs, status};
    int nl = 0;
    k_bpp_init<<<dim3((max_t + 255) / 256, H), 256, 0, st>>>(b);
    ++nl;
    SolveArgs sv{};
    sv.L = L;
    sv.offsets = offsets;
    sv.ldA = ldA;
    sv.status = status;
    sv.mode = SOLVE_VEC;
    sv.vin = f;
    sv.vout = x0;
    cudaError_t e = launch_trsv(sv, 1, H, st);
    if (e != cudaSuccess) return e;
    ++nl;
    const size_t smem = bpp_smem(ldA, zmax);
    e = cudaFuncSetAttribute(k_bpp_step, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_refine_apply, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    SolveArgs sz{};
    sz.L = L;
    sz.offsets = offsets;
    sz.ldA = ldA;
    sz.status = status;
    sz.mode = SOLVE_UNIT_Z;
    sz.zlist = zlist;
    sz.nz = nz;
    sz.W = W;
    sz.zmax = zmax;
    sz.done = piv;          // piv[4h] is the done flag
    sz.done_stride = 4;
    for (int it = 0; it < max_iter; ++it) {
        if (it > 0) {
            // columns H^{-1} e_z for the zero set chosen by the previous step
            e = launch_trsv(sz, 32, H, st);
            if (e != cudaSuccess) return e;
            ++nl;
        }
        k_bpp_step<<<H, 512, smem, st>>>(b);
        ++nl;
    }
    k_bpp_finish<<<(H + 127) / 128, 128, 0, st>>>(b, H);
    ++nl;
    for (int it = 0; it < refine_iters; ++it) {
        k_rowmass<<<dim3((n + 7) / 8, H), 256, 0, st>>>(L2, x, offsets, n, ldA, u, status);
        k_colresid<<<dim3((max_t + 63) / 64, H), 256, 0, st>>>(L2, u, x, zflag, offsets, n, ldA, hs, r, status);
        SolveArgs s3 = sv;
        s3.vin = r;
        s3.vout = d0;
        e = launch_trsv(s3, 1, H, st);
        if (e != cudaSuccess) return e;
        k_refine_apply<<<H, 512, smem, st>>>(b, d0);
        nl += 4;
    }
    if (launches) *launches = nl;
    return cudaGetLastError();
}

cudaError_t launch_beta_out(float* x, const int32_t* offsets, int H, int max_t, float* beta, const int32_t* status,
                            cudaStream_t st) {
    dim3 grid((max_t + 255) / 256, H);
    k_beta_out<<<grid, 256, 0, st>>>(x, offsets, beta, status);
    return cudaGetLastError();
}

}  // namespace kvc
