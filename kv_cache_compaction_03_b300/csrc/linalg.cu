// Batched dense solvers for the two fits of the compaction ("Fast KV
// Compaction via Attention Matching", section 2, "Ajustement du biais et des
// valeurs"):
//   k_chol          in-place lower Cholesky of H = A'^T A' + mu I or of
//                   M = X^T X + lambda I (one CTA per head)
//   k_nnls_bpp      min_{w>=0} 1/2 w^T H w - f^T w by block principal pivoting;
//                   each pivoting step solves the free-set system through the
//                   full factor of H and a Schur complement on the zero set
//   k_rowmass / k_colresid / k_nnls_correct
//                   iterative refinement of w with the residual
//                   A'^T (1 - A' w) + mu (1 - w) taken from A' directly
//   k_beta_out      beta = log w
//   k_cholsolve     C_v = M^{-1} R (columns split across CTAs)
// All matrices are row-major fp32; a CTA-wide routine is called by every
// thread of the block.
#include "common.cuh"

namespace kvc {

// ------------------------------------------------------------ CTA routines
// In-place lower Cholesky of the n x n matrix A (leading dim lda), right-
// looking, NB-wide panels.  smem: NB*(NB+1) + n*NB floats.  Returns false
// (uniformly across the block) if a pivot is not positive or not finite.
template <int NB>
__device__ bool cta_chol(float* A, int n, int64_t lda, float* smem, int* sflag) {
    float* Dg = smem;
    float* Pn = smem + NB * (NB + 1);
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) *sflag = 0;
    __syncthreads();
    for (int k0 = 0; k0 < n; k0 += NB) {
        const int kb = min(NB, n - k0);
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            Dg[i * (NB + 1) + j] = (j <= i) ? A[(int64_t)(k0 + i) * lda + k0 + j] : 0.f;
        }
        __syncthreads();
        if (tid < 32) {
            const int lane = tid;
            for (int j = 0; j < kb; ++j) {
                const float djj = Dg[j * (NB + 1) + j];
                if (!(djj > 0.f) || !isfinite(djj)) {
                    if (lane == 0) *sflag = 1;
                    break;
                }
                const float r = sqrtf(djj);
                __syncwarp();
                if (lane == 0) Dg[j * (NB + 1) + j] = r;
                for (int i = j + 1 + lane; i < kb; i += 32) Dg[i * (NB + 1) + j] /= r;
                __syncwarp();
                for (int i = j + 1 + lane; i < kb; i += 32) {
                    const float lij = Dg[i * (NB + 1) + j];
                    for (int k = j + 1; k <= i; ++k) Dg[i * (NB + 1) + k] -= lij * Dg[k * (NB + 1) + j];
                }
                __syncwarp();
            }
        }
        __syncthreads();
        if (*sflag) return false;
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            if (j <= i) A[(int64_t)(k0 + i) * lda + k0 + j] = Dg[i * (NB + 1) + j];
        }
        const int m = n - k0 - kb;
        for (int r = tid; r < m; r += nt) {
            float* row = A + (int64_t)(k0 + kb + r) * lda + k0;
            float x[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                if (j < kb) {
                    float v = row[j];
#pragma unroll
                    for (int p = 0; p < NB; ++p)
                        if (p < j) v -= x[p] * Dg[j * (NB + 1) + p];
                    x[j] = v / Dg[j * (NB + 1) + j];
                } else {
                    x[j] = 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                if (j < kb) row[j] = x[j];
                Pn[r * NB + j] = x[j];
            }
        }
        __syncthreads();
        // trailing update, lower triangle, 4x4 register blocks
        const int m4 = (m + 3) / 4;
        const int nblk = m4 * (m4 + 1) / 2;
        for (int bidx = tid; bidx < nblk; bidx += nt) {
            int bi = (int)((sqrtf(8.f * (float)bidx + 1.f) - 1.f) * 0.5f);
            while (bi * (bi + 1) / 2 > bidx) --bi;
            while ((bi + 1) * (bi + 2) / 2 <= bidx) ++bi;
            const int bj = bidx - bi * (bi + 1) / 2;
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
            const int ri = bi * 4, rj = bj * 4;
#pragma unroll 4
            for (int p = 0; p < NB; ++p) {
                float pi[4], pj[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) pi[a] = (ri + a < m) ? Pn[(ri + a) * NB + p] : 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) pj[c] = (rj + c < m) ? Pn[(rj + c) * NB + p] : 0.f;
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(pi[a], pj[c], acc[a][c]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int i = ri + a;
                if (i >= m) continue;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = rj + c;
                    if (j < m && j <= i) A[(int64_t)(k0 + kb + i) * lda + k0 + kb + j] -= acc[a][c];
                }
            }
        }
        __syncthreads();
    }
    return true;
}

// Solve L Y = B in place (B: n x nrhs, leading dim ldb; L lower, lda).
// smem: NB*(NB+1) floats.
template <int NB>
__device__ void cta_trsm_lower(const float* L, int n, int64_t lda, float* B, int nrhs, int64_t ldb, float* Dg) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int k0 = 0; k0 < n; k0 += NB) {
        const int kb = min(NB, n - k0);
        __syncthreads();
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            Dg[i * (NB + 1) + j] = (j <= i) ? L[(int64_t)(k0 + i) * lda + k0 + j] : 0.f;
        }
        __syncthreads();
        for (int c = tid; c < nrhs; c += nt) {
            float y[NB];
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                if (i < kb) {
                    float v = B[(int64_t)(k0 + i) * ldb + c];
#pragma unroll
                    for (int p = 0; p < NB; ++p)
                        if (p < i) v -= Dg[i * (NB + 1) + p] * y[p];
                    y[i] = v / Dg[i * (NB + 1) + i];
                    B[(int64_t)(k0 + i) * ldb + c] = y[i];
                }
            }
        }
        __syncthreads();
        const int rows = n - k0 - kb;
        const int64_t tot = (int64_t)rows * nrhs;
        for (int64_t e = tid; e < tot; e += nt) {
            const int r = k0 + kb + (int)(e / nrhs), c = (int)(e % nrhs);
            const float* lr = L + (int64_t)r * lda + k0;
            float v = B[(int64_t)r * ldb + c];
            for (int p = 0; p < kb; ++p) v -= lr[p] * B[(int64_t)(k0 + p) * ldb + c];
            B[(int64_t)r * ldb + c] = v;
        }
    }
    __syncthreads();
}

// Solve L^T X = Y in place.
template <int NB>
__device__ void cta_trsm_upper_t(const float* L, int n, int64_t lda, float* B, int nrhs, int64_t ldb, float* Dg) {
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int kend = n; kend > 0; kend -= NB) {
        const int k0 = max(0, kend - NB);
        const int kb = kend - k0;
        __syncthreads();
        for (int e = tid; e < kb * kb; e += nt) {
            const int i = e / kb, j = e % kb;
            Dg[i * (NB + 1) + j] = (j <= i) ? L[(int64_t)(k0 + i) * lda + k0 + j] : 0.f;
        }
        __syncthreads();
        for (int c = tid; c < nrhs; c += nt) {
            float x[NB];
#pragma unroll
            for (int ii = NB - 1; ii >= 0; --ii) {
                if (ii < kb) {
                    float v = B[(int64_t)(k0 + ii) * ldb + c];
#pragma unroll
                    for (int p = 0; p < NB; ++p)
                        if (p > ii && p < kb) v -= Dg[p * (NB + 1) + ii] * x[p];
                    x[ii] = v / Dg[ii * (NB + 1) + ii];
                    B[(int64_t)(k0 + ii) * ldb + c] = x[ii];
                } else {
                    x[ii] = 0.f;
                }
            }
        }
        __syncthreads();
        const int64_t tot = (int64_t)k0 * nrhs;
        for (int64_t e = tid; e < tot; e += nt) {
            const int r = (int)(e / nrhs), c = (int)(e % nrhs);
            float v = B[(int64_t)r * ldb + c];
            for (int p = 0; p < kb; ++p) v -= L[(int64_t)(k0 + p) * lda + r] * B[(int64_t)(k0 + p) * ldb + c];
            B[(int64_t)r * ldb + c] = v;
        }
    }
    __syncthreads();
}

template <int NB>
__device__ __forceinline__ void cta_cholsolve(const float* L, int n, int64_t lda, float* B, int nrhs, int64_t ldb,
                                              float* Dg) {
    cta_trsm_lower<NB>(L, n, lda, B, nrhs, ldb, Dg);
    cta_trsm_upper_t<NB>(L, n, lda, B, nrhs, ldb, Dg);
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
// grid H, block 1024.  Factor the t_h x t_h lower triangle of mats[h].
template <int NB>
__global__ void __launch_bounds__(1024) k_chol(float* __restrict__ mats, const int32_t* __restrict__ offsets,
                                               int64_t ldA, int32_t* __restrict__ status) {
    const int h = blockIdx.x;
    if (!head_ok(status, h)) return;
    extern __shared__ float sm[];
    __shared__ int sflag;
    const int t = offsets[h + 1] - offsets[h];
    if (!cta_chol<NB>(mats + (int64_t)h * ldA * ldA, t, ldA, sm, &sflag)) {
        if (threadIdx.x == 0) set_status(status, h, KVC_ERR_NOT_SPD);
    }
}

// C_v = M^{-1} R for 16 columns per CTA.  grid (D/16, H), block 256.
template <int D>
__global__ void __launch_bounds__(256) k_cholsolve(const float* __restrict__ L, const float* __restrict__ R,
                                                   const int32_t* __restrict__ offsets, int64_t ldA,
                                                   float* __restrict__ Cv, const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    __shared__ float Dg[32 * 33];
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int c0 = blockIdx.x * 16;
    float* B = Cv + (int64_t)off * D + c0;
    for (int e = threadIdx.x; e < t * 16; e += blockDim.x) {
        const int i = e / 16, c = e % 16;
        B[(int64_t)i * D + c] = R[((int64_t)off + i) * D + c0 + c];
    }
    cta_cholsolve<32>(L + (int64_t)h * ldA * ldA, t, ldA, B, 16, D, Dg);
}

// ------------------------------------------------------------ NNLS

// Free-set solution for the current zero set: x = H^{-1}(rhs + E_Z nu) with nu
// chosen so x_Z = 0.  On entry sx holds H^{-1} rhs; on exit sx = x and
// snu[k] = nu_k (the gradient on the zero set).  Rebuilds W and S when
// `rebuild` is set.  Returns false if (H^{-1})_ZZ is not numerically SPD.
__device__ bool schur_apply(const NnlsArgs& a, int h, int t, int nz, const int* zl, bool rebuild, float* sx,
                            float* snu, float* sm_chol, int* sflag) {
    if (nz == 0) return true;
    const int64_t ldW = a.zmax;
    float* W = a.W + (int64_t)h * a.ldA * ldW;
    float* S = a.S + (int64_t)h * ldW * ldW;
    const float* L = a.L + (int64_t)h * a.ldA * a.ldA;
    if (rebuild) {
        for (int64_t e = threadIdx.x; e < (int64_t)t * nz; e += blockDim.x) {
            const int i = (int)(e / nz), k = (int)(e % nz);
            W[(int64_t)i * ldW + k] = (i == zl[k]) ? 1.f : 0.f;
        }
        __syncthreads();
        cta_cholsolve<32>(L, t, a.ldA, W, nz, ldW, sm_chol);
        for (int e = threadIdx.x; e < nz * nz; e += blockDim.x) {
            const int r = e / nz, c = e % nz;
            S[(int64_t)r * ldW + c] = W[(int64_t)zl[r] * ldW + c];
        }
        __syncthreads();
        if (!cta_chol<16>(S, nz, ldW, sm_chol, sflag)) return false;
    }
    for (int k = threadIdx.x; k < nz; k += blockDim.x) snu[k] = -sx[zl[k]];
    __syncthreads();
    cta_cholsolve<16>(S, nz, ldW, snu, 1, 1, sm_chol);
    for (int i = threadIdx.x; i < t; i += blockDim.x) {
        float v = sx[i];
        const float* wr = W + (int64_t)i * ldW;
        for (int k = 0; k < nz; ++k) v = fmaf(wr[k], snu[k], v);
        sx[i] = v;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < nz; k += blockDim.x) sx[zl[k]] = 0.f;
    __syncthreads();
    return true;
}

// Rebuild the sorted zero-set list from the flags; returns |Z|.
__device__ int build_zlist(const int8_t* zf, int t, int* zl, int zmax, int* sbuf) {
    // simple ordered compaction: thread chunks + scan
    const int chunk = (t + blockDim.x - 1) / blockDim.x;
    const int j0 = min(t, (int)threadIdx.x * chunk), j1 = min(t, j0 + chunk);
    int c = 0;
    for (int j = j0; j < j1; ++j) c += zf[j] != 0;
    // exclusive scan over the block
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

// grid H, block 1024.  Dynamic smem: 3*ldA floats + zmax ints + chol scratch.
__global__ void __launch_bounds__(1024) k_nnls_bpp(NnlsArgs a) {
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return;
    extern __shared__ float sm[];
    const int off = a.offsets[h];
    const int t = a.offsets[h + 1] - off;
    float* sx0 = sm;                          // H^{-1} f
    float* sx = sx0 + a.ldA;                  // current iterate
    float* sy = sx + a.ldA;                   // gradient on the zero set
    float* snu = sy + a.ldA;                  // [zmax]
    int* zl = reinterpret_cast<int*>(snu + a.zmax);
    float* sm_chol = reinterpret_cast<float*>(zl + a.zmax);   // 16*17 + zmax*16 floats
    __shared__ int sbuf[33];
    __shared__ int sflag, s_best, s_budget, s_nbad, s_maxbad, s_done;
    __shared__ float sred[32];
    int8_t* zf = a.zflag + off;
    const float* L = a.L + (int64_t)h * a.ldA * a.ldA;

    for (int i = threadIdx.x; i < t; i += blockDim.x) {
        sx0[i] = a.f[off + i];
        zf[i] = 0;
    }
    if (threadIdx.x == 0) {
        s_best = t + 1;
        s_budget = 3;
        s_done = 0;
    }
    __syncthreads();
    cta_cholsolve<32>(L, t, a.ldA, sx0, 1, 1, sm_chol);
    const float fmax = block_max_abs(a.f + off, t, sred);
    int it = 0;
    int nz = 0;
    for (; it < a.max_iter; ++it) {
        nz = build_zlist(zf, t, zl, a.zmax, sbuf);
        if (nz > a.zmax) {
            if (threadIdx.x == 0) set_status(a.status, h, KVC_ERR_NNLS_MAXITER);
            break;
        }
        for (int i = threadIdx.x; i < t; i += blockDim.x) {
            sx[i] = sx0[i];
            sy[i] = 0.f;
        }
        __syncthreads();
        if (!schur_apply(a, h, t, nz, zl, true, sx, snu, sm_chol, &sflag)) {
            if (threadIdx.x == 0) set_status(a.status, h, KVC_ERR_NOT_SPD);
            break;
        }
        for (int k = threadIdx.x; k < nz; k += blockDim.x) sy[zl[k]] = snu[k];
        __syncthreads();
        const float xmax = block_max_abs(sx, t, sred);
        const float tolx = 1e-6f * xmax, toly = 1e-6f * fmax;
        if (threadIdx.x == 0) {
            s_nbad = 0;
            s_maxbad = -1;
        }
        __syncthreads();
        int nb = 0, mb = -1;
        for (int i = threadIdx.x; i < t; i += blockDim.x) {
            const bool bad = zf[i] ? (sy[i] < -toly) : (sx[i] < -tolx);
            if (bad) {
                ++nb;
                mb = max(mb, i);
            }
        }
        if (nb) {
            atomicAdd(&s_nbad, nb);
            atomicMax(&s_maxbad, mb);
        }
        __syncthreads();
        const int nbad = s_nbad;
        if (nbad == 0) {
            if (threadIdx.x == 0) s_done = 1;
            __syncthreads();
            break;
        }
        bool full = false;
        if (threadIdx.x == 0) {
            if (nbad < s_best) {
                s_best = nbad;
                s_budget = 3;
                sflag = 1;
            } else if (s_budget > 0) {
                --s_budget;
                sflag = 1;
            } else {
                sflag = 0;
            }
        }
        __syncthreads();
        full = sflag != 0;
        const int maxbad = s_maxbad;
        for (int i = threadIdx.x; i < t; i += blockDim.x) {
            const bool bad = zf[i] ? (sy[i] < -toly) : (sx[i] < -tolx);
            if (bad && (full || i == maxbad)) zf[i] = zf[i] ? 0 : 1;
        }
        __syncthreads();
    }
    if (!s_done && head_ok(a.status, h) && threadIdx.x == 0) set_status(a.status, h, KVC_ERR_NNLS_MAXITER);
    for (int i = threadIdx.x; i < t; i += blockDim.x) a.x[off + i] = zf[i] ? 0.f : fmaxf(sx[i], 0.f);
    if (threadIdx.x == 0) {
        a.hs[h].nzero = nz;
        a.hs[h].iters = it;
    }
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

// x += H_FF^{-1} r_F via the stored factor and Schur complement.  grid H, block 1024.
__global__ void __launch_bounds__(1024) k_nnls_correct(NnlsArgs a, const float* __restrict__ r) {
    const int h = blockIdx.x;
    if (!head_ok(a.status, h)) return;
    extern __shared__ float sm[];
    const int off = a.offsets[h];
    const int t = a.offsets[h + 1] - off;
    float* sd = sm;
    float* snu = sd + a.ldA;
    int* zl = reinterpret_cast<int*>(snu + a.zmax);
    float* sm_chol = reinterpret_cast<float*>(zl + a.zmax);
    __shared__ int sbuf[33];
    __shared__ int sflag;
    const int nz = build_zlist(a.zflag + off, t, zl, a.zmax, sbuf);
    if (nz > a.zmax) return;
    for (int i = threadIdx.x; i < t; i += blockDim.x) sd[i] = r[off + i];
    __syncthreads();
    cta_cholsolve<32>(a.L + (int64_t)h * a.ldA * a.ldA, t, a.ldA, sd, 1, 1, sm_chol);
    schur_apply(a, h, t, nz, zl, false, sd, snu, sm_chol, &sflag);
    for (int i = threadIdx.x; i < t; i += blockDim.x)
        if (!a.zflag[off + i]) a.x[off + i] += sd[i];
}

// beta = log w (w clamped at 0; -inf where w = 0).  grid ceil(maxsum/256).
__global__ void k_beta_out(float* __restrict__ x, const int32_t* __restrict__ offsets, int H, float* __restrict__ beta,
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
static size_t chol_smem(int nb, int n) { return (size_t)(nb * (nb + 1) + (size_t)n * nb) * sizeof(float); }

cudaError_t launch_chol(float* mats, const int32_t* offsets, int H, int max_t, int64_t ldA, int32_t* status,
                        cudaStream_t st) {
    cudaError_t e;
    if (max_t <= 1024) {
        size_t smem = chol_smem(32, max_t);
        e = cudaFuncSetAttribute(k_chol<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_chol<32><<<H, 1024, smem, st>>>(mats, offsets, ldA, status);
    } else if (max_t <= 2048) {
        size_t smem = chol_smem(16, max_t);
        e = cudaFuncSetAttribute(k_chol<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_chol<16><<<H, 1024, smem, st>>>(mats, offsets, ldA, status);
    } else {
        size_t smem = chol_smem(8, max_t);
        e = cudaFuncSetAttribute(k_chol<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_chol<8><<<H, 1024, smem, st>>>(mats, offsets, ldA, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_cholsolve(int d, const float* L, const float* R, const int32_t* offsets, int H, int64_t ldA,
                             float* Cv, const int32_t* status, cudaStream_t st) {
    dim3 grid(d / 16, H);
    if (d == 128)
        k_cholsolve<128><<<grid, 256, 0, st>>>(L, R, offsets, ldA, Cv, status);
    else
        k_cholsolve<64><<<grid, 256, 0, st>>>(L, R, offsets, ldA, Cv, status);
    return cudaGetLastError();
}

static size_t nnls_smem(int64_t ldA, int zmax) {
    return (size_t)(3 * ldA + zmax) * sizeof(float) + (size_t)zmax * sizeof(int) +
           chol_smem(16, zmax) + 32 * 33 * sizeof(float);
}

cudaError_t launch_nnls(const NnlsArgs& a, int H, cudaStream_t st) {
    size_t smem = nnls_smem(a.ldA, a.zmax);
    cudaError_t e = cudaFuncSetAttribute(k_nnls_bpp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_nnls_bpp<<<H, 1024, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_nnls_refine(const NnlsArgs& a, const float* L2, float* u, float* r, int H, int n, int max_t,
                               cudaStream_t st) {
    k_rowmass<<<dim3((n + 7) / 8, H), 256, 0, st>>>(L2, a.x, a.offsets, n, a.ldA, u, a.status);
    k_colresid<<<dim3((max_t + 63) / 64, H), 256, 0, st>>>(L2, u, a.x, a.zflag, a.offsets, n, a.ldA, a.hs, r,
                                                          a.status);
    size_t smem = nnls_smem(a.ldA, a.zmax);
    cudaError_t e = cudaFuncSetAttribute(k_nnls_correct, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_nnls_correct<<<H, 1024, smem, st>>>(a, r);
    return cudaGetLastError();
}

cudaError_t launch_beta_out(float* x, const int32_t* offsets, int H, int max_t, float* beta, const int32_t* status,
                            cudaStream_t st) {
    dim3 grid((max_t + 255) / 256, H);
    k_beta_out<<<grid, 256, 0, st>>>(x, offsets, H, beta, status);
    return cudaGetLastError();
}

size_t nnls_smem_bytes(int64_t ldA, int zmax) { return nnls_smem(ldA, zmax); }

}  // namespace kvc
