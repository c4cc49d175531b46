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
//   k_sweep_pivot   grid (blocks, H): every CTA sweeps the 64 x 64 pivot
//                   block in registers (64 scalar sweeps, giving -P), then
//                   computes U_i = A_ik P for its row block i (stored
//                   transposed) and copies V_i = A_ki (row block k)
//   k_sweep_update  grid (lower tiles, H): every 64 x 64 tile on or below
//                   the diagonal is updated from U, V and P (128 threads, an
//                   8 x 4 register tile each; both operand tiles are 64
//                   contiguous 256-byte rows); on a head's last block the
//                   stored result is negated, so the matrix ends as +H^{-1}
//   k_sweep_mirror  copies the lower triangle into the upper one
//   k_symv          y = H^{-1} v for every head (one warp per row)
//   k_apply_inverse C_v = M^{-1} R (the least-squares fit of C_v when M is
//                   inverted by the same sweeps)
// The sweep keeps the symmetric matrix in its lower triangle (row-major,
// leading dimension ldA); an entry above the diagonal is read from its
// mirror image.  The finished inverse is stored in full.
#include "common.cuh"

namespace kvc {

namespace {
constexpr int SB = 64;     // sweep block

struct SweepArgs {
    float* A;                 // [H][ldA][ldA]
    float* U;                 // [H][64][ldA]  U^T: U[p][r] = (A_ik P)[r][p]
    float* V;                 // [H][64][ldA]
    float* P;                 // [H][64][64]
    const int32_t* offsets;
    int64_t ldA;
    int k0;                   // first row of the pivot block
    int32_t* status;
};


// grid (blocks, H), block 256.  Thread (ii, cq) holds row ii, columns
// 16 cq .. 16 cq + 15 of the pivot block in registers; the 64 scalar sweeps
// run as 4 x 16 with the inner 16 unrolled, so the column the sweep pivots on
// has a static register index (and the loop body stays small).
constexpr int kPS = SB + 4;      // padded smem row, 16-byte aligned

__global__ void __launch_bounds__(256) k_sweep_pivot(SweepArgs s) {
    const int h = blockIdx.y;
    if (!head_ok(s.status, h)) return;
    const int t = s.offsets[h + 1] - s.offsets[h];
    const int k0 = s.k0;
    if (k0 >= t) return;
    const int r0 = blockIdx.x * SB;
    if (r0 >= t) return;
    __shared__ __align__(16) float rowb[2][SB];
    __shared__ __align__(16) float Ps[SB][kPS];     // A_ik (rows r0.., columns k0..)
    __shared__ __align__(16) float Pn[SB][kPS];     // P
    __shared__ int bad;
    const float* A = s.A + (int64_t)h * s.ldA * s.ldA;
    const int tid = threadIdx.x;
    const int ii = tid >> 2, cq = tid & 3;          // row ii, columns 16 cq + m
    // the pivot block: its stored lower triangle, staged through Pn
    for (int e = tid; e < SB * SB; e += 256) {
        const int r = e / SB, c = e % SB;
        if (c <= r) Pn[r][c] = (k0 + r < t && k0 + c < t) ? A[(int64_t)(k0 + r) * s.ldA + k0 + c] : (r == c ? 1.f : 0.f);
    }
    __syncthreads();
    float a[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int c = 16 * cq + m;
        a[m] = (c <= ii) ? Pn[ii][c] : Pn[c][ii];
    }
    if (r0 > k0) {
        for (int e = tid; e < SB * SB; e += 256) {
            const int rr = e / SB, c = e % SB;
            const int r = r0 + rr, col = k0 + c;
            Ps[rr][c] = (r < t && col < t) ? A[(int64_t)r * s.ldA + col] : 0.f;
        }
    } else if (r0 < k0) {
        // A_ik above the diagonal: the transpose of the stored tile (k, i)
        for (int e = tid; e < SB * SB; e += 256) {
            const int c = e / SB, rr = e % SB;
            const int r = r0 + rr, col = k0 + c;
            Ps[rr][c] = (r < t && col < t) ? A[(int64_t)col * s.ldA + r] : 0.f;
        }
    }
    if (tid == 0) bad = 0;
    __syncthreads();     // Pn is rewritten below
    // 64 scalar sweeps of the pivot block; the block stays symmetric, so row
    // p also provides column p
    for (int pb = 0; pb < 4; ++pb) {
#pragma unroll
        for (int m0 = 0; m0 < 16; ++m0) {
            const int p = 16 * pb + m0;
            float* rb = rowb[p & 1];
            if (ii == p) {
#pragma unroll
                for (int m = 0; m < 16; m += 4)
                    *reinterpret_cast<float4*>(rb + 16 * cq + m) = make_float4(a[m], a[m + 1], a[m + 2], a[m + 3]);
            }
            __syncthreads();
            float d = rb[p];
            if (!(d > 0.f) || !isfinite(d)) {
                if (tid == 0) bad = 1;
                d = 1.f;
            }
            // reciprocal: hardware approximation plus one Newton step (~1 ulp)
            float inv;
            asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(d));
            inv = inv * fmaf(-d, inv, 2.f);
            if (ii != p) {
                // a_ic -= a_ip a_pc / d; column p itself becomes a_ip / d
                const float f = rb[ii] * inv;
#pragma unroll
                for (int m = 0; m < 16; m += 4) {
                    const float4 r4 = *reinterpret_cast<const float4*>(rb + 16 * cq + m);
                    a[m] = fmaf(-f, r4.x, a[m]);
                    a[m + 1] = fmaf(-f, r4.y, a[m + 1]);
                    a[m + 2] = fmaf(-f, r4.z, a[m + 2]);
                    a[m + 3] = fmaf(-f, r4.w, a[m + 3]);
                }
                if (cq == pb) a[m0] = f;
            } else {
                // row p becomes a_pc / d, the pivot -1 / d
#pragma unroll
                for (int m = 0; m < 16; ++m) a[m] *= inv;
                if (cq == pb) a[m0] = -inv;
            }
        }
    }
    __syncthreads();
    if (bad) {
        if (blockIdx.x == 0 && tid == 0) set_status(s.status, h, KVC_ERR_NOT_SPD);
        return;
    }
#pragma unroll
    for (int m = 0; m < 16; m += 4)
        *reinterpret_cast<float4*>(&Pn[ii][16 * cq + m]) = make_float4(-a[m], -a[m + 1], -a[m + 2], -a[m + 3]);
    __syncthreads();
    if (r0 == k0) {
        float* Ph = s.P + (int64_t)h * SB * SB;
        for (int e = tid; e < SB * SB; e += 256) Ph[e] = Pn[e / SB][e % SB];
        return;
    }
    // U_i = A_ik P  (rows r0 .. r0+63), V_i = A_ki = A_ik^T
    float acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m] = 0.f;
#pragma unroll 4
    for (int p = 0; p < SB; ++p) {
        const float x = Ps[ii][p];
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 q = *reinterpret_cast<const float4*>(&Pn[p][16 * cq + m]);
            acc[m] = fmaf(x, q.x, acc[m]);
            acc[m + 1] = fmaf(x, q.y, acc[m + 1]);
            acc[m + 2] = fmaf(x, q.z, acc[m + 2]);
            acc[m + 3] = fmaf(x, q.w, acc[m + 3]);
        }
    }
    float* Uh = s.U + (int64_t)h * SB * s.ldA + r0;
#pragma unroll
    for (int m = 0; m < 16; ++m) Uh[(int64_t)(16 * cq + m) * s.ldA + ii] = acc[m];
    float* Vh = s.V + (int64_t)h * SB * s.ldA + r0;
    for (int e = tid; e < SB * SB; e += 256) {
        const int c = e / SB, rr = e % SB;
        Vh[(int64_t)c * s.ldA + rr] = Ps[rr][c];
    }
}

__device__ __forceinline__ void tri_tile(int p, int& I, int& J) {
    int i = (int)((sqrtf(8.f * (float)p + 1.f) - 1.f) * 0.5f);
    while (i * (i + 1) / 2 > p) --i;
    while ((i + 1) * (i + 2) / 2 <= p) ++i;
    I = i;
    J = p - i * (i + 1) / 2;
}

constexpr int kUpdThreads = 128;
constexpr int kUS = SB + 4;      // padded smem row: 16-byte aligned

// grid (blocks * (blocks + 1) / 2, H), block 128: tile (bi >= bj) of the lower triangle.
__global__ void __launch_bounds__(kUpdThreads) k_sweep_update(SweepArgs s) {
    const int h = blockIdx.y;
    if (!head_ok(s.status, h)) return;
    const int t = s.offsets[h + 1] - s.offsets[h];
    const int k0 = s.k0;
    if (k0 >= t) return;
    int bi, bj;
    tri_tile(blockIdx.x, bi, bj);
    const int ri = bi * SB, rj = bj * SB;
    if (ri >= t) return;
    const bool last = k0 + SB >= t;        // this head's last pivot block: store +H^{-1}
    const float sg = last ? -1.f : 1.f;
    float* A = s.A + (int64_t)h * s.ldA * s.ldA;
    const float* Uh = s.U + (int64_t)h * SB * s.ldA;     // U^T [64][ldA]
    const float* Vh = s.V + (int64_t)h * SB * s.ldA;
    const float* Ph = s.P + (int64_t)h * SB * SB;
    const int tid = threadIdx.x;
    const bool pi = (ri == k0), pj = (rj == k0);
    if (pi || pj) {
        // pivot row / column / block: copies, no products
        for (int e = tid; e < SB * SB; e += kUpdThreads) {
            const int r = e / SB, c = e % SB;
            if (ri + r >= t || rj + c >= t) continue;
            float v;
            if (pi && pj) v = -Ph[e];
            else if (pj) v = Uh[(int64_t)c * s.ldA + ri + r];        // A_ik = U_i
            else v = Uh[(int64_t)r * s.ldA + rj + c];               // A_kj = U_j^T
            A[(int64_t)(ri + r) * s.ldA + rj + c] = sg * v;
        }
        return;
    }
    __shared__ __align__(16) float Ut[SB][kUS];     // Ut[p][r] = U_i[r][p]
    __shared__ __align__(16) float Vs[SB][kUS];     // Vs[p][c] = V[p][rj + c]
    {
        float4 ru[8], rv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + kUpdThreads * q;           // float4 index: row e / 16, column 4 (e % 16)
            const int p = e >> 4, c4 = (e & 15) * 4;
            ru[q] = *reinterpret_cast<const float4*>(Uh + (int64_t)p * s.ldA + ri + c4);
            rv[q] = *reinterpret_cast<const float4*>(Vh + (int64_t)p * s.ldA + rj + c4);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = tid + kUpdThreads * q;
            const int p = e >> 4, c4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(&Ut[p][c4]) = ru[q];
            *reinterpret_cast<float4*>(&Vs[p][c4]) = rv[q];
        }
    }
    __syncthreads();
    const int ty = tid >> 4, tx = tid & 15;          // rows 8 ty .., columns 4 tx ..
    float acc[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 4
    for (int p = 0; p < SB; ++p) {
        const float4 u0 = *reinterpret_cast<const float4*>(&Ut[p][ty * 8]);
        const float4 u1 = *reinterpret_cast<const float4*>(&Ut[p][ty * 8 + 4]);
        const float4 v0 = *reinterpret_cast<const float4*>(&Vs[p][tx * 4]);
        const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float v[4] = {v0.x, v0.y, v0.z, v0.w};
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(u[a], v[c], acc[a][c]);
    }
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int r = ri + ty * 8 + a;
        if (r >= t) continue;
        float* row = A + (int64_t)r * s.ldA + rj + tx * 4;
        if (rj + tx * 4 + 4 <= t) {
            float4 o = *reinterpret_cast<float4*>(row);
            o.x = sg * (o.x - acc[a][0]);
            o.y = sg * (o.y - acc[a][1]);
            o.z = sg * (o.z - acc[a][2]);
            o.w = sg * (o.w - acc[a][3]);
            *reinterpret_cast<float4*>(row) = o;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (rj + tx * 4 + c < t) row[c] = sg * (row[c] - acc[a][c]);
        }
    }
}

// Upper triangle <- lower triangle.  grid (blocks * (blocks - 1) / 2 + blocks, H), block 256.
__global__ void __launch_bounds__(256) k_sweep_mirror(float* __restrict__ Am, const int32_t* __restrict__ offsets,
                                                      int64_t ldA, const int32_t* __restrict__ status) {
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

// C[off + i][c] = sum_j Minv[i][j] R[off + j][c] (C_v from the explicit
// inverse).  grid (ceil(max_t / 64), H), block 256: a CTA computes 64 rows x
// D columns, each thread 4 rows x D/16 columns, in 64-column steps of j.
template <int D>
__global__ void __launch_bounds__(256) k_apply_inverse(const float* __restrict__ Minv, const float* __restrict__ R,
                                                       const int32_t* __restrict__ offsets, int64_t ldA,
                                                       float* __restrict__ C, const int32_t* __restrict__ status) {
    const int h = blockIdx.y;
    if (!head_ok(status, h)) return;
    const int off = offsets[h];
    const int t = offsets[h + 1] - off;
    const int i0 = blockIdx.x * SB;
    if (i0 >= t) return;
    __shared__ float Ms[SB][SB + 1];
    __shared__ __align__(16) float Rs[SB][D];
    const float* Mh = Minv + (int64_t)h * ldA * ldA;
    constexpr int CW = D / 16;                 // columns per thread
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    float acc[4][CW];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < CW; ++c) acc[a][c] = 0.f;
    for (int j0 = 0; j0 < t; j0 += SB) {
        __syncthreads();
        for (int e = threadIdx.x; e < SB * SB; e += 256) {
            const int r = e / SB, c = e % SB;
            Ms[r][c] = (i0 + r < t && j0 + c < t) ? Mh[(int64_t)(i0 + r) * ldA + j0 + c] : 0.f;
        }
        for (int e = threadIdx.x; e < SB * D; e += 256) {
            const int r = e / D, c = e % D;
            Rs[r][c] = (j0 + r < t) ? R[((int64_t)off + j0 + r) * D + c] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int p = 0; p < SB; ++p) {
            float m[4], r[CW];
#pragma unroll
            for (int a = 0; a < 4; ++a) m[a] = Ms[ty * 4 + a][p];
#pragma unroll
            for (int c = 0; c < CW; ++c) r[c] = Rs[p][tx + 16 * c];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < CW; ++c) acc[a][c] = fmaf(m[a], r[c], acc[a][c]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = i0 + ty * 4 + a;
        if (i >= t) continue;
#pragma unroll
        for (int c = 0; c < CW; ++c) C[((int64_t)off + i) * D + tx + 16 * c] = acc[a][c];
    }
}

}  // namespace

int sweep_launches(int max_t) { return 2 * ((max_t + SB - 1) / SB) + 1; }

// H^{-1} in place for every head (max_t bounds t_h).  U, V: [H][64][ldA],
// P: [H][64][64] scratch.
cudaError_t launch_sweep_inverse(float* A, const int32_t* offsets, int H, int max_t, int64_t ldA, float* U, float* V,
                                 float* P, int32_t* status, cudaStream_t st) {
    const int nb = (max_t + SB - 1) / SB;
    const int ntri = nb * (nb + 1) / 2;
    for (int k = 0; k < nb; ++k) {
        SweepArgs s{A, U, V, P, offsets, ldA, k * SB, status};
        k_sweep_pivot<<<dim3(nb, H), 256, 0, st>>>(s);
        k_sweep_update<<<dim3(ntri, H), kUpdThreads, 0, st>>>(s);
    }
    k_sweep_mirror<<<dim3(ntri, H), 256, 0, st>>>(A, offsets, ldA, status);
    return cudaGetLastError();
}

// C_v = M^{-1} R from the explicit inverse: C [sum t][d], R [sum t][d].
cudaError_t launch_apply_inverse(int d, const float* Minv, const float* R, const int32_t* offsets, int H, int max_t,
                                 int64_t ldA, float* C, const int32_t* status, cudaStream_t st) {
    dim3 grid((max_t + SB - 1) / SB, H);
    if (d == 128)
        k_apply_inverse<128><<<grid, 256, 0, st>>>(Minv, R, offsets, ldA, C, status);
    else
        k_apply_inverse<64><<<grid, 256, 0, st>>>(Minv, R, offsets, ldA, C, status);
    return cudaGetLastError();
}

cudaError_t launch_symv(const float* Hinv, const float* v, const int32_t* offsets, int H, int max_t, int64_t ldA,
                        float* y, const int32_t* done, int done_stride, const int32_t* status, cudaStream_t st) {
    k_symv<<<dim3((max_t + 7) / 8, H), 256, 0, st>>>(Hinv, v, offsets, ldA, y, done, done_stride, status);
    return cudaGetLastError();
}

}  // namespace kvc
