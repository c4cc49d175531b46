// Explicit inverse of the NNLS matrix H = A'^T A' + mu I ("Fast KV
// Compaction via Attention Matching", section 2, fitting beta by NNLS): the
// block-principal-pivoting NNLS works entirely with H^{-1} (its columns for
// the zero set, the unconstrained solution H^{-1} f and refinement steps), so
// one inverse replaces every triangular solve.
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
//                   computes U_i = A_ik P for its row block i and copies
//                   V_i = A_ki (row block k)
//   k_sweep_update  grid (lower tiles, H): every 64 x 64 tile on or below
//                   the diagonal is updated from U, V and P (64 threads, an
//                   8 x 8 register tile each); on a head's last block the
//                   stored result is negated, so the matrix ends as +H^{-1}
//   k_sweep_mirror  copies the lower triangle into the upper one
//   k_symv          y = H^{-1} v for every head (one warp per row)
// The sweep keeps the symmetric matrix in its lower triangle (row-major,
// leading dimension ldA); an entry above the diagonal is read from its
// mirror image.  The finished inverse is stored in full.
#include "common.cuh"

namespace kvc {

namespace {
constexpr int SB = 64;     // sweep block

struct SweepArgs {
    float* A;                 // [H][ldA][ldA]
    float* U;                 // [H][ldA][64]
    float* V;                 // [H][64][ldA]
    float* P;                 // [H][64][64]
    const int32_t* offsets;
    int64_t ldA;
    int k0;                   // first row of the pivot block
    int32_t* status;
};

// Entry (r, c) of the symmetric matrix kept in its lower triangle; rows and
// columns past t read as the identity.
__device__ __forceinline__ float load_sym(const float* A, int64_t ldA, int r, int c, int t) {
    if (r >= t || c >= t) return (r == c) ? 1.f : 0.f;
    return (r >= c) ? A[(int64_t)r * ldA + c] : A[(int64_t)c * ldA + r];
}

// grid (blocks, H), block 256.
__global__ void __launch_bounds__(256) k_sweep_pivot(SweepArgs s) {
    const int h = blockIdx.y;
    if (!head_ok(s.status, h)) return;
    const int t = s.offsets[h + 1] - s.offsets[h];
    const int k0 = s.k0;
    if (k0 >= t) return;
    const int r0 = blockIdx.x * SB;
    if (r0 >= t) return;
    __shared__ float rowb[2][SB];
    __shared__ float Ps[SB][SB + 1];      // A_ik (rows r0.., columns k0..)
    __shared__ float Pn[SB][SB + 1];      // P
    __shared__ int bad;
    const float* A = s.A + (int64_t)h * s.ldA * s.ldA;
    const int tid = threadIdx.x;
    const int ii = tid >> 2, cq = tid & 3;   // row ii, columns cq + 4m
    float a[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) a[m] = load_sym(A, s.ldA, k0 + ii, k0 + cq + 4 * m, t);
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
    // 64 scalar sweeps of the pivot block; the block stays symmetric, so row
    // p also provides column p
#pragma unroll
    for (int p = 0; p < SB; ++p) {
        float* rb = rowb[p & 1];
        if (ii == p) {
#pragma unroll
            for (int m = 0; m < 16; ++m) rb[cq + 4 * m] = a[m];
        }
        __syncthreads();
        float d = rb[p];
        if (!(d > 0.f) || !isfinite(d)) {
            if (tid == 0) bad = 1;
            d = 1.f;
        }
        const float inv = 1.f / d;
        if (ii != p) {
            // a_ic -= a_ip a_pc / d; column p itself becomes a_ip / d
            const float f = rb[ii] * inv;
#pragma unroll
            for (int m = 0; m < 16; ++m) a[m] = fmaf(-f, rb[cq + 4 * m], a[m]);
            if (cq == (p & 3)) a[p >> 2] = f;
        } else {
            // row p becomes a_pc / d, the pivot -1 / d
#pragma unroll
            for (int m = 0; m < 16; ++m) a[m] *= inv;
            if (cq == (p & 3)) a[p >> 2] = -inv;
        }
    }
    __syncthreads();
    if (bad) {
        if (blockIdx.x == 0 && tid == 0) set_status(s.status, h, KVC_ERR_NOT_SPD);
        return;
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) Pn[ii][cq + 4 * m] = -a[m];
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
    for (int p = 0; p < SB; ++p) {
        const float x = Ps[ii][p];
#pragma unroll
        for (int m = 0; m < 16; ++m) acc[m] = fmaf(x, Pn[p][cq + 4 * m], acc[m]);
    }
    float* Uh = s.U + ((int64_t)h * s.ldA + r0) * SB;
#pragma unroll
    for (int m = 0; m < 16; ++m) Uh[ii * SB + cq + 4 * m] = acc[m];
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

constexpr int kUpdThreads = 64;
constexpr int kUS = SB + 4;      // padded smem row: 16-byte aligned, spreads the transposed stores

// grid (blocks * (blocks + 1) / 2, H), block 64: tile (bi >= bj) of the lower triangle.
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
    const float* Uh = s.U + (int64_t)h * s.ldA * SB;
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
            else if (pj) v = Uh[(int64_t)(ri + r) * SB + c];          // A_ik = U_i
            else v = Uh[(int64_t)(rj + c) * SB + r];                 // A_kj = U_j^T
            A[(int64_t)(ri + r) * s.ldA + rj + c] = sg * v;
        }
        return;
    }
    __shared__ __align__(16) float Ut[SB][kUS];     // Ut[p][r] = U_i[r][p]
    __shared__ __align__(16) float Vs[SB][kUS];     // Vs[p][c] = V[p][rj + c]
    for (int e = tid; e < SB * SB; e += kUpdThreads) {
        const int r = e / SB, p = e % SB;
        Ut[p][r] = Uh[(int64_t)(ri + r) * SB + p];
        const int pp = e / SB, c = e % SB;
        Vs[pp][c] = Vh[(int64_t)pp * s.ldA + rj + c];
    }
    __syncthreads();
    const int ty = tid >> 3, tx = tid & 7;          // rows 8 ty .., columns 8 tx ..
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[a][c] = 0.f;
#pragma unroll 4
    for (int p = 0; p < SB; ++p) {
        const float4 u0 = *reinterpret_cast<const float4*>(&Ut[p][ty * 8]);
        const float4 u1 = *reinterpret_cast<const float4*>(&Ut[p][ty * 8 + 4]);
        const float4 v0 = *reinterpret_cast<const float4*>(&Vs[p][tx * 8]);
        const float4 v1 = *reinterpret_cast<const float4*>(&Vs[p][tx * 8 + 4]);
        const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[a][c] = fmaf(u[a], v[c], acc[a][c]);
    }
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int r = ri + ty * 8 + a;
        if (r >= t) continue;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int col = rj + tx * 8 + c;
            if (col < t) {
                float* p = A + (int64_t)r * s.ldA + col;
                *p = sg * (*p - acc[a][c]);
            }
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

}  // namespace

int sweep_launches(int max_t) { return 2 * ((max_t + SB - 1) / SB) + 1; }

// H^{-1} in place for every head (max_t bounds t_h).  U: [H][ldA][64],
// V: [H][64][ldA], P: [H][64][64] scratch.
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

cudaError_t launch_symv(const float* Hinv, const float* v, const int32_t* offsets, int H, int max_t, int64_t ldA,
                        float* y, const int32_t* done, int done_stride, const int32_t* status, cudaStream_t st) {
    k_symv<<<dim3((max_t + 7) / 8, H), 256, 0, st>>>(Hinv, v, offsets, ldA, y, done, done_stride, status);
    return cudaGetLastError();
}

}  // namespace kvc
