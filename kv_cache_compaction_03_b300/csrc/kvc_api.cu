// extern "C" entry points of libkvc: argument checks, workspace carving and
// the launch sequence of the compaction steps ("Fast KV Compaction via
// Attention Matching", section 2).  Everything is enqueued on the caller's
// stream; nothing here allocates, frees or synchronises.
#include <atomic>
#include <cmath>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"

namespace kvc {
cudaError_t launch_validate(const int32_t*, const int32_t*, int, int, int, int, int, int, int32_t*, HeadScalars*,
                            cudaStream_t);
cudaError_t launch_attn_fwd_simt(int, int, const void*, const void*, const void*, int, int, int, float, float*, float*,
                                 int32_t*, int, const float*, cudaStream_t);
cudaError_t launch_colscore_simt(int, int, const void*, const void*, const float*, int, int, int, float, float*,
                                 const int32_t*, int, const float*, cudaStream_t);
cudaError_t launch_select(const float*, int, int, const int32_t*, int, int, int, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_shift_idx(int32_t*, const int32_t*, int, int, int, int, const int32_t*, cudaStream_t);
cudaError_t launch_gather(int, int, const void*, const void*, bool, int, int, int, const int32_t*, const int32_t*,
                          void*, float*, void*, int64_t, const int32_t*, const float*, int64_t, float*, cudaStream_t);
cudaError_t launch_masslogits_tc(int d, const void* Q, const void* Ck, const float* lse2, const int32_t* offsets,
                                 int H, int n, int max_t, int64_t ldA, float c2, float* L2, void* Ah, void* Al,
                                 float* colpart, int64_t part_stride, double* sqpart, int32_t* status, int qdiv,
                                 long long wait_limit, const float* bk, cudaStream_t st);
cudaError_t launch_colsum_total(const float* part, int ntiles, int64_t stride, const int32_t* offsets, float* b,
                                int H, int max_cols, const int32_t* status, cudaStream_t st);
cudaError_t launch_masslogits(int, int, const void*, const void*, const float*, const int32_t*, int, int, int, int64_t,
                              float, float*, const int32_t*, int, const float*, cudaStream_t);
cudaError_t launch_attend(int, int, const void*, int, const void*, const float*, const float*, const int32_t*, int,
                          float, float*, int32_t*, cudaStream_t);
cudaError_t launch_attend_decode(int, int, const void*, int, const void*, const float*, const float*, const int32_t*,
                                 int, float, float*, int32_t*, cudaStream_t);
int attend_decode_max_queries();
size_t omp_workspace_bytes(int dtype, int H, int n, int T, int max_t);
size_t omp_order_offset(int dtype, int H, int n, int T, int max_t);
int omp_launches(int dtype, int max_t, int nf);
cudaError_t launch_colmean_simt(int dtype, int d, const void* Q, const void* K, const float* lse2, int H, int n, int T,
                                float c2, float* out, const int32_t* status, cudaStream_t st);
int tam_max_segments();
cudaError_t launch_tam_plan(const float* alpha, int H, int T, const int32_t* bounds, int S, double c,
                            const int32_t* offsets, uint8_t* pivot, int32_t* seg_bud, int32_t* seg_keep,
                            int32_t* seg_off, int32_t* status, cudaStream_t st);
cudaError_t launch_tam_kept(const uint8_t* pivot, int H, int T, int max_t, const int32_t* idx,
                            const int32_t* offsets, uint8_t* kp, int32_t* plist, int32_t* npk,
                            const int32_t* status, cudaStream_t st);
cudaError_t launch_tam_fix_g(float* G, int64_t ldA, float* f, const uint8_t* kp, const int32_t* plist,
                             const int32_t* npk, const int32_t* offsets, int H, int max_t, const int32_t* status,
                             cudaStream_t st);
cudaError_t launch_tam_fix_m(float* M, int64_t ldA, float* R, const float* Vsel, int d, const uint8_t* kp,
                             const int32_t* plist, const int32_t* npk, const int32_t* offsets, int H, int max_t,
                             const int32_t* status, cudaStream_t st);
cudaError_t launch_select_seg(const float* score, int H, int T, const int32_t* offsets, const int32_t* bounds,
                              int nseg, const uint8_t* pivot, const int32_t* seg_keep, const int32_t* seg_off,
                              int32_t* idx_out, int32_t* status, cudaStream_t st);
cudaError_t launch_omp_select(int dtype, int d, const void* Q, const void* K, const float* lse2, float c2, int H,
                              int n, int T, int max_t, const int32_t* offsets, int keep_first, int keep_last,
                              void* ws, int32_t* idx_out, int32_t* status, long long wait_limit, cudaStream_t st);
cudaError_t launch_gram_sym_tc(const void* Ah, const void* Al, const int32_t* offsets, int H, int n, int max_t,
                               int64_t ld, float* C, int64_t ldc, int32_t* status, long long wait_limit,
                               cudaStream_t st);
cudaError_t launch_gram_rect_tc(int d, const void* Ah, const void* Al, const void* Bh, const void* Bl,
                                const int32_t* offsets, int H, int n, int max_t, int64_t ld, float* C,
                                int32_t* status, long long wait_limit, cudaStream_t st);
cudaError_t launch_split_hilo(bool exp_mode, const float* X, int H, int rows, int64_t ld, const int32_t* offsets,
                              int cols, int max_cols, void* Xh, void* Xl, float* part, float* colsum, double* sqpart,
                              const int32_t* status, cudaStream_t st);
cudaError_t launch_ridge_g(float*, const float*, const int32_t*, int, int64_t, float, const double*, int64_t, float*,
                           HeadScalars*, int32_t*,
                           cudaStream_t);
cudaError_t launch_ridge_m(int, float*, float*, const float*, const int32_t*, int, int64_t, float, HeadScalars*,
                           int32_t*, cudaStream_t);
cudaError_t launch_xsoftmax(const float*, const float*, const int32_t*, int, int, int64_t, void*, void*,
                            const int32_t*, cudaStream_t);
cudaError_t launch_chol(float*, const int32_t*, int, int, int64_t, float*, int32_t*, cudaStream_t);
int chol_launches(int max_t);
cudaError_t launch_cholsolve(int, const float*, const float*, const float*, const int32_t*, int, int64_t, float*,
                             const int32_t*,
                             cudaStream_t);
cudaError_t launch_nnls_all(const float* Hinv, const float* f, const int32_t* offsets, int H, int n, int max_t,
                            int64_t ldA, const float* L2, float* x, float* x0, int8_t* zflag, int32_t* zlist,
                            int32_t* nz, float* S, int32_t* piv, float* r, float* d0, HeadScalars* hs,
                            int zmax, int max_iter, int refine_iters, void* rpart_ws, const uint8_t* fixed,
                            int32_t* status, cudaStream_t st, int* launches);
cudaError_t launch_sweep_inverse(float* A, const int32_t* offsets, int H, int max_t, int64_t ldA, float* U,
                                 void* split, float* P, int32_t* status, long long wait_limit, cudaStream_t st);
int sweep_launches(int max_t);
size_t apply_inverse_tc_scratch(int H, int64_t ldA, int d);
size_t refine_part_bytes(int H, int n, int max_t, int64_t ldA);
cudaError_t launch_apply_inverse_tc(int d, const float* Minv, const float* R, const int32_t* offsets, int H,
                                    int max_t, int64_t ldA, void* split, float* C, int32_t* status,
                                    long long wait_limit, cudaStream_t st);
cudaError_t launch_attn_fwd_tc(int d, const void* Q, const void* K, const void* V16, const int32_t* vexp, int H,
                               int n, int T, float c2, float* O, float* lse2, int32_t* status, int qdiv,
                               long long wait_limit, const float* bias2, cudaStream_t st);
cudaError_t launch_v_to_f16(const void* V, bool v_f32, int H, int64_t per_head, uint32_t* vmax, void* V16,
                            int32_t* vexp, int32_t* status, cudaStream_t st);
cudaError_t launch_colscore_tc(int d, const void* Q, const void* K, const float* lse2, int H, int n, int T,
                               float c2, float* score, int32_t* status, int qdiv, long long wait_limit,
                               const float* bias2, cudaStream_t st);
bool tc_maps_available();
cudaError_t launch_beta_out(float*, const int32_t*, int, int, float*, const int32_t*, const float*, const int32_t*, int,
                            cudaStream_t);
cudaError_t launch_bias_log2(const float* bias, int H, int T, float* bias2, int32_t* status, cudaStream_t st);

constexpr int kMaxT = 4096;     // largest budget the per-head solvers support
constexpr int kMaxHeads = 65535;  // heads index grid.y
constexpr int kMaxStages = 32;

// Optional per-stage CUDA events (KVC_FLAG_STAGE_TIMING), recorded on the
// caller's stream between stages; read back by kvc_stage_times.  One record
// per host thread (the last timed call).
struct StageLog {
    bool created = false;
    int n = 0;
    int launches = 0;
    const char* names[kMaxStages];
    int counts[kMaxStages];
    cudaEvent_t ev[kMaxStages + 1];
};
static thread_local StageLog g_log;
static thread_local int g_last_launches = 0;

struct StageClock {
    bool on;
    cudaStream_t st;
    int launches = 0;
    StageClock(bool enable, cudaStream_t s) : on(enable), st(s) {
        if (!on) return;
        if (!g_log.created) {
            for (int i = 0; i <= kMaxStages; ++i) cudaEventCreate(&g_log.ev[i]);
            g_log.created = true;
        }
        g_log.n = 0;
        cudaEventRecord(g_log.ev[0], st);
    }
    void stage(const char* name, int count) {
        launches += count;
        if (!on || g_log.n >= kMaxStages) return;
        g_log.names[g_log.n] = name;
        g_log.counts[g_log.n] = count;
        cudaEventRecord(g_log.ev[g_log.n + 1], st);
        ++g_log.n;
    }
    void finish() {
        g_last_launches = launches;
        if (on) g_log.launches = launches;
    }
};

// One stage of the launch sequence: an NVTX range named after the stage
// around its launches (for timeline tools), the launch error check, and the
// optional stage event.
#define KVC_STAGE(name, count, call)                   \
    do {                                               \
        nvtxRangePushA(name);                          \
        cudaError_t _e = (call);                       \
        nvtxRangePop();                                \
        if (_e != cudaSuccess) return KVC_ERR_CUDA;    \
        clk.stage(name, count);                        \
    } while (0)

struct Layout {
    int64_t ldA;
    int zmax;
    size_t O, lse2, score, L2, Ah, Al, Oh, Ol, bpart, sqpart, Vsel, Ckw, G, dinv, swV, swP, rpart, b, f, x, x0, d0, r, R, zflag, zlist, nz, piv, S, hs, omp;
    size_t msplit;                                 // bf16 terms of M^{-1} and R for the C_v product
    size_t V16, vexp, vmax;                        // the values in fp16 for the attention pass (bf16 input)
    size_t bias2, bk;                              // key biases (log2 units): padded per head, and of the kept keys
    size_t tO, tlse, talpha, tkeep, toff, tkp, tpl, tnp;     // thought-aware planning (n_win > 0)
    size_t total;
};

static size_t carve(size_t& cur, size_t bytes) {
    size_t at = (size_t)round_up((int64_t)cur, 256);
    cur = at + bytes;
    return at;
}

// Window queries and segments of the thought-aware planner; none otherwise.
// `biased`: the keys carry input biases and the values are fp32 (a compacted
// cache, compacted again).
struct TamShape {
    int n_win = 0, nseg = 0;
    bool biased = false;
};

// Inputs and outputs of the thought-aware planner.
struct TamInputs {
    const void* Q_win;          // [H][n_win][d] dtype
    int n_win;
    const int32_t* bounds;      // device [nseg + 1]
    int nseg;
    double c;
    int32_t* seg_budgets;       // device [H][nseg]
    uint8_t* pivots;            // device [H][T]
};

static Layout make_layout(const kvc_problem& p, const kvc_params& prm, TamShape ts = TamShape{}) {
    Layout L{};
    const size_t H = p.H, n = p.n, T = p.T, d = p.d, mt = p.max_t;
    L.ldA = round_up(p.max_t, 64);
    L.zmax = std::max(1, std::min(prm.nnls_max_zero, p.max_t));
    const size_t ldA = (size_t)L.ldA, zm = (size_t)L.zmax;
    size_t c = 0;
    L.O = carve(c, H * n * d * 4);
    L.lse2 = carve(c, H * n * 4);
    L.score = carve(c, H * T * 4);
    L.L2 = carve(c, H * n * ldA * 4);
    L.Ah = carve(c, H * n * ldA * 2);         // A' (then X) as bf16 hi / lo terms
    L.Al = carve(c, H * n * ldA * 2);
    L.Oh = carve(c, H * n * d * 2);           // O as bf16 hi / lo terms
    L.Ol = carve(c, H * n * d * 2);
    L.bpart = carve(c, ((n + 127) / 128) * H * mt * 4);   // column sums of A' per 128-query tile
    L.sqpart = carve(c, ((n + 127) / 128) * (ldA / 64) * H * 8);  // sums of A'^2 per CTA of the mass pass
    L.Vsel = carve(c, H * mt * d * 4);
    L.Ckw = carve(c, H * ldA * d * 2);
    L.G = carve(c, H * ldA * ldA * 4);
    L.dinv = carve(c, H * ldA * 64 * 4);      // Cholesky diagonal inverses; sweep U panel
    L.swV = carve(c, 6 * H * 64 * ldA * 2);   // sweep: U^T and V as three bf16 terms each
    L.swP = carve(c, 4 * H * 64 * 64 * 4);    // sweep: pivot block inverse, next block inputs, its inverse
    L.b = carve(c, H * mt * 4);
    L.f = carve(c, H * mt * 4);
    L.x = carve(c, H * mt * 4);
    L.x0 = carve(c, H * mt * 4);
    L.d0 = carve(c, H * mt * 4);
    L.r = carve(c, H * mt * 4);
    L.rpart = carve(c, refine_part_bytes(p.H, p.n, p.max_t, L.ldA));   // residual partials per row block
    L.R = carve(c, H * mt * d * 4);
    L.zflag = carve(c, H * mt);
    L.zlist = carve(c, H * zm * 4);
    L.nz = carve(c, H * 4);
    L.piv = carve(c, H * 16);
    L.S = carve(c, H * zm * zm * 4);
    L.hs = carve(c, H * sizeof(HeadScalars));
    // the terms of M^{-1} and R are needed only after the last reader of the
    // mass logits and the A' / X terms: they share that span when it is large enough
    {
        const size_t need = apply_inverse_tc_scratch((int)H, (int64_t)ldA, (int)d);
        const size_t span = L.Al + H * n * ldA * 2 - L.L2;
        L.msplit = need <= span ? L.L2 : carve(c, need);
    }
    // the fp16 values are read by the attention passes only, before the mass
    // logits are written: they share that span when it is large enough
    if (p.dtype == KVC_DTYPE_BF16) {
        const size_t need = H * T * d * 2;
        const size_t span = L.Al + H * n * ldA * 2 - L.L2;
        L.V16 = need <= span ? L.L2 : carve(c, need);
        L.vexp = carve(c, H * 4);
        L.vmax = carve(c, H * 4);
    }
    if (ts.biased) {
        L.bias2 = carve(c, H * (size_t)round_up(p.T, 256) * 4);
        L.bk = carve(c, H * mt * 4);
    }
    // key selection by matching pursuit: the relative mass of every key and the pursuit's state
    L.omp = (prm.flags & KVC_FLAG_SELECT_OMP) ? carve(c, omp_workspace_bytes(p.dtype, p.H, p.n, p.T, p.max_t)) : 0;
    if (ts.n_win > 0) {
        L.tO = carve(c, H * (size_t)ts.n_win * d * 4);
        L.tlse = carve(c, H * (size_t)ts.n_win * 4);
        L.talpha = carve(c, H * T * 4);
        L.tkeep = carve(c, H * (size_t)ts.nseg * 4);
        L.toff = carve(c, H * (size_t)ts.nseg * 4);
        L.tkp = carve(c, H * mt);
        L.tpl = carve(c, H * mt * 4);
        L.tnp = carve(c, H * 4);
    }
    L.total = (size_t)round_up((int64_t)c, 256);
    return L;
}

static bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

static kvc_status check_problem(const kvc_problem* p) {
    if (!p) return KVC_ERR_INVALID_ARG;
    if (p->H < 1 || p->H > kMaxHeads || p->n < 1 || p->T < 1) return KVC_ERR_INVALID_ARG;
    if (p->d != 64 && p->d != 128) return KVC_ERR_INVALID_ARG;
    if (p->dtype != KVC_DTYPE_BF16 && p->dtype != KVC_DTYPE_F32) return KVC_ERR_INVALID_ARG;
    if (p->max_t < 1 || p->max_t > p->T || p->max_t > kMaxT) return KVC_ERR_INVALID_ARG;
    return KVC_OK;
}

// T_total: the length of the whole cache the forced ranges count positions of.
static kvc_status check_params(const kvc_params& q, int64_t T_total) {
    if (!(q.scale >= 0.f) || !std::isfinite(q.scale)) return KVC_ERR_INVALID_ARG;
    if (!(q.eps_mu > 0.f) || !(q.eps_lambda > 0.f) || !std::isfinite(q.eps_mu) || !std::isfinite(q.eps_lambda))
        return KVC_ERR_INVALID_ARG;
    if (q.nnls_max_iter < 1 || q.nnls_max_zero < 1 || q.refine_iters < 0 || q.wait_timeout_us < 1)
        return KVC_ERR_INVALID_ARG;
    if (q.keep_first < 0 || q.keep_last < 0 ||
        (q.flags & ~(KVC_FLAG_STAGE_TIMING | KVC_FLAG_CHOLESKY_CV | KVC_FLAG_SELECT_OMP)) != 0)
        return KVC_ERR_INVALID_ARG;
    if ((int64_t)q.keep_first + q.keep_last > T_total) return KVC_ERR_INVALID_ARG;
    return KVC_OK;
}

// The caller's wait limit in SM clock cycles of the current device (its
// peak clock: at a lower clock the limit lasts longer).  The clock rate is
// queried once per device and kept (the query is not free on every call).
static long long wait_cycles(uint32_t us) {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> khz_of[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
    int khz = dev >= 0 ? khz_of[dev].load(std::memory_order_relaxed) : 0;
    if (khz <= 0) {
        if (dev < 0 || cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0)
            khz = 2032000;
        if (dev >= 0) khz_of[dev].store(khz, std::memory_order_relaxed);
    }
    return (long long)us * khz / 1000;
}

static float log2_scale(const kvc_problem& p, float scale) {
    const double s = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)p.d);
    return (float)(s * 1.4426950408889634);
}

}  // namespace kvc

using namespace kvc;

#define KVC_TRY(call)                                  \
    do {                                               \
        cudaError_t _e = (call);                       \
        if (_e != cudaSuccess) return KVC_ERR_CUDA;    \
    } while (0)

extern "C" {

kvc_status kvc_default_params(kvc_params* prm) {
    if (!prm) return KVC_ERR_INVALID_ARG;
    std::memset(prm, 0, sizeof(*prm));
    prm->scale = 0.f;
    prm->eps_mu = 1e-2f;
    prm->eps_lambda = 1e-2f;
    prm->nnls_max_iter = 32;
    prm->nnls_max_zero = 512;
    prm->refine_iters = 1;
    prm->wait_timeout_us = 1000000u;
    return KVC_OK;
}

kvc_status kvc_workspace_size(const kvc_problem* p, const kvc_params* prm, size_t* bytes) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK || !bytes) return KVC_ERR_INVALID_ARG;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if ((s = check_params(q, p->T)) != KVC_OK) return s;
    *bytes = make_layout(*p, q).total;
    return KVC_OK;
}

kvc_status kvc_workspace_offset(const kvc_problem* p, const kvc_params* prm, int32_t item, size_t* offset) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK || !offset) return KVC_ERR_INVALID_ARG;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    // the layout does not depend on the forced ranges, which may count the
    // positions of a longer cache (the per-chunk problem of a chunked call)
    if ((s = check_params(q, INT64_MAX)) != KVC_OK) return s;
    const Layout L = make_layout(*p, q);
    switch (item) {
        case 0: *offset = L.O; break;
        case 1: *offset = L.lse2; break;
        case 2: *offset = L.score; break;
        case 3: *offset = L.x; break;
        case 4: *offset = L.hs; break;
        case 5:
            if (!(q.flags & KVC_FLAG_SELECT_OMP)) return KVC_ERR_INVALID_ARG;
            *offset = L.omp + omp_order_offset(p->dtype, p->H, p->n, p->T, p->max_t);
            break;
        case 6: *offset = L.L2; break;
        default: return KVC_ERR_INVALID_ARG;
    }
    return KVC_OK;
}

}  // extern "C"

namespace kvc {

// The launch sequence of one compaction over the heads of *p.  `chunks` > 1
// when each head of *p is one of `chunks` contiguous chunks of a longer cache
// (heads head * chunks + c share the reference queries of `head`).  With
// bias_in the keys carry input biases ([H][T] fp32) and V is fp32 (a
// compacted cache compacted again).  The arguments have been checked by the
// caller.
static kvc_status enqueue_compact(const kvc_problem* p, const kvc_params& q, int chunks, const void* Q_ref,
                                  const void* K, const void* V, const int32_t* budgets, const int32_t* offsets,
                                  int32_t* idx_out, void* C_k, float* beta, float* C_v, int32_t* head_status,
                                  void* workspace, size_t workspace_bytes, cudaStream_t st,
                                  const TamInputs* tam = nullptr, const float* bias_in = nullptr) {
    const Layout L = make_layout(*p, q, tam ? TamShape{tam->n_win, tam->nseg} : TamShape{0, 0, bias_in != nullptr});
    if (!workspace || workspace_bytes < L.total) return KVC_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return KVC_ERR_ALIGN;

    char* ws = static_cast<char*>(workspace);
    float* O = (float*)(ws + L.O);
    float* lse2 = (float*)(ws + L.lse2);
    float* score = (float*)(ws + L.score);
    float* L2 = (float*)(ws + L.L2);
    float* Vsel = (float*)(ws + L.Vsel);
    float* G = (float*)(ws + L.G);
    float* dinv = (float*)(ws + L.dinv);
    float* b = (float*)(ws + L.b);
    float* f = (float*)(ws + L.f);
    float* x = (float*)(ws + L.x);
    float* r = (float*)(ws + L.r);
    float* R = (float*)(ws + L.R);
    int8_t* zflag = (int8_t*)(ws + L.zflag);
    int32_t* zlist = (int32_t*)(ws + L.zlist);
    int32_t* nzv = (int32_t*)(ws + L.nz);
    int32_t* piv = (int32_t*)(ws + L.piv);
    float* x0 = (float*)(ws + L.x0);
    float* d0 = (float*)(ws + L.d0);
    float* S = (float*)(ws + L.S);
    HeadScalars* hs = (HeadScalars*)(ws + L.hs);

    const int H = p->H, n = p->n, T = p->T, d = p->d, dt = p->dtype, mt = p->max_t;
    const int qdiv = chunks;
    const float c2 = log2_scale(*p, q.scale);
    const long long wl = wait_cycles(q.wait_timeout_us);

    StageClock clk(q.flags & KVC_FLAG_STAGE_TIMING, st);
    KVC_STAGE("validate", 1,
              launch_validate(budgets, offsets, H, T, mt, chunks, q.keep_first, q.keep_last, head_status, hs, st));
    const bool biased = bias_in != nullptr;
    float* bias2 = biased ? (float*)(ws + L.bias2) : nullptr;
    float* bk = biased ? (float*)(ws + L.bk) : nullptr;
    if (biased) KVC_STAGE("bias", 1, launch_bias_log2(bias_in, H, T, bias2, head_status, st));
    // bf16 inputs take the tensor-core passes (tcgen05/TMEM/TMA); fp32 inputs
    // the FFMA passes (a tf32 contraction would not keep fp32 accuracy).
    const bool omp = (q.flags & KVC_FLAG_SELECT_OMP) != 0;
    uint8_t* kp = tam ? (uint8_t*)(ws + L.tkp) : nullptr;      // kept rows that are pivots
    const int32_t* vexp = dt == KVC_DTYPE_BF16 ? (const int32_t*)(ws + L.vexp) : nullptr;
    if (dt == KVC_DTYPE_BF16) {
        KVC_STAGE("v_f16", 2,
                  launch_v_to_f16(V, biased, H, (int64_t)T * d, (uint32_t*)(ws + L.vmax), ws + L.V16,
                                  (int32_t*)(ws + L.vexp), head_status, st));
        KVC_STAGE("attn_fwd", 1,
                  launch_attn_fwd_tc(d, Q_ref, K, ws + L.V16, vexp, H, n, T, c2, O, lse2, head_status, qdiv, wl, bias2,
                                     st));
        if (!omp)
            KVC_STAGE("colscore", 1,
                      launch_colscore_tc(d, Q_ref, K, lse2, H, n, T, c2, score, head_status, qdiv, wl, bias2, st));
    } else {
        KVC_STAGE("attn_fwd", 1,
                  launch_attn_fwd_simt(dt, d, Q_ref, K, V, H, n, T, c2, O, lse2, head_status, qdiv, bias2, st));
        if (!omp)
            KVC_STAGE("colscore", 1,
                      launch_colscore_simt(dt, d, Q_ref, K, lse2, H, n, T, c2, score, head_status, qdiv, bias2, st));
    }
    if (tam) {
        float* Ow = (float*)(ws + L.tO);
        float* lw = (float*)(ws + L.tlse);
        float* alpha = (float*)(ws + L.talpha);
        int32_t* skeep = (int32_t*)(ws + L.tkeep);
        int32_t* soff = (int32_t*)(ws + L.toff);
        // (the tensor-core pass tiles queries by 128; shorter windows take the FFMA pass)
        if (dt == KVC_DTYPE_BF16 && tam->n_win >= 128)
            KVC_STAGE("win_attn", 1,
                      launch_attn_fwd_tc(d, tam->Q_win, K, ws + L.V16, vexp, H, tam->n_win, T, c2, Ow, lw, head_status,
                                         1, wl, nullptr, st));
        else
            KVC_STAGE("win_attn", 1,
                      launch_attn_fwd_simt(dt, d, tam->Q_win, K, V, H, tam->n_win, T, c2, Ow, lw, head_status, 1,
                                           nullptr, st));
        KVC_STAGE("win_alpha", 1,
                  launch_colmean_simt(dt, d, tam->Q_win, K, lw, H, tam->n_win, T, c2, alpha, head_status, st));
        KVC_STAGE("tam_plan", 1,
                  launch_tam_plan(alpha, H, T, tam->bounds, tam->nseg, tam->c, offsets, tam->pivots,
                                  tam->seg_budgets, skeep, soff, head_status, st));
        KVC_STAGE("select", 1,
                  launch_select_seg(score, H, T, offsets, tam->bounds, tam->nseg, tam->pivots, skeep, soff, idx_out,
                                    head_status, st));
    } else if (omp)
        KVC_STAGE("omp", omp_launches(dt, mt, (int)std::min<int64_t>(T, (int64_t)q.keep_first + q.keep_last)),
                  launch_omp_select(dt, d, Q_ref, K, lse2, c2, H, n, T, mt, offsets, q.keep_first, q.keep_last,
                                    ws + L.omp, idx_out, head_status, wl, st));
    else
        KVC_STAGE("select", 1,
                  launch_select(score, H, T, offsets, chunks, q.keep_first, q.keep_last, idx_out, head_status, st));
    void* Ckw = ws + L.Ckw;
    const bool tc = dt == KVC_DTYPE_BF16;
    KVC_STAGE("gather", 1,
              launch_gather(dt, d, K, V, biased, H, T, mt, offsets, idx_out, C_k, Vsel, tc ? Ckw : nullptr, L.ldA,
                            head_status, bias2, round_up(T, 256), bk, st));
    if (chunks > 1)
        KVC_STAGE("shift_idx", 1, launch_shift_idx(idx_out, offsets, H, T, mt, chunks, head_status, st));
    int32_t* plist = tam ? (int32_t*)(ws + L.tpl) : nullptr;   // kept pivot rows, per head
    int32_t* npk = tam ? (int32_t*)(ws + L.tnp) : nullptr;
    if (tam)
        KVC_STAGE("tam_kept", 1,
                  launch_tam_kept(tam->pivots, H, T, mt, idx_out, offsets, kp, plist, npk, head_status, st));
    if (tc) {
        // the kept keys' per-head copy has ldA rows per head; the map sees H * ldA rows
        // the log-masses, A' as bf16 hi / lo terms and the column-sum partials of b in one pass
        KVC_STAGE("masslogits", 1,
                  launch_masslogits_tc(d, Q_ref, Ckw, lse2, offsets, H, n, mt, L.ldA, c2, L2, ws + L.Ah, ws + L.Al,
                                       (float*)(ws + L.bpart), (int64_t)H * mt, (double*)(ws + L.sqpart), head_status,
                                       qdiv, wl, bk, st));
        KVC_STAGE("colsum", 1,
                  launch_colsum_total((float*)(ws + L.bpart), (n + 127) / 128, (int64_t)H * mt, offsets, b, H, mt,
                                      head_status, st));
    } else {
        KVC_STAGE("masslogits", 1,
                  launch_masslogits(dt, d, Q_ref, C_k, lse2, offsets, H, n, mt, L.ldA, c2, L2, head_status, qdiv,
                                    bk, st));
        KVC_STAGE("split_a", 2,
                  launch_split_hilo(true, L2, H, n, L.ldA, offsets, 0, mt, ws + L.Ah, ws + L.Al,
                                    (float*)(ws + L.bpart), b, (double*)(ws + L.sqpart), head_status, st));
    }
    KVC_STAGE("gram_a", 1,
              launch_gram_sym_tc(ws + L.Ah, ws + L.Al, offsets, H, n, mt, L.ldA, G, L.ldA, head_status, wl, st));
    // mu from the exact squares of A' (parts per CTA of the pass that formed A')
    const int64_t sq_count = (int64_t)((n + 127) / 128) * (tc ? (mt + 127) / 128 : L.ldA / 64);
    KVC_STAGE("ridge_g", 1,
              launch_ridge_g(G, b, offsets, H, L.ldA, q.eps_mu, (const double*)(ws + L.sqpart), sq_count, f, hs,
                             head_status, st));
    if (tam)
        KVC_STAGE("tam_fix_g", 2, launch_tam_fix_g(G, L.ldA, f, kp, plist, npk, offsets, H, mt, head_status, st));
    KVC_STAGE("inv_h", sweep_launches(mt),
              launch_sweep_inverse(G, offsets, H, mt, L.ldA, dinv, ws + L.swV, (float*)(ws + L.swP),
                                   head_status, wl, st));
    int nnls_launches = 0;
    KVC_STAGE("nnls", nnls_launches,
              launch_nnls_all(G, f, offsets, H, n, mt, L.ldA, L2, x, x0, zflag, zlist, nzv, S, piv, r, d0, hs,
                              L.zmax, q.nnls_max_iter, q.refine_iters, ws + L.rpart, kp, head_status, st,
                              &nnls_launches));
    KVC_STAGE("beta", 1, launch_beta_out(x, offsets, H, mt, beta, head_status, bias_in, idx_out, T, st));
    KVC_STAGE("xsoftmax", 1,
              launch_xsoftmax(L2, x, offsets, H, n, L.ldA, ws + L.Ah, ws + L.Al, head_status, st));
    KVC_STAGE("gram_x", 1,
              launch_gram_sym_tc(ws + L.Ah, ws + L.Al, offsets, H, n, mt, L.ldA, G, L.ldA, head_status, wl, st));
    KVC_STAGE("split_o", 1,
              launch_split_hilo(false, O, H, n, d, nullptr, d, d, ws + L.Oh, ws + L.Ol, nullptr, nullptr, nullptr,
                                head_status, st));
    KVC_STAGE("xto", 1,
              launch_gram_rect_tc(d, ws + L.Ah, ws + L.Al, ws + L.Oh, ws + L.Ol, offsets, H, n, mt, L.ldA, R,
                                  head_status, wl, st));
    KVC_STAGE("ridge_m", 2, launch_ridge_m(d, G, R, Vsel, offsets, H, L.ldA, q.eps_lambda, hs, head_status, st));
    if (tam)
        KVC_STAGE("tam_fix_m", 2,
                  launch_tam_fix_m(G, L.ldA, R, Vsel, d, kp, plist, npk, offsets, H, mt, head_status, st));
    if (q.flags & KVC_FLAG_CHOLESKY_CV) {
        KVC_STAGE("chol_m", chol_launches(mt), launch_chol(G, offsets, H, mt, L.ldA, dinv, head_status, st));
        KVC_STAGE("cholsolve", 1, launch_cholsolve(d, G, dinv, R, offsets, H, L.ldA, C_v, head_status, st));
    } else {
        KVC_STAGE("inv_m", sweep_launches(mt),
                  launch_sweep_inverse(G, offsets, H, mt, L.ldA, dinv, ws + L.swV, (float*)(ws + L.swP),
                                       head_status, wl, st));
        KVC_STAGE("apply_minv", 3,
                  launch_apply_inverse_tc(d, G, R, offsets, H, mt, L.ldA, ws + L.msplit, C_v, head_status, wl, st));
    }
    clk.finish();
    return KVC_OK;
}

// Whole-cache problem *p split into `chunks` chunks: the per-chunk problem.
static kvc_status chunk_problem(const kvc_problem* p, int32_t chunks, kvc_problem* pc) {
    if (!p || chunks < 1 || p->T < 1 || p->T % chunks != 0) return KVC_ERR_INVALID_ARG;
    if ((int64_t)p->H * chunks > kMaxHeads) return KVC_ERR_INVALID_ARG;
    *pc = *p;
    pc->H = p->H * chunks;
    pc->T = p->T / chunks;
    return check_problem(pc);
}

static kvc_status check_buffers(const void* Q_ref, const void* K, const void* V, const int32_t* budgets,
                                const int32_t* offsets, const int32_t* idx_out, const void* C_k, const float* beta,
                                const float* C_v, const int32_t* head_status) {
    if (!Q_ref || !K || !V || !budgets || !offsets || !idx_out || !C_k || !beta || !C_v || !head_status)
        return KVC_ERR_INVALID_ARG;
    if (!aligned(Q_ref, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(C_k, 16) || !aligned(C_v, 16) ||
        !aligned(beta, 4) || !aligned(idx_out, 4) || !aligned(budgets, 4) || !aligned(offsets, 4) ||
        !aligned(head_status, 4))
        return KVC_ERR_ALIGN;
    return KVC_OK;
}

}  // namespace kvc

extern "C" {

kvc_status kvc_compact(const kvc_problem* p, const kvc_params* prm, const void* Q_ref, const void* K, const void* V,
                       const int32_t* budgets, const int32_t* offsets, int32_t* idx_out, void* C_k, float* beta,
                       float* C_v, int32_t* head_status, void* workspace, size_t workspace_bytes,
                       kvc_stream_t stream) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK) return s;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if ((s = check_params(q, p->T)) != KVC_OK) return s;
    if ((s = check_buffers(Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status)) != KVC_OK) return s;
    return enqueue_compact(p, q, 1, Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status, workspace,
                           workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

static kvc_status check_tam(const kvc_problem* p, const kvc_params& q, const void* Q_win, int32_t n_win,
                            const int32_t* bounds, int32_t nseg, float c) {
    if (!Q_win || !bounds || n_win < 1 || nseg < 1 || nseg > tam_max_segments() || nseg > p->T) return KVC_ERR_INVALID_ARG;
    if (!(c > 0.f) || !std::isfinite(c)) return KVC_ERR_INVALID_ARG;
    if (q.keep_first != 0 || q.keep_last != 0 || (q.flags & KVC_FLAG_SELECT_OMP)) return KVC_ERR_INVALID_ARG;
    if (!aligned(Q_win, 16) || !aligned(bounds, 4)) return KVC_ERR_ALIGN;
    return KVC_OK;
}

kvc_status kvc_workspace_size_tam(const kvc_problem* p, const kvc_params* prm, int32_t n_win, int32_t nseg,
                                  size_t* bytes) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK || !bytes || n_win < 1 || nseg < 1 || nseg > tam_max_segments()) return KVC_ERR_INVALID_ARG;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if ((s = check_params(q, p->T)) != KVC_OK) return s;
    *bytes = make_layout(*p, q, TamShape{n_win, nseg}).total;
    return KVC_OK;
}

kvc_status kvc_compact_tam(const kvc_problem* p, const kvc_params* prm, const void* Q_ref, const void* K,
                           const void* V, const void* Q_win, int32_t n_win, const int32_t* seg_bounds, int32_t nseg,
                           float pivot_c, const int32_t* budgets, const int32_t* offsets, int32_t* idx_out, void* C_k,
                           float* beta, float* C_v, int32_t* head_status, int32_t* seg_budgets_out,
                           uint8_t* pivots_out, void* workspace, size_t workspace_bytes, kvc_stream_t stream) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK) return s;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if ((s = check_params(q, p->T)) != KVC_OK) return s;
    if ((s = check_tam(p, q, Q_win, n_win, seg_bounds, nseg, pivot_c)) != KVC_OK) return s;
    if (!seg_budgets_out || !pivots_out) return KVC_ERR_INVALID_ARG;
    if (!aligned(seg_budgets_out, 4)) return KVC_ERR_ALIGN;
    if ((s = check_buffers(Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status)) != KVC_OK) return s;
    const TamInputs tam{Q_win, n_win, seg_bounds, nseg, (double)pivot_c, seg_budgets_out, pivots_out};
    return enqueue_compact(p, q, 1, Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status, workspace,
                           workspace_bytes, reinterpret_cast<cudaStream_t>(stream), &tam);
}

kvc_status kvc_workspace_size_biased(const kvc_problem* p, const kvc_params* prm, size_t* bytes) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK || !bytes) return KVC_ERR_INVALID_ARG;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if ((s = check_params(q, p->T)) != KVC_OK) return s;
    *bytes = make_layout(*p, q, TamShape{0, 0, true}).total;
    return KVC_OK;
}

kvc_status kvc_compact_biased(const kvc_problem* p, const kvc_params* prm, const void* Q_ref, const void* K,
                              const float* bias, const float* V, const int32_t* budgets, const int32_t* offsets,
                              int32_t* idx_out, void* C_k, float* beta, float* C_v, int32_t* head_status,
                              void* workspace, size_t workspace_bytes, kvc_stream_t stream) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK) return s;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if ((s = check_params(q, p->T)) != KVC_OK) return s;
    if (q.flags & KVC_FLAG_SELECT_OMP) return KVC_ERR_INVALID_ARG;
    if (!bias) return KVC_ERR_INVALID_ARG;
    if (!aligned(bias, 4)) return KVC_ERR_ALIGN;
    if ((s = check_buffers(Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status)) != KVC_OK) return s;
    return enqueue_compact(p, q, 1, Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status, workspace,
                           workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr, bias);
}

kvc_status kvc_workspace_size_chunked(const kvc_problem* p, const kvc_params* prm, int32_t chunks, size_t* bytes) {
    kvc_problem pc;
    const kvc_status s = chunk_problem(p, chunks, &pc);
    if (s != KVC_OK || !bytes) return KVC_ERR_INVALID_ARG;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if (check_params(q, p->T) != KVC_OK) return KVC_ERR_INVALID_ARG;
    *bytes = make_layout(pc, q).total;
    return KVC_OK;
}

kvc_status kvc_compact_chunked(const kvc_problem* p, const kvc_params* prm, int32_t chunks, const void* Q_ref,
                               const void* K, const void* V, const int32_t* budgets, const int32_t* offsets,
                               int32_t* idx_out, void* C_k, float* beta, float* C_v, int32_t* head_status,
                               void* workspace, size_t workspace_bytes, kvc_stream_t stream) {
    kvc_status s = check_problem(p);
    if (s != KVC_OK) return s;
    kvc_problem pc;
    if ((s = chunk_problem(p, chunks, &pc)) != KVC_OK) return s;
    kvc_params q;
    if (prm) q = *prm; else kvc_default_params(&q);
    if ((s = check_params(q, p->T)) != KVC_OK) return s;
    if (q.flags & KVC_FLAG_SELECT_OMP) return KVC_ERR_INVALID_ARG;      // the pursuit runs on whole caches only
    if ((s = check_buffers(Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status)) != KVC_OK) return s;
    return enqueue_compact(&pc, q, chunks, Q_ref, K, V, budgets, offsets, idx_out, C_k, beta, C_v, head_status,
                           workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

kvc_status kvc_attend(const kvc_problem* p, const void* Q, int32_t n_q, const void* C_k, const float* beta,
                      const float* C_v, const int32_t* offsets, float* O_out, int32_t* head_status, float scale,
                      kvc_stream_t stream) {
    if (!p || p->H < 1 || p->H > kMaxHeads || (p->d != 64 && p->d != 128) || n_q < 1 ||
        (p->dtype != KVC_DTYPE_BF16 && p->dtype != KVC_DTYPE_F32) || !(scale >= 0.f) || !std::isfinite(scale))
        return KVC_ERR_INVALID_ARG;
    if (!Q || !C_k || !beta || !C_v || !offsets || !O_out || !head_status) return KVC_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(C_k, 16) || !aligned(C_v, 16) || !aligned(O_out, 16) || !aligned(beta, 4) ||
        !aligned(offsets, 4) || !aligned(head_status, 4))
        return KVC_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    KVC_TRY(cudaMemsetAsync(head_status, 0, sizeof(int32_t) * p->H, st));
    // few queries per head (decode): a cluster of CTAs splits each head's keys;
    // many queries: query tiles per head
    if (n_q <= attend_decode_max_queries())
        KVC_TRY(launch_attend_decode(p->dtype, p->d, Q, n_q, C_k, beta, C_v, offsets, p->H, log2_scale(*p, scale),
                                     O_out, head_status, st));
    else
        KVC_TRY(launch_attend(p->dtype, p->d, Q, n_q, C_k, beta, C_v, offsets, p->H, log2_scale(*p, scale), O_out,
                              head_status, st));
    return KVC_OK;
}

kvc_status kvc_stage_times(int32_t* n_stages, float* ms, const char** names, int32_t* counts, int32_t* launches,
                           int32_t cap) {
    if (!n_stages || cap < 0 || (cap > 0 && (!ms || !names || !counts))) return KVC_ERR_INVALID_ARG;
    if (launches) *launches = g_last_launches;
    if (!g_log.created || g_log.n == 0) {
        *n_stages = 0;
        return KVC_OK;
    }
    if (cudaEventSynchronize(g_log.ev[g_log.n]) != cudaSuccess) return KVC_ERR_CUDA;
    const int m = g_log.n < cap ? g_log.n : cap;
    for (int i = 0; i < m; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_log.ev[i], g_log.ev[i + 1]) != cudaSuccess) return KVC_ERR_CUDA;
        ms[i] = t;
        names[i] = g_log.names[i];
        counts[i] = g_log.counts[i];
    }
    *n_stages = g_log.n;
    return KVC_OK;
}

const char* kvc_status_string(kvc_status s) {
    switch (s) {
        case KVC_OK: return "ok";
        case KVC_ERR_INVALID_ARG: return "invalid argument";
        case KVC_ERR_ALIGN: return "pointer not aligned";
        case KVC_ERR_WORKSPACE: return "workspace missing or too small";
        case KVC_ERR_CUDA: return "CUDA launch or runtime error";
        case KVC_ERR_NOALLOC_LIMIT: return "problem needs more scratch than the fixed no-allocation array holds";
        case KVC_ERR_BAD_BUDGET: return "bad budget or offsets for this head";
        case KVC_ERR_NOT_SPD: return "matrix not positive definite";
        case KVC_ERR_NNLS_MAXITER: return "NNLS iteration or zero-set cap reached";
        case KVC_ERR_NONFINITE: return "non-finite value";
        case KVC_ERR_TIMEOUT: return "device-side wait timed out";
        case KVC_ERR_DEBUG_BOUNDS: return "debug build: index outside its buffer (access skipped)";
    }
    return "unknown status";
}

#ifdef KVC_DEBUG
const char* kvc_version(void) { return "kvc 0.2.0 sm_103a debug"; }
#else
const char* kvc_version(void) { return "kvc 0.2.0 sm_103a"; }
#endif

}  // extern "C"
