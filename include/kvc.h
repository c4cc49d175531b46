/*
 * kvc.h - C ABI of the B300 Attention Matching KV-cache compaction library.
 *
 * The method is the one described on "Fast KV Compaction via Attention
 * Matching" (gist.science explainer of arXiv 2602.16284), section 2
 * ("Objectif principal", "Pipeline algorithmique"): for every KV head, a cache
 * of T keys/values and n reference queries Q_ref are reduced to t < T entries
 * (C_k = selected original keys, a per-key scalar bias beta, refitted values
 * C_v) so that softmax(q C_k^T/sqrt(d) + beta) C_v and
 * sum_i exp(q C_k[i]/sqrt(d) + beta_i) reproduce the full cache's attention
 * output and attention mass for the reference queries.
 *
 * Conventions shared by every entry point
 *  - All pointers marked "device" are CUDA device pointers on the current
 *    device; "host" pointers are ordinary host memory.
 *  - The caller owns every buffer.  kvc_compact / kvc_attend allocate nothing
 *    and free nothing; scratch comes from the caller's workspace.
 *  - Work is enqueued asynchronously on `stream`; no call synchronises the
 *    stream.  Outputs are valid once the stream reaches that point.
 *  - Tensors are row-major with the head dimension d contiguous; heads are
 *    packed back to back (head h of Q starts at element h*n*d).
 *  - Q/K/V/C_k are `dtype` (bf16 or fp32); every other float is fp32.
 *  - The return value reports argument, alignment, workspace and launch
 *    errors only (nothing is enqueued when it is not KVC_OK).  Numerical
 *    outcomes are written per head into `head_status` (device int32 [H]);
 *    a head whose status is not KVC_OK has unspecified outputs.
 *  - No C++ exception crosses this interface.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvc_stream_t;  /* cudaStream_t; NULL = legacy default stream */

typedef enum kvc_status {
    KVC_OK = 0,
    /* call-level errors (return value) */
    KVC_ERR_INVALID_ARG = 1,   /* bad size, null pointer, unsupported d/dtype     */
    KVC_ERR_ALIGN = 2,         /* a tensor pointer is not 16-byte aligned          */
    KVC_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required       */
    KVC_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed       */
    KVC_ERR_NOALLOC_LIMIT = 5, /* kvc_compact_noalloc: the problem needs more
                                  scratch than KVC_NOALLOC_SCRATCH_BYTES           */
    /* per-head outcomes (head_status) */
    KVC_ERR_BAD_BUDGET = 16,   /* t_h outside [1, min(T, max_t)], offsets not the
                                  exclusive prefix sum of budgets, or more forced
                                  keys than t_h                                     */
    KVC_ERR_NOT_SPD = 17,      /* a Cholesky pivot was not positive                 */
    KVC_ERR_NNLS_MAXITER = 18, /* NNLS pivoting hit its iteration or set-size cap;
                                  the head's outputs are not written; workspace
                                  item W holds the last clamped iterate        */
    KVC_ERR_NONFINITE = 19,    /* NaN/Inf in the inputs or an intermediate          */
    KVC_ERR_TIMEOUT = 20,      /* a bounded device-side wait gave up (after
                                  kvc_params.wait_timeout_us, one second by
                                  default); the kernel released its resources
                                  and left the head unfinished                 */
    KVC_ERR_DEBUG_BOUNDS = 21  /* debug build only (libkvc_debug.so, compiled
                                  with KVC_DEBUG): a kernel found an index read
                                  from data outside the buffer it addresses and
                                  skipped the access                           */
} kvc_status;

typedef enum kvc_dtype { KVC_DTYPE_BF16 = 0, KVC_DTYPE_F32 = 1 } kvc_dtype;

/* Shape of one call.  H independent KV heads (1 <= H <= 65535), each with n
 * reference queries (for GQA, the group's query heads stacked), T cached
 * tokens, head dim d (64 or 128).  max_t bounds every per-head budget
 * (max_t <= min(T, 4096)). */
typedef struct kvc_problem {
    int32_t H;
    int32_t n;
    int32_t T;
    int32_t d;
    int32_t dtype;     /* kvc_dtype */
    int32_t max_t;
} kvc_problem;

/* Tuning / reading parameters.  kvc_default_params fills the defaults. */
typedef struct kvc_params {
    float scale;          /* logit scale; 0 -> 1/sqrt(d)                          */
    float eps_mu;         /* NNLS ridge toward w = 1: mu = eps_mu * tr(G)/t (1e-2) */
    float eps_lambda;     /* C_v ridge toward V[idx]: lambda = eps_lambda *
                             tr(X^T X)/t (1e-2)                                   */
    int32_t nnls_max_iter;  /* block-pivoting iterations (default 32)             */
    int32_t nnls_max_zero;  /* cap on weights held at zero (default 512)          */
    int32_t refine_iters;   /* NNLS iterative-refinement steps (default 1: the
                               residual is formed from A' itself and the ridge
                               from the exact squares of A', and one step
                               reaches the fixed point to ~1e-5 in beta)   */
    int32_t keep_first;     /* positions [0, keep_first) are always kept          */
    int32_t keep_last;      /* positions [T-keep_last, T) are always kept         */
    uint32_t flags;         /* KVC_FLAG_* bits; other bits must be 0              */
    uint32_t wait_timeout_us; /* limit of every bounded device-side wait of the
                             tensor-core kernels, in microseconds at the
                             device's peak SM clock (default 1000000, i.e.
                             one second; must be >= 1).  A wait that runs out
                             ends its kernel's work on that head: the kernel
                             waits (under its own one-second limit) for the
                             copies and tensor-core operations it has already
                             issued, releases its tensor memory and writes
                             KVC_ERR_TIMEOUT for the head.  Limits below about
                             half a millisecond are polled without suspending
                             the waiting thread.  Short limits are for tests
                             of that path: a limit below the normal latency
                             of a tile load times out on purpose.            */
} kvc_params;

/* kvc_params.flags: record a CUDA event on the stream after every stage of
 * kvc_compact, readable with kvc_stage_times (the events are created once per
 * host thread on first use and kept until exit). */
#define KVC_FLAG_STAGE_TIMING 1u
/* kvc_params.flags: solve the C_v normal equations with a blocked Cholesky
 * factorisation and two triangular solves instead of the default explicit
 * inverse by symmetric block sweeps (same results to rounding; the default is
 * faster because its block steps are shorter). */
#define KVC_FLAG_CHOLESKY_CV 2u
/* kvc_params.flags: choose the kept keys by orthogonal matching pursuit
 * instead of the highest RMS attention (page section 2, "Pipeline
 * algorithmique", key selection: keys picked greedily to best meet the
 * attention-mass objective, the weights then fitted by NNLS).  Atoms are the
 * columns p_j of the relative mass P_qj = exp(S_qj - lse_q) of all T keys,
 * the target is 1 per query; a step adds the key with the largest
 * <p_j, r> / ||p_j|| (ties to the lower position) where r is the residual of
 * the least-squares fit of 1 on the keys chosen so far; forced positions come
 * first.  beta and C_v are then fitted as usual.  With bf16 inputs every
 * step recomputes the correlations <p_j, r> on the tensor cores (Q K^T
 * again, weighted by r); with fp32 inputs the fp32 P of every head is kept
 * (H * T * n * 4 bytes of workspace).  Both keep an orthonormal basis
 * (H * max_t * n * 4 bytes); the selection order is readable at
 * kvc_workspace_offset item 5.  The pursuit is sequential over t: expect it
 * to cost far more than the default selection.  Not for kvc_compact_chunked. */
#define KVC_FLAG_SELECT_OMP 4u

/* Fill *prm with the defaults listed above.  Returns KVC_ERR_INVALID_ARG for a
 * null pointer. */
kvc_status kvc_default_params(kvc_params* prm);

/* Bytes of device workspace kvc_compact needs for problem *p (independent of
 * the budgets' values; sized by max_t).  Host-only; enqueues nothing. */
kvc_status kvc_workspace_size(const kvc_problem* p, const kvc_params* prm, size_t* bytes);

/* Byte offset, inside the workspace of kvc_compact for the same *p and *prm,
 * of an intermediate a caller may inspect after the call completes:
 *   0 O      fp32 [H][n][d]   reference outputs softmax(S) V
 *   1 LSE2   fp32 [H][n]      log2 of each query's attention mass
 *                             (lse in natural log = LSE2 * ln 2)
 *   2 SCORE  fp32 [H][T]      RMS attention score of every key
 *   3 W      fp32 [sum t]     NNLS weights w = exp(beta), offsets-indexed
 *   4 HEAD   32-byte records per head (ridges mu, lambda; NNLS zero-set
 *            size and iterations)
 *   5 ORDER  int32 [H][max_t]: keys in the order the pursuit chose them
 *            (KVC_FLAG_SELECT_OMP only; INVALID_ARG otherwise)
 *   6 L2     fp32 [H][n][ldA], ldA = max_t rounded up to a multiple of 64:
 *            log2 of the kept keys' relative mass A'_qi = exp(S_q,idx_i -
 *            lse_q) in columns i < t_h of head h (later columns
 *            unspecified).  Intact after the call only with
 *            KVC_FLAG_CHOLESKY_CV: the default C_v solve reuses this region
 *            for its operand terms once the log-masses have been read.
 * prm->keep_first / keep_last are not checked against p->T here (the layout
 * does not depend on them).
 * Host-only.  Errors: INVALID_ARG (bad problem/params or unknown item). */
kvc_status kvc_workspace_offset(const kvc_problem* p, const kvc_params* prm, int32_t item, size_t* offset);

/* Compact H KV heads (page section 2, "Pipeline algorithmique"):
 *   1. S = Q_ref K^T * scale, lse_q = log sum_j exp(S_qj), O = softmax(S) V;
 *   2. score_j = sqrt(mean_q exp(S_qj - lse_q)^2) (attention aggregated by RMS);
 *   3. idx = the t_h keys of largest float32 score (ties -> lower index;
 *      forced positions first), ascending; C_k = K[idx];
 *   4. w = exp(beta) >= 0 by NNLS on A'_qi = exp(S_q,idx_i - lse_q) against
 *      the relative mass target 1, with ridge mu ||w - 1||^2;
 *   5. C_v by least squares X C_v ~ O, X = softmax_i(S_q,idx_i + beta_i), with
 *      ridge lambda ||C_v - V[idx]||^2, through X^T X, X^T O and Cholesky.
 *
 * Arguments (device unless stated):
 *   p, prm     host; problem shape and parameters (prm NULL -> defaults)
 *   Q_ref      [H][n][d] dtype          K, V  [H][T][d] dtype   (16B aligned)
 *   budgets    int32 [H]: t_h, 1 <= t_h <= min(T, max_t)
 *   offsets    int32 [H+1]: exclusive prefix sum of budgets (offsets[0] = 0);
 *              head h's outputs occupy rows [offsets[h], offsets[h+1])
 *   idx_out    int32 [sum t]: kept positions, ascending within a head
 *   C_k        [sum t][d] dtype: exact copies of the kept K rows
 *   beta       fp32 [sum t]: log w, -INFINITY where w = 0
 *   C_v        fp32 [sum t][d]
 *   head_status int32 [H]: KVC_OK or a per-head outcome above
 *   workspace  device scratch of at least kvc_workspace_size bytes, 256B aligned
 * Errors: INVALID_ARG, ALIGN, WORKSPACE, CUDA (nothing enqueued on the first
 * three).  Calls that share a workspace must not overlap on the GPU. */
kvc_status kvc_compact(const kvc_problem* p, const kvc_params* prm,
                       const void* Q_ref, const void* K, const void* V,
                       const int32_t* budgets, const int32_t* offsets,
                       int32_t* idx_out, void* C_k, float* beta, float* C_v,
                       int32_t* head_status,
                       void* workspace, size_t workspace_bytes, kvc_stream_t stream);

/* Size of the fixed device scratch array behind kvc_compact_noalloc (64 MiB).
 * Every GPU that loads this library holds one such array until the process
 * exits. */
#define KVC_NOALLOC_SCRATCH_BYTES (64u << 20)

/* kvc_compact without a workspace argument, for callers that cannot allocate
 * device memory: an engine whose allocator has reserved the device's memory
 * and forbids other allocations, a latency-critical path where cudaMalloc /
 * cudaFree would synchronise the device, or a C program with no device
 * allocator.  The page has no counterpart of this entry point; it is an
 * interface convenience only.
 *
 * Arguments, outputs, per-head statuses and results are those of
 * kvc_compact.  Differences:
 *  - The scratch is a library-owned device array of KVC_NOALLOC_SCRATCH_BYTES.
 *    A problem whose kvc_workspace_size exceeds it is rejected with
 *    KVC_ERR_NOALLOC_LIMIT, and nothing is enqueued.
 *  - The call allocates and frees nothing: no cudaMalloc, no cudaFree and no
 *    allocating library routine.  prm->flags must not ask for stage timing,
 *    since that creates events (INVALID_ARG).
 *  - The first call on a device looks up the array's device address with
 *    that device current, and caches it. Make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents.  The kernels write every scratch value before reading it.
 *    Calls whose work overlaps on the GPU (different streams, or different
 *    host threads without ordering) race on the array: order them, or use
 *    kvc_compact with separate workspaces.
 * Errors: those of kvc_compact, plus NOALLOC_LIMIT. */
kvc_status kvc_compact_noalloc(const kvc_problem* p, const kvc_params* prm,
                               const void* Q_ref, const void* K, const void* V,
                               const int32_t* budgets, const int32_t* offsets,
                               int32_t* idx_out, void* C_k, float* beta, float* C_v,
                               int32_t* head_status, kvc_stream_t stream);

/* Chunked compaction (page section 2, "Compaction par blocs": the full
 * context is prefilled, its KV cache is cut into contiguous chunks, each
 * chunk is compacted on its own, and the compacted chunks are concatenated).
 *
 * *p describes the whole cache: H KV heads of T positions, n reference
 * queries per head, max_t bounding every per-chunk budget.  Each head's cache
 * is split into `chunks` equal chunks of Tc = T / chunks positions (T must be
 * a multiple of chunks; max_t <= Tc).  Chunk c of head h is compacted exactly
 * as kvc_compact compacts one head of Tc positions, against all n reference
 * queries of head h.  Chunks are indexed g = h * chunks + c throughout.
 *
 * Arguments (device unless stated):
 *   p, prm     host; whole-cache shape, parameters (prm NULL -> defaults);
 *              H * chunks <= 65535
 *   chunks     host; number of chunks per head, >= 1 (1 = kvc_compact)
 *   Q_ref      [H][n][d] dtype       K, V  [H][T][d] dtype   (16B aligned)
 *   budgets    int32 [H*chunks]: t_g, 1 <= t_g <= min(Tc, max_t)
 *   offsets    int32 [H*chunks+1]: exclusive prefix sum of budgets.  The rows
 *              of head h's merged compact cache are [offsets[h*chunks],
 *              offsets[(h+1)*chunks]), chunk by chunk; that range is what
 *              kvc_attend reads with per-head offsets offsets[h*chunks].
 *   idx_out    int32 [sum t]: kept positions in the WHOLE cache (c*Tc plus
 *              the position inside chunk c), ascending within a chunk and so
 *              within a head
 *   C_k, beta, C_v   as in kvc_compact, per chunk
 *   head_status int32 [H*chunks]: per-chunk outcomes as in kvc_compact
 *   workspace  at least kvc_workspace_size_chunked bytes, 256B aligned
 * prm->keep_first / keep_last count positions of the whole cache: chunk c
 * keeps the part of [0, keep_first) and of [T - keep_last, T) inside it.
 * Errors: INVALID_ARG (also T not a multiple of chunks, max_t > Tc, too many
 * chunks), ALIGN, WORKSPACE, CUDA (nothing enqueued on the first three).
 * Workspace offsets (kvc_workspace_offset) are those of the per-chunk problem
 * {H*chunks, n, Tc, d, dtype, max_t}, whose intermediates are per chunk. */
kvc_status kvc_compact_chunked(const kvc_problem* p, const kvc_params* prm, int32_t chunks,
                               const void* Q_ref, const void* K, const void* V,
                               const int32_t* budgets, const int32_t* offsets,
                               int32_t* idx_out, void* C_k, float* beta, float* C_v,
                               int32_t* head_status,
                               void* workspace, size_t workspace_bytes, kvc_stream_t stream);

/* Compact a cache that carries per-key biases and fp32 values: a compacted
 * cache, compacted again.  This is the step of periodic compaction
 * ("Thought-Aware KV Cache Compaction" explainer, section 2 D "Compaction
 * periodique": every P new tokens the t compacted entries plus the P new
 * tokens are compacted back to t, so the cache stays between t and t + P;
 * "Fast KV Compaction via Attention Matching", section 4, "Compaction en
 * ligne": repeated compaction during decoding).
 *
 * The caller concatenates, per head, the compacted entries (C_k, beta, C_v of
 * an earlier call) and the new tokens (their keys, bias 0, their values in
 * fp32).  The steps are those of kvc_compact with the biases in the logits,
 * S_qj = q . K_j * scale + bias_j, so that the targets (attention mass and
 * outputs of the reference queries) are those of the cache as it stands:
 *   1. lse and O = softmax(S) V over the biased cache;
 *   2. key scores sqrt(mean_q exp(S_qj - lse_q)^2); the t_h largest kept;
 *   3. w' >= 0 by the NNLS on A'_qi = exp(S_q,idx_i - lse_q) (biases
 *      included) with ridge mu ||w' - 1||^2, so that the fit scales the kept
 *      entries' existing weights and pulls toward "no change";
 *   4. beta_out = bias_idx + log w' (-INFINITY where w' = 0 or the bias
 *      is -INFINITY);
 *   5. C_v by least squares against O with ridge lambda ||C_v - V[idx]||^2.
 * Keeping every entry (t_h = T) returns the cache unchanged (beta = bias,
 * C_v = V, up to rounding).
 *
 * Arguments as kvc_compact, except (device):
 *   K        [H][T][d] dtype (the kept keys are exact copies of these rows)
 *   bias     fp32 [H][T] natural-log units; -INFINITY switches an entry off
 *            (its attention is 0); NaN or +INFINITY -> NONFINITE for the head;
 *            4-byte aligned
 *   V        fp32 [H][T][d], 16-byte aligned
 *   workspace at least kvc_workspace_size_biased bytes
 * A head whose every key is switched off gets NONFINITE.  KVC_FLAG_SELECT_OMP
 * must be unset (INVALID_ARG); keep_first / keep_last apply as in kvc_compact.
 * Errors: INVALID_ARG, ALIGN, WORKSPACE, CUDA (nothing enqueued on the first
 * three). */
kvc_status kvc_compact_biased(const kvc_problem* p, const kvc_params* prm,
                              const void* Q_ref, const void* K, const float* bias, const float* V,
                              const int32_t* budgets, const int32_t* offsets,
                              int32_t* idx_out, void* C_k, float* beta, float* C_v,
                              int32_t* head_status,
                              void* workspace, size_t workspace_bytes, kvc_stream_t stream);

/* Bytes of workspace kvc_compact_biased needs.  Host-only.  Errors:
 * INVALID_ARG. */
kvc_status kvc_workspace_size_biased(const kvc_problem* p, const kvc_params* prm, size_t* bytes);

/* Bytes of workspace kvc_compact_chunked needs for *p cut into `chunks`
 * chunks per head (that of the per-chunk problem).  Host-only.
 * Errors: INVALID_ARG. */
kvc_status kvc_workspace_size_chunked(const kvc_problem* p, const kvc_params* prm, int32_t chunks, size_t* bytes);

/* Thought-aware compaction ("Thought-Aware KV Cache Compaction" explainer,
 * section 2, on top of Attention Matching): B, segment budgets, and C, pivot
 * protection.  The segments are given (the page finds them in the text).
 *   - alpha_j = mean over the n_win window queries (the last tokens'
 *     queries) of softmax_j(q K^T * scale): the attention key j receives.
 *   - Pivots: alpha_j > pivot_c * mean_j alpha_j.  They are kept with
 *     beta = 0 and C_v = V exactly.
 *   - Segment i = positions [seg_bounds[i], seg_bounds[i+1]) keeps its pivots
 *     and t_i other keys, t_i ~ sqrt(w_i) * n_i of the budget left after all
 *     pivots (w_i = sum of alpha over the segment, n_i its non-pivot count),
 *     capped at n_i with the excess re-shared, made integral by largest
 *     remainder (ties to the lower segment); computed in double.
 *   - Inside a segment, the t_i keys of highest RMS attention over the
 *     reference queries (as kvc_compact).
 *   - beta and C_v as kvc_compact, with the pivots held fixed: the NNLS and
 *     the least squares run over the other kept keys and the pivots'
 *     contribution moves to the targets (ridges over all kept keys).
 * Arguments as kvc_compact, plus (device unless stated):
 *   Q_win       [H][n_win][d] dtype, 16B aligned; n_win >= 1 (host)
 *   seg_bounds  int32 [nseg+1], shared by every head: 0 = b_0 < ... < b_nseg
 *               = T; 1 <= nseg <= 1024 (host).  Checked on the device: a head
 *               gets BAD_BUDGET if they are not so
 *   pivot_c     host; the threshold factor c > 0
 *   budgets     t_h per head, pivots included (BAD_BUDGET if a head has more
 *               pivots than t_h)
 *   seg_budgets_out int32 [H][nseg]: t_i (non-pivot keys kept per segment)
 *   pivots_out  uint8 [H][T]: 1 where alpha_j is above the threshold
 *   workspace   at least kvc_workspace_size_tam bytes
 * prm->keep_first / keep_last must be 0 and KVC_FLAG_SELECT_OMP unset.
 * Errors: INVALID_ARG, ALIGN, WORKSPACE, CUDA.  Intermediates: the
 * kvc_workspace_offset items of the same *p and *prm. */
kvc_status kvc_compact_tam(const kvc_problem* p, const kvc_params* prm,
                           const void* Q_ref, const void* K, const void* V,
                           const void* Q_win, int32_t n_win,
                           const int32_t* seg_bounds, int32_t nseg, float pivot_c,
                           const int32_t* budgets, const int32_t* offsets,
                           int32_t* idx_out, void* C_k, float* beta, float* C_v,
                           int32_t* head_status, int32_t* seg_budgets_out, uint8_t* pivots_out,
                           void* workspace, size_t workspace_bytes, kvc_stream_t stream);

/* Bytes of workspace kvc_compact_tam needs.  Host-only.  Errors: INVALID_ARG. */
kvc_status kvc_workspace_size_tam(const kvc_problem* p, const kvc_params* prm, int32_t n_win, int32_t nseg,
                                  size_t* bytes);

/* Read a compacted cache with a per-key bias (page section 2 objective, and
 * section 5 on use with standard attention kernels):
 *   O_out[h][q] = softmax_i(Q[h][q] . C_k[i] * scale + beta[i]) C_v[i]
 * over head h's rows i in [offsets[h], offsets[h+1]).
 *   p          host; H, d, dtype are read (n, T, max_t ignored)
 *   Q          [H][n_q][d] dtype;  C_k [sum t][d] dtype;  beta fp32 [sum t];
 *   C_v        fp32 [sum t][d];  offsets int32 [H+1] (device)
 *   O_out      fp32 [H][n_q][d]
 *   head_status int32 [H]: KVC_OK, BAD_BUDGET (empty or inconsistent range),
 *              NONFINITE (every bias -inf for some query)
 *   scale      logit scale; 0 -> 1/sqrt(d)
 * With n_q <= 16 (decode: one new token per query head of a group) each head
 * is split over a cluster of 8 CTAs that stream its keys and merge their
 * partial softmax states on chip; with more queries each CTA takes a tile of
 * 64 queries of one head.  Both give the same result up to fp32 rounding.
 * 1 <= H <= 65535.
 * Errors: INVALID_ARG, ALIGN, CUDA. */
kvc_status kvc_attend(const kvc_problem* p, const void* Q, int32_t n_q,
                      const void* C_k, const float* beta, const float* C_v,
                      const int32_t* offsets, float* O_out, int32_t* head_status,
                      float scale, kvc_stream_t stream);

/* Device time of each stage of the last kvc_compact call made on this host
 * thread with KVC_FLAG_STAGE_TIMING (measuring instrumentation; no
 * counterpart on the page).  Blocks until that call's last stage finished.
 *   n_stages  out: number of stages recorded (0 if no timed call yet)
 *   ms, names, counts  out, host arrays of `cap` entries: stage duration in
 *             milliseconds, static stage name, kernel launches in the stage
 *   launches  out (may be NULL): kernel launches of the last kvc_compact call
 *             (timed or not) on this thread
 * Errors: INVALID_ARG (null n_stages, or null arrays with cap > 0), CUDA. */
kvc_status kvc_stage_times(int32_t* n_stages, float* ms, const char** names, int32_t* counts,
                           int32_t* launches, int32_t cap);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* kvc_status_string(kvc_status s);

/* Library version string, e.g. "kvc 0.1.0 sm_103a". */
const char* kvc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H_ */
