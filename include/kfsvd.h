/*
 * kfsvd.h - C ABI of libkfsvd.so: curvature-whitened truncated SVD of linear layers with
 * global rank allocation, on one NVIDIA Blackwell GPU (sm_103a).
 *
 * The calls follow the statement of the problem in
 *   LASER: Loss-Aware Singular-value Decomposition and Rank Allocation for Efficient
 *   Low-Precision Vision-Language Models (technical summary, Methodology 1 and 2),
 *   UniRank: Unified Rank Allocation for Low-Rank LLM Compression (section 2.1), and
 *   Swift-SVD: Theoretical Optimality Meets Practical Efficiency in Low-Rank LLM
 *   Compression (section 2A):
 * given a weight W (d_in x d_out, y = x W) and calibration activations A and output
 * gradients Gr, estimate the K-FAC factors X = A^T A / N and G = Gr^T Gr / N, whiten
 * W~ = S_x W S_g with S_x^T S_x = X and S_g S_g^T = G, take the spectrum of W~, keep the
 * components with the largest estimated loss increase 1/2 sigma^2 under a global parameter
 * budget (each kept pair costs d_in + d_out), and map the kept factors back:
 * U = S_x^-1 U~_r Sigma_r, V = V~_r^T S_g^-1, so that W ~= U V.
 *
 * Conventions shared by every call:
 *  - All matrix pointers are DEVICE pointers to caller-owned memory; matrices are
 *    row-major with an explicit leading dimension in elements (ld >= columns).
 *  - Every call is asynchronous on the caller's CUDA stream (`stream`, a cudaStream_t;
 *    NULL is the legacy default stream).  Nothing is copied between host and device
 *    except by kf_sync_status.
 *  - Argument errors (null pointers, sizes, leading dimensions, alignment, workspace too
 *    small) are detected on the host before any launch and returned synchronously; the
 *    text is available from kf_last_error().
 *  - Numerical failures found on the device (a Cholesky pivot <= 0, Jacobi not converged,
 *    a device-side wait that gave up) are recorded in the context's device status word;
 *    the first one wins.  kf_sync_status() synchronises the stream and returns it.
 *  - Scratch memory is passed in by the caller as `workspace` / `workspace_bytes`; each
 *    call has a *_workspace_size() query.  The library allocates nothing per call; the
 *    context owns a few bytes of device status and one pinned host word.
 *  - A context may be used by one host thread at a time.
 */
#ifndef KFSVD_H
#define KFSVD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KF_API __attribute__((visibility("default")))
#else
#define KF_API
#endif

typedef struct CUstream_st* kf_stream_t; /* identical to cudaStream_t */

typedef enum {
  KF_OK = 0,
  KF_ERR_INVALID = 1,         /* bad argument: null pointer, size, ld, alignment, mode   */
  KF_ERR_WORKSPACE = 2,       /* workspace_bytes smaller than the matching *_size query  */
  KF_ERR_CUDA = 3,            /* a CUDA runtime call or kernel launch failed            */
  KF_ERR_NOT_SPD = 4,         /* Cholesky met a pivot <= 0 or not finite (info = index)  */
  KF_ERR_NO_CONVERGENCE = 5,  /* Jacobi did not converge within max_sweeps (info = unit) */
  KF_ERR_TIMEOUT = 6,         /* a bounded device-side wait gave up (info = site code)   */
  KF_ERR_UNSUPPORTED = 7      /* device is not compute capability 10.x/11.x, or size cap */
} kf_status;

typedef enum { KF_BF16 = 0, KF_F32 = 1 } kf_dtype;
typedef enum { KF_QUANT_NONE = 0, KF_QUANT_INT8_TOKEN = 1 } kf_quant;
typedef enum {
  KF_KEY_HALF_SIGMA2 = 0,   /* 1/2 sigma^2: the K-FAC estimate of the loss increase */
  KF_KEY_PER_PARAM = 1,     /* 1/2 sigma^2 / (m + n): score per parameter cost */
  KF_FIXED_RANK = 2,        /* a given rank per unit, no sort */
  KF_KEY_ENERGY_RATIO = 3   /* sigma_i^2 / sum_j sigma_j^2 of the unit (UniRank's local significance) */
} kf_alloc_mode;
typedef enum { KF_SIDE_RIGHT = 0, KF_SIDE_LEFT = 1 } kf_side;

/* whiten() flags: reuse factors that an earlier whiten() call already wrote into the
 * same buffers (e.g. q, k and v share the input factor S_x). */
#define KF_REUSE_SX 1u
#define KF_REUSE_SG 2u
#define KF_REUSE_SINV 4u
/* whiten() flags: the three bfloat16 planes of S_x (S_g) that the previous whiten() call left
 * in the same workspace are reused instead of split again.  Valid only when that call had the
 * same workspace pointer, the same m and n, and the same factor (units that share an input or
 * output factor, e.g. the attention heads of one layer, taken one after the other). */
#define KF_REUSE_SX_PLANES 8u
#define KF_REUSE_SG_PLANES 16u

typedef struct kf_ctx kf_ctx;

/* Creates a context on `device` (made current for the call).  Fails with
 * KF_ERR_UNSUPPORTED on GPUs older than compute capability 10.0. */
KF_API kf_status kf_create(int device, kf_ctx** out);
KF_API void kf_destroy(kf_ctx* ctx);

/* Message of the last failing call made on this host thread ("" if none). */
KF_API const char* kf_last_error(void);

/* Number of CUDA kernels this library has launched in the process so far (all contexts,
 * all streams); differences of two readings count the launches of the calls between. */
KF_API uint64_t kf_launch_count(void);

/* Synchronises `stream`, then returns and clears the device status word.  *info (may be
 * NULL) receives the detail: the global pivot index for KF_ERR_NOT_SPD, the unit index
 * for KF_ERR_NO_CONVERGENCE, the wait site for KF_ERR_TIMEOUT. */
KF_API kf_status kf_sync_status(kf_ctx* ctx, kf_stream_t stream, int32_t* info);

/* Limit, in nanoseconds of device wall-clock time, of each wait inside the tensor-core
 * pipeline (a stage of operands arriving, an accumulator being consumed) for later calls on
 * this context; 0 restores the default of 4 s.  A wait that runs out records KF_ERR_TIMEOUT
 * (info = wait site) in the status word, and the kernel stops issuing work, waits for what
 * it already started (on the 4 s limit), releases its tensor memory and returns; its output
 * is then incomplete.  The context stays usable: the next call with a long enough limit
 * computes normally.  A short limit is for testing the failure path. */
KF_API kf_status kf_set_wait_limit(kf_ctx* ctx, uint64_t limit_ns);

/* Measurement aid: launches a kernel that keeps every FP32 FMA pipe of the device busy
 * (8 CTAs of 256 threads per SM, 16 independent fma chains per thread, `iters` steps) and
 * returns in *flops the flops it executes (2 per fma); the caller times the launch on
 * `stream` with CUDA events to measure the FP32 SIMT roof of the Gram and Jacobi kernels.
 * sink: device float[8], written only in a case that does not occur (keeps the work live). */
KF_API kf_status kf_fp32_fma_probe(kf_ctx* ctx, int64_t iters, float* sink, double* flops, kf_stream_t stream);

/* Side whose Gram matrix the spectrum is taken from: KF_SIDE_RIGHT (W~^T W~, n x n) when
 * d_out <= d_in, else KF_SIDE_LEFT (W~ W~^T, m x m). */
KF_API kf_side kf_gram_side(int64_t m, int64_t n);

/* ------------------------------------------------------------------------------------
 * (1) kfac_accumulate - step 1: stream calibration rows into a K-FAC factor.
 * LASER Methodology 1 (X, G are activation and gradient covariances estimated on a
 * calibration set; quantisation-aware whitening estimates them from quantised
 * activations); Swift-SVD 2A (the covariance is aggregated batch by batch).
 *
 * act:     n_tokens x d rows (one token per row), dtype KF_BF16 or KF_F32, leading
 *          dimension ld; 16-byte aligned, ld * sizeof(dtype) a multiple of 16.
 * quant:   KF_QUANT_INT8_TOKEN fake-quantises every row first: s = max|row| / 127,
 *          q = clamp(rint(x / s), -127, 127), value s * q rounded to bfloat16 (float32
 *          arithmetic, a zero row stays zero).
 * cov_sum: d x d float32 (ldc), caller-initialised (zero before the first chunk).  The
 *          lower triangle including the diagonal (i >= j) is incremented by
 *          sum_t a_ti a_tj; entries above the diagonal are neither read nor written.
 * Products of bfloat16 values are exact and accumulate in float32 on the tensor cores,
 * 2048 tokens per tensor-core pass; the partial sums are added with IEEE float32 adds
 * (relative error of a diagonal entry about 5e-6 at 131072 tokens).  Float32 rows are split
 * into two bfloat16 terms (three products: hi*hi + hi*lo + lo*hi).
 * ---------------------------------------------------------------------------------- */
KF_API size_t kfac_accumulate_workspace_size(kf_dtype dtype, kf_quant quant, int64_t d);
KF_API kf_status kfac_accumulate(kf_ctx* ctx, const void* act, kf_dtype dtype, int64_t n_tokens,
                          int64_t d, int64_t ld, kf_quant quant, float* cov_sum, int64_t ldc,
                          void* workspace, size_t workspace_bytes, kf_stream_t stream);

/* Step 1a on its own: the per-token INT8 fake quantisation that kfac_accumulate applies with
 * KF_QUANT_INT8_TOKEN (LASER Methodology 1, quantisation-aware whitening), for callers that
 * need the quantised rows themselves (the empirical-Fisher pass reads the same quantised
 * activations the covariance was built from).  in: n_tokens x d rows (KF_BF16 or KF_F32,
 * leading dimension ld); out: n_tokens x d bfloat16, leading dimension d, caller-owned.  Every
 * row is quantised over its full width d (the scale is max|row| / 127). */
KF_API kf_status fake_quant_rows(kf_ctx* ctx, const void* in, kf_dtype dtype, int64_t n_tokens, int64_t d,
                                 int64_t ld, void* out, kf_stream_t stream);

/* Step 1, tail: turns a finished sum into the damped factor, in place:
 * C = sum / n_tokens (lower triangle mirrored to the full matrix), then
 * C += lambda * mean(diag(C)) * I.  Call once per site after its last kfac_accumulate. */
KF_API kf_status kf_finalize_covariance(kf_ctx* ctx, float* cov, int64_t ldc, int64_t d,
                                 int64_t n_tokens, float lambda, kf_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (2)+(3) whiten - Cholesky factors and the curvature-weighted weight.
 * LASER Methodology 1: W~ = S_x W S_g with S_x, S_g Cholesky factors of X and G.
 *
 * X:     m x m damped input factor (ldx), G: n x n damped output factor (ldg); may point
 *        at a diagonal block of a larger factor (per-head units).
 * W:     m x n weight (d_in x d_out), KF_BF16 or KF_F32, leading dimension ldw.
 * Sx:    m x m out, S_x = chol_lower(X)^T (upper triangular, zeros below the diagonal).
 * Sg:    n x n out, S_g = chol_lower(G) (lower triangular, zeros above).
 * Sinv:  s x s out, inverse of the Gram-side factor (S_g^-1 for KF_SIDE_RIGHT, S_x^-1 for
 *        KF_SIDE_LEFT; see kf_gram_side), needed by unwhiten().
 * Wt:    m x n float32 out, W~ = S_x W S_g, computed on the tensor cores with every float32
 *        operand split into three bfloat16 planes (the full 24-bit significand) and the K
 *        range summed 1024 at a time inside the tensor cores, partials in float32.
 * flags: KF_REUSE_* skip recomputing a factor already present in its buffer.
 * A pivot <= 0 sets KF_ERR_NOT_SPD on the device (raise lambda and retry).
 * ---------------------------------------------------------------------------------- */
KF_API size_t whiten_workspace_size(int64_t m, int64_t n);
KF_API kf_status whiten(kf_ctx* ctx, const float* X, int64_t ldx, int64_t m, const float* G,
                 int64_t ldg, int64_t n, const void* W, kf_dtype w_dtype, int64_t ldw,
                 uint32_t flags, float* Sx, int64_t ldsx, float* Sg, int64_t ldsg, float* Sinv,
                 int64_t ldsi, float* Wt, int64_t ldwt, void* workspace,
                 size_t workspace_bytes, kf_stream_t stream);

/* factor_covariances - step 2 for many factors at once: the Cholesky factor of each damped
 * covariance and, where asked, the inverse of that factor, each job an independent chain of
 * launches on one of the context's internal streams (forked from and joined back into
 * `stream`, so the call is ordered on it like any other).  A group of units then calls
 * whiten() with KF_REUSE_SX | KF_REUSE_SG | KF_REUSE_SINV.  The factorisations are chains of
 * small launches (64 x 64 diagonal blocks, panels, tensor-core trailing updates), so running
 * the chains side by side shortens the step to about the longest chain.
 * Per job: A (n x n, lda, lower triangle read) the damped factor; S (lds) out: the lower
 * Cholesky factor L (upper = 0, as S_g) or L^T (upper = 1, as S_x), zeros in the other
 * triangle; Sinv (ldsi, may be NULL) out: the inverse of S (L^-1 or L^-T).  A non-positive
 * pivot sets KF_ERR_NOT_SPD as in whiten().  The jobs' outputs must not overlap. */
typedef struct {
  const float* A;
  int64_t lda, n;
  float* S;
  int64_t lds;
  float* Sinv;    /* may be NULL */
  int64_t ldsi;
  int32_t upper;
} kf_factor_job;
KF_API size_t factor_covariances_workspace_size(int32_t n_jobs, const kf_factor_job* jobs);
KF_API kf_status factor_covariances(kf_ctx* ctx, int32_t n_jobs, const kf_factor_job* jobs, void* workspace,
                                    size_t workspace_bytes, kf_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (4) whitened_svd - spectrum of W~ through its Gram matrix.
 * LASER Methodology 1 (SVD of W~); Swift-SVD 2A (one eigendecomposition of the Gram of
 * the aggregated output instead of repeated SVDs).
 *
 * Batched: all problems of one call must have the same s = min(m, n) (s <= 16384).
 * Unlike the other calls, whitened_svd waits on the stream once per Jacobi sweep (from the
 * third on): it reads a 4-byte convergence flag and launches no further sweep once every
 * problem of the call has converged.
 * For each problem: C = W~^T W~ (KF_SIDE_RIGHT) or W~ W~^T (KF_SIDE_LEFT) in float32;
 * C = Q Lambda Q^T by blocked parallel cyclic Jacobi (32-wide blocks, round-robin pairing,
 * one sweep of plane rotations per 64 x 64 pair problem in shared memory, the block rotations
 * applied to C and Q on the tensor cores with every float32 operand as three bfloat16 planes,
 * float32-accurate) until every block pair has
 * |c_pq| <= tol * sqrt(c_pp c_qq) (or below a float32 rounding floor).  The vectors are then
 * sorted by their Rayleigh values ||W~ q|| / ||q|| (evaluated on W~ itself, not on C) and
 * refined by two passes of windowed Rayleigh-Ritz: every window of 128 consecutive vectors
 * is rotated by the eigenvectors of the exact Gram of its images (W~ q_i, float64 sums), the
 * second pass with windows offset by 64.  This removes the rounding drift of the Jacobi
 * rotations from the singular values (float32-level relative accuracy on the leading ones).
 * sigma:  s floats out, descending.
 * vecs:   s x s out (ldv): column i is the unit-norm Gram-side singular vector of sigma[i]
 *         (a right singular vector of W~ for KF_SIDE_RIGHT, a left one otherwise).
 * sweeps: device int out (may be NULL): sweeps used.  Not converged within max_sweeps
 *         sets KF_ERR_NO_CONVERGENCE (results are still written).
 * ---------------------------------------------------------------------------------- */
typedef struct {
  const float* Wt;   /* m x n, ldw */
  int64_t m, n, ldw;
  float* sigma;      /* s */
  float* vecs;       /* s x s, ldv */
  int64_t ldv;
  int32_t* sweeps;   /* device, may be NULL */
} kf_svd_problem;

/* Optional timing of whitened_svd's phases, measured with CUDA events recorded on the
 * caller's stream, plus the rotation-application work the Jacobi kernel executed (pairs
 * whose coupling fell below the threshold are skipped and do no work). */
typedef struct {
  float gram_ms, jacobi_ms, rayleigh_ms, refine_ms;  /* refine: windowed refinement + final sort */
  int64_t jacobi_steps;          /* solve + apply launch pairs issued */
  double jacobi_apply_flops;     /* executed tensor-core flops of the rotation products (bfloat16 plane products,
                                    2 M N K per MMA) */
  float jacobi_solve_ms;         /* summed device time of the pair-solve launches */
  float jacobi_apply_ms;         /* summed device time of the rotation-apply launches */
  int64_t jacobi_apply_launches; /* number of rotation-apply launches timed */
  double jacobi_apply_bytes;     /* algorithmic bytes of the rotation apply: C and Qt read and written once per
                                    executed task (a C super-tile moves 64 KB in and 64 or 128 KB out, a Qt
                                    panel 32 KB in and out) */
} kf_svd_profile;

/* Enables (1) or disables (0) recording of the profile by later whitened_svd calls. */
KF_API kf_status kf_svd_profile_enable(kf_ctx* ctx, int enable);
/* Synchronises the stream of the last profiled whitened_svd call and returns its profile. */
KF_API kf_status kf_svd_profile_read(kf_ctx* ctx, kf_svd_profile* out);

KF_API size_t whitened_svd_workspace_size(int32_t n_problems, int64_t m_max, int64_t n_max, int64_t s);
KF_API kf_status whitened_svd(kf_ctx* ctx, int32_t n_problems, const kf_svd_problem* problems,
                       float tol, int32_t max_sweeps, void* workspace, size_t workspace_bytes,
                       kf_stream_t stream);

/* ------------------------------------------------------------------------------------
 * (5a) score_and_allocate - global sort-and-truncate rank allocation.
 * UniRank 2.1 (all scores pooled and sorted descending; kept singular pairs each cost
 * m + n parameters; accumulate until the budget is reached) and LASER Methodology 2
 * (greedy global selection, score per parameter cost).
 *
 * sigma:      device, the units' spectra concatenated; unit u owns
 *             sigma[seg_offset[u] .. seg_offset[u+1]) in descending order.
 * seg_offset: device int64[n_units + 1]; cost: device int64[n_units] (m_u + n_u; every cost
 *             must be >= 0, so that the kept components form a prefix of the sorted list).
 * mode:       KF_KEY_HALF_SIGMA2: key 0.5f * (sigma * sigma);
 *             KF_KEY_PER_PARAM:  that divided by (float)cost[u];
 *             KF_KEY_ENERGY_RATIO: (sigma * sigma) / (sum of the unit's sigma^2);
 *             KF_FIXED_RANK:     ranks[u] = min(fixed_rank[u], length of unit u).
 * The keys are sorted descending (ties: lower unit, then lower component index first): the
 * 64-bit words (~key_bits << 32 | component id) are built in id order and sorted by a stable
 * device LSD radix sort over the score word (four 8-bit passes), which leaves equal scores in
 * id order; the prefix sum of costs in that order is cut at the longest prefix with
 * sum <= budget.  Each pass and the cost prefix are single launches whose 4096-key tiles
 * chain their offsets by a decoupled look-back; its waits are bounded (4 s), and one that ran
 * out would be reported as KF_ERR_TIMEOUT by kf_sync_status.
 * ranks:      device int32[n_units] out: kept components per unit.
 * cut:        device float[2] out (may be NULL): score of the last kept and of the first
 *             dropped component (NaN where there is none).
 * used:       device int64 out (may be NULL): parameters of the kept components.
 * Integer results are deterministic and bit-identical for identical sigma input.
 * ---------------------------------------------------------------------------------- */
KF_API size_t score_and_allocate_workspace_size(int64_t n_components, int32_t n_units);
KF_API kf_status score_and_allocate(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset,
                             const int64_t* cost, int32_t n_units, int64_t n_components,
                             int64_t budget, kf_alloc_mode mode, const int32_t* fixed_rank,
                             int32_t* ranks, float* cut, int64_t* used, void* workspace,
                             size_t workspace_bytes, kf_stream_t stream);

/* score_and_allocate_weighted - the same allocation with every key multiplied by a per-unit
 * weight: UniRank 2.1's aggregated score s_{l,i} = I_l sigma_{l,i}^2 / ||Sigma_l||_F^2 is
 * KF_KEY_ENERGY_RATIO with unit_weight = I_l (the layer's functional importance, computed by
 * the caller from forward passes); any other scoring mode may be weighted the same way.
 * unit_weight: device float[n_units], finite and >= 0 (a negative or NaN weight counts as 0);
 * NULL means 1 for every unit.  KF_FIXED_RANK is rejected.  The energy of a unit is the float64
 * sum of its sigma^2 rounded to float32; every key is then formed in float32 with one rounding
 * per operation (square, divide, multiply by the weight).  Workspace as for
 * score_and_allocate (score_and_allocate_workspace_size covers every mode). */
KF_API kf_status score_and_allocate_weighted(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset,
                                             const int64_t* cost, int32_t n_units, int64_t n_components,
                                             int64_t budget, kf_alloc_mode mode, const float* unit_weight,
                                             int32_t* ranks, float* cut, int64_t* used, void* workspace,
                                             size_t workspace_bytes, kf_stream_t stream);

/* score_and_allocate_keys - sort-and-truncate over per-component keys computed elsewhere
 * (UniRank 2.1's procedure with any score, e.g. LASER Methodology 2's empirical-Fisher scores
 * from empirical_fisher_accumulate).  keys: device float[n_components] laid out like sigma
 * (unit u owns keys[seg_offset[u] .. seg_offset[u+1])), >= 0 (a negative or NaN key counts as
 * 0), in any order within a unit.  Ties: lower unit, then lower component index first.
 * ranks: kept components per unit; keep: device uint8[n_components] out (may be NULL), 1 for
 * every kept component (the kept set of a unit need not be a prefix of its spectrum);
 * cut / used as for score_and_allocate.  Workspace: score_and_allocate_workspace_size. */
KF_API kf_status score_and_allocate_keys(kf_ctx* ctx, const float* keys, const int64_t* seg_offset,
                                         const int64_t* cost, int32_t n_units, int64_t n_components,
                                         int64_t budget, int32_t* ranks, uint8_t* keep, float* cut,
                                         int64_t* used, void* workspace, size_t workspace_bytes,
                                         kf_stream_t stream);

/* score_and_allocate_hybrid - sort-and-truncate on Swift-SVD's hybrid score (section B,
 * Dynamic Rank Allocation Strategy: s_i = beta_i^alpha (log(e + eps*_{k,i}))^(1 - alpha),
 * combining the layer's end-to-end importance beta_i with the closed-form loss eps*_{k,i} of
 * the layer truncated to rank k).  Keyed per component: component k (0-based) of unit u gets
 * the unit's score at rank k, with eps*_k = sum_{j >= k} sigma_j^2 the energy the truncation
 * drops (float64, summed one term at a time from the unit's last component upward), key =
 * (float)(beta_u^alpha * pow(log(e + eps*_k), 1 - alpha)) in float64; the keys are sorted
 * descending (ties: lower unit, then lower component) and cut at the budget as in
 * score_and_allocate, so the next component always goes to the unit whose current
 * truncation scores highest.  eps*_k never increases along a unit, so neither do its keys
 * and the kept set is a prefix of its spectrum (ranks[u] components).
 * importance: device float[n_units] (beta; NULL means 1 for every unit; a value that is not
 *             positive gives the unit keys 0).
 * alpha:      in [0, 1] (KF_ERR_INVALID otherwise): 1 ranks units by beta alone, 0 by the
 *             residual loss alone.  The grid search over alpha and the retention ratio that the
 *             paper runs on validation data is the caller's.
 * sigma, seg_offset, cost, ranks, cut, used and the workspace as for score_and_allocate; the
 * scale of sigma matters (eps* enters through log(e + eps*)). */
KF_API kf_status score_and_allocate_hybrid(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset,
                                           const int64_t* cost, int32_t n_units, int64_t n_components,
                                           int64_t budget, const float* importance, double alpha,
                                           int32_t* ranks, float* cut, int64_t* used, void* workspace,
                                           size_t workspace_bytes, kf_stream_t stream);

/* score_and_allocate_noalloc - score_and_allocate for callers that cannot allocate device
 * memory: for example a host framework that has already handed all device memory to its own
 * pool, or a caller that must not trigger a device allocation (which may synchronise the
 * device) in the middle of a job.  It takes no workspace and allocates nothing: its scratch
 * is a 25 MiB file-scope device array of the library, held on every GPU that uses it until
 * the process exits.  With CUDA's lazy module loading (the default) the array is reserved
 * on a device when the library's allocation code is first used there: the first launch of
 * any allocation kernel (score_and_allocate and its variants) or this call's first address
 * lookup.  A caller that must not allocate after some point should make one call (of this
 * entry point or of score_and_allocate) on each device before it.  The papers have no counterpart; this is
 * a packaging variant of (5a) with identical results.
 * Limit: n_components <= 1048576 (2^20); larger calls return KF_ERR_UNSUPPORTED before any
 * launch.  The first call on a device looks up the array's device address (once per
 * device); make that first call before any stream capture.  Every call reuses the same
 * array (the parts that must start at zero are cleared by each call): calls that overlap on
 * the GPU, on any stream or context of the same device, race and must be serialised. */
KF_API kf_status score_and_allocate_noalloc(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset,
                                            const int64_t* cost, int32_t n_units, int64_t n_components,
                                            int64_t budget, kf_alloc_mode mode, const int32_t* fixed_rank,
                                            int32_t* ranks, float* cut, int64_t* used, kf_stream_t stream);

/* kf_hybrid_ffn_budget - LASER's hybrid FFN budget: the parameters left for the low-rank
 * factors once the dense channels are paid for, max(budget - dense_cost, 0), with
 * dense_cost = sum_i d_model[i] n_dense[i] over the dense projections (a dense channel of a
 * gate or up projection keeps its d_model weights) written to *dense_cost (may be NULL).
 * Host arrays of n entries; returns -1 (message in kf_last_error) for a negative n or entry,
 * or a null array with n > 0.  Host arithmetic, no device work. */
KF_API int64_t kf_hybrid_ffn_budget(int64_t budget, int32_t n, const int64_t* d_model, const int64_t* n_dense,
                                    int64_t* dense_cost);

/* ------------------------------------------------------------------------------------
 * (5b) unwhiten - rank-r factors in the original space.
 * LASER Methodology 1: the low-rank factors of W~ are mapped back to the original space.
 *
 * The r leading columns of vecs are re-orthonormalised (CholeskyQR2) first.
 * KF_SIDE_RIGHT (vecs = V~): U = W (S_g V~_r)          (= S_x^-1 U~_r Sigma_r),
 *                            V = V~_r^T S_g^-1.
 * KF_SIDE_LEFT  (vecs = U~): U = S_x^-1 U~_r Sigma_r,
 *                            V = Sigma_r^-1 (U~_r^T S_x) W   (= V~_r^T S_g^-1).
 * Sx, Sg, Sinv as written by whiten(); sigma, vecs as written by whitened_svd().  Only the
 * Gram-side factor is read (Sg for KF_SIDE_RIGHT, Sx for KF_SIDE_LEFT); the other one may be
 * NULL (its leading dimension is then ignored), so a caller can free it after whiten().
 * U: m x r float32 out (ldu); V: r x n float32 out (ldvo).  0 <= r <= min(m, n).
 * ---------------------------------------------------------------------------------- */
KF_API size_t unwhiten_workspace_size(int64_t m, int64_t n, int32_t r);
KF_API kf_status unwhiten(kf_ctx* ctx, const void* W, kf_dtype w_dtype, int64_t ldw, int64_t m,
                   int64_t n, const float* Sx, int64_t ldsx, const float* Sg, int64_t ldsg,
                   const float* Sinv, int64_t ldsi, const float* sigma, const float* vecs,
                   int64_t ldv, int32_t r, float* U, int64_t ldu, float* V, int64_t ldvo,
                   void* workspace, size_t workspace_bytes, kf_stream_t stream);

/* ------------------------------------------------------------------------------------
 * empirical_fisher_accumulate - LASER Methodology 2's component importance: the
 * contribution of each singular pair to the empirical-Fisher quadratic loss, evaluated with
 * the calibration gradients in the original space.  For the factors U (m x r, column i =
 * u_i) and V (r x n, row i = v_i) of all the components to be scored (unwhiten with r =
 * min(m, n) gives every component):
 *   score_sum[i] += sum_t (a_t . u_i)^2 (g_t . v_i)^2      (float64)
 * over the n_tokens rows of act (n_tokens x m, lda) and grad (n_tokens x n, ldg), bfloat16 or
 * float32.  The score is score_sum / (2 N) after the last chunk.  The projections run on the
 * tensor cores with U and V split into hi + lo bfloat16 planes (about 3e-5 relative per
 * projection); the squares and sums are float64, in a fixed order (deterministic).
 * ---------------------------------------------------------------------------------- */
/* empirical_fisher_finalize: keys[i] = (float)(score_sum[i] / (2 n_tokens)) for i < n (IEEE
 * float64 division, rounded to nearest float32): the scores as float32 sort keys for
 * score_and_allocate_keys, n_tokens the calibration tokens accumulated. */
KF_API kf_status empirical_fisher_finalize(kf_ctx* ctx, const double* score_sum, int64_t n, int64_t n_tokens,
                                           float* keys, kf_stream_t stream);
KF_API size_t empirical_fisher_workspace_size(int64_t m, int64_t n, int32_t r);
KF_API kf_status empirical_fisher_accumulate(kf_ctx* ctx, const void* act, kf_dtype act_dtype, int64_t lda,
                                             const void* grad, kf_dtype grad_dtype, int64_t ldg,
                                             int64_t n_tokens, int64_t m, int64_t n, const float* U,
                                             int64_t ldu, const float* V, int64_t ldv, int32_t r,
                                             double* score_sum, void* workspace, size_t workspace_bytes,
                                             kf_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Swift-SVD activation-only route (Swift-SVD 2A): the rank-k W_k minimising
 * ||A W - A W_k||_F is W V_k V_k^T, with V_k the top-k eigenvectors of the covariance of the
 * layer output C = (1/N) sum_t y_t^T y_t, y_t = a_t W; no gradient factor, no Cholesky.
 *
 * activation_covariance: C (n x n float32, ldc, full matrix) = W^T X W for the activation
 *   second moment X (m x m float32, ldx, full symmetric, e.g. kfac_accumulate's sum
 *   finalised with lambda = 0) and W (m x n, KF_BF16 or KF_F32).  Since
 *   sum_t (a_t W)^T (a_t W) = W^T (sum_t a_t^T a_t) W this is the output covariance, with the
 *   token stream read once per activation site (shared by every matrix reading that site).
 *   Tensor cores, float32 operands as three bfloat16 planes (float32-level accuracy).
 * activation_eig: eigenpairs of every C_i by the blocked Jacobi solver of whitened_svd
 *   applied to C itself (Rayleigh quotients q.Cq / q.q, windowed Rayleigh-Ritz refinement
 *   on C); sigma = sqrt(max(lambda, 0)) descending (the singular values of Y / sqrt(N)),
 *   vecs column i = the unit-norm eigenvector of sigma[i].  Same-n problems per call
 *   (n <= 16384); waits on the stream once per sweep like whitened_svd.
 * activation_factors: U = W V_r (m x r, tensor cores, W and V_r as hi + lo bfloat16 planes)
 *   and V = V_r^T (r x n), V_r the first r columns of vecs; U V = W V_r V_r^T.
 * The ranks come from score_and_allocate on the concatenated sigma (1/2 sigma^2 is half the
 * activation-aware loss increase per dropped component, m + n parameters per kept pair).
 * ---------------------------------------------------------------------------------- */
typedef struct {
  const float* C;    /* n x n, ldc (lower triangle read) */
  int64_t n, ldc;
  float* sigma;      /* n */
  float* vecs;       /* n x n, ldv */
  int64_t ldv;
  int32_t* sweeps;   /* device, may be NULL */
} kf_sym_problem;

KF_API size_t activation_covariance_workspace_size(int64_t m, int64_t n);
KF_API kf_status activation_covariance(kf_ctx* ctx, const float* X, int64_t ldx, int64_t m, const void* W,
                                       kf_dtype w_dtype, int64_t ldw, int64_t n, float* C, int64_t ldc,
                                       void* workspace, size_t workspace_bytes, kf_stream_t stream);
KF_API size_t activation_eig_workspace_size(int32_t n_problems, int64_t n);
KF_API kf_status activation_eig(kf_ctx* ctx, int32_t n_problems, const kf_sym_problem* problems, float tol,
                                int32_t max_sweeps, void* workspace, size_t workspace_bytes, kf_stream_t stream);
KF_API size_t activation_factors_workspace_size(int64_t m, int64_t n, int32_t r);
KF_API kf_status activation_factors(kf_ctx* ctx, const void* W, kf_dtype w_dtype, int64_t ldw, int64_t m, int64_t n,
                                    const float* vecs, int64_t ldv, int32_t r, float* U, int64_t ldu, float* V,
                                    int64_t ldvo, void* workspace, size_t workspace_bytes, kf_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Index plumbing for subsets chosen by a keep mask (the empirical-Fisher kept components, the
 * hybrid FFN's channel split).
 * gather_rows_cols: dst[i][j] = src[row_idx ? row_idx[i] : i][col_idx ? col_idx[j] : j] for
 *   i < rows, j < cols; src (src_rows x src_cols, lds) and dst (ldd) of the same dtype
 *   (KF_BF16 or KF_F32), indices device int64.  An index outside src writes 0 and sets
 *   KF_ERR_INVALID (info 151) in the status word.
 * compact_mask: idx[0 .. *count) = the positions p < n whose mask byte is nonzero (want = 1)
 *   or zero (want = 0), in increasing order; idx has room for n entries; count is device.
 * ---------------------------------------------------------------------------------- */
KF_API kf_status gather_rows_cols(kf_ctx* ctx, const void* src, kf_dtype dtype, int64_t lds, int64_t src_rows,
                                  int64_t src_cols, const int64_t* row_idx, int64_t rows, const int64_t* col_idx,
                                  int64_t cols, void* dst, int64_t ldd, kf_stream_t stream);
KF_API kf_status compact_mask(kf_ctx* ctx, const uint8_t* mask, int64_t n, int32_t want, int64_t* idx,
                              int64_t* count, kf_stream_t stream);

/* ------------------------------------------------------------------------------------
 * channel_errors - LASER's hybrid FFN channel selection (Hybrid SVD-quantisation for FFNs:
 * a temporary SVD of the gate and up projections finds the "SVD-friendly" hidden channels,
 * those it reconstructs with low error; the others stay dense).  For W (m x n, a gate or up
 * projection, column j = hidden channel j), the temporary factors U (m x r, ldu) and V
 * (r x n, ldv) and the input factor X (m x m float32, full symmetric):
 *   err_sum[j] += d_j^T X d_j,  d_j = (W - U V)[:, j]        (float64, deterministic)
 * the mean squared error of channel j's pre-activation over the calibration inputs.  Call it
 * for gate and then up with the same err_sum (zeroed first) so that the errors of a channel
 * add; keys (float[n], may be NULL) receives float(err_sum) after the addition.  Products on
 * the tensor cores with U, V, X and W - U V as three bfloat16 planes each.  r = 0 scores the
 * dense weight itself.  The split follows from score_and_allocate_keys on keys with one unit,
 * cost 1 per channel and budget = the number of dense channels: the kept mask marks the
 * dense channels (the largest errors; equal errors keep the lower index dense), the rest
 * are SVD-friendly.
 * ---------------------------------------------------------------------------------- */
KF_API size_t channel_errors_workspace_size(int64_t m, int64_t n, int32_t r);
KF_API kf_status channel_errors(kf_ctx* ctx, const void* W, kf_dtype w_dtype, int64_t ldw, int64_t m, int64_t n,
                                const float* U, int64_t ldu, const float* V, int64_t ldv, int32_t r,
                                const float* X, int64_t ldx, double* err_sum, float* keys, void* workspace,
                                size_t workspace_bytes, kf_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KFSVD_H */
