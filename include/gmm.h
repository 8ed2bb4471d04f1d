/*
 * gmm.h -- C ABI of the B300 (sm_103a) GMM EM-step library.
 *
 * One call runs one Expectation-Maximization iteration of a Gaussian mixture
 * with spherical or diagonal covariance over N points in D dimensions and K
 * components, without ever storing the N x K responsibility matrix: memory
 * beyond X is O(K * D) (plus O(N) floats when K > 1024, see gmm_em_step).
 * A second call returns every point's m largest responsibilities.
 *
 * The method (web pages it is described on):
 *  - "Flash-GMM: A Memory-Efficient Kernel for Scalable Soft Clustering",
 *    section 2: mixture density, E-step responsibilities in log space
 *    (log-sum-exp), M-step for N_k, pi_k, mu_k and the variance; section 3:
 *    the N x K responsibility matrix is what a naive GPU EM must store and
 *    re-read; conclusion: multi-assignment from the final responsibilities.
 *  - "ML0094 GMM vs K-Means": EM steps, soft assignment.
 *  - "GMMXX" README, "Covariance Coverage": parameter shapes (K,) for
 *    spherical and (K, D) for diagonal variances.
 *
 * Conventions for every entry point
 *  - X is row-major N x D, contiguous, on the device, either float32 or
 *    bfloat16 (x_dtype).  Its base address must be 16-byte aligned.
 *  - Parameters are float32 device arrays: log_weights (K), means (K x D
 *    row-major), vars (K for spherical, K x D for diagonal).  Log-weights need
 *    not be normalised; a log-weight of -inf marks a dead component.
 *  - All array arguments are caller-owned device pointers unless stated; the
 *    library never frees them.  Work is enqueued on `stream` (a cudaStream_t,
 *    NULL = legacy default stream) and the call returns without waiting,
 *    unless opts->loglik_on_host is set.
 *  - The library keeps one internal workspace per device (O(K * D) bytes
 *    times the number of SMs, plus O(N) floats when K > 1024, plus, for a
 *    tied covariance of bf16 data, one D x D float matrix per 8192 rows).  It is grown
 *    on demand with cudaMalloc, so a call that needs a bigger workspace
 *    synchronises the device first; gmm_workspace_bytes() reports the size
 *    and gmm_reserve() allocates it up front.  Calls on different streams of
 *    one device must not overlap in time (they share the workspace).
 *  - Return value: GMM_OK (0) or a negative gmm_status_t.  Argument errors are
 *    found on the host before anything is enqueued.  Device-side conditions
 *    (non-finite or non-positive parameters, a synchronisation wait that ran
 *    out) are recorded in a device status word; they are returned by the call
 *    itself when it synchronises (loglik_on_host), otherwise by
 *    gmm_stream_status().  gmm_last_error() gives the message of the last
 *    failure on the calling thread.  There is no fallback path: a failure is
 *    reported, never silently computed another way.
 */
#ifndef GMM_B300_H
#define GMM_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Covariance types.  TIED: one full D x D covariance shared by all
 * components ("GMMXX" README, "Covariance Coverage": tied, shape (D, D));
 * vars / new_vars are then that D x D matrix (row-major, symmetric positive
 * definite).  gmm_em_step, gmm_predict_topm and gmm_assign_threshold take
 * all three; gmm_em_step_host and gmm_em_step_noalloc take SPHERICAL and
 * DIAG. */
typedef enum { GMM_SPHERICAL = 0, GMM_DIAG = 1, GMM_TIED = 2 } gmm_cov_t;
typedef enum { GMM_F32 = 0, GMM_BF16 = 1 } gmm_dtype_t;

/* Arithmetic of the two tensor-core contractions (logits and statistics).
 *  FAST:    half-precision (fp16) operands with fp32 accumulation, one pass.
 *           Data are scaled by a power of two so that |x|^2 fits fp16 (bf16
 *           data then stay exact); float32 data are also shifted by the mean
 *           of the component means.
 *  PRECISE: every operand split into two fp16 parts (hi + lo, 22 significant
 *           bits), three products per contraction (hi*hi + hi*lo + lo*hi),
 *           fp32 accumulation; data shifted and scaled as above.
 *  AUTO:    FAST for bf16 X, PRECISE for float32 X. */
typedef enum { GMM_PREC_AUTO = 0, GMM_PREC_FAST = 1, GMM_PREC_PRECISE = 2 } gmm_precision_t;

typedef enum {
    GMM_OK = 0,
    GMM_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, N < 1, D < 1, ... */
    GMM_ERR_UNSUPPORTED = -2,   /* a shape outside the supported window */
    GMM_ERR_NONFINITE = -3,     /* a parameter is NaN/inf, or a variance <= 0 */
    GMM_ERR_CUDA = -4,          /* a CUDA runtime call failed */
    GMM_ERR_TIMEOUT = -5,       /* a device-side wait exceeded its bound */
    GMM_ERR_RANGE = -6,         /* data too large for the FAST operand range */
    GMM_ERR_CAPACITY = -7       /* gmm_assign_threshold: more entries than the output holds */
} gmm_status_t;

/* Launch plan of one EM step (or top-m pass).
 *  CLUSTER: one pass over X; the CTAs that hold the 128-component slices of
 *           one point tile form a thread-block cluster and exchange their
 *           per-row normalisers through distributed shared memory
 *           (K <= 1024; above that, the normaliser pass below runs with
 *           clusters of 8 slices and per-cluster partial normalisers).
 *  SPLIT:   two passes; the first computes every slice's per-row normaliser
 *           independently (no clusters) into an N x slices buffer, a small
 *           kernel combines them, and the second pass recomputes the logits
 *           and accumulates the statistics with the normaliser read from
 *           memory.  1.5 times the tensor-core work, no cross-CTA waits,
 *           N * ceil(K / 128) + N extra floats of workspace.
 *  AUTO:    CLUSTER for K <= 1024.  Above that the EM step takes two passes
 *           either way, and AUTO runs its normaliser pass as in SPLIT (no
 *           clusters) when the N x ceil(K / 128) normalisers fit in 4 GiB,
 *           else in clusters of 8; the top-m pass keeps clusters of 8. */
typedef enum { GMM_PLAN_AUTO = 0, GMM_PLAN_CLUSTER = 1, GMM_PLAN_SPLIT = 2 } gmm_plan_t;

typedef struct {
    int32_t precision;       /* gmm_precision_t, default AUTO */
    float reg_covar;         /* added to every new variance, default 1e-6 */
    float var_floor;         /* new variance = max(v, var_floor) + reg_covar, default 0 */
    float x_absmax;          /* > 0: caller's bound on max |X| (skips a scan of X) */
    int32_t loglik_on_host;  /* 1: total_loglik is a host pointer; the call waits
                                for the stream and reports device-side errors */
    int32_t plan;            /* gmm_plan_t, default AUTO */
    int32_t wait_limit;      /* polls each device-side wait makes before it gives
                                up and the call reports GMM_ERR_TIMEOUT; 0 (the
                                default) = about 4 million (a few seconds).  Small
                                values exist to test the failure path. */
    int32_t approx_top_k;    /* gmm_em_step only: 0 (the default) or >= K = exact
                                EM; 1 <= k < K: approximate top-k EM (see
                                gmm_em_step) */
    int32_t topm_refine;     /* gmm_refine_t, default AUTO: the direct-form
                                refinement of the top-m candidates (see
                                gmm_predict_topm) */
} gmm_opts;

/* Refinement of the top-m candidates (gmm_predict_topm, gmm_assign_threshold,
 * approximate top-k EM).  AUTO: on for PRECISE, off for FAST.  The
 * refinement gathers each candidate's (mu, 1/s2) row, 8 bytes per feature,
 * candidate and point (from L2), which on 10M x 128 bf16 points with m = 4
 * adds about 2.5 ms to a 22 ms FAST pass.  It needs a further 1 KB per
 * component of workspace. */
typedef enum { GMM_REFINE_AUTO = 0, GMM_REFINE_ON = 1, GMM_REFINE_OFF = 2 } gmm_refine_t;

/* Fill *opts with the defaults listed above. */
void gmm_default_opts(gmm_opts *opts);

/*
 * One EM iteration ("Flash-GMM", section 2; "ML0094 GMM vs K-Means").
 *   E-step: r_ik = pi_k N(x_i | mu_k, Sigma_k) / sum_j pi_j N(x_i | mu_j, Sigma_j)
 *   M-step: N_k = sum_i r_ik;  new log-weight = log(N_k / N);
 *           new mean mu_k' = sum_i r_ik x_i / N_k;
 *           diagonal:  s2_kd' = sum_i r_ik (x_id - mu_kd')^2 / N_k
 *           spherical: s2_k'  = sum_i r_ik ||x_i - mu_k'||^2 / (D N_k)
 *           tied:      Sigma' = sum_k sum_i r_ik (x_i - mu_k')(x_i - mu_k')^T / N
 *           then s2' = max(s2', var_floor) + reg_covar (tied: on the
 *           diagonal of Sigma').
 *   A component with N_k < 1e-30 keeps its mean and variance (tied: its
 *   mean; it adds nothing to Sigma'); its new log-weight is -inf.
 *   total_loglik = sum_i log sum_k pi_k N(x_i | mu_k, Sigma_k), evaluated at
 *   the INPUT parameters (a by-product of the E-step), as one double; a
 *   device pointer unless opts->loglik_on_host.
 * Outputs may alias the corresponding inputs (all inputs are consumed before
 * the first output is written).  Statistics are reduced in a fixed order:
 * repeated calls give bit-identical results.
 * Supported: 1 <= D <= 128, 1 <= K <= 8192 (K <= 1024 in a single pass over
 * X; above that the E-step's normaliser is computed in a first pass and kept
 * in an N-float buffer), N >= 1.  PRECISE at D > 64 reads the parameter
 * image again for every 128-point tile (it does not fit on chip beside the
 * data); it is slower per element than at D <= 64.
 *
 * Approximate top-k EM (opts->approx_top_k = k, 1 <= k < K; the "GMMXX"
 * README's training option approx_top_k): each point keeps its k largest
 * logits l_ik and its responsibilities are normalised over those k only,
 *   r_ik = exp(l_ik) / sum_{j kept} exp(l_ij)  (0 for the others),
 * equal logits kept by the lower index first; the M-step above then runs
 * with these responsibilities.  total_loglik stays the exact one (all K
 * components).  The E-step is the top-m pass of gmm_predict_topm (m = k,
 * same arithmetic); the statistics are gathered per component in point
 * order (bit-identical on repeated calls), the variance in a second pass
 * over the kept pairs.  Needs k <= 16, N < 2^31, SPHERICAL or DIAG, and a
 * workspace of about 16 N k bytes more.
 */
int gmm_em_step(const void *X, int64_t N, int32_t D, int32_t K, int32_t cov_type,
                int32_t x_dtype, const float *log_weights, const float *means,
                const float *vars, float *new_log_weights, float *new_means,
                float *new_vars, double *total_loglik, const gmm_opts *opts,
                void *stream);

/*
 * Top-m soft assignment (the multi-assignment of "Flash-GMM", conclusion:
 * boundary vectors go to several posting lists, read off the final
 * responsibilities).  For every point i, resp_out[i*m + j] and
 * idx_out[i*m + j] (j < m) are its j-th largest responsibility r_ik
 * (normalised over all K components, not over the m kept) and the component
 * index k, in descending order of r; equal responsibilities are ordered by
 * the lower index first.  m = 1 is the hard label (predict).  total_loglik
 * (may be NULL) receives sum_i log p(x_i) as in gmm_em_step.
 * Two stages.  The tensor-core pass selects each point's m candidates from
 * the expanded-form logits and normalises over all K.  When refinement is on
 * (opts->topm_refine) and the covariance is SPHERICAL or DIAG, the
 * candidates' logits are then recomputed in fp32 from the direct form  log pi_k - 1/2 sum_d [log(2 pi s2_kd) + (x_d - mu_kd)^2 / s2_kd]
 * ("Flash-GMM", section 2), the candidates' total share R (the sum of their
 * responsibilities from the pass) is divided among them by these logits,
 * the list is sorted again, and total_loglik becomes
 * sum_i [log sum_{j kept} exp(l_ij) - log R_i].  The direct form does not
 * lose the digits that the expanded form cancels away at sharply fitted
 * components (|x|^2 / s2 large).  Which components are kept is the pass's.
 * gmm_em_step with approx_top_k and gmm_assign_threshold run the same two
 * stages.
 * Supported: 1 <= m <= min(K, 16); other limits as gmm_em_step.
 */
int gmm_predict_topm(const void *X, int64_t N, int32_t D, int32_t K, int32_t cov_type,
                     int32_t x_dtype, const float *log_weights, const float *means,
                     const float *vars, int32_t m, float *resp_out, int32_t *idx_out,
                     double *total_loglik, const gmm_opts *opts, void *stream);

/*
 * Threshold multi-assignment ("Flash-GMM", conclusion: border vectors are
 * assigned to several clusters using the responsibilities), as compressed
 * rows for posting lists: every (point, component) pair whose responsibility
 * reaches a threshold.
 *   For every point i, the components k with r_ik >= tau among the point's
 *   max_per_point largest responsibilities, in descending order of r (equal
 *   values: lower k first).  When tau > 1 / (max_per_point + 1) this is every
 *   k with r_ik >= tau, since the responsibilities of a point sum to one.
 *   offsets (N + 1 int64, device): point i's entries are
 *   [offsets[i], offsets[i+1]); offsets[N] is the total.  idx_out (int32) and
 *   resp_out (float32), device, hold `capacity` entries.  If the total
 *   exceeds capacity, offsets are still written, the entries are not, and
 *   the device status reports GMM_ERR_CAPACITY (read offsets[N] and call
 *   again with room for it).
 * Supported: 0 < tau <= 1, 1 <= max_per_point <= min(K, 16); other limits
 * as gmm_predict_topm.  The total log-likelihood is not computed.
 */
int gmm_assign_threshold(const void *X, int64_t N, int32_t D, int32_t K, int32_t cov_type,
                         int32_t x_dtype, const float *log_weights, const float *means,
                         const float *vars, float tau, int32_t max_per_point, int64_t *offsets,
                         int32_t *idx_out, float *resp_out, int64_t capacity,
                         const gmm_opts *opts, void *stream);

/*
 * gmm_em_step_host -- the same EM step as gmm_em_step for X held in HOST
 * memory, possibly larger than the GPU's ("Flash-GMM", introduction and
 * contributions: the kernel's memory does not grow with N, so the data set
 * may exceed the device; streaming X in chunks is this library's way of
 * feeding such a data set).
 *  - X_host: row-major N x D (x_dtype), contiguous, in host memory; it should
 *    be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to run
 *    asynchronously.  Parameters and outputs are device pointers exactly as
 *    for gmm_em_step; they may alias the same way.
 *  - The rows go to the GPU in chunks of chunk_rows rows (rounded down to a
 *    multiple of 128; 0 picks 1,048,576) through two device staging buffers:
 *    chunk c + 1 is copied on an internal stream while chunk c is processed
 *    on `stream`.  The statistics of all chunks add into the same partials,
 *    so the result equals one gmm_em_step over all N rows up to the order of
 *    the floating-point sums.
 *  - opts->x_absmax > 0 is required: the FAST operand scale must be fixed
 *    before the first chunk is seen (GMM_ERR_INVALID_ARG otherwise).
 *  - The workspace grows by two staging buffers of chunk_rows rows.  The
 *    host buffer must stay valid and unchanged until the stream has passed
 *    this call.  Error behaviour as gmm_em_step.
 */
int gmm_em_step_host(const void *X_host, int64_t N, int32_t D, int32_t K, int32_t cov_type,
                     int32_t x_dtype, const float *log_weights, const float *means,
                     const float *vars, float *new_log_weights, float *new_means,
                     float *new_vars, double *total_loglik, int64_t chunk_rows,
                     const gmm_opts *opts, void *stream);

/*
 * gmm_em_step_noalloc -- the same EM step as gmm_em_step, for callers that
 * cannot allocate device memory while they run: for example a process whose
 * device memory is handed out up front by its own allocator, or a code path
 * that must not call cudaMalloc/cudaFree because those calls can synchronise
 * the whole device.  The web pages describing the method have no counterpart
 * of this entry point.
 *  - Allocates nothing.  All scratch comes from one 24 MiB array compiled into
 *    this library; every GPU that loads the library keeps those 24 MiB
 *    reserved until the process exits.  The caller passes inputs and outputs
 *    exactly as for gmm_em_step.
 *  - Limits: K <= 1024 (larger K needs an N-sized buffer) and the statistics
 *    of the problem must fit the array; when they fit only partly the step
 *    runs on fewer thread blocks (gmm_plan_info reports how many: at D = 128,
 *    K = 1024 the array holds 11 of the 15 tile groups of a B300).  Larger problems are rejected with
 *    GMM_ERR_UNSUPPORTED and a message in gmm_last_error().
 *  - The first call with a given device current looks up the array's device
 *    address (cudaGetSymbolAddress) and sets kernel attributes; make that
 *    first call before any stream capture.
 *  - All calls share the one array, and it keeps the last call's contents
 *    (each call clears the parts that must start at zero).  Calls whose work
 *    overlaps on the GPU, on any streams, race on that array: serialise them.
 *  - Device-side conditions (non-finite parameters, timeouts) are reported
 *    only when opts->loglik_on_host is set (the call then waits for the
 *    stream); gmm_stream_status() does not see them.
 */
int gmm_em_step_noalloc(const void *X, int64_t N, int32_t D, int32_t K, int32_t cov_type,
                        int32_t x_dtype, const float *log_weights, const float *means,
                        const float *vars, float *new_log_weights, float *new_means,
                        float *new_vars, double *total_loglik, const gmm_opts *opts,
                        void *stream);

/* Bytes of internal workspace a call with these arguments needs. */
size_t gmm_workspace_bytes(int64_t N, int32_t D, int32_t K, int32_t cov_type,
                           int32_t x_dtype, const gmm_opts *opts);

/* Allocate the workspace for such calls now (on the current device). */
int gmm_reserve(int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                const gmm_opts *opts);

/* Wait for `stream` and return the device-side status of the calls enqueued
 * on it so far (GMM_OK, GMM_ERR_NONFINITE, GMM_ERR_TIMEOUT, GMM_ERR_RANGE),
 * then clear it. */
int gmm_stream_status(void *stream);

/* Message of the last failure on the calling thread ("" if none). */
const char *gmm_last_error(void);

/* Free the internal workspace of every device (call when idle). */
void gmm_release(void);

/* Launch plan of an EM step with these arguments on the current device (for
 * measurement and tests; no work is enqueued).  Fills info[0..7]:
 *   [0] CTAs per thread-block cluster (component slices sharing a point tile;
 *       two-pass plan: of the EM step's normaliser pass)
 *   [1] tile groups of the statistics pass (co-resident clusters, or CTAs per
 *       slice in the two-pass plan)
 *   [2] 1 when the step takes two passes (K > 1024, or plan SPLIT)
 *   [3] tile groups of the normaliser pass (two-pass plan; else 0)
 *   [4] tiles between flushes of the statistics from tensor memory
 *   [5] threads per CTA of the E-step kernel
 *   [6] tile groups gmm_em_step_noalloc would use (its scratch array holds the
 *       per-group statistics; 0 where that entry point refuses the shape)
 *   [7] 128-point tiles of the data set
 * info is a host array of at least 8 int32.  Returns GMM_OK or an error code. */
int gmm_plan_info(int64_t N, int32_t D, int32_t K, int32_t cov_type, int32_t x_dtype,
                  const gmm_opts *opts, int32_t *info);

/* Number of kernel launches the last successful call enqueued. */
int32_t gmm_last_launch_count(void);

/* Timing of the main (fused E-step + statistics) kernel, for measurement:
 * after gmm_profile_begin(), each call on this thread records a CUDA event
 * pair around every launch of that kernel on its stream; gmm_profile_end()
 * waits for those events and returns the summed device time in milliseconds
 * and the number of launches, then stops recording. */
void gmm_profile_begin(void);
int gmm_profile_end(double *main_kernel_ms, int32_t *launches);

#ifdef __cplusplus
}
#endif
#endif /* GMM_B300_H */
