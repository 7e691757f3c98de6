/*
 * prm.h -- C ABI of libprm: the Periodic Row-wise Muon (PR-Muon) and MuonBP
 * optimizer step for the 2-D weight matrices of a model, on one GB300 GPU.
 *
 * Method sources (cited by title and section):
 *   [SMDiT]  "Scaling Muon for Diffusion Transformers": abstract, and the
 *            PaperDaily walkthrough of it -- section "Periodic Row-wise Muon"
 *            (Fig. 3 update rule with refresh indicator rho_t, Fig. 4 RowNorm
 *            R_eps), section "Distributed co-design" (Fig. 8 column statistics
 *            of tall matrices) and the cost note (NS5 Theta(5 r^2 c)).
 *   [MuonBP] "MuonBP: Faster Muon via Block-Periodic Orthogonalization",
 *            abstract (blockwise orthogonalisation, periodic full
 *            orthogonalisation, two step sizes).
 *
 * Conventions for every call:
 *   - Return value: PRM_OK (0) or one of the PRM_ERR_* codes below; no call
 *     throws, aborts or prints. prm_last_error() gives a one-line reason.
 *   - "device" pointers are CUDA global-memory addresses on the context's
 *     device; "host" pointers are ordinary CPU memory.
 *   - Ownership: the caller owns every tensor and the workspace. The library
 *     keeps non-owning pointers from prm_register_matrices / prm_set_workspace
 *     until the next registration or prm_destroy.
 *   - Streams are passed as `void*` holding a cudaStream_t (NULL = legacy
 *     default stream). Work is enqueued asynchronously; argument errors are
 *     returned at once, asynchronous CUDA errors on a later call or from
 *     prm_sync_status().
 *   - One context per stream; a context is not thread-safe.
 */
#ifndef PRM_H
#define PRM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PRM_API __attribute__((visibility("default")))
#else
#define PRM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define PRM_OK                 0
#define PRM_ERR_INVALID_ARG    1  /* null pointer, K < 1, t < 0, eps <= 0, beta outside [0,1), ... */
#define PRM_ERR_SHAPE          2  /* rows/cols < 1, MuonBP long side < blocks, pitch < cols */
#define PRM_ERR_ALIGNMENT      3  /* a pointer is not 16-byte aligned */
#define PRM_ERR_NOT_REGISTERED 4  /* step before prm_register_matrices / prm_set_workspace */
#define PRM_ERR_CUDA           5  /* a CUDA runtime or driver call failed */
#define PRM_ERR_TIMEOUT        6  /* a device-side bounded wait gave up (error word set) */
#define PRM_ERR_OOM            7  /* host allocation failed */
#define PRM_ERR_WORKSPACE      8  /* workspace missing or smaller than prm_workspace_bytes() */
#define PRM_ERR_UNSUPPORTED    9  /* no sm_100-family device, or a size beyond a kernel limit */

/* ---- enums ------------------------------------------------------------ */
#define PRM_FP32 0   /* gradient element type: float32 */
#define PRM_BF16 1   /* gradient element type: bfloat16 */
#define PRM_FP16 2   /* float16: the Gram-stage output of the standalone NS5 stages */

#define PRM_MODE_PRMUON 0   /* [SMDiT] Fig. 3: NS5 when t % K == 0, else gamma * R_eps */
#define PRM_MODE_MUONBP 1   /* [MuonBP]: full NS5 when t % K == 0, else NS5 per block */

typedef struct prm_ctx prm_ctx;

/* One 2-D weight matrix, stored row-major with rows x cols elements.
 *   param     float32, device, read and written in place (W).
 *   momentum  float32, device, read and written in place (M); starts at zero
 *             for a fresh run; together with t it is the whole optimizer state.
 *   grad      device, read only (G), element type grad_dtype.
 *   rows/cols m and n, both >= 1. m <= n is "wide" (rows are the short-side
 *             vectors), m > n is "tall" (columns are).
 *   shape_scale  per-matrix multiplier of the step size; <= 0 selects the
 *             default sqrt(max(1, rows / cols)).
 * All three pointers must be 16-byte aligned. */
typedef struct {
  float*      param;
  float*      momentum;
  const void* grad;
  int32_t     grad_dtype;
  int32_t     reserved;    /* must be 0 */
  int64_t     rows;
  int64_t     cols;
  float       shape_scale;
  float       reserved2;   /* must be 0 */
} prm_matrix_desc;

/* Creates a context bound to CUDA device `cuda_device` (must be compute
 * capability 10.3, sm_103a). *out receives the handle; free it with
 * prm_destroy. Errors: INVALID_ARG (out NULL), CUDA, UNSUPPORTED, OOM. */
PRM_API int prm_create(prm_ctx** out, int cuda_device);

/* Releases the context and its internal device tables. Never frees caller
 * buffers (tensors or workspace). NULL is accepted and ignored. */
PRM_API int prm_destroy(prm_ctx* ctx);

/* Registers `count` matrices (count >= 0; 0 clears the registration) and
 * plans the step: RowNorm launch groups by exact shape, NS5 groups by the
 * wide orientation r x c (tall matrices are orthogonalised transposed, as the
 * cost Theta(5 r^2 c) of [SMDiT]'s cost note implies), and -- when
 * muonbp_blocks = P > 0 -- the [MuonBP] blocks: P contiguous pieces along each
 * matrix's long side, the last taking the remainder. muonbp_blocks = 0
 * disables MuonBP mode for this registration.
 * The descriptor array is copied (host memory, read only).
 * Registration resets the workspace binding: call prm_set_workspace again.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, CUDA, OOM. */
PRM_API int prm_register_matrices(prm_ctx* ctx, const prm_matrix_desc* descs, int count,
                          int muonbp_blocks);

/* Caps the workspace that the next prm_register_matrices plans.
 *   max_bytes = SIZE_MAX: no cap -- every NS5 group's buffers are live at
 *     once and the five rounds of all groups run together (POLY once per
 *     short side r).
 *   max_bytes = 0 (the default): automatic -- plans up to 16 GiB stay whole;
 *     larger ones are split as with a 4 GiB cap (on the 15B-shaped DiT set
 *     this is ~10 % faster than one 75 GB plan, the power-capped SM clock
 *     running higher on the smaller per-launch working sets).
 *   otherwise: the refresh (and the MuonBP block step) is split into
 *     sequential sub-plans of whole matrices, each sized to fit `max_bytes`;
 *     a sub-plan holds at least one matrix, so a single matrix larger than
 *     the cap still gets the room it needs -- prm_workspace_bytes reports the
 *     actual need.
 * Results do not depend on the split. This is the single-GPU counterpart of
 * the bucketed refresh of [SMDiT] section "Distributed co-design" (at most a
 * bounded number of matrices materialised at a time). Errors: INVALID_ARG. */
PRM_API int prm_set_workspace_limit(prm_ctx* ctx, size_t max_bytes);

/* How the NS5 rounds of the next prm_register_matrices are evaluated. Both
 * forms compute the same five rounds X <- a X + (b A + c A A) X, A = X X^T,
 * of [SMDiT] section "Periodic Row-wise Muon"; they differ in rounding only.
 *   PRM_NS_FORM_AUTO (the default): NS5 groups whose wide shape r x c is
 *     wide enough for it to save at least 10 % of the executed flops
 *     (c >= 1.37 r at r = 2048, c >= 1.9 r for r <= 256; square matrices
 *     never) take the Gram route -- the rounds run in legs of at most
 *     three; a leg starts from an explicit X_s, iterates only r x r matrices
 *     (Q_j = P_j ... P_1 and T_j = Q_j X_s X_s^T, all symmetric, fp16 with
 *     fp32 accumulation) and ends with X_e = Q_L X_s. Per matrix a leg of L
 *     rounds costs 4 r^2 c + O(L r^3) flops instead of L (4 r^2 c + 2 r^3):
 *     for the five default rounds at r = 2048 about 40 % fewer executed
 *     flops on c = 4 r, 23 % on c = 2 r. The other groups, and every group
 *     when c = 0 in ns_coeffs, take the direct route.
 *   PRM_NS_FORM_DIRECT: every group evaluates the five rounds on X itself.
 * Errors: INVALID_ARG (unknown form). */
#define PRM_NS_FORM_AUTO   0
#define PRM_NS_FORM_DIRECT 1
PRM_API int prm_set_ns_form(prm_ctx* ctx, int form);

/* Pure helper: which NS5 evaluation the planner gives an m x n matrix under
 * `form`: 2 when the short side is below 64 (in either form: fp32 rounds on
 * CUDA cores, see below), 1 for the Gram route, 0 for the direct rounds on
 * tensor cores; -PRM_ERR_INVALID_ARG for m or n < 1 or an unknown form. (The
 * Gram route also needs c != 0 in ns_coeffs at step time.)
 *
 * Short sides below 64: such a matrix fills at most a quarter of the tensor
 * cores' 256-wide tile, and with so few elements the bf16 rounding of X and
 * of the r x r products no longer averages out. These matrices run the five
 * rounds A = X X^T, P = a I + b A + c A A, X <- P X in fp32 on CUDA cores
 * (sums in a fixed order), in both forms and in MuonBP block steps alike. */
PRM_API int prm_ns_route(int64_t m, int64_t n, int form);

/* Bytes of device scratch the registered plan needs (NS5 operands in bf16,
 * Gram / polynomial matrices, norm and column partial sums). *bytes (host)
 * receives the size; 0 when nothing is registered. */
PRM_API int prm_workspace_bytes(const prm_ctx* ctx, size_t* bytes);

/* Hands the library a caller-allocated device buffer of `bytes` bytes,
 * 256-byte aligned, at least prm_workspace_bytes(). Its contents need not be
 * initialised and are overwritten by every step. Errors: INVALID_ARG,
 * ALIGNMENT, WORKSPACE. */
PRM_API int prm_set_workspace(prm_ctx* ctx, void* dev_ptr, size_t bytes);

/* One optimizer step at index t over every registered matrix, enqueued on
 * `stream`:
 *   M <- beta * M + G                              (momentum)
 *   PRM_MODE_PRMUON ([SMDiT] Fig. 3 / Fig. 4):
 *     t % K == 0: D = NS5(M), eta = lr
 *     otherwise : D = R_eps(M), each short-side vector divided by
 *                 max(||v||_2, eps), eta = lr * gamma
 *   PRM_MODE_MUONBP ([MuonBP]): t % K == 0: D = NS5(M), eta = lr;
 *                 otherwise D = NS5 of each block on its own, eta = lr * gamma
 *   W <- W * (1 - lr * wd) - eta * s * D           (decoupled weight decay)
 * NS5: X = M / (||M||_F + 1e-7) (transposed if tall), then five rounds of
 * A = X X^T, B = b A + c A A, X <- a X + B X, in bf16 operands with fp32
 * accumulation (evaluated as X <- P X with P = a I + B formed as a completed
 * square, see the standalone stages below). ns_coeffs (host, 3 floats: a, b, c) may be NULL for the
 * default quintic (3.4445, -4.7750, 2.0315) -- the pages print no
 * coefficients, so this default is a stated choice.
 * Preconditions: t >= 0, K >= 1 (K = 1 is vanilla Muon), 0 <= beta < 1,
 * eps > 0, finite lr / wd / gamma. Errors: INVALID_ARG, NOT_REGISTERED,
 * WORKSPACE, CUDA (launch failures). A device-side wait that gave up is
 * reported by prm_sync_status(), not here (reading it needs a sync).
 * A step is not atomic: when a CUDA error comes back, the kernels enqueued
 * before the failing launch still run, so some matrices may hold the updated
 * W and M and others the old ones; re-running the step would apply the
 * momentum twice to the former. Every step reuses the one workspace, so
 * steps on different streams must be ordered by the caller (events). */
PRM_API int prm_step(prm_ctx* ctx, int64_t t, int K, float gamma, float lr, float wd, float beta,
             float eps, const float* ns_coeffs, int mode, void* stream);

/* Pure helper: 1 if step t takes the refresh / full-NS5 branch, 0 if it takes
 * the RowNorm / block branch ([SMDiT] Fig. 3 refresh indicator; the same rule
 * in both modes). Returns -PRM_ERR_INVALID_ARG for t < 0, K < 1 or an unknown
 * mode. */
PRM_API int prm_branch(int64_t t, int K, int mode);

/* Synchronises `stream` and reads the device error word that bounded waits
 * inside the NS5 kernels set when they give up. Returns PRM_OK, TIMEOUT or
 * CUDA; clears the word. */
PRM_API int prm_sync_status(prm_ctx* ctx, void* stream);

/* Test and debugging aid: writes to host_out (host, rows * cols floats,
 * row-major) the direction D of the most recent prm_step for registered
 * matrix `idx` -- NS5(M_t) on a refresh / full step, the NS5 of each MuonBP
 * block on a block step, R_eps(M_t) on a RowNorm step ([SMDiT] Fig. 3 and
 * Fig. 4), before the step size s * eta is applied. D is recomputed from the
 * matrix's momentum with the step's own kernels, so the momentum must still
 * hold M_t: call it before the next step and before anything else writes the
 * momentum. The NS5 directions are recomputed by the step's own (deterministic)
 * kernels from the same momentum, so they are the bf16 values the step applied;
 * the RowNorm direction is the fp32 quotient M / max(||v||, eps), which the
 * step folds into one coefficient with s * eta. Synchronises the device,
 * allocates and frees its own scratch (the matrix's size twice, plus the NS5
 * workspace of that one matrix) and runs on the legacy default stream; not
 * for use inside a stream capture. Errors: INVALID_ARG (NULL, idx out of
 * range, no step since registration), NOT_REGISTERED, OOM, CUDA, TIMEOUT. */
PRM_API int prm_debug_last_direction(prm_ctx* ctx, int idx, float* host_out);

/* Test aid for the bounded waits: in the next RowNorm step, the one-launch
 * tall-matrix kernel does not publish the inverse column norms of column
 * stripe `stripe` (stripes of 128 columns, numbered across the tall matrices
 * of one shape in registration order; a stripe beyond them withholds
 * nothing), so that stripe's update tiles wait wait_limit_s seconds (in
 * (0, 2]) for a flag that nothing sets, give up and leave that stripe of W
 * unchanged; prm_sync_status then reports PRM_ERR_TIMEOUT and the context
 * stays usable. The momentum update of the step completes. No effect on
 * refresh steps (it stays armed for the next RowNorm step) or on views that
 * take the three-launch form. Errors: INVALID_ARG. */
PRM_API int prm_debug_withhold_tall_norms(prm_ctx* ctx, int stripe, double wait_limit_s);

/* ---- allocation-free RowNorm step for one tall matrix -------------------
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory when the update runs (a host process whose
 * allocator owns all device memory and refuses new allocations mid-step, an
 * integration that cannot afford cudaMalloc's implicit synchronisation, a
 * plugin that only receives the tensors it updates). It performs the same
 * RowNorm step as prm_step does for a tall matrix on a non-refresh step
 * (momentum, column norms, update; fp32 parameter and momentum updated in
 * place, gradient fp32 or bf16, all row-major and contiguous on the current
 * device), but takes its scratch from a fixed 4 MiB array compiled into the
 * library instead of a workspace: it calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   Limits: rows > cols (tall), ceil(rows / 256) * cols + cols <= 1,048,576
 *   floats (e.g. up to 32768 x 4096 or 20480 x 5120); larger shapes return
 *   PRM_ERR_UNSUPPORTED. shape_scale <= 0 selects sqrt(rows / cols).
 *   Every call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress, which allocates nothing); the first call on a
 *   device also loads the library's device code there, so make that first
 *   call before any stream capture. Every call shares the array and finds
 *   the previous call's contents in it (each call writes every element it
 *   reads before reading it): calls whose work may overlap on the GPU (other
 *   streams, unordered host threads) race and must not be issued.
 *   Errors: INVALID_ARG, SHAPE, UNSUPPORTED, CUDA. */
PRM_API int prm_rownorm_tall_step_noalloc(float* param, float* momentum, const void* grad,
                                          int grad_dtype, int64_t rows, int64_t cols, float gamma,
                                          float lr, float wd, float beta, float eps,
                                          float shape_scale, void* stream);

/* ---- AdamW for the non-matrix parameters -----------------------------
 * [SMDiT] (scaling-study section) keeps biases, normalisation parameters and
 * other non-matrix parameters on AdamW; its reference [3] (Loshchilov and
 * Hutter) is decoupled weight decay. The pages print no formula; this is the
 * plain reading of that reference:
 *   m <- b1 m + (1 - b1) g ;  v <- b2 v + (1 - b2) g^2
 *   p <- p (1 - lr wd) - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
 * over `n` elements of flat device buffers: param, exp_avg (m), exp_avg_sq (v)
 * fp32, updated in place; grad (read only) fp32 or bf16 per grad_dtype.
 * t >= 1 counts steps from 1 (bias correction). Hyper-parameters are doubles:
 * 1 - b1, 1 - b2 and the bias corrections are formed in double on the host
 * and rounded once to fp32. Any n >= 0 and any alignment
 * (16-byte aligned buffers take the vector path). Asynchronous on `stream`.
 * Errors: INVALID_ARG (t < 1, n < 0, NULL pointer with n > 0, b1 / b2 outside
 * [0, 1), eps <= 0, non-finite lr / wd), CUDA. */
PRM_API int prm_adamw_step(float* param, float* exp_avg, float* exp_avg_sq, const void* grad,
                           int grad_dtype, int64_t n, int64_t t, double lr, double beta1, double beta2,
                           double eps, double wd, void* stream);

/* ---- kernel timing (benchmarks) --------------------------------------
 * When enabled, every kernel family launched by prm_step is bracketed by a
 * pair of CUDA events recorded on the launching stream, and its algorithmic
 * work is accumulated: for the GEMM families the FLOPs they execute --
 * 2 M N K per matrix for COMBINE; for the symmetric r x r outputs (GRAM,
 * POLY and the Gram route's updates) the share of 2 r r K that their upper
 * 256 x 256 super-blocks cover, nb (nb + 1) / 2 of nb^2 with
 * nb = ceil(r / 256) (36 / 64 at r = 2048; the lower ones are mirrored, not
 * multiplied); for the fp32 rounds of short sides below 64 the FLOPs of
 * their Gram pairs, P X and P; bytes for the memory-bound ones (RowNorm
 * 18 B per parameter with bf16 gradients, 20 B with fp32; prep 12 / 14 B).
 * The refresh's parameter update runs in the epilogue of the last COMBINE
 * launch and is timed with it. Families: */
#define PRM_FAMILY_ROWNORM_WIDE 0
#define PRM_FAMILY_ROWNORM_TALL 1
#define PRM_FAMILY_NS_PREP      2
#define PRM_FAMILY_NS_GRAM      3
#define PRM_FAMILY_NS_POLY      4
#define PRM_FAMILY_NS_COMBINE   5
#define PRM_FAMILY_NS_SYM       6  /* Gram route: Q <- P Q, T <- P T */
#define PRM_FAMILY_NS_SMALL     7  /* NS5 of short sides below 64 (fp32, CUDA cores; executed flops) */
#define PRM_FAMILY_COUNT        8

/* enable = 1 clears the records and starts recording; 0 stops. */
PRM_API int prm_profile(prm_ctx* ctx, int enable);

/* Totals since the last prm_profile(ctx, 1) for one family (or -1 for all):
 * *total_ms summed event time, *records bracketed launches of that family,
 * *kernels individual kernel launches inside them, *work the algorithmic
 * FLOPs or bytes. Waits for the recorded events (host-blocking). */
PRM_API int prm_profile_read(prm_ctx* ctx, int family, double* total_ms, int64_t* records,
                             int64_t* kernels, double* work);

/* Last error message of this context (or of the last failed prm_create when
 * ctx is NULL). Never NULL; owned by the library. */
PRM_API const char* prm_last_error(const prm_ctx* ctx);

/* ---- standalone building blocks ---------------------------------------
 * The stages of NS5 on caller buffers, for users who want the orthogonaliser
 * without the optimizer state, and for kernel-level tests. A batch holds
 * `batch` matrices of r x c (r <= c) bf16 values stored row-major with row
 * pitch `ldc` elements (ldc >= c, ldc % 8 == 0), matrix i at offset
 * i * r * ldc; r x r matrices use pitch `ldr` (ldr >= r, ldr % 8 == 0).
 * All pointers are device, 16-byte aligned; bf16 values are passed as
 * uint16_t bit patterns. `scale` (device, batch floats) may be NULL for 1.
 * [SMDiT] section "Periodic Row-wise Muon": one NS5 round is
 * A = X X^T, B = b A + c A A, X' = a X + B X. The library evaluates it as
 * X' = P X with P = a I + b A + c A A written as a completed square: for
 * c != 0, C = sqrt|c| A + sgn(c) b / (2 sqrt|c|) I and
 * P = sgn(c) C C + (a - b^2 / (4c)) I (exact: C is a polynomial in A); for
 * c = 0, P = b A + a I comes straight from the Gram stage. The three calls
 * below are those stages:
 *   prm_ns_gram(gain = sqrt|c|, diag = sgn(c) b / (2 sqrt|c|), PRM_FP16) -> C
 *   prm_ns_poly(gain = sgn(c), diag = a - b^2 / (4c), PRM_FP16)          -> P
 *   prm_ns_combine                                                       -> X'
 * (for c = 0: prm_ns_gram(gain = b, diag = a, PRM_BF16) -> P, then
 * prm_ns_combine). C is kept in fp16: its diagonal holds the shift
 * b / (2 sqrt|c|), next to which bf16 would lose most of sqrt|c| A_ii. */

/* C[i] = gain * scale[i]^2 * X[i] X[i]^T + diag * I  (symmetric; tensor
 * cores, tcgen05), written as out_dtype (PRM_BF16 or PRM_FP16). Errors:
 * INVALID_ARG (also non-finite gain / diag, other out_dtype), ALIGNMENT,
 * CUDA, UNSUPPORTED. */
PRM_API int prm_ns_gram(const uint16_t* X, uint16_t* C, const float* scale, float gain, float diag,
                int out_dtype, int batch, int64_t r, int64_t c, int64_t ldc, int64_t ldr, void* stream);

/* P[i] = gain * C[i] C[i] + diag * I   (C symmetric, of type in_dtype:
 * PRM_BF16 or PRM_FP16; P bf16, must not alias C). */
PRM_API int prm_ns_poly(const uint16_t* C, uint16_t* P, float gain, float diag, int in_dtype, int batch,
                int64_t r, int64_t ldr, void* stream);

/* Xout[i] = scale[i] * P[i] X[i]  (Xout must not alias X). */
PRM_API int prm_ns_combine(const uint16_t* X, const uint16_t* P, uint16_t* Xout, const float* scale,
                   int batch, int64_t r, int64_t c, int64_t ldc, int64_t ldr, void* stream);

/* Bytes of workspace prm_newton_schulz needs for `batch` matrices of m x n. */
PRM_API int prm_newton_schulz_workspace(int batch, int64_t m, int64_t n, size_t* bytes);

/* out[i] = NS_steps(in[i]) for `batch` fp32 matrices of m x n (row-major,
 * contiguous, device), tall inputs orthogonalised transposed; the result is
 * fp32. steps >= 1, ns_coeffs NULL for the default quintic. Evaluated in the
 * PRM_NS_FORM_AUTO form (prm_set_ns_form): shapes wide enough take the Gram
 * route, in legs of at most three rounds. The call synchronises `stream`
 * before returning (its launch tables are freed). */
PRM_API int prm_newton_schulz(const float* in, float* out, int batch, int64_t m, int64_t n,
                      const float* ns_coeffs, int steps, void* workspace, size_t ws_bytes,
                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PRM_H */
