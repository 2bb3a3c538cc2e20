/*
 * dyra.h -- C ABI of the B300 (sm_103a) DyRA linear layer.
 *
 * The layer approximates Y = X W + b by
 *
 *     Y ~= X W_hat + b + L R,        L = X P,   R = (L^T L + lambda I)^-1 (L^T X) W_res
 *
 * W_hat is a static structured approximation of W (truncated-SVD low rank U V, or
 * Monarch), W_res = W - W_hat, P = W_res R0^T (R0 R0^T)^-1 is fixed offline, and R is
 * recomputed for every sample by one alternating-least-squares step.
 *
 * Sources: "DyRA: Dynamic Residual Approximation for Efficient Matrix Multiplication in
 * DNNs" -- section-by-section summary page: 2.2 (dynamic residual approximation, ridge),
 * 2.3 (one-step ALS, Proposition 1, cost), 2.4 (fused kernels, Cholesky for small r and
 * Newton-Schulz for larger r), Appendix B (truncated SVD, Monarch); and the blog digest
 * "DyRA：用输入相关的残差修正加速大模型的矩阵乘法": residual-split equations
 * (W = W_hat + W_res, XW = X W_hat + X W_res), the rank-r objective
 * min ||X W_res - L R||_F^2 with the ALS order of operations, the one-step form
 * XW ~ X W_hat + L(1) R(1), and the offline / online flow (R0 = top right singular vectors
 * of W_res, prepared once).
 *
 * Conventions for every call:
 *   - All matrices are row-major. X is [batch, n, d], Y is [batch, n, m].
 *   - "host" pointers are ordinary CPU memory; "device" pointers are CUDA global memory
 *     of the layer's device. The library never takes ownership of a caller pointer.
 *   - A call that returns an error status has launched nothing and changed no caller
 *     buffer, except where stated. Nothing prints, exits or traps.
 *   - Every forward call is asynchronous on the caller's stream and allocates nothing.
 */
#ifndef DYRA_H_
#define DYRA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DYRA_ABI_VERSION 3

typedef enum dyra_status {
  DYRA_OK = 0,
  DYRA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shapes            */
  DYRA_ERR_UNSUPPORTED = 2,   /* valid request that this library does not implement     */
  DYRA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (see dyra_last_error) */
  DYRA_ERR_OOM = 4,           /* device or host allocation failed in dyra_prepare       */
  DYRA_ERR_NOT_SPD = 5,       /* reported by dyra_workspace_status: some L^T L + lambda I
                                 was not positive definite                               */
  DYRA_ERR_TIMEOUT = 6,       /* a bounded in-kernel wait gave up (kernel returned early) */
  DYRA_ERR_WORKSPACE = 7,     /* workspace too small or misaligned                      */
  DYRA_ERR_NO_DEVICE = 8      /* no usable sm_103 device                                */
} dyra_status;

typedef enum dyra_static_kind {
  DYRA_STATIC_LOWRANK = 0,    /* W_hat = U V, U: d x k, V: k x m (truncated SVD)        */
  DYRA_STATIC_MONARCH = 1,    /* W_hat = blockdiag(B1) . stride permutation . blockdiag(B2) */
  DYRA_STATIC_BLAST = 2       /* nb x nb blocks, block (i,j) = U_i S_ij V_j^T: row bases U_i
                                 [d/nb x t] shared along block row i, column bases V_j
                                 [m/nb x t] shared along block column j, a t x t middle matrix
                                 per block (summary page Appendix B; blog structured-methods
                                 section), fitted by alternating exact minimisations of
                                 ||W - W_hat||_F from truncated SVDs, 10 sweeps             */
} dyra_static_kind;

typedef enum dyra_dtype {
  DYRA_F32 = 0,               /* X, Y, factors fp32; fp32 SIMT kernels                  */
  DYRA_BF16 = 1               /* X, Y, factors bf16; fp32 accumulation on tcgen05        */
} dyra_dtype;

typedef enum dyra_solver {
  DYRA_SOLVE_AUTO = 0,        /* Cholesky if r <= 64, else Newton-Schulz                 */
  DYRA_SOLVE_CHOLESKY = 1,    /* exact SPD solve, r <= 64 (bf16: elimination without
                                 pivoting, whose pivots are Cholesky's; f32: fp64)       */
  DYRA_SOLVE_NEWTON_SCHULZ = 2 /* ns_iters steps of X <- X (2I - G X) after Jacobi scaling */
} dyra_solver;

/* Input-aware static decomposition (summary page Appendix B; blog section
 * "已有结构化矩阵方法分工有何不同": calibration activations define an input-side transform S, the
 * weight is written W = (W S) S^-1 and W S is truncated by its SVD). In this library's
 * row-vector convention y = x W that is W_hat = S^-T TSVD_k(S^T W). Low-rank layers only. */
typedef enum dyra_input_aware {
  DYRA_INPUT_AWARE_NONE = 0,      /* plain truncated SVD of W                                */
  DYRA_INPUT_AWARE_DIAG = 1,      /* S = diag(rms of each input channel over calib rows)     */
  DYRA_INPUT_AWARE_CHOLESKY = 2   /* S = lower Cholesky factor of calib^T calib / n_calib
                                     (needs n_calib >= d and a full-rank calibration set)    */
} dyra_input_aware;

/* Activation applied to the layer's output, Y = act(X W_hat + b + L R), in the output
 * kernel's epilogue (bf16 layers only). GELU is the erf form x Phi(x) of the ViT / DINOv3 MLP
 * blocks (summary page Appendix D: every linear layer of those models is replaced). */
typedef enum dyra_activation {
  DYRA_ACT_NONE = 0,
  DYRA_ACT_GELU = 1
} dyra_activation;

/* Arguments of dyra_prepare / dyra_fit. All pointers are HOST pointers to float64, read
 * only during the call. Zero-initialise the struct and set what you need. */
typedef struct dyra_prepare_args {
  const double *W;      /* [d, m] dense weight (required)                                 */
  const double *b;      /* [m] bias, or NULL for zero bias                                */
  int d, m;             /* input / output features                                        */
  dyra_static_kind kind;
  int k;                /* LOWRANK: static rank, 0 <= k < min(d, m).
                           MONARCH: block count nb, d % nb == 0 and m % nb == 0
                           (W_hat[(a,i),(c,j)] = B1[a][i,c] B2[c][a,j]).
                           BLAST: blocks per side nb, d % nb == 0 and m % nb == 0        */
  int r;                /* residual rank, 1 <= r <= 256 (bf16) / 1 <= r <= 64 (f32)      */
  const double *R0;     /* [r, m] fixed initial right factor, full row rank, or NULL for
                           the top-r right singular vectors of W_res                     */
  const double *F1;     /* optional static factors (both or neither):                     */
  const double *F2;     /*   LOWRANK: F1 = U [d, k], F2 = V [k, m]
                             MONARCH: F1 = B1 [nb, d/nb, nb], F2 = B2 [nb, nb, m/nb]
                           BLAST: F1 = U [nb, d/nb, t], F2 = V [nb, m/nb, t] (and F3)
                           NULL: fitted here (truncated SVD / blockwise rank-1 SVD /
                           BLAST alternating fit)                                         */
  double ridge;         /* lambda >= 0 added to the diagonal of L^T L (absolute)          */
  dyra_solver solver;
  int ns_iters;         /* Newton-Schulz iterations (0 => 8)                             */
  dyra_dtype dtype;
  int device;           /* CUDA device ordinal the layer lives on                        */
  int fit_threads;      /* host threads for the fit, 0 => hardware concurrency           */
  const double *calib;  /* [n_calib, d] calibration activations (input_aware != NONE)     */
  int n_calib;
  dyra_input_aware input_aware; /* ignored when F1/F2 are given                           */
  dyra_activation activation;   /* applied to Y (bf16 layers); NONE for a plain linear    */
  double als_t;         /* ALS iterations t of the correction (summary page 3.3 / Figure 9;
                           blog ablation: t = 1.5 updates L, R, L): 1, 1.5, 2, ... 8 (bf16
                           layers); 0 => 1, the pages' default one-step form. A further
                           L-update from R solves P = W_res R^T (R R^T)^-1, L = X P; a further
                           R-update repeats the one-step R-update from the new L.          */
  int blast_t;          /* BLAST: rank t of every block's middle matrix, 1 <= t <= min(d,
                           m) / nb (bf16 kernels: d / nb % 64 == 0, t % 32 == 0, t <= 256) */
  const double *F3;     /* BLAST with F1/F2 given: middle matrices S [nb, nb, t, t]       */
} dyra_prepare_args;

/* Read-only description of a prepared layer (the shapes and options of dyra_prepare). */
typedef struct dyra_layer_desc {
  int d, m, k, r;
  dyra_static_kind kind;
  dyra_dtype dtype;
  dyra_solver solver;   /* resolved (never AUTO)                                          */
  int ns_iters;
  double ridge;
  int device;
  int kernels_per_forward; /* kernel launches one dyra_linear_forward enqueues           */
  dyra_activation activation;
  double als_t;
} dyra_layer_desc;

typedef struct dyra_layer dyra_layer;   /* opaque; owns its device copies of the factors */

/* Offline preparation (synchronous, not meant for the timed path): static fit of W (unless
 * F1/F2 are given), W_res = W - W_hat, R0 (unless given), P = W_res R0^T (R0 R0^T)^-1, and
 * upload of the factors in the layer's dtype to `device`.
 * Passages: blog digest, section "没有训练时离线准备和在线计算是什么" (offline: static
 * structured factors, residual, fixed initial right factor R0 = top right singular vectors of
 * W_res, precomputed left projection, once per layer) and section "DyRA 的整体流程是怎样的"
 * (the offline stage of the flow); section "静态分支与残差如何拆分" (W = W_hat + W_res);
 * summary page Appendix B (truncated SVD; Monarch by a truncated SVD of each block of the
 * rearranged weight, also the blog's section "已有结构化矩阵方法分工有何不同"). P is the
 * least-squares L-update of the blog's section "残差乘积的低秩优化目标是什么" with R = R0. On success *out owns the layer;
 * free it with dyra_layer_destroy. Errors: INVALID_ARG (shapes, null W, r out of range,
 * R0 rank deficient), UNSUPPORTED (a shape the kernels do not take), NO_DEVICE, OOM, CUDA. */
dyra_status dyra_prepare(const dyra_prepare_args *args, dyra_layer **out);

/* The offline step alone, on the host (no device needed; same passages as dyra_prepare): the static fit (unless F1/F2
 * are given), W_res, R0 (unless given) and P, in float64, written to caller-owned host
 * buffers (any may be NULL; sizes as in dyra_export / dyra_export_factors). dtype, solver
 * and device are not used. Lets a CPU machine prepare factors that dyra_prepare later
 * uploads through F1/F2/R0. Errors: INVALID_ARG, OOM. */
dyra_status dyra_fit(const dyra_prepare_args *args, double *W_hat, double *W_res, double *P,
                     double *R0, double *F1, double *F2);

/* Frees a layer from dyra_prepare (waits for the layer's device to finish its work first).
 * NULL is a no-op. Packaging: the pages have no counterpart. */
void dyra_layer_destroy(dyra_layer *layer);

/* Fills *out with the layer's shapes and resolved options. Errors: INVALID_ARG (NULL).
 * Packaging: the pages have no counterpart. */
dyra_status dyra_layer_info(const dyra_layer *layer, dyra_layer_desc *out);

/* Host float64 copies of what dyra_prepare computed (before rounding to the device dtype):
 * the offline quantities of the blog's section "没有训练时离线准备和在线计算是什么".
 * Any pointer may be NULL. Sizes: W_hat, W_res [d, m]; P [d, r]; R0 [r, m];
 * F1/F2 as in dyra_prepare_args. */
dyra_status dyra_export(const dyra_layer *layer, double *W_hat, double *W_res, double *P,
                        double *R0);
dyra_status dyra_export_factors(const dyra_layer *layer, double *F1, double *F2);

/* Bytes of device workspace dyra_linear_forward needs for (batch, n): the per-sample
 * rank-r intermediates of the online step (blog section "残差乘积的低秩优化目标是什么":
 * every intermediate passes through a rank-r channel, never the full residual product).
 * Errors: INVALID_ARG (null pointers, negative sizes). */
dyra_status dyra_workspace_size(const dyra_layer *layer, int batch, int n, size_t *bytes);

/* The online step: Y = X W_hat + b + L R per sample, with L = X P (L-update from R0) and
 * R = (L^T L + lambda I)^-1 (L^T X) W_res (R-update), one least-squares system per sample.
 * Passages: blog digest, section "一次迭代的近似形式与额外代价" (one ALS iteration, L then R,
 * XW ~ X W_hat + L(1) R(1)), section "残差乘积的低秩优化目标是什么" (the objective
 * min ||X W_res - L R||_F^2 and the order of operations: input projected to r first, then
 * multiplied by the residual), section "DyRA 的整体流程是怎样的" (online stage: static branch,
 * thin product for L, least-squares R, fused accumulation; Cholesky for small r and
 * Newton-Schulz for large r; the residual product never written to memory); summary page
 * 2.2 (ridge) and 2.4 (solver choice).
 * X: device [batch, n, d], Y: device [batch, n, m], both in the layer's
 * dtype, 16-byte aligned, rows densely packed. workspace: device, >= dyra_workspace_size
 * bytes, 256-byte aligned, owned by the caller; it must not be shared by two forwards that
 * may run at the same time. Enqueues every kernel on `stream` and returns without waiting.
 * batch == 0 or n == 0 is a no-op. A sample whose
 * L^T L + lambda I is not positive definite (e.g. an all-zero sample with lambda = 0) gets
 * R = 0 -- its rows of Y are the static branch plus b -- and is counted in the status word
 * that dyra_workspace_status reads. Errors (nothing launched): INVALID_ARG, WORKSPACE, CUDA. */
dyra_status dyra_linear_forward(const dyra_layer *layer, const void *X, int batch, int n,
                                void *Y, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/* A transformer MLP block with both linear layers replaced (summary page Appendix D: the
 * evaluated ViT / DINOv3 models replace every linear layer; summary page 3.2: end-to-end
 * latency): H = fc1(X), with fc1's own activation (GELU for an MLP block), then Y = fc2(H),
 * each layer's correction computed from its own input, both enqueued on `stream`.
 * X: device [batch, n, fc1.d]; H: device [batch, n, fc1.m], caller-owned, overwritten; Y:
 * device [batch, n, fc2.m]; all in the layers' dtype (bf16), 16-byte aligned. workspace:
 * >= max(dyra_workspace_size(fc1), dyra_workspace_size(fc2)) bytes, used by one layer after
 * the other; its status words (dyra_workspace_status) count both layers. Errors (nothing
 * launched): INVALID_ARG (fc1.m != fc2.d, different dtype or device, null pointers),
 * WORKSPACE, CUDA. */
dyra_status dyra_mlp_forward(const dyra_layer *fc1, const dyra_layer *fc2, const void *X,
                             int batch, int n, void *H, void *Y, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Same step (same passages as dyra_linear_forward) from HOST buffers: copies X_host -> X_dev,
 * runs the forward, copies Y_dev -> Y_host. The samples are independent (one least-squares
 * system each), so a large batch is cut into up to 8 groups of whole samples whose copies in,
 * forwards and copies out overlap: the copies run on two streams the layer owns, the forwards
 * on `stream`, and `stream` waits for the last copy out, so work enqueued on `stream` after
 * this call (or a synchronisation of `stream`) sees Y_host written. Use page-locked host
 * memory (pageable memory makes the copies synchronous). X_dev / Y_dev are device staging
 * buffers owned by the caller; the workspace's status words count every group. Calls on one
 * layer from several host threads are serialised. */
dyra_status dyra_linear_forward_host(const dyra_layer *layer, const void *X_host, int batch,
                                     int n, void *Y_host, void *X_dev, void *Y_dev,
                                     void *workspace, size_t workspace_bytes,
                                     cudaStream_t stream);

/* The same forward (same streams, same kernels; same passages as dyra_linear_forward) that
 * also records two events around every kernel it launches (the pages time only whole
 * models, summary page 3.2; this is the per-kernel measurement): events[2i] just before kernel i and events[2i + 1] just after it, both
 * on `stream`, so cudaEventElapsedTime(events[2i], events[2i + 1]) is kernel i's
 * device time. count = kernels_per_forward; max_events must be >= 2 * count. *recorded
 * receives 2 * count. Called while `stream` is being captured into a CUDA graph, the records
 * become event-record nodes (cudaEventRecordExternal), so every replay of the graph times
 * its kernels. Errors as dyra_linear_forward, plus INVALID_ARG for too few events. */
dyra_status dyra_linear_forward_profiled(const dyra_layer *layer, const void *X, int batch,
                                         int n, void *Y, void *workspace,
                                         size_t workspace_bytes, cudaStream_t stream,
                                         cudaEvent_t *events, int max_events, int *recorded);

/* Name of kernel `i` of the forward (static string), or NULL for an index out of range or a
 * NULL layer. Packaging: the pages have no counterpart. */
const char *dyra_kernel_name(const dyra_layer *layer, int i);

/* Per-sample solve status (summary page 2.2: the R-update is a least-squares solve with an
 * optional ridge; a sample whose L^T L + lambda I is not positive definite has no Cholesky
 * factor, this library's reading is R = 0 for it).
 * Synchronises `stream`, then reads the status word the last forward on `workspace` left:
 * *not_spd_samples = samples that fell back to the static branch, *timeouts = bounded
 * in-kernel waits that gave up. Returns DYRA_ERR_TIMEOUT if *timeouts > 0, else
 * DYRA_ERR_NOT_SPD if *not_spd_samples > 0, else DYRA_OK. */
dyra_status dyra_workspace_status(const dyra_layer *layer, const void *workspace,
                                  cudaStream_t stream, int *not_spd_samples, int *timeouts);

/* Intermediates a forward leaves in its workspace, for tests that check each kernel: the
 * quantities of the blog's section "残差乘积的低秩优化目标是什么" (L, L^T L, L^T X, R). */
typedef enum dyra_buffer {
  DYRA_BUF_T = 0,      /* [batch, n, ld] = [X F1 | L] (bf16: F1 columns padded to a multiple
                          of 64; Monarch: the permuted X BD1 in place of X F1)              */
  DYRA_BUF_C = 1,      /* bf16 path: C^T = X^T L, [batch, d, r] fp32; f32 path: C = L^T X,
                          [batch, r, d] fp32                                                */
  DYRA_BUF_G = 2,      /* L^T L without lambda, [batch, r, r] (fp32 / fp64)                */
  DYRA_BUF_GINV = 3,   /* (L^T L + lambda I)^-1, [batch, r, r] (bf16 / fp64)               */
  DYRA_BUF_B = 4,      /* f32 path only: B = C W_res, [batch, r, m] fp32                    */
  DYRA_BUF_R = 5,      /* R = (L^T L + lambda I)^-1 C W_res, [batch, r, m] (bf16 / fp32)     */
  DYRA_BUF_CS = 6      /* bf16 path only: (L^T L + lambda I)^-1 C, [batch, r, d] bf16       */
} dyra_buffer;

/* Byte offset of intermediate `which` inside the workspace for (batch, n) and its row
 * stride in elements. Returns UNSUPPORTED for a buffer the layer's path does not have. */
dyra_status dyra_workspace_tensor(const dyra_layer *layer, int batch, int n, int which,
                                  size_t *offset_bytes, int *ld);

/* Bytes of the library's static device scratch (see dyra_linear_forward_static). */
#define DYRA_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* dyra_linear_forward for callers that cannot allocate device memory: code running inside
 * an allocator that must not re-enter itself, a host that forbids cudaMalloc after start-up
 * (fixed-budget serving processes), or plugins handed only input and output buffers. The
 * pages have no counterpart of this call; it is a packaging variant of the forward.
 * It runs the same kernels as dyra_linear_forward, with the workspace taken from a static
 * device array of DYRA_STATIC_SCRATCH_BYTES bytes that the library image carries: every GPU
 * that loads the library holds that array until the process exits. It calls no cudaMalloc,
 * cudaFree or other device-allocating routine. X, Y: as in dyra_linear_forward (device,
 * caller-owned). The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with the layer's device current); make that first call before any
 * stream capture. The address is cached together with the device's current CUDA context and
 * looked up again when that context changes (after cudaDeviceReset, say). All calls share the one array and it keeps the previous call's contents;
 * the forward clears its own status words, so the layer's samples that were not positive
 * definite are not readable afterwards through this entry point. Two calls whose work can
 * overlap on the GPU (different streams, or different layers on one device) race on the
 * array: serialise them. Errors: WORKSPACE (with dyra_last_error naming the sizes) when
 * (batch, n) needs more scratch than the array holds -- dyra_workspace_size gives the need --
 * otherwise as dyra_linear_forward. */
dyra_status dyra_linear_forward_static(const dyra_layer *layer, const void *X, int batch, int n,
                                       void *Y, cudaStream_t stream);

/* Self-test of the failure path (packaging: the pages have no counterpart). Launches one
 * CTA whose bounded mbarrier wait -- the same wait every kernel of the forward uses, with
 * its limit set to limit_us microseconds instead of 2 s -- runs on a barrier that nothing
 * arrives on. The wait gives up, counts itself in status_words[1] and the kernel returns.
 * status_words: device, at least 2 ints, 4-byte aligned, caller-owned; zeroed by this call.
 * Synchronises `stream`. Returns DYRA_ERR_TIMEOUT when the wait gave up (the designed
 * outcome), DYRA_OK if it did not, INVALID_ARG for limit_us outside [1, 2000000] or a bad
 * pointer, CUDA on a launch error. */
dyra_status dyra_selftest_bounded_wait(int limit_us, int *status_words, cudaStream_t stream);

/* Text of a status code (static string). Packaging: the pages have no counterpart. */
const char *dyra_status_string(dyra_status status);
/* Text of the last CUDA/driver error seen by this thread inside the library ("" if none).
 * Packaging: the pages have no counterpart. */
const char *dyra_last_error(void);
/* DYRA_ABI_VERSION of the loaded library. */
int dyra_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DYRA_H_ */
