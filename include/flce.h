/*
 * libflce -- chunked fused LM-head cross-entropy on one GB300 (sm_103a).
 *
 * Given hidden states h[N,H] and the LM-head weight W[V,H] (bf16, row-major),
 * the library computes, without ever storing the N x V logit matrix:
 *
 *   z[i,v]  = sum_k h[i,k] W[v,k]
 *   lse[i]  = log sum_v exp(z[i,v])
 *   m[i]    = (targets[i] != ignore_index)
 *   logp[i] = m[i] * (z[i,targets[i]] - lse[i])          (0 on ignored rows)
 *   n_valid = sum_i m[i]
 *   loss    = -sum_i m[i] w[i] logp[i] / n_valid         (0 when n_valid == 0)
 *   D[i,v]  = (exp(z[i,v] - lse[i]) - [v == targets[i]]) * m[i] * w[i] * grad_scale
 *   dH      = D W            dW = D^T h
 *
 * Sources: Unsloth, "Reinforcement Learning GRPO with 7x longer context",
 * section "Flattened sequence-length chunking" (rows are the flattened batch x
 * context tokens, taken in chunks; each chunk's logits are hidden @ lm_head,
 * upcast to fp32, log-softmaxed, and the completion token's log-prob is
 * gathered) and section "Offloading activations for log-softmax" (the
 * backward recomputes the chunk's logits instead of storing them); TRL v1.13
 * article "Training Beyond 1M Tokens", loss section (256 rows per chunk,
 * chunk losses summed) and speed & memory section (bf16 operands on the
 * tensor cores).  With w = 1 the loss is the masked mean NLL; with per-token
 * weights (e.g. GRPO advantages) it is -sum(w logp)/sum(mask).
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers on the current CUDA device unless
 *     stated otherwise; the caller owns every buffer and the stream; the
 *     library never frees caller memory.
 *   - bf16 arrays are passed as uint16_t bit patterns (flce_bf16).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous and stream-ordered; nothing is synchronised unless
 *     stated.
 *   - Host-side argument checks return a status before any launch.  No C++
 *     exception crosses this interface.
 *   - H must be a multiple of 8 and h, W, D-type buffers 16-byte aligned
 *     (TMA rows are 16-byte aligned), else FLCE_ERR_UNSUPPORTED.
 *   - N, H, V must each be < 2^31.
 *   - Not thread-safe for concurrent calls from several host threads while
 *     profiling is enabled.
 *   - CUDA graphs: flce_forward(_ex), flce_backward(_ex),
 *     flce_forward_backward, the distillation and e4m3 entry points can be
 *     captured into a CUDA graph and replayed
 *     when they are given a caller workspace, FLCE_VALIDATE is unset,
 *     profiling is off, and one eager call of the same kind has run on the
 *     device first (it sets kernel attributes and caches the device's
 *     co-resident cluster count).
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(FLCE_BUILDING_LIBRARY) && defined(__GNUC__)
#define FLCE_API __attribute__((visibility("default")))
#else
#define FLCE_API
#endif

typedef uint16_t flce_bf16;

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,  /* null/ill-sized argument, workspace too small */
  FLCE_ERR_BAD_TARGET = 2,   /* validation mode: a target outside [0,V) */
  FLCE_ERR_UNSUPPORTED = 3,  /* shape/alignment the kernels do not handle */
  FLCE_ERR_OOM = 4,          /* library-side workspace allocation failed */
  FLCE_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  FLCE_ERR_TIMEOUT = 6       /* a kernel's bounded wait ran out (device error word) */
} flce_status;

/*
 * Logit transforms applied elementwise to z before the log-softmax, in this
 * order: multiply, divide, soft-cap, temperature.  Source: Unsloth,
 * "Reinforcement Learning GRPO with 7x longer context", section "Flattened
 * sequence-length chunking": the chunked selective log-softmax takes
 * logit_scale_multiply, logit_scale_divide, logit_softcapping and
 * temperature (the page prints neither their order nor their defaults; the
 * order of its call is taken, and 0 disables the first three).
 *   scale_multiply  y *= scale_multiply           (0 = off; must be >= 0)
 *   scale_divide    y /= scale_divide             (0 = off; must be >= 0)
 *   softcap         y = softcap * tanh(y/softcap) (0 = off; must be >= 0)
 *   temperature     y /= temperature              (1 = off; must be > 0)
 * lse and logp are those of y; the backward's D carries dy/dz.  Invalid
 * values return FLCE_ERR_INVALID_ARG.
 */
typedef struct flce_logit_transform {
  float scale_multiply;
  float scale_divide;
  float softcap;
  float temperature;
} flce_logit_transform;

/*
 * Forward: per-token log-probs, log-sum-exp, masked (weighted) mean loss.
 *
 *   h        [N,H] bf16, row-major (row i = token i of the flattened batch).
 *   W        [V,H] bf16, row-major (the lm_head weight).
 *   targets  [N] int64; each in [0,V) or == ignore_index.  A target outside
 *            [0,V) that is not ignore_index is never read out of bounds: its
 *            row's logp is NaN (and so is the loss) unless FLCE_VALIDATE=1 is
 *            set in the environment, in which case the call synchronises the
 *            stream after a check kernel and returns FLCE_ERR_BAD_TARGET
 *            before any GEMM runs.
 *   weights  [N] fp32 per-token weights, or NULL for all ones.
 *   N, H, V  sizes (N may be 0).
 *   chunk_rows  rows per chunk (the pages' chunk size, 256 in TRL).  The
 *            forward keeps logits in tensor memory only, so its workspace is
 *            O(N * splits) whatever chunk_rows is; results do not depend on it.
 *   ignore_index  target value that marks a row without loss (-100 in PyTorch).
 *   out_logp [N] fp32 or NULL.  0 on ignored rows.
 *   out_lse  [N] fp32 or NULL.  Computed for every row, ignored or not;
 *            flce_backward needs it.
 *   out_loss [1] fp32 or NULL.
 *   out_n_valid [1] int64 or NULL: the exact count of non-ignored rows.
 *   workspace, workspace_bytes: device scratch of at least
 *            flce_workspace_bytes(N,H,V,chunk_rows) bytes, 256-byte aligned;
 *            or NULL, in which case the call allocates it stream-ordered
 *            (cudaMallocAsync) and frees it (cudaFreeAsync) on `stream`.
 * At least one of out_logp, out_lse, out_loss, out_n_valid must be non-NULL.
 */
FLCE_API flce_status flce_forward(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                         const float* weights, int64_t N, int64_t H, int64_t V,
                         int64_t chunk_rows, int64_t ignore_index, float* out_logp,
                         float* out_lse, float* out_loss, int64_t* out_n_valid,
                         void* workspace, size_t workspace_bytes, void* stream);

/* flce_forward with a logit transform (NULL = identity). */
FLCE_API flce_status flce_forward_ex(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                     const float* weights, int64_t N, int64_t H, int64_t V,
                                     int64_t chunk_rows, int64_t ignore_index,
                                     const flce_logit_transform* transform, float* out_logp,
                                     float* out_lse, float* out_loss, int64_t* out_n_valid,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * flce_forward_ex with flags (0 = flce_forward_ex).
 *   FLCE_FORWARD_SKIP_IGNORED: the GEMM covers the non-ignored rows only
 *     (the row skipping of the Unsloth page's "Flattened sequence-length
 *     chunking" applied to the forward).  Ignored rows get out_lse = NaN
 *     (not computed) and out_logp = 0; flce_backward never reads their lse.
 *     The rows are found and gathered on the device (no host sync), in
 *     blocks of 4,096 rows of h inside the workspace that
 *     flce_workspace_bytes reports.  Calls with N < 2,048 rows
 *     (FLCE_SKIP_MIN_ROWS overrides the bound), or with FLCE_COMPACT=0,
 *     compute every row as flce_forward_ex does.
 * Other flag bits: FLCE_ERR_INVALID_ARG.
 */
#define FLCE_FORWARD_SKIP_IGNORED 1u
FLCE_API flce_status flce_forward_ex2(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                                      const float* weights, int64_t N, int64_t H, int64_t V,
                                      int64_t chunk_rows, int64_t ignore_index,
                                      const flce_logit_transform* transform, uint32_t flags,
                                      float* out_logp, float* out_lse, float* out_loss,
                                      int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                                      void* stream);

/*
 * Backward: dH = D W and dW = D^T h with
 *   D[i,v] = (exp(z[i,v] - lse[i]) - [v == targets[i]]) * m[i] * w[i] * grad_scale.
 *
 *   lse      [N] fp32 from flce_forward (same h, W).
 *   grad_scale  g, applied literally.  The library does not divide by n_valid:
 *            for the gradient of the mean loss pass g = dLoss / n_valid.  An
 *            arbitrary per-token upstream gradient dL/dlogp[i] is obtained with
 *            weights[i] = -dL/dlogp[i] and g = 1.
 *   dH       [N,H] bf16 output (overwritten; ignored rows get 0), or NULL to
 *            skip the dH GEMM.
 *   dW       [V,H] fp32 output (overwritten), or NULL to skip the dW GEMM
 *            (frozen lm_head).
 *   chunk_rows  the dlogits memory bound: the workspace holds at most
 *            C x V bf16 dlogits, C = chunk_rows rounded up to 128 (plus dH
 *            fp32 partials and gathered rows, together no larger): extra
 *            memory O(chunk_rows * V), never O(N * V).  Within that bound the
 *            backward walks blocks of R >= C rows and, inside each block,
 *            vocabulary slabs of Vs columns with R * Vs <= C * V, choosing R
 *            by a time model (flce_backward_plan); dW is read-modified-
 *            written once per row block, and dH is summed over the slabs in
 *            fp32 and rounded to bf16 once.  Results do not depend on
 *            chunk_rows beyond fp32 summation order.
 * Other arguments as in flce_forward.  Rows with an out-of-range target get
 * D = softmax * w * g (no one-hot term); FLCE_VALIDATE=1 rejects them.
 */
FLCE_API flce_status flce_backward(const flce_bf16* h, const flce_bf16* W, const int64_t* targets,
                          const float* weights, const float* lse, float grad_scale,
                          flce_bf16* dH, float* dW, int64_t N, int64_t H, int64_t V,
                          int64_t chunk_rows, int64_t ignore_index, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Forward and backward of the mean loss in one call, without the backward's
 * logits recompute.  The pages' chunked loops recompute each chunk's logits
 * in the backward; this call is an addition of this library (no counterpart
 * on the pages) that trades that GEMM for memory inside the same budget.
 * Per block of R rows over the whole vocabulary, one GEMM computes the online
 * log-sum-exp (as flce_forward) and keeps exp(u - chunk max) in bf16 plus the
 * maximum of every 32-column chunk; once the rows' lse is known, one
 * elementwise pass turns them into the dlogits in place (the target column
 * from its exact fp32 logit), and the dH / dW GEMMs follow.  That is
 * 6 N V H instead of 8 N V H tensor FLOPs; the extra rounding of the stored
 * exponentials (bf16) is of the same size as that of the bf16 dlogits.
 *
 *   Outputs as flce_forward_ex (out_logp, out_lse, out_loss, out_n_valid may
 *   be NULL) and flce_backward_ex (dH and/or dW), with
 *     dH, dW = grad_scale * d(loss) / d(h, W),  loss = -sum m w logp / n_valid
 *   (grad_scale = 1 for the plain mean loss; zero gradients when n_valid = 0).
 *   chunk_rows sets the block: R = C = chunk_rows rounded up to 128 rows,
 *   stored as R x ldD bf16 exponentials (ldD = V rounded up to 32) plus
 *   R x ldD / 32 fp32 maxima (1/16 of that).  When C is below 2,048 rows
 *   (and below N), the call runs flce_forward_ex and the tiled backward
 *   instead, with grad_scale / n_valid applied on the device.
 *   Ignored rows: the blocks run over a permutation that puts the
 *   non-ignored rows first (written on the device; FLCE_COMPACT=0 keeps
 *   the row order).  Every row gets its lse when out_lse is given; with
 *   out_lse NULL the forward GEMM covers the non-ignored rows only.  The
 *   dH / dW GEMMs cover the non-ignored rows only, and the ignored rows' dH
 *   is zero.  The block's rows of h are gathered into the workspace (R x H
 *   bf16 more).
 *   Workspace: flce_forward_backward_workspace_bytes, or NULL.
 */
FLCE_API flce_status flce_forward_backward(const flce_bf16* h, const flce_bf16* W,
                                           const int64_t* targets, const float* weights,
                                           int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                                           int64_t ignore_index,
                                           const flce_logit_transform* transform,
                                           float grad_scale, float* out_logp, float* out_lse,
                                           float* out_loss, int64_t* out_n_valid, flce_bf16* dH,
                                           float* dW, void* workspace, size_t workspace_bytes,
                                           void* stream);

/* Workspace bytes of flce_forward_backward for these sizes (0 on invalid). */
FLCE_API size_t flce_forward_backward_workspace_bytes(int64_t N, int64_t H, int64_t V,
                                                      int64_t chunk_rows);

/* flce_backward with a logit transform (NULL = identity); `lse` must come
 * from flce_forward_ex with the same transform. */
FLCE_API flce_status flce_backward_ex(const flce_bf16* h, const flce_bf16* W,
                                      const int64_t* targets, const float* weights,
                                      const float* lse, float grad_scale, flce_bf16* dH, float* dW,
                                      int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                                      int64_t ignore_index, const flce_logit_transform* transform,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * A gradient scale held in device memory, so that a caller can pass the
 * incoming gradient of the loss and the count the forward produced without
 * synchronising the host (no counterpart on the pages: the mean loss of the
 * TRL and Unsloth loops divides by the token count; here the division happens
 * on the device).  The dlogits are multiplied by
 *   grad_scale * (*scale) / max(*count, 1),
 * where a NULL scale or count stands for 1 (and no division).  Both are read
 * by the kernels when they run, in stream order.
 */
typedef struct flce_device_scale {
  const float* scale;    /* [1] fp32 device, 4-byte aligned, or NULL */
  const int64_t* count;  /* [1] int64 device, 8-byte aligned, or NULL (e.g. out_n_valid) */
} flce_device_scale;

/* flce_backward_ex with D's scale grad_scale * (*scale) / max(*count, 1) from
 * device memory (device_scale may be NULL: grad_scale alone).  For the
 * gradient of the mean loss with an incoming gradient dLoss on the device:
 * grad_scale = 1, scale = &dLoss, count = the forward's out_n_valid. */
FLCE_API flce_status flce_backward_ex2(const flce_bf16* h, const flce_bf16* W,
                                       const int64_t* targets, const float* weights,
                                       const float* lse, float grad_scale,
                                       const flce_device_scale* device_scale, flce_bf16* dH,
                                       float* dW, int64_t N, int64_t H, int64_t V,
                                       int64_t chunk_rows, int64_t ignore_index,
                                       const flce_logit_transform* transform, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* Multiply dH ([n_dH] bf16, rounded to nearest even) and dW ([n_dW] fp32) in
 * place by *scale (a device fp32 scalar) -- e.g. gradients that
 * flce_forward_backward computed for an incoming gradient of 1, once the
 * real one is known on the device.  A scale of exactly 1 moves no data.
 * Either array may be NULL with its count 0; arrays 16-byte aligned. */
FLCE_API flce_status flce_scale_grads(flce_bf16* dH, int64_t n_dH, float* dW, int64_t n_dW,
                                      const float* scale, void* stream);

/*
 * Distillation: a student head (h_s [N,H_s], W_s [V,H_s]) learns a frozen
 * teacher head's (h_t [N,H_t], W_t [V,H_t]) token distribution.  Source: TRL
 * v1.13 article, speed & memory section: the distillation trainer computes
 * every chunk twice, once with the student's head and once with the
 * teacher's.  Reading taken (the page names no formula): per row
 *   kl[i] = m[i] * KL(p_t || p_s) = m[i] * sum_v p_t (log p_t - log p_s),
 *   loss  = sum_i m[i] w[i] kl[i] / sum_i m[i],
 * with p = softmax of the transformed logits of each head (the same
 * transform for both, e.g. a temperature) and m[i] = (targets[i] !=
 * ignore_index), or 1 for every row when targets == NULL (targets are
 * otherwise unused).  Both heads run in one tile pipeline (student and
 * teacher logits of a tile sit side by side in tensor memory); the forward
 * never stores either head's logits.  Outputs (each may be NULL, not all):
 * out_kl [N], out_lse_s [N], out_lse_t [N] fp32, out_loss, out_n_valid.
 * Other arguments and conventions as in flce_forward; the workspace size is
 * flce_kd_workspace_bytes.
 */
FLCE_API flce_status flce_kd_forward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                     const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                     const int64_t* targets, const float* weights, int64_t N,
                                     int64_t V, int64_t chunk_rows, int64_t ignore_index,
                                     const flce_logit_transform* transform, float* out_kl,
                                     float* out_lse_s, float* out_lse_t, float* out_loss,
                                     int64_t* out_n_valid, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * flce_kd_forward / flce_jsd_forward with flags (0 = the plain call).
 *   FLCE_FORWARD_SKIP_IGNORED: with targets given, both heads' GEMMs skip
 *     the ignored rows (as flce_forward_ex2): their kl / jsd is 0 and their
 *     out_lse_s, out_lse_t and out_kl_sm are NaN (not computed), which the
 *     backwards never read.  Calls with N < 2,048 rows (FLCE_SKIP_MIN_ROWS
 *     overrides the bound) or with FLCE_COMPACT=0 compute every row.  The
 *     workspace is flce_kd_workspace_bytes.
 * Other flag bits: FLCE_ERR_INVALID_ARG.
 */
FLCE_API flce_status flce_kd_forward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                         const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                         const int64_t* targets, const float* weights, int64_t N,
                                         int64_t V, int64_t chunk_rows, int64_t ignore_index,
                                         const flce_logit_transform* transform, uint32_t flags,
                                         float* out_kl, float* out_lse_s, float* out_lse_t,
                                         float* out_loss, int64_t* out_n_valid, void* workspace,
                                         size_t workspace_bytes, void* stream);
FLCE_API flce_status flce_jsd_forward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                          const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                          const int64_t* targets, const float* weights, int64_t N,
                                          int64_t V, int64_t chunk_rows, int64_t ignore_index,
                                          float beta, const flce_logit_transform* transform,
                                          uint32_t flags, float* out_jsd, float* out_lse_s,
                                          float* out_lse_t, float* out_kl_sm, float* out_loss,
                                          int64_t* out_n_valid, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * Student gradients of the distillation loss (the teacher is frozen):
 *   D[i,v] = (p_s[i,v] - p_t[i,v]) * m[i] * w[i] * grad_scale * dy/dz_s,
 *   dH_s = D W_s ([N,H_s] bf16, or NULL),  dW_s = D^T h_s ([V,H_s] fp32, or NULL),
 * recomputing both heads' logits chunk by chunk (chunk_rows as in
 * flce_backward).  lse_s / lse_t come from flce_kd_forward (or
 * flce_kd_forward_ex2).  Where targets mark ignored rows, the chunks run
 * over the non-ignored rows only (both heads' rows gathered per chunk); the
 * ignored rows' lse are never read and their dH_s rows are 0.  workspace is
 * flce_kd_workspace_bytes.
 */
FLCE_API flce_status flce_kd_backward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                      const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                      const int64_t* targets, const float* weights,
                                      const float* lse_s, const float* lse_t, float grad_scale,
                                      flce_bf16* dH_s, float* dW_s, int64_t N, int64_t V,
                                      int64_t chunk_rows, int64_t ignore_index,
                                      const flce_logit_transform* transform, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* flce_kd_backward with D's scale grad_scale * (*scale) / max(*count, 1) from
 * device memory (see flce_device_scale; NULL: grad_scale alone). */
FLCE_API flce_status flce_kd_backward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                          const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                          const int64_t* targets, const float* weights,
                                          const float* lse_s, const float* lse_t, float grad_scale,
                                          const flce_device_scale* device_scale, flce_bf16* dH_s,
                                          float* dW_s, int64_t N, int64_t V, int64_t chunk_rows,
                                          int64_t ignore_index,
                                          const flce_logit_transform* transform, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * Jensen-Shannon distillation.  Source: TRL v1.13 article, section "Other
 * changes in v1.13": a fused linear JSD loss is among TRL's fused losses; the
 * page gives no formula.  Reading taken: per row, the generalised
 * Jensen-Shannon divergence with mixture weight beta in (0, 1) (1/2 is the
 * textbook JSD):
 *   M      = beta * p_t + (1 - beta) * p_s,
 *   jsd[i] = m[i] * (beta * KL(p_t || M) + (1 - beta) * KL(p_s || M)),
 *   loss   = sum_i m[i] w[i] jsd[i] / sum_i m[i],
 * with p_s, p_t, m[i], the logit transform, weights and the two heads as in
 * flce_kd_forward.  Small beta approaches beta * KL(p_t || p_s) (the KL
 * calls); beta near 1 approaches (1 - beta) * KL(p_s || p_t).
 *
 * flce_jsd_forward needs both heads' final log-sum-exp before it can form M,
 * so it runs both heads twice: once for the log-sum-exp (as
 * flce_kd_forward), once for the mixture terms.  Outputs (each may be NULL,
 * not all): out_jsd [N], out_lse_s [N], out_lse_t [N], out_kl_sm [N] fp32
 * (KL(p_s || M) of every row, masked or not: flce_jsd_backward needs it),
 * out_loss, out_n_valid.  beta outside (0, 1) -> FLCE_ERR_INVALID_ARG.
 */
FLCE_API flce_status flce_jsd_forward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                      const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                      const int64_t* targets, const float* weights, int64_t N,
                                      int64_t V, int64_t chunk_rows, int64_t ignore_index,
                                      float beta, const flce_logit_transform* transform,
                                      float* out_jsd, float* out_lse_s, float* out_lse_t,
                                      float* out_kl_sm, float* out_loss, int64_t* out_n_valid,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Student gradients of the Jensen-Shannon loss (the teacher is frozen):
 *   D[i,v] = (1 - beta) p_s[i,v] (ln(p_s[i,v] / M[i,v]) - kl_sm[i]) * m[i] w[i] grad_scale
 *            * f'(z_s[i,v]),
 *   dH_s = D W_s, dW_s = D^T h_s,
 * with lse_s, lse_t, kl_sm from flce_jsd_forward or flce_jsd_forward_ex2
 * (same beta and transform).  Memory, tiling and the skipping of ignored
 * rows as flce_kd_backward.
 */
FLCE_API flce_status flce_jsd_backward(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                       const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                       const int64_t* targets, const float* weights,
                                       const float* lse_s, const float* lse_t, const float* kl_sm,
                                       float beta, float grad_scale, flce_bf16* dH_s, float* dW_s,
                                       int64_t N, int64_t V, int64_t chunk_rows,
                                       int64_t ignore_index, const flce_logit_transform* transform,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* flce_jsd_backward with D's scale grad_scale * (*scale) / max(*count, 1)
 * from device memory (see flce_device_scale; NULL: grad_scale alone). */
FLCE_API flce_status flce_jsd_backward_ex2(const flce_bf16* h_s, const flce_bf16* W_s, int64_t H_s,
                                           const flce_bf16* h_t, const flce_bf16* W_t, int64_t H_t,
                                           const int64_t* targets, const float* weights,
                                           const float* lse_s, const float* lse_t, const float* kl_sm,
                                           float beta, float grad_scale,
                                           const flce_device_scale* device_scale, flce_bf16* dH_s,
                                           float* dW_s, int64_t N, int64_t V, int64_t chunk_rows,
                                           int64_t ignore_index,
                                           const flce_logit_transform* transform, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * GRPO per-token objective on the sampled tokens' log-probs.  Source: TRL
 * v1.13 article, section "Other changes in v1.13": a fused linear GRPO loss is
 * among TRL's fused losses; the page gives no formula.  Reading taken (the
 * GRPO objective with a clipped probability ratio and the k3 estimate of the
 * KL divergence to a reference policy), per row i with m[i] = (targets[i] !=
 * ignore_index), or 1 for every row when targets == NULL:
 *   r[i]     = exp(logp[i] - old_logp[i])      (1 when old_logp == NULL)
 *   obj[i]   = min(r A, clip(r, 1 - eps_low, 1 + eps_high) A),  A = advantages[i]
 *   kl[i]    = exp(ref - logp) - (ref - logp) - 1   (0 when beta == 0)
 *   token[i] = m[i] (beta kl[i] - obj[i]),  loss = sum_i token[i] / sum_i m[i]
 * and weights[i] = -d token[i] / d logp[i] (0 on masked rows).  old_logp and
 * ref_logp are constants.  The loss's gradients are then
 *   flce_backward(h, W, targets, weights, lse, 1 / n_valid, ...);
 * with old_logp == NULL and beta == 0, weights = m A (the GRPO-style
 * advantage-weighted loss).
 *
 *   logp, advantages [N] fp32 (logp from flce_forward); old_logp, ref_logp
 *   [N] fp32 or NULL (ref_logp required when beta > 0); eps_low in [0, 1),
 *   eps_high >= 0, beta >= 0, else FLCE_ERR_INVALID_ARG.  Outputs (each may
 *   be NULL, not all): out_token_loss [N], out_weights [N] fp32, out_loss [1]
 *   fp32, out_n_valid [1] int64.  Workspace: flce_grpo_workspace_bytes(N),
 *   or NULL (stream-ordered allocation).
 */
FLCE_API flce_status flce_grpo_token_loss(const float* logp, const float* old_logp,
                                          const float* ref_logp, const float* advantages,
                                          const int64_t* targets, int64_t N, int64_t ignore_index,
                                          float eps_low, float eps_high, float beta,
                                          float* out_token_loss, float* out_weights,
                                          float* out_loss, int64_t* out_n_valid, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* Workspace bytes of flce_grpo_token_loss for N rows (0 on invalid N). */
FLCE_API size_t flce_grpo_workspace_bytes(int64_t N);

/*
 * The GRPO loss of flce_grpo_token_loss and its gradients in one call,
 * without the backward's logits recompute (an addition of this library, as
 * flce_forward_backward): per block of rows, the forward GEMM keeps the
 * exponentials, the block's log-probs give its token losses and backward
 * weights w = -d(token loss)/d(logp), and the dlogits pass and the dH / dW
 * GEMMs use those weights.
 *   loss = sum m * token / sum m  (out_loss [1], or NULL),
 *   dH, dW = grad_scale * d(loss) / d(h, W),
 *   out_logp [N] and out_token_loss [N] fp32 or NULL; out_n_valid int64 or NULL.
 * advantages [N] fp32 (required), old_logp / ref_logp [N] fp32 or NULL, and
 * eps_low, eps_high, beta as flce_grpo_token_loss (ref_logp required when
 * beta > 0).  Blocks, row compaction (ignored rows are skipped in every
 * GEMM: no lse is returned), the fallback for budgets under 2,048 rows and
 * the workspace (flce_forward_backward_workspace_bytes) are those of
 * flce_forward_backward.
 */
FLCE_API flce_status flce_grpo_forward_backward(const flce_bf16* h, const flce_bf16* W,
                                                const int64_t* targets, const float* advantages,
                                                const float* old_logp, const float* ref_logp,
                                                float eps_low, float eps_high, float beta, int64_t N,
                                                int64_t H, int64_t V, int64_t chunk_rows,
                                                int64_t ignore_index,
                                                const flce_logit_transform* transform,
                                                float grad_scale, float* out_logp,
                                                float* out_token_loss, float* out_loss,
                                                int64_t* out_n_valid, flce_bf16* dH, float* dW,
                                                void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of the distillation calls (flce_kd_* and flce_jsd_*) for
 * these sizes. */
FLCE_API size_t flce_kd_workspace_bytes(int64_t N, int64_t H_s, int64_t H_t, int64_t V,
                                        int64_t chunk_rows);

/*
 * e4m3 (fp8) operands for the forward log-prob path.  Source: Unsloth, "Reinforcement
 * Learning GRPO with 7x longer context", introduction: its RL features combine
 * with float8 training (FP8 RL).  The forward alone is offered in e4m3 -- it
 * serves log-probs that need no gradient (e.g. reference or old-policy
 * log-probs in RL); the backward stays bf16, since dlogits with a 3-bit
 * mantissa cannot keep gradients within 1 % (relative Frobenius).
 *
 * flce_quantize_e4m3_rows: x [rows, cols] bf16 -> q [rows, cols] e4m3 bytes
 * and scale [rows] fp32 with scale = max|x_row| / 448 (1 for an all-zero row)
 * and q = e4m3(x / scale), round to nearest even, saturating.  cols % 16 == 0.
 *
 * flce_forward_e4m3: flce_forward_ex on the dequantised operands, i.e. with
 * z[i,v] = (sum_k q_h[i,k] q_W[v,k]) * h_scale[i] * W_scale[v], computed by
 * e4m3 tensor-core MMAs (kind::f8f6f4) into fp32.  h8 [N,H], W8 [V,H] e4m3
 * row-major; h_scale [N], W_scale [V] fp32 (W_scale 16-byte aligned);
 * H % 16 == 0.  Other arguments as in flce_forward_ex.
 */
FLCE_API flce_status flce_quantize_e4m3_rows(const flce_bf16* x, int64_t rows, int64_t cols,
                                             uint8_t* q, float* scale, void* stream);

FLCE_API flce_status flce_forward_e4m3(const uint8_t* h8, const float* h_scale, const uint8_t* W8,
                                       const float* W_scale, const int64_t* targets,
                                       const float* weights, int64_t N, int64_t H, int64_t V,
                                       int64_t chunk_rows, int64_t ignore_index,
                                       const flce_logit_transform* transform, float* out_logp,
                                       float* out_lse, float* out_loss, int64_t* out_n_valid,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward that allocates nothing (no counterpart on the source pages: the
 * method itself does not need it).
 *
 * For callers that may not allocate device memory at all: runtimes that hand
 * out every byte of device memory from a fixed pool of their own (an
 * allocation behind their back breaks their accounting or fails), and
 * services that must keep a constant footprint from start-up on (an
 * allocation on the hot path could fail under memory pressure or stall on the
 * allocator).  Same arguments and results as flce_forward with workspace =
 * NULL, except that no workspace is allocated: the call uses a 16 MiB scratch
 * array that the library keeps in device memory on every device that loads it,
 * for the life of the process.
 *   - The forward's scratch is about N * (4 + 8 * S) bytes for S vocabulary
 *     splits; this call uses as many splits as fit in 16 MiB (results equal
 *     flce_forward's up to fp32 rounding of the split combine).  It returns
 *     FLCE_ERR_UNSUPPORTED, before any launch, only when one split does not
 *     fit: about 12 bytes per row, so N above about 1.39 million rows.
 *   - The first call on each device (and the first after the device's
 *     context was rebuilt, e.g. by a reset) looks up the array's device
 *     address with cudaGetSymbolAddress, which may also create the device's
 *     primary context; make that first call before any stream capture.
 *   - All calls share the one array: calls whose kernels may overlap on the
 *     GPU (different streams without ordering between them) race on it and
 *     must not be issued.  Each call writes every scratch word it reads, so
 *     what an earlier call left there does not affect the result.
 *   - Makes no cudaMalloc/cudaFree or other allocating call.
 */
FLCE_API flce_status flce_forward_static_scratch(const flce_bf16* h, const flce_bf16* W,
                                                 const int64_t* targets, const float* weights,
                                                 int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                                                 int64_t ignore_index, float* out_logp,
                                                 float* out_lse, float* out_loss,
                                                 int64_t* out_n_valid, void* stream);

/* The backward's tiling for these sizes (host-only; no device is touched).
 * Output of flce_backward_plan. */
typedef struct flce_backward_plan_info {
  int64_t rows_per_block;   /* R: rows whose dlogits are held at once */
  int64_t vocab_per_slab;   /* Vs: vocabulary columns per slab (V when one slab) */
  int64_t row_blocks;       /* ceil(N / R) */
  int64_t vocab_slabs;      /* ceil(V / Vs) */
  int64_t dh_splits;        /* k-splits of the dH GEMM (fp32 partial sets) */
  int64_t dlogits_bytes;    /* bytes of the dlogits block: R * row pitch * 2 */
  int64_t workspace_bytes;  /* flce_backward's whole workspace for these sizes */
  int64_t dlogits_buffers;  /* 1, or 2 when the row blocks run pipelined: slab s + 1's dlogits
                               formed while slab s's dH and dW run (both gradients wanted,
                               several slabs; dlogits_bytes covers both buffers) */
  int64_t dh_wide;          /* 1 when the dH GEMM runs 256 x 512 tiles on SM pairs (one slab, at
                               least two waves of 256 x 256 tiles), else 0 */
} flce_backward_plan_info;

/* Backward tiling that flce_backward uses for N, H, V, chunk_rows when it
 * computes both dH and dW (under the current run-time options) on a GPU that
 * holds `workers` persistent tile workers (CTAs for cta_group 1, CTA pairs
 * for cta_group 2; 152 SMs give 152 or 76).  workers <= 0 or cta_group == 0:
 * query the current device and the FLCE_CTA_GROUP setting.  workspace_bytes
 * covers the tiling of a call that computes only one of the gradients too.
 * FLCE_ERR_INVALID_ARG on invalid sizes or a NULL out. */
FLCE_API flce_status flce_backward_plan(int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                                        int32_t workers, int32_t cta_group,
                                        flce_backward_plan_info* out);

/* Workspace bytes that both flce_forward and flce_backward need for these
 * sizes on the current device (0 on invalid sizes).  Host-only; if no device
 * can be queried it assumes 152 SMs. */
FLCE_API size_t flce_workspace_bytes(int64_t N, int64_t H, int64_t V, int64_t chunk_rows);

/* Static, human-readable name of a status. */
FLCE_API const char* flce_status_string(flce_status s);

/* Synchronises `stream`, then reads and clears the library's device error
 * word on the current device: FLCE_ERR_TIMEOUT if a kernel gave up a bounded
 * wait since the last call, FLCE_ERR_CUDA if the stream reports an error,
 * else FLCE_OK. */
FLCE_API flce_status flce_device_status(void* stream);

/*
 * Run-time options (no counterpart on the source pages: they select among
 * equivalent schedules of the same computation, or add checks).
 *
 * One process-wide table that every entry point reads when it is called.
 * Each option starts from its environment variable (read once, when the
 * library first consults an option), else from its built-in default; after
 * that only flce_set_option changes it.  Results depend on no option beyond
 * fp32 rounding of summation orders, except FLCE_OPT_VALIDATE (an extra
 * check).  Setting an option while another host thread is inside a call is
 * allowed but gives that call either value.
 */
typedef enum flce_option {
  FLCE_OPT_CTA_GROUP = 0,   /* FLCE_CTA_GROUP: 2 = SM-pair GEMMs (default), 1 = one SM per tile */
  FLCE_OPT_COMPACT,         /* FLCE_COMPACT: 1 = backwards (and flagged forwards) skip ignored
                               rows (default), 0 = every row */
  FLCE_OPT_VALIDATE,        /* FLCE_VALIDATE: 1 = check targets first (one stream sync;
                               FLCE_ERR_BAD_TARGET), 0 = no check (default) */
  FLCE_OPT_PDL,             /* FLCE_PDL: 1 = programmatic dependent launch of the GEMMs
                               (default), 0 = plain stream order */
  FLCE_OPT_D_TMA,           /* FLCE_D_TMA: 1 = dlogits written through TMA boxes (default),
                               0 = per-thread stores */
  FLCE_OPT_WIDE_EPILOGUE,   /* FLCE_WIDE_EPILOGUE: 1 = 8 epilogue warps in the two-head
                               dlogits modes (default), 0 = 4 */
  FLCE_OPT_BWD_ROWS,        /* FLCE_BWD_ROWS: backward row block R (clamped to the budget);
                               0 = the planner's choice (default) */
  FLCE_OPT_FWD_SPLITS,      /* FLCE_FWD_SPLITS: forward vocabulary splits; 0 = planner (default) */
  FLCE_OPT_DH_SPLITS,       /* FLCE_DH_SPLITS: dH k-splits (1..16); 0 = planner (default) */
  FLCE_OPT_DH_GROUP,        /* FLCE_DH_GROUP: row tiles per dH raster group (default 8);
                               0 = all row tiles */
  FLCE_OPT_FWD_BLOCK_ROWS,  /* FLCE_FWD_BLOCK_ROWS: rows per forward launch, rounded up to a
                               tile; -1 = 16 row tiles (default), 0 = all rows in one launch */
  FLCE_OPT_SKIP_MIN_ROWS,   /* FLCE_SKIP_MIN_ROWS: fewest rows for which a forward skips
                               ignored rows (default 2,048) */
  FLCE_OPT_FUSE_DH_DW,      /* FLCE_FUSE_DH_DW: 1 = a vocabulary slab's dH and dW GEMMs run in one
                               launch when the backward has several slabs (default),
                               0 = always two launches */
  FLCE_OPT_DW_EPILOGUE_WARPS,  /* FLCE_DW_EPILOGUE_WARPS: epilogue warps of the dW GEMM at
                                  short K (at most 1,024 rows): 16 (default) or 8 */
  FLCE_OPT_PIPELINE,        /* FLCE_PIPELINE: 1 = a backward of several vocabulary slabs runs
                               each row block in one launch, its units ordered by device-side
                               counters (default), 0 = two launches per slab.  The launch's
                               SM pairs draw units in an order in which every wait points to
                               earlier units, so it completes on however many SMs other work
                               leaves it; each wait is bounded (FLCE_ERR_TIMEOUT) */
  FLCE_OPT_DH_WIDE,         /* FLCE_DH_WIDE: 1 = the dH GEMM of a one-slab backward runs 256 x
                               512 tiles on SM pairs (default), 0 = 256 x 256 */
  FLCE_OPT_GRID_WORKERS,    /* FLCE_GRID_WORKERS: persistent workers (CTAs, or CTA pairs) that
                               each GEMM launch starts, 1..4,096; 0 = as many as the device
                               holds at once (default).  Plans stay those of the device's
                               count: fewer workers leave SMs to other work; more start as
                               resident ones retire (the round-robin units of a GEMM run
                               in further waves; in the pipelined backward, whose workers
                               draw units, the late ones find them taken).  Results do not
                               depend on it */
  FLCE_OPT_COUNT
} flce_option;

/* Set option `opt` to `value` for every later call in this process.
 * FLCE_ERR_INVALID_ARG (nothing changed) for an unknown option or a value
 * outside the range listed above. */
FLCE_API flce_status flce_set_option(flce_option opt, int64_t value);

/* Current value of option `opt` into *value (a host pointer).
 * FLCE_ERR_INVALID_ARG for an unknown option or a NULL value. */
FLCE_API flce_status flce_get_option(flce_option opt, int64_t* value);

/* Diagnostic of the kernels' bounded waits (failure detection without a GPU
 * fault).  Launches one warp that waits, through the same bounded-wait
 * routine as the GEMM pipelines, on an mbarrier nothing arrives on, giving up
 * after `limit_cycles` SM clock cycles (1 .. 2e9).  Synchronises `stream`.
 * Returns FLCE_OK when the wait gave up and returned as designed; the device
 * error word is then set, so the next flce_device_status returns
 * FLCE_ERR_TIMEOUT (and clears it).  The CUDA context stays usable. */
FLCE_API flce_status flce_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/* ---- profiling (CUDA events around each launch, on the launch stream) ---- */

/* Enable (1) or disable (0) per-kernel event timing; enabling clears totals. */
FLCE_API flce_status flce_profile_enable(int enable);

/* Number of kernel kinds the profiler distinguishes. */
FLCE_API int flce_profile_num_kinds(void);

/* Static name of kernel kind `kind` (NULL if out of range). */
FLCE_API const char* flce_profile_kind_name(int kind);

/* Synchronises on the recorded events and returns the accumulated device
 * time (ms) and launch count of kernel kind `kind` since profiling was
 * enabled.  Host pointers. */
FLCE_API flce_status flce_profile_read(int kind, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
