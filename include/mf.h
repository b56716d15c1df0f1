/*
 * mf.h -- packed native-resolution joint attention for NVIDIA B300 (sm_103a).
 *
 * The operation (Mage-Flow, "An Efficient Native-Resolution Foundation Model
 * for Image Generation and Editing"; review page, section "Native-Resolution
 * MMDiT"; Hugging Face paper page, Highlights "Native resolution" and
 * "System-level speed"; model card, section "Architecture"):
 *
 *   Images of different sizes become 16x-downsampled latent grids of
 *   (H/16)*(W/16) tokens (review, section "Mage-VAE": patchification is
 *   absorbed into the tokenizer).  Each sample's text tokens and image tokens
 *   are concatenated [text; image] and samples are packed back to back under a
 *   token budget.  Joint self-attention runs inside each sample only, confined
 *   by cumulative per-sample offsets (cu_seqlens) instead of a mask, with
 *   per-sample 2D rotary embedding on Q and K.
 *
 * RoPE layout (the pages name per-sample 2D RoPE but not its layout; this
 * library fixes it): head_dim split in half, the first half rotated by the
 * token's latent row, the second half by its column; pair (2i, 2i+1) of a half
 * turns at frequency theta^(-2i/(head_dim/2)); x0' = x0 cos - x1 sin,
 * x1' = x0 sin + x1 cos; text tokens are not rotated.  Image token j of a
 * sample (0-based, row-major, row = index along the height) has
 * (row, col) = (j / (W/16), j % (W/16)).
 *
 * Conventions shared by every call:
 *   - Device tensors are caller-owned and contiguous.  Q, K, V, O, dO, dQ, dK,
 *     dV are bf16 [total_tokens, heads, head_dim] (row stride heads*head_dim),
 *     16-byte aligned.  LSE is float32 [heads, total_tokens], natural log of
 *     the scaled logits' sum of exponentials.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     launch is enqueued on it.  Only mf_check synchronizes it (to read the
 *     status word); mf_pack_plan and the attention calls never do.
 *   - The library allocates no device memory: the caller passes workspaces
 *     sized by the *_workspace_size calls.  It keeps no state besides a
 *     per-thread copy of the last CUDA error message.
 *   - Arguments are validated before anything is launched; a bad argument
 *     returns MF_ERR_INVALID_ARG and leaves every buffer untouched.
 *   - Every wait inside a kernel is bounded (a few seconds).  A kernel that
 *     gives up sets the plan's device status word and exits cleanly;
 *     mf_check() reports it as MF_ERR_TIMEOUT, and mf_last_cuda_error() then
 *     names the kernel, the barrier of the first timeout and how many CTAs
 *     gave up.  Every plan carries its own status: check each plan whose
 *     kernels ran.
 *   - softmax_scale <= 0 selects 1/sqrt(head_dim).
 *   - Precision: Q, K, V, O and the gradients are bf16 with fp32
 *     accumulation.  The logit product R(Q) R(K)^T is computed from fp16
 *     rotated rows (R(Q) pre-multiplied by softmax_scale * log2 e), whose
 *     finer significand keeps the rotation's rounding error 8x below bf16's.
 *     Domain: every rotated, scaled value must stay within the fp16 range
 *     (|s log2(e) R(q)|, |R(k)| <= 65504); a value beyond it is reported as
 *     MF_ERR_RANGE by mf_check, never saturated silently.
 *   - Samples are independent for any input: no value of one sample, finite
 *     or not, reaches another sample's outputs.
 *   - head_dim must be 64 or 128 (MF_ERR_UNSUPPORTED otherwise).
 */
#ifndef MF_H_
#define MF_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MF_API __attribute__((visibility("default")))
#else
#define MF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MF_OK = 0,
  MF_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misaligned pointer, short workspace */
  MF_ERR_UNSUPPORTED = 2, /* head_dim not 64/128, too many samples, grid side > 1024 */
  MF_ERR_BUDGET = 3,      /* not even the first sample fits the token budget */
  MF_ERR_CUDA = 4,        /* a CUDA call failed; see mf_last_cuda_error() */
  MF_ERR_TIMEOUT = 5,     /* a kernel's bounded wait expired (reported by mf_check) */
  MF_ERR_RANGE = 6        /* a rotated, scaled Q or K value left the fp16 range of the
                             logit MMA (|value| > 65504; reported by mf_check) */
} mf_status;

/* One sample of a pack: text length in tokens, image height and width in
 * pixels (positive multiples of 16, or both 0 for a text-only sample with
 * text_len > 0), and its latent frames: 1 (or 0) for a
 * generation sample, 2 for an edit sample, whose source and target latents
 * (the same size) follow its text as frames 0 and 1 (review, editing-model
 * section: (h, w, f) positions tell source tokens from target tokens). */
typedef struct {
  int32_t text_len;
  int32_t height;
  int32_t width;
  int32_t frames;
} mf_sample;

/* Largest supported pack (samples) and latent grid side. */
#define MF_MAX_SAMPLES 4096
#define MF_MAX_GRID 1024
/* Rows per attention tile; the work list counts tiles of this size. */
#define MF_TILE 128

/* A pack plan.  Filled by mf_pack_plan; every pointer points into the
 * caller's plan workspace (device memory) and stays valid as long as it. */
typedef struct {
  int32_t n_samples;    /* samples packed: the longest prefix within the budget */
  int32_t total_tokens; /* cu_seqlens[n_samples] */
  int32_t max_seqlen;   /* max_i L_i */
  int32_t max_grid;     /* max_i max(H_i/16, W_i/16) */
  int32_t head_dim;     /* head_dim the RoPE table was built for */
  int32_t n_tiles;      /* sum_i ceil(L_i / MF_TILE) */
  int32_t n_pairs;      /* sum_i ceil(L_i / (2 * MF_TILE)): forward work units */
  int32_t *cu_seqlens;  /* device int32 [n_samples + 1], exclusive scan of L_i */
  int32_t *pos;         /* device int32 [total_tokens][2]: (row, col); text = (-1, -1) */
  int32_t *frame;       /* device int32 [total_tokens]: latent frame; text = -1 */
  int32_t rope_axes;    /* 2: (row, col) RoPE; 3: (frame, row, col) RoPE */
  float *rope_cs;       /* device float32 [grid][a/2][2]: cos, sin of p * theta^(-2i/a) for the
                           row/col slices of a dims (a = head_dim/2 with 2 axes, 7 head_dim/16
                           with 3), grid > max_grid */
  float *rope_f;        /* device float32 [2][head_dim/16][2]: the frame slice's table (3 axes;
                           NULL with 2) */
  int32_t *order;       /* device int32 [n_samples][4]: (sample, first tile, first tile pair, 0),
                           longest sample first */
  int32_t *status;      /* device int32 status word written by kernels that time out */
} mf_plan;

/* Bytes of device workspace mf_pack_plan needs for this request.  Validates
 * the request like mf_pack_plan (same error codes); `samples` is host memory. */
MF_API mf_status mf_pack_plan_workspace_size(const mf_sample *samples, int32_t n_samples,
                                      int32_t token_budget, int32_t head_dim, int32_t rope_axes,
                                      size_t *bytes);

/* Plan a pack (review, section "Native-Resolution MMDiT": variable-length
 * latent token rows packed under a fixed token budget, unpadded text, per-
 * sample cumulative offsets).  The longest prefix of `samples` whose total
 * token count is <= token_budget is packed (token_budget 0 = no budget).
 *   samples      host array [n_samples]; 0 <= n_samples <= MF_MAX_SAMPLES
 *   head_dim     64 or 128 (sizes the RoPE table)
 *   rope_axes    2: the first half of head_dim turns by the latent row, the
 *                second by the column; 3: head_dim is cut into frame | row |
 *                col slices of head_dim/8, 7 head_dim/16 and 7 head_dim/16
 *                dims (the edit model's (h, w, f) positions).  Pair i of an
 *                a-dim slice turns at theta^(-2i/a) times the token's index on
 *                that axis.  Edit samples (frames = 2) need 3.
 *   rope_theta   RoPE base (> 0; 10000 is the usual value)
 *   workspace    device memory of at least mf_pack_plan_workspace_size bytes,
 *                256-byte aligned
 *   plan_out     host struct, filled on success
 * The host computes the plan's scalars (packed count, total tokens, maxima,
 * tile and tile-pair counts) from `samples` and returns without waiting on
 * `stream`; the device prefix scan, the per-token id expansion and the RoPE
 * table run on `stream`.  The scan recomputes the scalars and, if they differ
 * from the host's, sets the status word so that mf_check fails with
 * MF_ERR_CUDA.  `samples` is copied with cudaMemcpyAsync: pageable memory is
 * free for reuse on return, page-locked memory only once `stream` has run
 * the copy.
 * Errors: MF_ERR_INVALID_ARG (null pointer, text_len < 0, H or W not a
 * positive multiple of 16 (both 0 needs text_len > 0), frames not in
 * {0, 1, 2}, frames = 2 with
 * rope_axes 2, rope_axes not 2 or 3, total tokens >= 2^31, short or
 * misaligned workspace), MF_ERR_UNSUPPORTED, MF_ERR_BUDGET, MF_ERR_CUDA. */
MF_API mf_status mf_pack_plan(const mf_sample *samples, int32_t n_samples, int32_t token_budget,
                       int32_t head_dim, int32_t rope_axes, float rope_theta, void *workspace,
                       size_t workspace_bytes, mf_plan *plan_out, void *stream);

/* Bytes of device workspace mf_attn_fwd needs: an fp16 rotated copy R(K)
 * [total_tokens, heads, head_dim] (the streamed operand of the logit
 * product) and the attention kernel's 256-byte work counter. */
MF_API mf_status mf_attn_fwd_workspace_size(int32_t total_tokens, int32_t heads, int32_t head_dim,
                                            size_t *bytes);

/* Forward: for every sample i and head h,
 *   O = softmax(s * R(Q) R(K)^T) V,  LSE = logsumexp(s * R(Q) R(K)^T)  (rows)
 * over that sample's tokens only, R = the 2D rotation above.
 *   q, k, v     device bf16 [plan->total_tokens, heads, head_dim]
 *   workspace   device memory of mf_attn_fwd_workspace_size bytes, 256-byte
 *               aligned (contents on entry are ignored; a first kernel writes
 *               the rotated K copy that the attention kernel streams, while
 *               each Q tile is rotated in the attention kernel's prologue and
 *               never written back)
 *   o           device bf16, same shape (written)
 *   lse         device float32 [heads, plan->total_tokens] (written)
 * Errors: MF_ERR_INVALID_ARG (null/misaligned pointer, heads < 1, head_dim
 * different from the plan's, short workspace), MF_ERR_UNSUPPORTED,
 * MF_ERR_CUDA.  A rotated value beyond the fp16 range shows up as
 * MF_ERR_RANGE from mf_check. */
MF_API mf_status mf_attn_fwd(const void *q, const void *k, const void *v, const mf_plan *plan,
                      int32_t heads, int32_t head_dim, float softmax_scale, void *workspace,
                      size_t workspace_bytes, void *o, float *lse, void *stream);

/* Bytes of device workspace mf_attn_bwd needs: float32 row dots
 * D = rowsum(dO * O) [heads, total_tokens], a float32 dQ accumulator
 * [total_tokens, heads, head_dim], an fp16 rotated copy s log2(e) R(Q) of the
 * same shape (the streamed operand of the backward's logit product) and the
 * attention kernel's 256-byte work counter (each section 256-byte aligned). */
MF_API mf_status mf_attn_bwd_workspace_size(int32_t total_tokens, int32_t heads, int32_t head_dim,
                                     size_t *bytes);

/* Backward of mf_attn_fwd with respect to the un-rotated inputs:
 *   P = exp(s R(Q) R(K)^T - LSE);  dV = P^T dO;  dP = dO V^T;
 *   D = rowsum(dO * O);  dS = P * (dP - D);
 *   dQ = R^T (s dS R(K));  dK = R^T (s dS^T R(Q))
 *   q, k, v, o, dout  device bf16 [total_tokens, heads, head_dim]
 *   lse               device float32 [heads, total_tokens] from mf_attn_fwd
 *   workspace         device memory of mf_attn_bwd_workspace_size bytes,
 *                     256-byte aligned (contents on entry are ignored; each
 *                     K tile is rotated in the attention kernel's prologue
 *                     and never written back)
 *   dq, dk, dv        device bf16 [total_tokens, heads, head_dim] (written)
 * Errors as mf_attn_fwd, plus a short workspace (MF_ERR_INVALID_ARG). */
MF_API mf_status mf_attn_bwd(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, const mf_plan *plan, int32_t heads,
                      int32_t head_dim, float softmax_scale, void *workspace,
                      size_t workspace_bytes, void *dq, void *dk, void *dv, void *stream);

/* Size of the fixed device scratch behind mf_attn_bwd_noalloc (128 MiB). */
#define MF_NOALLOC_SCRATCH_BYTES (128u * 1024u * 1024u)

/* mf_attn_bwd for callers that cannot allocate device memory.  (The Mage-Flow
 * pages have no counterpart: this is a deployment convenience of the
 * library.)  Some callers cannot call cudaMalloc where they run the backward:
 * an engine plugin whose execute step may not allocate, a runtime whose pool
 * already owns all device memory, or a latency-critical loop that avoids
 * cudaMalloc because it can synchronize the device.  This call takes the same
 * arguments as mf_attn_bwd minus the workspace and uses instead a fixed
 * MF_NOALLOC_SCRATCH_BYTES array of device memory that the library reserves
 * on every GPU that loads it, held until the process exits.  It allocates
 * nothing itself.
 *   - A call looks up that array's device address on the current device
 *     (a device reset reloads the library's GPU code, and the array may then
 *     sit elsewhere) and caches it per device.  A call made while `stream`
 *     is capturing uses the cached address instead, so make a first call on
 *     each device before any stream capture.
 *   - Packs whose backward workspace (mf_attn_bwd_workspace_size) exceeds
 *     MF_NOALLOC_SCRATCH_BYTES return MF_ERR_UNSUPPORTED without launching;
 *     use mf_attn_bwd with a caller workspace for those.
 *   - Every call on a device shares the one array.  Each call overwrites what
 *     it needs before reading it, so earlier contents never leak into a
 *     result, but calls that overlap on the GPU (e.g. on two streams at once)
 *     race on the array and must be serialized by the caller.
 * Other arguments, results and errors as mf_attn_bwd. */
MF_API mf_status mf_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                     const float *lse, const void *dout, const mf_plan *plan,
                                     int32_t heads, int32_t head_dim, float softmax_scale,
                                     void *dq, void *dk, void *dv, void *stream);

/* The memory-bound chains around one joint-attention block, each one fused
 * pass over HBM (review, kernel-fusion section: normalisation, adaptive
 * modulation, RoPE application, gating and the residual add run fused
 * instead of as separate kernels).  The pages give no exact form; the
 * plainest reading for a diffusion-transformer block is used.  The
 * projections around them are plain matrix products left to the caller
 * (e.g. cuBLAS):
 *     y   = mf_norm_modulate(x)               LN(x) (1 + scale_s) + shift_s
 *     qkv = y W_qkv                           [q | k | v], each [heads, head_dim]
 *     o   = mf_attn_fwd_qkv(qkv)              RoPE fused into its first pass
 *     z   = o W_o
 *     out = mf_gate_residual(x, z)            x + gate_s * z
 * Modulation vectors are per sample of the plan (s = the sample a token
 * belongs to), bf16 [n_samples, hidden]; x, y, z, out are bf16
 * [total_tokens, hidden], 16-byte aligned.
 *
 * mf_norm_modulate: LayerNorm over the hidden size without affine (mean and
 * population variance of the row, eps inside the square root, fp32), then
 * the modulation, rounded to bf16.  hidden in {1024, 2048, 3072, 4096, 6144,
 * 8192} (else MF_ERR_UNSUPPORTED). */
MF_API mf_status mf_norm_modulate(const void *x, const mf_plan *plan, int32_t hidden, const void *shift,
                                  const void *scale, float eps, void *y, void *stream);

/* out = x + gate_s * z in fp32, rounded to bf16 (hidden a multiple of 8;
 * out may be x). */
MF_API mf_status mf_gate_residual(const void *x, const void *z, const mf_plan *plan, int32_t hidden,
                                  const void *gate, void *out, void *stream);

/* mf_attn_fwd on the output of a QKV projection: qkv is bf16
 * [total_tokens, 3 * heads * head_dim], each row [q | k | v] with every
 * third ordered [head][dim].  The first pass reads q and k from those rows
 * and rotates them into the workspace (so the split and the RoPE cost no
 * extra pass), and the attention kernel reads v in place.  Workspace, o, lse
 * and errors as mf_attn_fwd. */
MF_API mf_status mf_attn_fwd_qkv(const void *qkv, const mf_plan *plan, int32_t heads, int32_t head_dim,
                                 float softmax_scale, void *workspace, size_t workspace_bytes, void *o,
                                 float *lse, void *stream);

/* Classifier-free guidance over a pack whose samples come in (conditional,
 * unconditional) pairs: samples 2p and 2p + 1 are the two branches of prompt
 * p, run in one packed forward (review, section on CFG).  For the image rows
 * of each pair (the rows with an image position; they end each sample, so
 * row j from the end of one pairs with row j from the end of the other):
 *     out[cond row] = u + guidance * (c - u)
 * in fp32, rounded to bf16.  The pages do not print the combination; this is
 * the standard reading.  Other rows of `out` are left untouched, and `out`
 * may be `o` itself.
 *   o, out   device bf16 [plan->total_tokens, heads, head_dim]
 * Errors: as mf_attn_fwd's argument checks, MF_ERR_INVALID_ARG for an odd
 * sample count or a non-finite guidance; a pair whose image sizes differ is
 * skipped and mf_check reports MF_ERR_INVALID_ARG. */
MF_API mf_status mf_cfg_combine(const void *o, const mf_plan *plan, int32_t heads, int32_t head_dim,
                                float guidance, void *out, void *stream);

/* Synchronize `stream`, then read and clear the plan's device status word:
 * MF_OK, MF_ERR_TIMEOUT, MF_ERR_RANGE, MF_ERR_INVALID_ARG (a mismatched CFG
 * pair), or MF_ERR_CUDA for a failed synchronization, a misaligned shared-
 * memory window or a device pack scan that disagreed with the host's plan. */
MF_API mf_status mf_check(const mf_plan *plan, void *stream);

/* Profiling aid: the next mf_attn_fwd or mf_attn_bwd call made by this
 * thread records `start_event` on its stream right before its main attention
 * kernel and `stop_event` right after it (cudaEvent_t handles created by the
 * caller; both NULL clears the request).  The request is consumed by that
 * one call.  This lets a caller time the tensor-core kernel alone, without
 * the backward's pre- and post-processing kernels.  MF_ERR_INVALID_ARG if
 * exactly one of the two is NULL. */
MF_API mf_status mf_record_main_kernel(void *start_event, void *stop_event);

/* Test aid for the timeout path (the Mage-Flow pages have no counterpart).
 * While `flags` is set, the attention calls made by this thread launch their
 * main kernel with the TMA producer dropping its streamed-tile loads:
 *   MF_DEBUG_DROP_FWD_KV   mf_attn_fwd issues no K/V tile loads,
 *   MF_DEBUG_DROP_BWD_QDO  mf_attn_bwd issues no q~/dO tile loads,
 * so the consumers' bounded waits run out (about 4 s), every warp leaves its
 * loop, the kernel frees its TMEM and exits, and mf_check reports
 * MF_ERR_TIMEOUT.  Nothing faults or hangs and the CUDA context stays usable.
 * The outputs of such a call are undefined.  0 restores normal operation.
 * MF_ERR_INVALID_ARG for unknown bits. */
#define MF_DEBUG_DROP_FWD_KV 1
#define MF_DEBUG_DROP_BWD_QDO 2
MF_API mf_status mf_debug_inject(int32_t flags);

/* Static description of a status code. */
MF_API const char *mf_status_string(mf_status status);

/* Message of the last CUDA error seen by this thread, or of the last timeout
 * mf_check reported ("" if none). */
MF_API const char *mf_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MF_H_ */
