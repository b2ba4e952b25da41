/*
 * flce.h — C ABI of the GB300 (sm_103a) fused linear cross-entropy library.
 *
 * Fused linear cross-entropy (FLCE) computes the language-model-head loss
 *
 *     z_iv  = h_i . w_v                      (logits Z = H W^T, never stored)
 *     lse_i = log sum_v exp(z_iv)
 *     loss  = sum_{i valid} (lse_i - z_{i,y_i}) / n      (reduction "mean")
 *
 * and its gradients
 *
 *     G     = (softmax(Z) - onehot(y)) * grad_scale / n   (rows of ignored tokens are 0)
 *     dH    = G W          dW = G^T H
 *
 * without writing the [N, V] logits to device memory.
 *
 * Sources: "Liger Kernel: Fused Triton Kernels for LLM Training", section "The
 * Architecture" (1. Fused Linear Cross-Entropy with Online LogSumExp: the
 * stable LSE, target-logit extraction, only the loss and per-token normalisers
 * kept; 2. In-Kernel Gradient Computation During the Backward Pass: softmax minus
 * one-hot, dL/dH = (dL/dZ) W, dL/dW = (dL/dZ)^T H, tile logits recomputed from the
 * saved LSE), with the 1/N mean factor of the same page's section
 * "Implementation: Simulating Fused Linear Cross-Entropy in Python"; GPU MODE
 * lecture 28 notes, cross-entropy section: the fused loss takes hidden states
 * (B*S, hidden), the LM-head weight (vocab, hidden) and labels, and replaces
 * PyTorch's cross entropy with reduction="mean".
 *
 * Conventions for every entry point
 *   - Matrices are dense, row-major, device memory: H is bf16 [N, D], W is bf16
 *     [V, D], labels are int32 [N]. bf16 values are passed as their uint16_t bit
 *     patterns. Every device pointer must be 16-byte aligned and D % 8 == 0 (the
 *     tensor-memory-access engine needs 16-byte row strides).
 *   - Ownership: the caller allocates and frees every buffer, the workspace
 *     included. The library allocates no device memory and keeps no pointer after
 *     a call returns (its tensor-memory-access descriptors are encoded on the host
 *     at each call and passed to the kernels by value).
 *   - Asynchrony: calls enqueue work on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream) and return before it finishes. Outputs are
 *     overwritten, never accumulated into.
 *   - Host-side errors are returned immediately and nothing is enqueued.
 *     Data-dependent errors found on the device (a label out of range, a wait
 *     that ran out of time) are written to the optional device word `status`;
 *     read it with flce_check_status(). When a device error is reported the
 *     outputs of that call are undefined, but no memory outside the given
 *     buffers is touched.
 *   - Labels equal to ignore_index contribute neither to the loss nor to the
 *     gradients and are not counted in n. If every label is ignored the loss
 *     and the gradients are 0 (not NaN); lse is still written for every token.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (host) and device status words. */
enum {
  FLCE_OK = 0,
  FLCE_ERR_NULL = 1,        /* a required pointer is NULL */
  FLCE_ERR_SHAPE = 2,       /* N, D or V < 1, or too large for int32 indexing */
  FLCE_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned, or D % 8 != 0 */
  FLCE_ERR_WORKSPACE = 4,   /* workspace smaller than flce_workspace_size() */
  FLCE_ERR_OPTION = 5,      /* an option is out of its range */
  FLCE_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed */
  FLCE_ERR_DEVICE = 7,      /* the current device is not an sm_103 GPU */
  FLCE_ERR_LABEL_RANGE = 8, /* device: a label is outside [0, V) and is not ignore_index */
  FLCE_ERR_TIMEOUT = 9      /* device: a pipeline wait exceeded timeout_ns */
};

/* FLCE_REDUCTION_NONE (per-token loss) is accepted by flce_forward and
 * flce_forward_noalloc only; flce_forward_backward rejects it with FLCE_ERR_OPTION. */
enum { FLCE_REDUCTION_MEAN = 0, FLCE_REDUCTION_SUM = 1, FLCE_REDUCTION_NONE = 2 };
enum { FLCE_DTYPE_F32 = 0, FLCE_DTYPE_BF16 = 1 };

typedef struct flce_options {
  int32_t ignore_index; /* label value that marks an ignored token; default -100 */
  int32_t reduction;    /* FLCE_REDUCTION_MEAN (default), _SUM, or _NONE (forward only) */
  float grad_scale;     /* upstream dL/dloss multiplying G; default 1 */
  float normalizer;     /* > 0: mean divides by this instead of the device-counted n
                           (a global token count for data-parallel callers); default 0 */
  int32_t dw_dtype;     /* dW element type: FLCE_DTYPE_F32 (default) or FLCE_DTYPE_BF16 */
  int32_t v_splits;     /* forward: vocabulary ranges per token block; 0 = planned */
  int64_t n_block;      /* backward: tokens per block (multiple of 128); 0 = planned */
  int64_t v_chunk;      /* backward: vocabulary ids per G chunk (multiple of 256); 0 = planned */
  int64_t timeout_ns;   /* limit of every device-side pipeline wait; 0 = 2 s */
  void* const* trace_events; /* optional array of caller-created cudaEvent_t: event 0 is
                                recorded on `stream` before the first kernel of a call and
                                event k after its k-th kernel (k <= trace_capacity - 1), so
                                that kernel k lasts elapsed(event k-1, event k); NULL = off */
  int32_t trace_capacity;    /* number of events in trace_events */
  int32_t reserved;          /* must be 0 */
} flce_options;

/* The execution plan the library will use for a problem on the current device. */
typedef struct flce_plan_info {
  int64_t n_block;           /* tokens per backward block */
  int64_t v_chunk;           /* vocabulary ids per G chunk */
  int32_t n_blocks;          /* backward token blocks */
  int32_t n_chunks;          /* backward vocabulary chunks */
  int32_t v_splits;          /* forward vocabulary ranges per 128-token block */
  int32_t kernel_launches;   /* kernels one call launches (the status reset is a memset, not counted) */
  size_t workspace_bytes;    /* the same value flce_workspace_size() returns */
  size_t plan_bytes;         /* workspace this plan actually touches on this device */
} flce_plan_info;

/* Fill *opt with the defaults listed above. */
void flce_default_options(flce_options* opt);

/*
 * Bytes of device workspace that flce_forward_backward and flce_forward need for
 * this problem and these options (opt may be NULL for the defaults). The
 * workspace holds the per-(token, vocabulary range) partial max/sum-exp pairs,
 * the target logits, per token the (max, 1 / sum, 1 - p of the target) the
 * gradient is formed from (16 bytes), one bf16 chunk of G ([n_block, v_chunk]) and, when the
 * vocabulary spans several chunks, an fp32 [n_block, D] dH accumulator (plus an
 * fp32 [V, D] dW accumulator only for bf16 dW with several token blocks). It is
 * the whole extra device memory of a call and is far below the N*V*4 bytes of
 * fp32 logits. Returns FLCE_OK and writes *bytes, or an error code
 * (FLCE_ERR_NULL, FLCE_ERR_SHAPE, FLCE_ERR_ALIGN for D % 8 != 0, FLCE_ERR_OPTION).
 */
int flce_workspace_size(int64_t N, int64_t D, int64_t V, const flce_options* opt, size_t* bytes);

/*
 * Bytes of device workspace that the forward-only calls (flce_forward,
 * flce_forward_fp8, flce_forward_shard) need: the forward pieces of
 * flce_workspace_size without the G chunk and the dH / dW accumulators,
 *     align256(8 * S * 256 * ceil(N / 256)) + 3 * align256(4 * N) + 256 bytes,
 * S = opt->v_splits (vocabulary ranges per 128-token block; 0 = the largest
 * count the planner can choose, min(ceil(V / 256), 128), so that the size does
 * not depend on the device). Independent of D. Same errors as flce_workspace_size.
 */
int flce_forward_workspace_size(int64_t N, int64_t D, int64_t V, const flce_options* opt,
                                size_t* bytes);

/*
 * Describe the plan for an (N, D, V) problem on the current device: token
 * blocks and vocabulary chunks of the backward pass, vocabulary ranges of the
 * forward pass, kernel launches per call, workspace bytes. want_dh / want_dw
 * (0 or 1) say which gradients the call will request; both 0 describes
 * flce_forward. Needs a current CUDA device (FLCE_ERR_CUDA / FLCE_ERR_DEVICE
 * otherwise); launches nothing.
 */
int flce_get_plan(int64_t N, int64_t D, int64_t V, const flce_options* opt, int32_t want_dh,
                  int32_t want_dw, flce_plan_info* info);

/*
 * Loss, per-token LSE and both gradients in one call: the fused linear
 * cross-entropy forward and backward of "Liger Kernel: Fused Triton Kernels for
 * LLM Training", section "The Architecture" (1. the logits tile by tile with an
 * online log-sum-exp and the target logit taken on the fly, only the loss and
 * the per-token log-sum-exp kept; 2. the logits recomputed from that
 * log-sum-exp, dL/dz = softmax - one-hot formed in the kernel, dL/dH = (dL/dz) W
 * and dL/dW = (dL/dz)^T H), with the 1/N mean of the page's Python simulation
 * and the argument layout of the GPU MODE lecture 28 notes, cross-entropy
 * section (hidden states (B*S, hidden), LM-head weight (vocab, hidden), labels).
 * The recompute takes the forward's per-token row maximum, sum of exponentials
 * and 1 - p of the target (the pieces of the log-sum-exp, kept in the workspace),
 * so that a confident token's gradient entry -scale * (1 - p) keeps fp32
 * precision.
 *   H       bf16 [N, D]   hidden states (input)
 *   W       bf16 [V, D]   LM-head weight (input)
 *   labels  int32 [N]     target ids in [0, V) or ignore_index (input)
 *   loss    fp32 [1]      scalar loss (output, required)
 *   lse     fp32 [N]      log-sum-exp of each token's logits (output, may be NULL)
 *   dH      bf16 [N, D]   dL/dH (output, may be NULL to skip the dH product)
 *   dW      [V, D]        dL/dW, fp32 or bf16 per opt->dw_dtype (output, may be NULL)
 *   workspace, ws_bytes   device scratch of at least flce_workspace_size() bytes
 *   status  int32 [1]     device status word (may be NULL); set to FLCE_OK at the
 *                         start of the call and to a device error code on failure
 *   stream  cudaStream_t
 */
int flce_forward_backward(const uint16_t* H, const uint16_t* W, const int32_t* labels, int64_t N,
                          int64_t D, int64_t V, const flce_options* opt, float* loss, float* lse,
                          uint16_t* dH, void* dW, void* workspace, size_t ws_bytes,
                          int32_t* status, void* stream);

/*
 * Forward only: the loss and (optionally) lse, without any gradient work (the
 * evaluation path): "Liger Kernel: Fused Triton Kernels for LLM Training",
 * section "The Architecture", 1. (chunked logits, online log-sum-exp, target
 * logit extraction; nothing of size N x V stored). Same arguments and rules as
 * flce_forward_backward, except that the workspace need only hold
 * flce_forward_workspace_size() bytes and that with reduction
 * FLCE_REDUCTION_NONE `loss` is fp32 [N]: each token's lse_i - z_{i,y_i}, and 0
 * for ignored tokens (the per-token loss of PyTorch's reduction="none", which the
 * GPU MODE lecture 28 notes' drop-in replaces).
 */
int flce_forward(const uint16_t* H, const uint16_t* W, const int32_t* labels, int64_t N, int64_t D,
                 int64_t V, const flce_options* opt, float* loss, float* lse, void* workspace,
                 size_t ws_bytes, int32_t* status, void* stream);

/*
 * FP8 operand variant (the lecture notes' open question on FP8 matrix units):
 * the logits are computed from E4M3 operands with per-tensor scales,
 *     z_iv = scale_h * scale_w * (H8_i . W8_v)     (E4M3 x E4M3, fp32 accumulate),
 * with tcgen05 kind::f8f6f4 for both logits products (the forward LSE pass and
 * the recompute of G); loss, lse and G follow from z exactly as in the bf16 path.
 * The gradient products take the bf16 tensors the FP8 operands were made from:
 * dH = G W and dW = G^T H (straight through the quantisation).
 *   H8 [N, D], W8 [V, D]  E4M3 bytes, row-major, 16-byte aligned, D % 16 == 0
 *   scale_h, scale_w      device pointers, each to one positive finite fp32 scale
 *                         (dequantised value = scale * e4m3), read by the kernels,
 *                         so a scale computed on the device (flce_quantize_e4m3)
 *                         needs no host round trip; 4-byte aligned. Only the
 *                         pointers are checked (FLCE_ERR_NULL, FLCE_ERR_ALIGN):
 *                         the values are read on the device, and a scale that
 *                         is not positive and finite gives meaningless outputs
 *   H, W                  bf16 [N, D], [V, D] (flce_forward_backward_fp8 only)
 * Other arguments, outputs, workspace (flce_workspace_size) and errors as in
 * flce_forward / flce_forward_backward.
 */
int flce_forward_fp8(const uint8_t* H8, const float* scale_h, const uint8_t* W8,
                     const float* scale_w,
                     const int32_t* labels, int64_t N, int64_t D, int64_t V,
                     const flce_options* opt, float* loss, float* lse, void* workspace,
                     size_t ws_bytes, int32_t* status, void* stream);
int flce_forward_backward_fp8(const uint8_t* H8, const float* scale_h, const uint8_t* W8,
                              const float* scale_w,
                              const uint16_t* H, const uint16_t* W, const int32_t* labels,
                              int64_t N, int64_t D, int64_t V, const flce_options* opt,
                              float* loss, float* lse, uint16_t* dH, void* dW, void* workspace,
                              size_t ws_bytes, int32_t* status, void* stream);

/*
 * Vocabulary shards: the local half of a vocabulary-parallel split (the lecture
 * notes' open question on vocabularies above a million ids, where the chunks grow
 * too large and the vocabulary has to be split). A device holding rows [v_offset, v_offset + V_shard) of W, as W_shard
 * ([V_shard, D] bf16, its row 0 being row v_offset of W), runs the two calls
 * below; the caller's collective combines the shards between them. labels hold
 * ids of the whole vocabulary [0, V_total) (or ignore_index) and are the same on
 * every shard; 0 <= v_offset, v_offset + V_shard <= V_total <= 2^30.
 *
 * flce_forward_shard writes, per token i (fp32 [N] each, 4-byte aligned):
 *   m[i]  = max over the shard's ids v of z_iv
 *   s[i]  = sum over the shard's ids v of exp(z_iv - m[i])
 *   zt[i] = z_{i,y_i} when y_i lies in the shard, else 0 (also 0 for ignored tokens)
 * The shards combine as  M_i = max_r m_r[i],  lse_i = M_i + log sum_r s_r[i] exp(m_r[i] - M_i),
 * z_t,i = sum_r zt_r[i]  (an all-reduce with max, then sums), and
 * loss = sum over non-ignored i of (lse_i - z_t,i) / n (sum: without the / n).
 *
 * flce_backward_shard takes that lse (fp32 [N], 4-byte aligned) and writes the
 * shard's part of the gradients, G_iv = (exp(z_iv - lse_i) - [v = y_i]) * scale
 * over the shard's ids (scale = grad_scale / n as in flce_forward_backward, n
 * counted from the labels, or the normalizer option). Having only lse, it forms
 * the target entry as p * scale - scale, so for a token whose p is close to 1 that
 * entry carries the fp32 rounding of lse (about 2^-24 |lse| of the scale), where
 * flce_forward_backward, which keeps 1 - p from its own forward, does not:
 *   dH_part  fp32 [N, D], 16-byte aligned: G W_shard; the caller sums the parts of
 *            all shards (then rounds to bf16 if it wants bf16 dH); nullable
 *   dW_shard [V_shard, D], fp32 or bf16 (dw_dtype): the shard's rows of dW; nullable
 * (not both null). Workspace: flce_workspace_size(N, D, V_shard, opt). Errors as in
 * flce_forward_backward, plus FLCE_ERR_SHAPE for a shard outside [0, V_total) and
 * FLCE_ERR_NULL for a missing m, s, zt or lse; a label outside [0, V_total) sets
 * FLCE_ERR_LABEL_RANGE in *status.
 */
int flce_forward_shard(const uint16_t* H, const uint16_t* W_shard, const int32_t* labels,
                       int64_t N, int64_t D, int64_t V_shard, int64_t v_offset, int64_t V_total,
                       const flce_options* opt, float* m, float* s, float* zt, void* workspace,
                       size_t ws_bytes, int32_t* status, void* stream);
int flce_backward_shard(const uint16_t* H, const uint16_t* W_shard, const int32_t* labels,
                        int64_t N, int64_t D, int64_t V_shard, int64_t v_offset, int64_t V_total,
                        const flce_options* opt, const float* lse, float* dH_part, void* dW_shard,
                        void* workspace, size_t ws_bytes, int32_t* status, void* stream);

/*
 * Per-tensor E4M3 quantisation on the device: the operand preparation the FP8
 * variant expects (the reading of the lecture notes' FP8 question that the FP8
 * entry points follow). Over the bf16 tensor x [n]:
 *     amax  = max_i |x_i|
 *     scale = amax / 448, computed in double and rounded to fp32 (1 if amax == 0)
 *     inv   = 448 / amax, computed in double, rounded to fp32 and capped at the
 *             largest finite fp32 (reached only for amax below about 1.3e-36;
 *             1 if amax == 0)
 *     q_i   = e4m3(x_i * inv), the product in fp32, rounded to the nearest
 *             code (ties to the even code), saturating at +-448; a zero result
 *             is encoded as +0
 * writes q (uint8 [n]), out[0] = scale and out[1] = amax (two device floats, the
 * first usable directly as scale_h / scale_w of the FP8 entry points). x must be
 * finite. n % 8 == 0, x and q 16-byte aligned, out 8-byte aligned. Enqueues a
 * 4-byte reset and two kernels on `stream`; no host synchronisation, no
 * allocation. Errors: FLCE_ERR_NULL, FLCE_ERR_SHAPE (n < 1), FLCE_ERR_ALIGN.
 */
int flce_quantize_e4m3(const uint16_t* x, int64_t n, uint8_t* q, float* out, void* stream);

/*
 * flce_forward, for callers that cannot allocate device memory at call time and
 * so cannot pass a workspace: for example a plugin whose host application owns
 * all device memory and gives it no allocator, or a server that reserved its
 * memory at start-up so that no call can fail with out-of-memory. The pages
 * have no counterpart of this entry point; it exists only for such callers.
 *   - Arguments and results are those of flce_forward without the workspace;
 *     the caller still passes H, W, labels, loss, lse and status.
 *   - Scratch is one 32 MiB array in device memory owned by the library. Every
 *     GPU that loads it keeps it until the process exits. The entry point calls
 *     no cudaMalloc, cudaFree or allocating library routine.
 *   - Set-up, once per device: the array is created when the CUDA runtime loads
 *     this part of the library on a device, which with CUDA's default lazy
 *     module loading is the first call on that device (the first call then also
 *     looks up the array's device address with that device current). That first
 *     call can therefore take 32 MiB of device memory and fail with
 *     FLCE_ERR_CUDA if none is left; every later call on the device allocates
 *     nothing. Callers that reserve memory up front should make the set-up call
 *         flce_forward_noalloc(NULL, NULL, NULL, 0, 0, 0, NULL, NULL, NULL, NULL, NULL)
 *     (it does only the set-up on the current device and returns FLCE_OK or
 *     FLCE_ERR_CUDA) on each device before reserving their pool, and before any
 *     stream capture.
 *   - Limit: the forward scratch, flce_forward_workspace_size() with the
 *     planned S (1 or 2 for large N), about 20 bytes per token and independent
 *     of D and V, must fit in 32 MiB: about 1.6 million tokens. A planned S is
 *     lowered until the partials fit; a caller's explicit opt->v_splits is kept.
 *     Problems that do not fit are rejected with FLCE_ERR_WORKSPACE before
 *     anything is enqueued.
 *   - Every call shares the one array, and it keeps the last call's contents.
 *     Nothing in it needs clearing between calls, because each call writes every
 *     scratch word before reading it. Calls whose work overlaps on the GPU (on
 *     different streams, or from different host threads) race on the array and
 *     give wrong results: serialise them.
 */
int flce_forward_noalloc(const uint16_t* H, const uint16_t* W, const int32_t* labels, int64_t N,
                         int64_t D, int64_t V, const flce_options* opt, float* loss, float* lse,
                         int32_t* status, void* stream);

/*
 * Cross-entropy over a given logits matrix: the unfused loss that fused linear
 * cross-entropy replaces (GPU MODE lecture 28 notes, cross-entropy section:
 * LigerCrossEntropyLoss(reduction="mean")(logits.view(-1, vocab), labels)).
 * Same loss, lse, ignore and scaling rules as flce_forward_backward, with z
 * given directly:
 *   logits   [N, V] fp32 or bf16 (dtype = FLCE_DTYPE_F32 / FLCE_DTYPE_BF16), row
 *            stride ld elements (ld >= V; ld * element size a multiple of 16)
 *   loss     fp32 [1], or fp32 [N] per-token losses with FLCE_REDUCTION_NONE
 *   lse      fp32 [N] (may be NULL)
 *   dlogits  [N, V] of the same dtype, row stride dld (may be NULL: no gradient;
 *            may equal logits with dld == ld: the gradient overwrites the logits
 *            row by row; must not otherwise overlap them). Not allowed with
 *            FLCE_REDUCTION_NONE.
 *   workspace of flce_ce_workspace_size() bytes (per-token loss, lse, scalars).
 * One read of the logits for the loss; for the gradient the row is read again
 * (mostly from L2) and dlogits written once.
 */
int flce_ce_workspace_size(int64_t N, int64_t V, const flce_options* opt, size_t* bytes);
int flce_ce_logits(const void* logits, int32_t dtype, int64_t ld, const int32_t* labels,
                   int64_t N, int64_t V, const flce_options* opt, float* loss, float* lse,
                   void* dlogits, int64_t dld, void* workspace, size_t ws_bytes, int32_t* status,
                   void* stream);

/*
 * Multiply dH (bf16, dh_elems elements) and dW (dw_dtype, dw_elems elements) in
 * place by the fp32 device scalar *scale, on `stream`. This is the backward step
 * of the drop-in loss (GPU MODE lecture 28 notes, cross-entropy section: the
 * fused loss replaces PyTorch's loss module, so autograd hands it dL/dloss):
 * flce_forward_backward computes the gradients for dL/dloss = 1, and this call
 * applies the actual upstream factor. When *scale == 1 the kernels exit without
 * touching memory (no host synchronisation is needed to find that out). Either
 * buffer may be NULL with 0 elements; sizes in bytes must be multiples of 16 and
 * pointers 16-byte aligned.
 */
int flce_scale_grads(uint16_t* dH, int64_t dh_elems, void* dW, int64_t dw_elems,
                     int32_t dw_dtype, const float* scale, void* stream);

/*
 * Synchronise `stream`, read the device status word and return it (FLCE_OK, or
 * the first device error a call recorded). Returns FLCE_ERR_CUDA if the stream
 * reports a CUDA error. status == NULL returns FLCE_OK after the synchronisation.
 */
int flce_check_status(const int32_t* status, void* stream);

/* Static English text for a return code. */
const char* flce_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
