/*
 * nc.h -- C ABI of libnc: one forward+backward training step of a
 * nanochat-style decoder-only GPT on one NVIDIA B300 (sm_103a).
 *
 * The model (all citations are to the nanochat pages this library restates):
 *   - token embedding `wte` and an untied output head `lm_head`
 *     (cosmicrealm "noao-chat-0-项目总体介绍" §2.1 item 3);
 *   - per block, pre-norm: a = norm(x); q,k,v = a Wq^T, a Wk^T, a Wv^T
 *     (bias-free, §2.1 item 5); half-split RoPE on q and k (§2.1 item 1:
 *     y1 = x1 cos + x2 sin, y2 = -x1 sin + x2 cos), then RMSNorm of q and k
 *     per head (§2.1 item 2); causal attention with grouped-query heads
 *     (§2.1 item 6; query head h reads kv head h / (n_head / n_kv_head));
 *     x += o Wo^T; x += relu(norm(x) Wfc^T)^2 Wproj^T (§2.1 item 4, with the
 *     4x hidden layer of woshipm nanochat analysis §五.1);
 *   - norm() is RMSNorm without gain, y = x / sqrt(mean(x^2) + eps)
 *     (§2.1 item 5); a final norm precedes lm_head;
 *   - loss: mean next-token cross-entropy over all B*T positions
 *     (devpress "用不到100美元，亲手训练一个属于你的GPT-2" §2.2 item 2);
 *   - fp32 master weights, cast to the compute dtype in the forward
 *     (devpress §4.2 "精度管理"; feinterview "nanochat：低成本跑通大模型训练全流程").
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are CUDA device pointers owned by the caller;
 *     *_host are host pointers owned by the caller.  Nothing is retained
 *     after a call returns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued on it; only calls that write a host pointer synchronise it.
 *   - Matrices are row-major with the last index contiguous.  Linear
 *     weights are stored W[out][in] and applied as y = x W^T.
 *   - Errors are returned as nc_status; no call aborts the process.  A
 *     model is not thread-safe: use one model per host thread / stream.
 */
#ifndef NC_H
#define NC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { NC_FP32 = 0, NC_BF16 = 1 };

typedef struct {
  int32_t depth;       /* number of blocks L                                  */
  int32_t n_embd;      /* residual width C = n_head * head_dim                */
  int32_t n_head;      /* query heads H                                       */
  int32_t n_kv_head;   /* key/value heads Hkv, H % Hkv == 0                   */
  int32_t head_dim;    /* hd; even; 64 or 128 in NC_BF16 mode                 */
  int32_t mlp_hidden;  /* F, the MLP width (4 * n_embd in the pages)          */
  int32_t vocab;       /* V                                                   */
  int32_t seq_len;     /* maximum T per call                                  */
  int32_t batch;       /* maximum B per call                                  */
  int32_t dtype;       /* compute dtype: NC_FP32 or NC_BF16                   */
  float rope_base;     /* RoPE base; 10000 when <= 0                          */
  float norm_eps;      /* RMSNorm eps; FLT_EPSILON when < 0                   */
  float init_std;      /* std of the N(0, std) init; 0.02 when <= 0           */
  /* Variants, both off when 0 (woshipm nanochat analysis §三.3 item 1 names a
   * "logit stabilisation" without defining it; read here as the soft-cap): */
  float logit_softcap; /* c > 0: every logit z becomes c * tanh(z / c) before
                          the softmax and in nc_forward_logits / decoding
                          outputs; must be finite and >= 0                   */
  int32_t embed_norm;  /* 1: RMSNorm (no gain, eps = norm_eps) of each
                          embedding row before the first block; 0 or 1       */
  /* The 8-bit training step (woshipm nanochat analysis §一.2 and §六.2 name
   * FP8 as a speed lever without a recipe): 1 makes every block's four
   * linear layers (q/k/v, output projection, MLP up and down) multiply E4M3
   * operands in the forward: the bf16 input activation and the fp32 master
   * weight are each quantised per tensor with current scaling (the
   * nc_op_quantize_fp8 rule; [Wq; Wk; Wv] is one tensor), products
   * accumulate in fp32 and are dequantised in the fused epilogues.  In the
   * backward their input gradients dX = dY W multiply E4M3 operands as well
   * (dY's bf16 value with its own per-tensor scale, W's forward codes read
   * transposed), and so do their weight gradients dW = dY^T X (the transposed
   * codes of dY and of the forward input); the quantisers pass gradients
   * through unchanged.  The lm_head, attention and norms stay bf16.  The
   * model then also holds every layer's transposed input codes,
   * batch * seq_len * (2 n_embd + n_head head_dim + mlp_hidden) bytes per
   * layer.  NC_BF16 only; n_embd and mlp_hidden multiples of 16; decoding
   * (nc_kv_cache_create) is not offered.  0: off.  */
  int32_t fp8;
} nc_config;

typedef struct nc_model nc_model;

typedef enum {
  NC_OK = 0,
  NC_ERR_CONFIG = 1,       /* invalid nc_config                                  */
  NC_ERR_ALLOC = 2,        /* device allocation failed                           */
  NC_ERR_ARG = 3,          /* NULL pointer, bad size or index                    */
  NC_ERR_TOKEN_RANGE = 4,  /* a token or target outside [0, vocab)               */
  NC_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed                  */
  NC_ERR_TIMEOUT = 6,      /* a bounded device-side wait expired                 */
  NC_ERR_UNSUPPORTED = 7   /* shape or mode this build does not implement        */
} nc_status;

/* Human-readable name of a status.  Never NULL. */
const char* nc_status_string(nc_status s);

/* Version string of this build (kernel set and target architecture). */
const char* nc_version(void);

/* ------------------------------------------------------------------------
 * Model lifetime.
 * nc_model_create validates `cfg`, allocates fp32 master weights (packed,
 * see nc_param_info), the compute-dtype weight copy and the activation
 * workspace for batch*seq_len tokens, and initialises every weight i.i.d.
 * N(0, init_std) from `seed` with the counter-based draw: SplitMix64
 * (Steele, Lea & Flood 2014), tensor j of the packed order using the stream
 * whose state starts at seed ^ ((j+1) * 0x9E3779B97F4A7C15), element e taking
 * output e; Box-Muller on (top 24 bits, bits 16..39) + 0.5 over 2^24 in fp64,
 * rounded once to float32.  Synchronous.  On failure *out is NULL.
 * ---------------------------------------------------------------------- */
nc_status nc_model_create(const nc_config* cfg, uint64_t seed, nc_model** out);
void nc_model_destroy(nc_model* m);
nc_status nc_model_config(const nc_model* m, nc_config* cfg_out);

/* Packed parameter layout (cosmicrealm "noao-chat-0-项目总体介绍" §2.1: the
 * untied embedding and output head, bias-free linears): wte[V,C]; per layer l:
 * Wq[H*hd,C], Wk[Hkv*hd,C], Wv[Hkv*hd,C], Wo[C,H*hd], Wfc[F,C], Wproj[C,F];
 * lm_head[V,C].  Wq/Wk/Wv are adjacent, so together they form one
 * [(H+2Hkv)*hd, C] matrix.  *n_tensors receives the number of tensors (2 + 6L)
 * and *n_elems the length of the packed vector (either may be NULL);
 * NC_ERR_ARG for a NULL model.  nc_param_info describes each tensor. */
nc_status nc_param_layout(const nc_model* m, int32_t* n_tensors, int64_t* n_elems);
/* The same call under its earlier name. */
nc_status nc_param_count(const nc_model* m, int32_t* n_tensors, int64_t* n_elems);
/* Tensor i: its name ("wte", "h3.wfc", "lm_head", ...), shape and element
 * offset in the packed vector.  `name` points to storage owned by the model. */
nc_status nc_param_info(const nc_model* m, int32_t i, const char** name,
                        int64_t* rows, int64_t* cols, int64_t* offset);
/* Copy all fp32 master weights (n_elems floats) to / from device memory. */
nc_status nc_get_params(const nc_model* m, float* dst_dev, void* stream);
nc_status nc_set_params(nc_model* m, const float* src_dev, void* stream);

/* ------------------------------------------------------------------------
 * The training step.
 * tokens_dev, targets_dev: int32 [B, T] (device).  1 <= B <= cfg.batch,
 * 1 <= T <= cfg.seq_len; position of token (b, t) is t.
 * loss_host: receives the mean cross-entropy over the B*T positions.
 * grads_dev: fp32, n_elems floats in the packed layout; OVERWRITTEN with
 * d(loss)/d(weights).  The weights are not updated.
 * Synchronises `stream` once at the end (to read the loss and the device
 * error flag).  A token or target outside [0, vocab) gives
 * NC_ERR_TOKEN_RANGE and leaves loss and grads unspecified.
 * ---------------------------------------------------------------------- */
nc_status nc_forward_backward(nc_model* m, const int32_t* tokens_dev,
                              const int32_t* targets_dev, int32_t B, int32_t T,
                              float* loss_host, float* grads_dev, void* stream);

/* The step for gradient accumulation over micro-batches (cosmicrealm
 * "noao-chat-0-项目总体介绍" §4.3: several forward + backward passes, then
 * one optimizer step): grads_dev = (accumulate ? grads_dev : 0) +
 * grad_scale * d(loss)/d(weights), loss being this call's mean cross-entropy
 * (written to loss_host unscaled).  With grad_scale = 1/k and accumulate set
 * on all but the first of k equal micro-batches, grads_dev ends as the
 * gradient of the mean loss over all of them.  grad_scale must be finite.
 * nc_forward_backward is this call with grad_scale = 1, accumulate = 0. */
nc_status nc_forward_backward_accumulate(nc_model* m, const int32_t* tokens_dev,
                                         const int32_t* targets_dev, int32_t B, int32_t T,
                                         float grad_scale, int32_t accumulate, float* loss_host,
                                         float* grads_dev, void* stream);

/* The same step with tokens and targets in (preferably pinned) host memory:
 * they are copied to the model's device buffers on `stream` first. */
nc_status nc_forward_backward_host(nc_model* m, const int32_t* tokens_host,
                                   const int32_t* targets_host, int32_t B, int32_t T,
                                   float* loss_host, float* grads_dev, void* stream);

/* Forward only: fp32 logits [B, T, V] (device, caller-owned).  Does not
 * synchronise; a token outside [0, vocab) sets the device error flag that
 * nc_last_error() reads. */
nc_status nc_forward_logits(nc_model* m, const int32_t* tokens_dev, int32_t B,
                            int32_t T, float* logits_dev, void* stream);

/* Forward only: per-position cross-entropy [B, T] fp32 (device). */
nc_status nc_forward_row_losses(nc_model* m, const int32_t* tokens_dev,
                                const int32_t* targets_dev, int32_t B, int32_t T,
                                float* losses_dev, void* stream);

/* Synchronise `stream` and turn the model's device error flag into a status
 * (NC_OK, NC_ERR_TOKEN_RANGE or NC_ERR_TIMEOUT); clears the flag. */
nc_status nc_last_error(nc_model* m, void* stream);

/* Number of kernels the last nc_forward_backward / nc_forward_logits call
 * enqueued (for launch accounting). */
int64_t nc_last_launch_count(const nc_model* m);

/* ------------------------------------------------------------------------
 * Kernel-level entry points.  Each runs one kernel of the step on caller
 * buffers so that it can be checked on its own.  `dtype` is NC_FP32 (float
 * buffers) or NC_BF16 (bfloat16 buffers, passed as void*).  No allocation
 * except where stated; all enqueue on `stream` without synchronising.
 * ---------------------------------------------------------------------- */

/* D[M,N] (op)= sum_k A(m,k) B(n,k).  A is [M][K] (a_kmajor=1) or [K][M]
 * (a_kmajor=0) with leading dimension lda (elements); B is [N][K]
 * (b_kmajor=1) or [K][N] (b_kmajor=0).  Epilogue `ep`:
 *   NC_EP_STORE     D (dtype) = acc
 *   NC_EP_STORE_F32 D (float) = acc
 *   NC_EP_ACCUM_F32 D (float) += acc          (residual add, dW accumulate)
 *   NC_EP_RELU2     D (dtype) = relu(acc), aux (dtype) = relu(acc)^2
 *   NC_EP_RELU2_BWD D (dtype) = acc * 2 * aux   (aux holds relu(u))
 *   NC_EP_RELU2_SQ  D (dtype) = relu(acc)^2      (aux unused)
 *   NC_EP_RELU2_SQ_BWD D (dtype) = acc * 2 * sqrt(aux)   (aux holds relu(u)^2;
 *                   sqrt(relu(u)^2) = relu(u), so the forward need not keep relu(u))
 * ldd / ldaux are leading dimensions in elements.  NC_BF16 runs the tcgen05
 * tensor-core kernel (lda, ldb multiples of 8, 16-byte aligned bases);
 * NC_FP32 runs exact fp32 FMA.  workspace may be NULL (see below). */
enum { NC_EP_STORE = 0, NC_EP_STORE_F32 = 1, NC_EP_ACCUM_F32 = 2,
       NC_EP_RELU2 = 3, NC_EP_RELU2_BWD = 4, NC_EP_RELU2_SQ = 5, NC_EP_RELU2_SQ_BWD = 6 };
nc_status nc_op_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K,
                     const void* A, int64_t lda, int32_t a_kmajor,
                     const void* B, int64_t ldb, int32_t b_kmajor,
                     int32_t ep, void* D, int64_t ldd, void* aux, int64_t ldaux,
                     void* workspace, size_t workspace_bytes, void* stream);
/* Device workspace (bytes) that lets an NC_BF16 GEMM with an fp32 epilogue
 * and few output tiles run stream-K: each CTA takes an equal share of the
 * (tile, k-block) work and tiles split between CTAs are summed afterwards in
 * CTA order (deterministic).  With a NULL or smaller workspace the GEMM runs
 * one CTA per output tile. */
size_t nc_gemm_workspace_bytes(void);

/* RMSNorm without gain over rows of x (float [rows, C]):
 * y (dtype) = x * rstd, rstd (float [rows]) = 1/sqrt(mean(x^2) + eps). */
nc_status nc_op_rmsnorm_fwd(int32_t dtype, int64_t rows, int32_t C, const float* x,
                            void* y, float* rstd, float eps, void* stream);
/* dx (float, accumulated: dx += ...) and dx_act (dtype copy of the result,
 * may be NULL) from dy (float [rows, C]), y (dtype) and rstd:
 * dx += rstd * (dy - y * mean(dy * y)). */
nc_status nc_op_rmsnorm_bwd(int32_t dtype, int64_t rows, int32_t C, const float* dy,
                            const void* y, const float* rstd, float* dx, void* dx_act,
                            void* stream);

/* RoPE angle table: cos_sin (float [T, hd/2, 2]) holds cos and sin of
 * theta[t][i] = t * rope_base^(-2i/hd), evaluated in fp64 and rounded once. */
nc_status nc_op_rope_table(int32_t T, int32_t hd, float rope_base, float* cos_sin,
                           void* stream);
/* In place on qkv (dtype [B*T, (H+2*Hkv)*hd]): RoPE on the H query and Hkv key
 * heads at position t = row % T, then RMSNorm of each of those head vectors;
 * rstd (float [B*T, H+Hkv]).  cos_sin from nc_op_rope_table with >= T rows. */
/* The same numbers as nc_op_rope_table, pair-major: pairs (float [hd/4, T, 4])
 * holds (cos_i, sin_i, cos_i+1, sin_i+1) for even i at each position.  hd % 4 == 0. */
nc_status nc_op_rope_table_pairs(int32_t T, int32_t hd, float rope_base, float* pairs, void* stream);
nc_status nc_op_rope_qknorm_fwd(int32_t dtype, int32_t B, int32_t T, int32_t H,
                                int32_t Hkv, int32_t hd, void* qkv, float* rstd,
                                const float* cos_sin, float eps, void* stream);
/* The q/k/v projection with the above fused into its epilogue (bf16 only):
 * qkv (bf16 [M, (H+2*Hkv)*hd], leading dimension ldqkv) = x (bf16 [M, K],
 * leading dimension ldx) times Wqkv^T (bf16 [(H+2*Hkv)*hd, K]), then for the
 * first H+Hkv heads of every row the rotary embedding at position row % T
 * followed by the per-head RMSNorm, computed from the fp32 accumulator; v is
 * stored as computed.  rstd (float [M, H+Hkv]).  cos_sin is the table of
 * nc_op_rope_table (pair_rows = 0) or of nc_op_rope_table_pairs built for
 * pair_rows >= T positions (faster: the epilogue's reads coalesce).  The rotation preserves the
 * sum of squares, so rstd is taken before rotating (cosmicrealm
 * "noao-chat-0-项目总体介绍" §2.1 items 1-2).  hd 64 or 128, (H+2*Hkv)*hd > 128,
 * 16-byte aligned buffers; NC_ERR_ARG / NC_ERR_UNSUPPORTED otherwise. */
nc_status nc_op_gemm_qkv_rope(int32_t M, int32_t K, int32_t T, int32_t H, int32_t Hkv,
                              int32_t hd, const void* x, int64_t ldx, const void* wqkv,
                              void* qkv, int64_t ldqkv, float* rstd, const float* cos_sin,
                              int32_t pair_rows, float eps, void* stream);
/* In place on dqkv: the backward of the above, given the saved (normalised)
 * qkv and rstd. */
nc_status nc_op_rope_qknorm_bwd(int32_t dtype, int32_t B, int32_t T, int32_t H,
                                int32_t Hkv, int32_t hd, void* dqkv, const void* qkv,
                                const float* rstd, const float* cos_sin, void* stream);

/* Causal GQA attention over the q, k, v column blocks of qkv (dtype
 * [B*T, (H+2*Hkv)*hd]); o (dtype [B*T, H*hd]); lse (float [B, H, T]). */
nc_status nc_op_attention_fwd(int32_t dtype, int32_t B, int32_t T, int32_t H,
                              int32_t Hkv, int32_t hd, const void* qkv, void* o,
                              float* lse, void* stream);
/* dqkv (dtype, same layout as qkv) from do_ (dtype [B*T, H*hd]).  workspace:
 * float [B*H*T] for rowsum(do * o). */
nc_status nc_op_attention_bwd(int32_t dtype, int32_t B, int32_t T, int32_t H,
                              int32_t Hkv, int32_t hd, const void* qkv, const void* o,
                              const float* lse, const void* do_, void* dqkv,
                              float* workspace, void* stream);
/* The bf16 attention backward with the backward of nc_op_rope_qknorm_fwd
 * folded into its output: the q and k blocks of dqkv receive the gradient with
 * respect to the projection output (before RoPE and the per-head RMSNorm),
 * given the saved normalised qkv, rstd (float [B*T, H+Hkv]) and the cos/sin
 * table; the v block is as from nc_op_attention_bwd.  Equivalent to
 * nc_op_attention_bwd followed by nc_op_rope_qknorm_bwd.  cos_sin is the table
 * of nc_op_rope_table (pair_rows = 0) or of nc_op_rope_table_pairs built for
 * pair_rows >= T positions (faster: a warp's reads of it coalesce).  hd 64 or
 * 128; NC_ERR_ARG for a NULL buffer or 0 < pair_rows < T. */
nc_status nc_op_attention_bwd_rope(int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t hd,
                                   const void* qkv, const void* o, const float* lse,
                                   const void* do_, void* dqkv, float* workspace,
                                   const float* rstd, const float* cos_sin, int32_t pair_rows,
                                   void* stream);

/* Cross-entropy on logits z (dtype [rows, V]) against targets (int32 [rows]):
 * row_loss (float [rows]) = logsumexp(z) - z[target]; z is overwritten in
 * place with (softmax(z) - onehot(target)) * grad_scale.  Targets outside
 * [0, V) set *err_dev |= 1 (err_dev int32, device, may be NULL). */
nc_status nc_op_cross_entropy(int32_t dtype, int64_t rows, int32_t V, void* z,
                              const int32_t* targets, float* row_loss, float grad_scale,
                              int32_t* err_dev, void* stream);
/* The same with the logit soft-cap: the loss is taken on c * tanh(z / c)
 * (softcap = c > 0, finite) and z is overwritten with the gradient with
 * respect to the raw logits, (softmax(zc) - onehot) * (1 - tanh(z / c)^2) *
 * grad_scale; softcap = 0 is nc_op_cross_entropy.  NC_ERR_ARG for a negative
 * or non-finite softcap. */
nc_status nc_op_cross_entropy_softcap(int32_t dtype, int64_t rows, int32_t V, void* z,
                                      const int32_t* targets, float* row_loss, float grad_scale,
                                      float softcap, int32_t* err_dev, void* stream);

/* x (float [n, C]) = float(round_dtype(wte[tokens[i]])) for wte float [V, C]. */
nc_status nc_op_embed_fwd(int32_t dtype, int64_t n, int32_t C, int32_t V,
                          const int32_t* tokens, const float* wte, float* x,
                          int32_t* err_dev, void* stream);
/* dwte (float [V, C]) = sum over i with tokens[i] == v of dx[i] (float [n, C]),
 * summed in increasing i; rows of ids not present are +0.0.  Deterministic.
 * A position whose id lies outside [0, V) adds to no row (this call does not
 * report it; the training step reports it as NC_ERR_TOKEN_RANGE).
 * scratch: at least nc_embed_bwd_scratch_bytes(n, C, V) bytes of device memory. */
size_t nc_embed_bwd_scratch_bytes(int64_t n, int32_t C, int32_t V);
nc_status nc_op_embed_bwd(int64_t n, int32_t C, int32_t V, const int32_t* tokens,
                          const float* dx, float* dwte, void* scratch, void* stream);

/* ------------------------------------------------------------------------
 * Embedding backward that allocates nothing.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory,
 * for example a host that gives this library only its input and output
 * buffers under a device-memory budget fixed in advance, or a process whose
 * allocator has already reserved the device's memory, where one more
 * cudaMalloc would fail.  nc_op_embed_bwd needs caller-provided scratch;
 * this variant computes the same result (bit for bit) using a scratch area
 * in a file-scope device array of NC_NOALLOC_SCRATCH_BYTES that every GPU
 * which loads the library keeps until the process exits.
 *  - Sizes whose scratch (nc_embed_bwd_scratch_bytes(n, C, V)) exceeds
 *    NC_NOALLOC_SCRATCH_BYTES are rejected with NC_ERR_UNSUPPORTED before any
 *    GPU work; NULL pointers, negative n or non-positive C or V give
 *    NC_ERR_ARG; n == 0 writes zeros to dwte.
 *  - The first call on a device looks up the array's device address (a
 *    one-time set-up per device, done with that device current); make that
 *    first call before any stream capture.  After cudaDeviceReset the array
 *    lives in a new context, and the next call looks its address up again.
 *  - It calls no cudaMalloc/cudaFree and no allocating library routine.
 *  - All calls share the one array, which keeps the last call's contents;
 *    the counters are zeroed on the stream at the start of every call.
 *    Calls that overlap on the GPU (different streams, or different host
 *    threads) race on the array: issue them in order on one stream.
 * Arguments are those of nc_op_embed_bwd without the scratch pointer.
 * ---------------------------------------------------------------------- */
#define NC_NOALLOC_SCRATCH_BYTES (64u << 20)
nc_status nc_op_embed_bwd_noalloc(int64_t n, int32_t C, int32_t V, const int32_t* tokens,
                                  const float* dx, float* dwte, void* stream);

/* ------------------------------------------------------------------------
 * Per-kernel-class device timing of the step.  While enabled, every kernel
 * the step enqueues is bracketed by CUDA events on the caller's stream, and
 * its class, algorithmic FLOPs and algorithmic HBM bytes are recorded.
 * nc_profile_enable(m, 1) starts (and zeroes) the accumulators, 0 stops.
 * nc_profile_read synchronises the recorded events and returns, for class
 * `cls`, the summed device milliseconds, the launch count and the summed
 * algorithmic FLOPs and bytes.
 * ---------------------------------------------------------------------- */
enum { NC_PROF_GEMM = 0, NC_PROF_ATTN_FWD = 1, NC_PROF_ATTN_BWD = 2, NC_PROF_NORM = 3,
       NC_PROF_ROPE = 4, NC_PROF_CE = 5, NC_PROF_EMBED = 6, NC_PROF_CAST = 7,
       NC_PROF_OTHER = 8,
       /* sub-classes of NC_PROF_GEMM (each GEMM is counted in one of these too) */
       NC_PROF_GEMM_FWD = 9, NC_PROF_GEMM_DX = 10, NC_PROF_GEMM_DW = 11, NC_PROF_GEMM_LM = 12,
       /* nc_optimizer_step: the matrices' Newton-Schulz iterations and Muon
          applies (concurrent on side streams, timed as one phase), and the
          elementwise kernels (momentum and norms, scaling, AdamW) */
       NC_PROF_OPT_NS = 13, NC_PROF_OPT_EW = 14,
       /* the 8-bit step's quantisation of GEMM operands (fp8 = 1) */
       NC_PROF_QUANT = 15,
       NC_PROF_CLASSES = 16 };
nc_status nc_profile_enable(nc_model* m, int32_t on);
nc_status nc_profile_read(nc_model* m, int32_t cls, double* ms, int64_t* launches,
                          double* flops, double* bytes);

/* ------------------------------------------------------------------------
 * Test hook.  Sets the time limit, in nanoseconds, of every bounded
 * mbarrier wait inside the tensor-core kernels (default 4 s).  When a wait
 * runs out, the kernel sets the timeout bit of the model's device error
 * flag (reported as NC_ERR_TIMEOUT), finishes its own in-flight copies and
 * MMAs (again bounded), frees its tensor memory and returns.
 * ---------------------------------------------------------------------- */
void nc_debug_set_wait_limit_ns(uint64_t ns);

/* Test hook for the timeout path.  on = 1 arms the next launch of the
 * single-CTA tensor-core GEMM kernel (see nc_debug_set_gemm_pair): its
 * MMA-issuing thread first waits on a barrier that nothing completes, so that
 * wait runs out after the limit above; the kernel then takes its timeout path
 * (error bit, drain of its own copies and MMAs under a fixed 2 s bound, TMEM
 * freed) and the call that reads the flag returns NC_ERR_TIMEOUT.  The
 * outputs of that GEMM are left unwritten.  The hook disarms itself at that
 * launch; on = 0 disarms it. */
void nc_debug_stall_next_gemm(int32_t on);

/* Test hook.  on = 0 makes every bf16 GEMM use the single-CTA kernel (128 x
 * 256 tiles); on = 1 (default) lets shapes with M >= 256 and N > 128 that do
 * not split K run on CTA pairs (256 x 256 tiles, tcgen05 cta_group::2).  Both
 * compute the same sums; the switch exists to test and time either path. */
void nc_debug_set_gemm_pair(int32_t on);

/* Test hook.  on = 1 (default): a bf16 model whose weight matrices all have
 * row counts that are multiples of 128 runs the optimizer's Newton-Schulz
 * iterations batched, one launch per product for all matrices of a shape; on
 * = 0 runs them matrix by matrix on side streams.  Both compute the same
 * products.  Read when a model allocates its optimizer state (its first
 * nc_optimizer_step), so it applies to models stepped after the call. */
void nc_debug_set_ns_batched(int32_t on);

/* Test hook.  on = 1 (default): a decode step replays a CUDA graph of the
 * step, captured once per batch size on an internal stream (its position
 * lives on the device, its tokens and logits pass through fixed buffers);
 * on = 0 enqueues the same kernels directly.  Both compute the same values. */
void nc_debug_set_decode_graph(int32_t on);

/* Test hook.  on = 1 (default): the decode kernels (skinny projections,
 * attention, combine) are launched with programmatic stream serialization, so
 * each may start while the previous kernel drains (a projection streams its
 * first weights then) and waits for it before touching its data; on = 0
 * launches them in plain stream order.  Both compute the same values.  Read
 * at launch time, so a step graph captured before the call keeps its form. */
void nc_debug_set_decode_pdl(int32_t on);

/* ------------------------------------------------------------------------
 * Optimizer step (cosmicrealm "noao-chat-0-项目总体介绍" §2.2 and §4.2;
 * woshipm nanochat analysis §六.1): the weight matrices (every Wq, Wk, Wv,
 * Wo, Wfc, Wproj) are updated by Muon, wte and lm_head by AdamW.  The pages
 * name the method and the learning rates; the constants below are those of the
 * published methods (Muon: Jordan et al. 2024; AdamW: Loshchilov & Hutter).
 *
 * Muon, per matrix W[rows, cols] with gradient G and momentum buffer M:
 *   M <- momentum M + G;  U = G + momentum M (nesterov) or M;
 *   X = U / (||U||_F + 1e-7), then ns_steps times X <- a X + (b A + c A^2) X
 *   with A = X X^T ((a, b, c) = (3.4445, -4.7750, 2.0315); a tall matrix is
 *   iterated as X <- a X + X (b A + c A^2) with A = X^T X, the same map);
 *   W <- W - lr_mult * matrix_lr * sqrt(max(1, rows/cols)) * X.
 *   The iteration runs in the model's compute dtype (bf16 products with fp32
 *   accumulation in NC_BF16 mode).
 * AdamW, per element of wte (lr = embedding_lr) and lm_head (unembedding_lr):
 *   m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
 *   W <- W - lr_mult * lr * (m/(1-b1^t) / (sqrt(v/(1-b2^t)) + eps) + wd W),
 *   t = the number of steps taken, counting this one.
 * ---------------------------------------------------------------------- */
typedef struct {
  float matrix_lr;       /* Muon learning rate (0.02)                          */
  float embedding_lr;    /* AdamW learning rate of wte (0.2)                   */
  float unembedding_lr;  /* AdamW learning rate of lm_head (0.004)             */
  float momentum;        /* Muon momentum in [0, 1) (0.95)                     */
  int32_t nesterov;      /* nonzero: the Nesterov form above (1)               */
  int32_t ns_steps;      /* Newton-Schulz iterations, 0..64 (5)                */
  float beta1, beta2;    /* AdamW moment decay rates in [0, 1) (0.9, 0.999)    */
  float adam_eps;        /* > 0 (1e-8)                                         */
  float weight_decay;    /* AdamW decoupled weight decay (0)                   */
} nc_optim_config;
/* Fill *oc with the defaults in parentheses above. */
void nc_optim_config_default(nc_optim_config* oc);
/* Apply one optimizer step to the model's fp32 master weights, given the
 * packed fp32 gradient `grads` (device, the layout of nc_forward_backward's
 * output); lr_mult (the caller's schedule value, e.g. warmup + cosine) scales
 * every learning rate.  The first call allocates the optimizer state on the
 * device and zeroes it; the state lives with the model.  Enqueued on `stream`
 * without synchronising; a bounded-wait timeout in a GEMM is reported by the
 * next call that reads the device error flag.  NC_ERR_ARG for NULL pointers or
 * out-of-range settings, NC_ERR_ALLOC if the state does not fit, and
 * NC_ERR_UNSUPPORTED for more than 384 weight matrices. */
nc_status nc_optimizer_step(nc_model* m, const nc_optim_config* oc, const float* grads,
                            float lr_mult, void* stream);
/* Zero the momentum and Adam moments and the step count. */
nc_status nc_optimizer_reset(nc_model* m, void* stream);
/* Optimizer steps taken since creation or the last reset (-1 for NULL). */
int64_t nc_optimizer_steps(const nc_model* m);
/* The orthogonalisation above on its own: x (float [rows, cols]) = `steps`
 * Newton-Schulz iterations from u / (||u||_F + 1e-7), computed in `dtype`.
 * workspace: nc_newton_schulz_workspace_bytes(dtype, rows, cols) bytes,
 * 256-byte aligned.  NC_BF16 needs rows, cols multiples of 8. */
size_t nc_newton_schulz_workspace_bytes(int32_t dtype, int32_t rows, int32_t cols);
/* D[m, n] (op)= sum_k A[m, k] W[n, k] for 1 <= M <= 32 rows (A [M][K], W
 * [N][K], both K-major), the decode step's projections: CUDA cores, one pass
 * over W, fp32 accumulation.  ep: NC_EP_STORE, NC_EP_STORE_F32,
 * NC_EP_ACCUM_F32 or NC_EP_RELU2_SQ.  K, lda, ldw multiples of 8, 16-byte
 * aligned A and W; NC_ERR_ARG otherwise. */
nc_status nc_op_gemm_rows(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* A,
                          int64_t lda, const void* W, int64_t ldw, int32_t ep, void* D,
                          int64_t ldd, void* stream);
nc_status nc_op_newton_schulz(int32_t dtype, int32_t rows, int32_t cols, int32_t steps,
                              const float* u, float* x, void* workspace, void* stream);

/* ------------------------------------------------------------------------
 * Incremental decoding with a key/value cache (woshipm nanochat analysis §三
 * item 4).  nc_prefill runs the forward over B prompts of T tokens
 * (positions 0..T-1), keeps every layer's keys (after RoPE and the QK norm)
 * and values, and writes the logits of each prompt's last position; every
 * nc_decode_step then feeds one token per sequence at the next position and
 * writes that position's logits.  The logits of prompt b at position t equal
 * row (b, t) of nc_forward_logits on the whole sequence (up to rounding).
 * The weights used are those cast by the last nc_prefill: after
 * nc_set_params or nc_optimizer_step, prefill again.  A decode step replays a
 * CUDA graph of the whole step (see nc_debug_set_decode_graph).
 * ---------------------------------------------------------------------- */
/* Allocate (or reuse, if large enough) the cache for max_batch sequences of
 * max_len positions and empty it.  1 <= max_batch <= cfg.batch,
 * 1 <= max_len <= cfg.seq_len; NC_ERR_UNSUPPORTED unless hd is 64 or 128 and
 * n_head / n_kv_head is 1, 2, 3, 4 or 8, and for an 8-bit model (cfg.fp8). */
nc_status nc_kv_cache_create(nc_model* m, int32_t max_batch, int32_t max_len);
/* tokens_dev: int32 [B, T]; logits_dev: fp32 [B, V] (device).  Replaces the
 * cache contents; B <= max_batch, T <= max_len.  Does not synchronise. */
nc_status nc_prefill(nc_model* m, const int32_t* tokens_dev, int32_t B, int32_t T,
                     float* logits_dev, void* stream);
/* tokens_dev: int32 [B], B = the prefill's B; logits_dev: fp32 [B, V].
 * NC_ERR_ARG when the cache is empty or full.  Does not synchronise. */
nc_status nc_decode_step(nc_model* m, const int32_t* tokens_dev, int32_t B, float* logits_dev,
                         void* stream);
/* Positions held per sequence (-1 for NULL). */
int32_t nc_kv_cache_length(const nc_model* m);

/* ------------------------------------------------------------------------
 * 8-bit floating-point GEMM (woshipm nanochat analysis §一.2 and §六.2: FP8
 * as a training speed lever; the pages fix no recipe).  Values are OCP FP8
 * E4M3 codes (1 sign, 4 exponent bits of bias 7, 3 mantissa bits; largest
 * finite 448, no infinities, 0x7f / 0xff NaN) with one fp32 scale per tensor.
 * ---------------------------------------------------------------------- */
/* Quantise n values of x_dev (dtype NC_FP32 or NC_BF16, device, 16-byte
 * aligned) to E4M3 codes in codes_dev (device, n bytes, 8-byte aligned):
 *   amax = max |x|;  scale = fl32(448 / amax), or 1 if that is not finite
 *   and positive;  code_i = E4M3(fl32(x_i * scale)), round to nearest even,
 *   saturating at +-448;  scale_inv = fl32(1 / scale).
 * stats_dev (device, 3 floats, 4-byte aligned) receives {amax, scale,
 * scale_inv}; element 0 is also the running maximum while the call runs.
 * Inputs must be finite.  n = 0 writes stats {0, 1, 1} only.  Does not
 * synchronise. */
nc_status nc_op_quantize_fp8(int32_t dtype, const void* x_dev, int64_t n, uint8_t* codes_dev,
                             float* stats_dev, void* stream);
/* D[M, N] = (*a_scale_inv) (*b_scale_inv) sum_k A(m, k) B(n, k) with A, B
 * E4M3 codes, both K-major: A[M][lda], B[N][ldb] bytes (lda, ldb >= K and
 * multiples of 16, bases 16-byte aligned).  The scales are device pointers
 * (e.g. element 2 of nc_op_quantize_fp8's stats).  fp32 accumulation on the
 * tensor cores; out_dtype NC_BF16 or NC_FP32 gives D's type, row pitch ldd
 * elements (16-byte aligned base and rows).  NC_ERR_ARG on a violated
 * precondition.  Does not synchronise. */
nc_status nc_op_gemm_fp8(int32_t M, int32_t N, int32_t K, const uint8_t* a_dev, int64_t lda,
                         const uint8_t* b_dev, int64_t ldb, const float* a_scale_inv_dev,
                         const float* b_scale_inv_dev, int32_t out_dtype, void* d_dev, int64_t ldd,
                         void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NC_H */
