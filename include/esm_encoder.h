/*
 * esm_encoder.h -- C ABI of the GB300 (sm_103a) ESM-2 encoder forward on packed
 * variable-length protein sequences.
 *
 * What is computed (sources are web pages; page title and section are named):
 *   * Packing: "生物大模型训练加速实战：基于PyTorch与NVIDIA BioNeMo的Transformer优化指南"
 *     (hotelren.com), section 3.2: a batch is the concatenation of its sequences'
 *     tokens plus cu_seqlens = cumsum([0] + lengths) and max_seqlen; the packed
 *     forward runs the token embedding and then every encoder layer over cu_seqlens.
 *   * The layer: same guide, section 3.1 (self-attention, LayerNorm, fc1, fc2 as one
 *     fused TransformerEngine encoder layer, padding mask, bshd or thd input), and the
 *     "NVIDIA ESM-2 TransformerEngine" walkthrough (mlqm.cn), sections on rotary
 *     position embedding (size hidden / heads), the padding mask with bshd input,
 *     fused QKV weights and the 1026-position / 33-token vocabulary.
 *   * Bidirectional attention: BioNeMo ESM-2 model card (docs.nvda.net.cn), model
 *     overview ("BERT-style bidirectional encoder"); output: one float vector per
 *     residue (section "输出").
 *   * FP8: the aikraft.ru TransformerEngine summary, "Рецепт FP8: Delayed Scaling"
 *     (E4M3 forward, amax history 16, max algorithm), and section 4.1 of the hotelren.com
 *     guide.
 *
 * Per layer (pre-LN):  y = LN1(x); [q|k|v] = y Wqkv^T + bqkv; RoPE(q, k);
 *   o = softmax(q k^T / sqrt(64)) v within each sequence; x += o Wo^T + bo;
 *   u = GELU(LN2(x) W1^T + b1); x += u W2^T + b2.   Output: LNf(x) (or x).
 * Readings where the pages are silent: LayerNorm eps from the config (1e-5), biased
 * variance; exact erf GELU; RoPE base from the config (10000), rotate-half pairs
 * (j, j + head_dim/2), positions restart at 0 at every sequence start; no dropout.
 *
 * Conventions for every call:
 *   * All device buffers belong to the caller; the library only borrows them for the
 *     duration of the (asynchronous) call on `stream`.  Pointers marked "device" must
 *     be device memory of the current device; "host" pointers are host memory.
 *   * Tensors are dense row-major.  Linear weights are [out_features, in_features].
 *     w_qkv rows are q | k | v, each block head-major (row h*64 + c).
 *   * Parameter dtype: float32 for ESM_FP32; bfloat16 for ESM_BF16 and ESM_FP8_E4M3
 *     (FP8 GEMM operands are quantised on the fly from the bf16 weights).
 *   * hidden_out dtype: float32 for ESM_FP32, bfloat16 otherwise.
 *   * Errors are returned, never thrown or trapped.  Host-side checks return at once.
 *     Errors the kernels detect (malformed cu_seqlens, token ids out of range, a
 *     bounded device wait that ran out) are latched in the handle and reported by
 *     esm_encoder_check(); outputs of such a call are unspecified but every access
 *     stays in bounds.
 *   * A handle is not thread-safe: do not call it from two host threads at once.
 *     Calls on one stream run in order; calls on different streams that share a
 *     workspace race.
 */
#ifndef ESM_ENCODER_H_
#define ESM_ENCODER_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ESM_API __attribute__((visibility("default")))
#else
#define ESM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* esm_stream_t;

typedef enum {
  ESM_OK = 0,
  ESM_ERR_INVALID_ARG = 1,    /* a pointer, size or config field is invalid          */
  ESM_ERR_UNSUPPORTED = 2,    /* device is not sm_103, or a geometry the kernels lack */
  ESM_ERR_BAD_CU_SEQLENS = 3, /* cu_seqlens not 0 = c0 <= c1 <= ... = T, or L > max   */
  ESM_ERR_TOKEN_RANGE = 4,    /* a token id outside [0, vocab)                        */
  ESM_ERR_WORKSPACE = 5,      /* workspace NULL, misaligned or smaller than required  */
  ESM_ERR_CUDA = 6,           /* a CUDA runtime call failed                           */
  ESM_ERR_TIMEOUT = 7         /* a bounded device-side wait gave up                   */
} esm_status;

typedef enum { ESM_FP32 = 0, ESM_BF16 = 1, ESM_FP8_E4M3 = 2, ESM_FP4_E2M1 = 3 } esm_precision;

/* Encoder geometry and numerics.  ESM-2 650M: {33, 1280, 20, 5120, 33, 1026, 1e-5,
 * 10000, 1, 1, ESM_BF16, 16}.  head_dim = hidden / heads must be 64 for ESM_BF16 and
 * ESM_FP8_E4M3 (and hidden a multiple of 256, ffn a multiple of 256); ESM_FP32 accepts
 * any even head_dim <= 64 with hidden <= 4096. */
typedef struct {
  int num_layers;
  int hidden;
  int heads;
  int ffn;
  int vocab;
  int max_positions;      /* upper bound of every sequence length (1026)            */
  float ln_eps;
  float rope_base;
  float emb_scale;        /* x = emb_scale * E[token]                                */
  int final_ln;           /* 1: apply the final LayerNorm; 0: return the residual   */
  esm_precision precision;
  int amax_history_len;   /* FP8 delayed scaling history length (1..1024)           */
} esm_config;

/* Device pointers to the weights.  The per-layer members point to HOST arrays of
 * num_layers DEVICE pointers (read during the call only). */
typedef struct {
  const void* emb;                 /* [vocab, hidden]                   */
  const void* const* ln1_g;        /* [hidden]                          */
  const void* const* ln1_b;        /* [hidden]                          */
  const void* const* w_qkv;        /* [3*hidden, hidden]                */
  const void* const* b_qkv;        /* [3*hidden]                        */
  const void* const* w_o;          /* [hidden, hidden]                  */
  const void* const* b_o;          /* [hidden]                          */
  const void* const* ln2_g;        /* [hidden]                          */
  const void* const* ln2_b;        /* [hidden]                          */
  const void* const* w_1;          /* [ffn, hidden]                     */
  const void* const* b_1;          /* [ffn]                             */
  const void* const* w_2;          /* [hidden, ffn]                     */
  const void* const* b_2;          /* [hidden]                          */
  const void* lnf_g;               /* [hidden] (ignored if final_ln==0) */
  const void* lnf_b;               /* [hidden]                          */
} esm_weights;

typedef struct esm_encoder esm_encoder_t;

/* Create a handle for `cfg` on the current CUDA device.  Fails with
 * ESM_ERR_UNSUPPORTED unless the device is compute capability 10.3 (GB300) and the
 * geometry is one the kernels implement.  Allocates a few KB of device state (the
 * error word and the FP8 scaling state).  *out is NULL on failure. */
ESM_API esm_status esm_encoder_create(const esm_config* cfg, esm_encoder_t** out);

/* Free the handle and its device state.  NULL is accepted. */
ESM_API void esm_encoder_destroy(esm_encoder_t* h);

/* Bytes of device workspace a forward over at most max_tokens packed tokens in at most
 * max_seqs sequences needs (for the padded call: max_tokens = B*S, max_seqs = B). */
ESM_API esm_status esm_encoder_workspace_size(const esm_encoder_t* h, int max_tokens, int max_seqs,
                                      size_t* bytes);

/* Packed (THD) forward -- the packed model forward of section 3.2 of the hotelren.com
 * guide: forward(input_ids, cu_seqlens, max_seqlen).
 *   token_ids   device int32 [total_tokens], each in [0, vocab)
 *   cu_seqlens  device int32 [num_seqs + 1], 0 = c0 <= ... <= c_B = total_tokens
 *   max_seqlen  >= every c_{i+1} - c_i and <= max_positions
 *   hidden_out  device [total_tokens, hidden]
 *   workspace   device, 256-byte aligned, >= esm_encoder_workspace_size(T, B)
 * total_tokens == 0 is a no-op.
 * The call only enqueues work on `stream` (kernels and one memset), so it can be captured
 * into a CUDA graph; make one uncaptured call with the same handle first (it performs the
 * one-time kernel configuration).  A graph bakes in the pointers and sizes it captured;
 * each replay also advances the FP8 delayed-scaling state. */
ESM_API esm_status esm_encoder_forward(esm_encoder_t* h, const esm_weights* w, const int32_t* token_ids,
                               const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                               int max_seqlen, void* hidden_out, void* workspace,
                               size_t workspace_bytes, esm_stream_t stream);

/* Same as esm_encoder_forward but token_ids, cu_seqlens and hidden_out are HOST
 * buffers: the call copies the inputs into the workspace, runs the forward and copies
 * the result back, all on `stream`, and returns after the stream has synchronised.
 * Pinned host memory gives asynchronous copies; pageable memory works too.  With pinned
 * buffers (and profiling off) the handle keeps CUDA graphs of whole calls, up to 8, keyed by
 * every pointer and size they bake in (host buffers, weights, workspace, the three sizes, the
 * per-layer precision).  The second call with a key captures it on an internal stream, and
 * later calls replay it on `stream`: the same work without ~170 separate kernel launches.  A
 * capture that fails falls back to launching the kernels; the first call of a key always does. */
ESM_API esm_status esm_encoder_forward_host(esm_encoder_t* h, const esm_weights* w,
                                    const int32_t* token_ids_host, const int32_t* cu_seqlens_host,
                                    int num_seqs, int total_tokens, int max_seqlen,
                                    void* hidden_out_host, void* workspace, size_t workspace_bytes,
                                    esm_stream_t stream);

/* Padded (BSHD) forward with a key padding mask -- the padding-mask / bshd input format
 * of the mlqm.cn walkthrough (attention-mask section) and section 3.1 of the hotelren.com
 * guide.  token_ids device int32 [B, S] (pad id anywhere past each length);
 * seq_lens device int32 [B], 1 <= len_b <= S <= max_positions.  Every row, padding
 * included, goes through the GEMMs; queries attend to keys < len_b only; output rows
 * b*S + s with s >= len_b are written as zero.  hidden_out device [B, S, hidden]. */
ESM_API esm_status esm_encoder_forward_padded(esm_encoder_t* h, const esm_weights* w,
                                      const int32_t* token_ids, const int32_t* seq_lens, int B,
                                      int S, void* hidden_out, void* workspace,
                                      size_t workspace_bytes, esm_stream_t stream);

/* Per-layer GEMM precision -- the layer_precision setting and the per-layer autocast
 * context (get_autocast_context(layer_number)) of the mlqm.cn walkthrough (mixed FP8 / FP4
 * section): each Transformer layer may run its linear maps in its own precision.
 * per_layer[num_layers]: for an ESM_FP8_E4M3 handle each entry is ESM_FP8_E4M3 (the
 * layer's four GEMMs take E4M3 operands with the handle's delayed scaling), ESM_BF16
 * (bf16 operands; the layer's scales are then left unchanged) or ESM_FP4_E2M1 (the layer's
 * four GEMMs take NVFP4 operands -- see esm_op_quantize_nvfp4 -- quantised in the call from
 * the bf16 LayerNorm outputs, attention output and GELU output and from the bf16 weights,
 * each tensor with its own current scale S = 448 * 6 / amax; block-scaled tcgen05 GEMMs);
 * attention and LayerNorm stay bf16 in every layer.  A handle of another precision accepts
 * only its own precision for every layer; ESM_FP4_E2M1 as a handle precision is
 * ESM_ERR_UNSUPPORTED.  num_layers must equal the config's.  Takes effect from the next
 * forward; default: every layer in the handle's precision. */
ESM_API esm_status esm_encoder_set_layer_precision(esm_encoder_t* h, const esm_precision* per_layer, int num_layers);

/* The NVFP4 tensor scales S of the last forward's FP4 layers (ESM_FP8_E4M3 handles): host_buf
 * float32 [num_layers * 8] in the tensor order {x_qkv, w_qkv, x_o, w_o, x_1, w_1, x_2, w_2}
 * (zero for layers that did not run in FP4); n must equal num_layers * 8.  Synchronises the
 * device. */
ESM_API esm_status esm_encoder_get_fp4_scales(const esm_encoder_t* h, float* host_buf, size_t n);

/* ---- masked-LM head (the step after the encoder) ----
 * The mlqm.cn walkthrough loads the model as AutoModelForMaskedLM and the BioNeMo ESM-2
 * model card (accuracy benchmark) scores it by masked-LM perplexity; the pages do not list
 * the head's layers.  Reading: the ESM-2 head of that model family,
 *   z = LN(GELU(h Wd^T + bd); ln_g, ln_b);  logits = z E^T + b_vocab,
 * with E the token embedding [vocab, hidden] (tied), and the loss per scored token
 * log(sum_v exp(logits_v)) - logits_target.
 * Pointers are device pointers in the handle's parameter dtype (bf16, or float32 for
 * ESM_FP32): dense_w [hidden, hidden] ([out, in]), dense_b, ln_g, ln_b [hidden],
 * emb [vocab, hidden], bias [vocab]; 16-byte aligned. */
typedef struct {
  const void* dense_w;
  const void* dense_b;
  const void* ln_g;
  const void* ln_b;
  const void* emb;
  const void* bias;
} esm_lm_head;

/* Workspace bytes esm_encoder_lm_head needs for total_tokens tokens (two [T, hidden]
 * activation buffers and a [T] float32 scratch). */
ESM_API esm_status esm_encoder_lm_head_workspace_size(const esm_encoder_t* h, int total_tokens, size_t* bytes);

/* Logits and masked cross-entropy of final hidden states.  hidden: device [T, hidden] in
 * the activation dtype (bf16; float32 for ESM_FP32), e.g. the output of
 * esm_encoder_forward.  targets: device int32 [T] with a token id in [0, vocab) for
 * scored positions and -100 elsewhere, or NULL (nothing scored).  Outputs (each may be
 * NULL): logits device float32 [T, vocab]; token_loss device float32 [T] (0 where not
 * scored); loss_sum device float32 scalar and count device int32 scalar (sum and number
 * of scored tokens, reduced in a fixed order: perplexity = exp(loss_sum / count)).
 * ESM_ERR_UNSUPPORTED when vocab > 64, the embedding does not fit shared memory (vocab x
 * hidden x element > 200 KB) or (bf16) hidden % 256 != 0.  A target outside [0, vocab)
 * and != -100 is not scored and latches ESM_ERR_TOKEN_RANGE (see esm_encoder_check). */
ESM_API esm_status esm_encoder_lm_head(esm_encoder_t* h, const esm_lm_head* head, const void* hidden,
                                       int total_tokens, const int32_t* targets, float* logits,
                                       float* token_loss, float* loss_sum, int* count, void* workspace,
                                       size_t workspace_bytes, esm_stream_t stream);

/* ---- masked-LM head backward (the loss end of a training step) ----
 * Gradients of the mean masked-LM loss L = loss_sum / count (the head and loss of
 * esm_encoder_lm_head) with respect to the hidden states and the head's parameters, so that
 * a training step runs from the loss: esm_encoder_forward_train -> esm_encoder_lm_head_backward
 * (d_hidden) -> esm_encoder_backward (d_hidden_out = d_hidden).  The head's forward is
 * recomputed inside the call.  ESM_BF16 handles (hidden % 256 == 0, vocab <= 64).
 * hidden: device bf16 [T, hidden] (e.g. hidden_out of the training forward); targets as for
 * esm_encoder_lm_head; d_hidden: device float32 [T, hidden] (overwritten); grads: device
 * float32 buffers shaped like the head's parameters (overwritten; grads->emb is the head's
 * part of the tied embedding's gradient: add esm_encoder_backward's grads->emb for the
 * total); loss_sum, count: device scalars or NULL (this call's scored-token loss sum and
 * count).  loss_count: device int32 scalar or NULL: the number of scored tokens the mean is
 * taken over.  NULL means this call's own count.  A data-parallel step passes the scored count
 * of the whole global batch (all ranks' counts summed first), so that every rank
 * differentiates the same loss, sum over all scored tokens / global count, and the ranks'
 * gradients summed over ranks are the batch gradient.  Unscored rows (target -100) get zero
 * gradient; with nothing scored (or loss_count <= 0) every gradient is zero.  Workspace: the
 * size query's bytes. */
typedef struct {
  float* dense_w;
  float* dense_b;
  float* ln_g;
  float* ln_b;
  float* emb;
  float* bias;
} esm_lm_head_grads;
ESM_API esm_status esm_encoder_lm_head_backward_workspace_size(const esm_encoder_t* h, int total_tokens,
                                                               size_t* bytes);
ESM_API esm_status esm_encoder_lm_head_backward(esm_encoder_t* h, const esm_lm_head* head, const void* hidden,
                                                int total_tokens, const int32_t* targets, float* d_hidden,
                                                const esm_lm_head_grads* grads, float* loss_sum, int* count,
                                                const int* loss_count, void* workspace, size_t workspace_bytes,
                                                esm_stream_t stream);

/* Synchronise `stream` and return (and clear) the first error the kernels latched
 * since the last check: ESM_ERR_BAD_CU_SEQLENS, ESM_ERR_TOKEN_RANGE, ESM_ERR_TIMEOUT
 * or ESM_OK. */
ESM_API esm_status esm_encoder_check(esm_encoder_t* h, esm_stream_t stream);

/* Packing indices only (bit-exact parity hook for section 3.2 packing): validates
 * cu_seqlens like the forward and writes pos_id[t] = t - c_{seg(t)} and seg_id[t]
 * (device int32 [total_tokens] each). */
ESM_API esm_status esm_encoder_debug_pack_index(esm_encoder_t* h, const int32_t* cu_seqlens, int num_seqs,
                                        int total_tokens, int max_seqlen, int32_t* pos_id,
                                        int32_t* seg_id, void* workspace, size_t workspace_bytes,
                                        esm_stream_t stream);

/* Failure-detection hook: one warp waits, through the bounded wait every kernel of the
 * library uses but with a limit of timeout_us microseconds (1..1000000), on an mbarrier
 * nothing arrives at.  The wait gives up, ESM_ERR_TIMEOUT is latched in the handle (read
 * it with esm_encoder_check) and the kernel returns: the context stays usable. */
ESM_API esm_status esm_encoder_debug_wait_timeout(esm_encoder_t* h, int timeout_us, esm_stream_t stream);

/* ---- single-operation hooks (the kernels the forward uses, exposed for parity) ---- */

/* y = LN(x) * gamma + beta per row.  x device float32 [rows, cols]; gamma, beta device
 * in the handle's parameter dtype [cols]; y device in the handle's activation dtype
 * (float32 for ESM_FP32, bfloat16 otherwise).  LayerNorm of the hotelren.com guide
 * section 3.1 / the aikraft.ru te.LayerNorm. */
ESM_API esm_status esm_op_layernorm(esm_encoder_t* h, const float* x, const void* gamma, const void* beta,
                            void* y, int rows, int cols, esm_stream_t stream);

typedef enum {
  ESM_EPI_BIAS_F32 = 0,   /* out float32 [M,N] = A B^T + bias                          */
  ESM_EPI_QKV_ROPE = 1,   /* out act [M,N], N = 3*hidden: A B^T + bias, RoPE on q|k   */
  ESM_EPI_RESIDUAL = 2,   /* out float32 [M,N] += A B^T + bias (the residual stream)  */
  ESM_EPI_GELU = 3        /* out act [M,N] = GELU(A B^T + bias)                        */
} esm_epilogue;

/* One GEMM of the layer with its fused epilogue: A [M,K] (activation dtype), B [N,K]
 * (parameter dtype), bias [N] (parameter dtype).  pos_id (device int32 [M]) gives each
 * row's position for ESM_EPI_QKV_ROPE and is ignored otherwise.  ESM_BF16 requires
 * K % 64 == 0 and N % 256 == 0; ESM_FP32 accepts any sizes.  (ESM_FP8_E4M3 handles
 * use the bf16 tensor-core GEMM here.) */
ESM_API esm_status esm_op_gemm(esm_encoder_t* h, esm_epilogue epi, const void* A, const void* B,
                       const void* bias, void* out, const int32_t* pos_id, int M, int N, int K,
                       esm_stream_t stream);

/* E4M3 forms of the two hooks above, for ESM_FP8_E4M3 handles.
 * esm_op_layernorm_e4m3: y[r, c] = E4M3(LN(x)[r, c] * (*scale)) (round to nearest even,
 *   saturating at +-448), max |LN(x)| folded into *amax with an atomic max (set it to 0
 *   first).  x device float32 [rows, cols]; gamma, beta device bf16; y device uint8 codes;
 *   scale, amax device float32 scalars.
 * esm_op_gemm_fp8: out = epilogue((A B^T) / ((*a_scale) (*b_scale)) + bias) with A
 *   [M, K] and B [N, K] device E4M3 codes, K % 128 == 0, N % 256 == 0; bias bf16; output
 *   as for esm_op_gemm (ESM_EPI_GELU writes bf16 here). */
ESM_API esm_status esm_op_layernorm_e4m3(esm_encoder_t* h, const float* x, const void* gamma, const void* beta,
                                         uint8_t* y, int rows, int cols, const float* scale, float* amax,
                                         esm_stream_t stream);
ESM_API esm_status esm_op_gemm_fp8(esm_encoder_t* h, esm_epilogue epi, const uint8_t* A, const uint8_t* B,
                                   const float* a_scale, const float* b_scale, const void* bias, void* out,
                                   const int32_t* pos_id, int M, int N, int K, esm_stream_t stream);

/* Variable-length bidirectional attention over packed sequences (section 3.2 of the
 * hotelren.com guide, thd format).  qkv device [T, 3*hidden] in the activation dtype
 * (q | k | v, head-major, RoPE already applied); o device [T, hidden].  Each token
 * attends to all tokens of its own sequence.  Uses the workspace for the work list. */
ESM_API esm_status esm_op_attention(esm_encoder_t* h, const void* qkv, const int32_t* cu_seqlens,
                            int num_seqs, int total_tokens, int max_seqlen, void* o,
                            void* workspace, size_t workspace_bytes, esm_stream_t stream);

/* ---- attention without any allocation ----
 * No counterpart on the pages: this entry point exists for callers that cannot allocate
 * device memory (a memory pool or allocator that owns the whole device, a plugin host that
 * hands out only its input and output buffers, a runtime that forbids allocation after
 * start-up).  It runs the same tcgen05 attention kernel as esm_op_attention on a bf16
 * handle, head_dim 64 (qkv device bf16 [T, 3*hidden], q | k | v head-major, RoPE applied,
 * 16-byte aligned; o device bf16 [T, hidden]; cu_seqlens device int32 [num_seqs + 1]),
 * without a handle or a workspace: its scratch is a fixed device array inside the library
 * (about 650 KB, held by every GPU that loads the library until the process exits), and
 * the kernel's TMA descriptor is encoded on the host for each call.
 * Limits: total_tokens <= ESM_NOALLOC_MAX_TOKENS, num_seqs <= ESM_NOALLOC_MAX_SEQS,
 * max_seqlen <= ESM_NOALLOC_MAX_TOKENS; larger sizes return ESM_ERR_INVALID_ARG.
 * hidden must be 64 * heads (ESM_ERR_UNSUPPORTED otherwise, or off sm_103).
 * status: device int32 or NULL.  When given, it receives (in stream order, after the
 * attention) ESM_OK, ESM_ERR_BAD_CU_SEQLENS if cu_seqlens was malformed (the offsets are
 * then clamped so every access stays in bounds, and o is not meaningful), or
 * ESM_ERR_TIMEOUT if a bounded device wait gave up.
 * The first call on each device looks up the array's device address (with that device
 * current) and caches it: make that first call before any stream capture.  Calls share
 * the array, so calls that overlap on the GPU (different streams) race. */
#define ESM_NOALLOC_MAX_TOKENS 65536
#define ESM_NOALLOC_MAX_SEQS 4096
ESM_API esm_status esm_op_attention_noalloc(const void* qkv, const int32_t* cu_seqlens, int num_seqs,
                                            int total_tokens, int max_seqlen, int hidden, int heads, void* o,
                                            int32_t* status, esm_stream_t stream);

/* ---- NVFP4 (block-scaled E2M1) operands and GEMM ----
 * The mlqm.cn walkthrough (section FP8与FP4混合精度支持) gives the encoder an fp4_recipe beside
 * the FP8 one; the pages give no FP4 format.  The format read here is the block-scaled FP4 of
 * the tensor cores: E2M1 values (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), one E4M3 scale per
 * block of 16 consecutive values along K, one fp32 tensor scale S = 448 * 6 / amax:
 *   sb = E4M3(max|block| / 6 * S),  q = E2M1(x * S / sb) (0 for an all-zero block),  x ~ q sb / S,
 * both roundings to nearest even, saturating.
 * esm_op_quantize_nvfp4: x device bf16 [rows, cols] (rows % 128 == 0, cols % 256 == 0, 16-byte
 *   aligned) -> codes device [rows, cols / 2] bytes (value k in the low nibble of byte k / 2 for
 *   even k), scales device [rows * cols / 16] bytes in 512-byte atoms of 128 rows x 64 values
 *   (atom (r / 128, k / 64) at ((r / 128) * (cols / 64) + k / 64) * 512, row r and 16-value block
 *   b inside it at (r % 32) * 16 + ((r % 128) / 32) * 4 + b), amax and scale device float scalars
 *   (overwritten: the tensor's max |x| and S).  Two kernels (amax, then codes and scales).
 * esm_op_gemm_nvfp4: v = (A B^T) / (a_scale b_scale) + bias for NVFP4 operands from
 *   esm_op_quantize_nvfp4 (A [M, K], B [N, K]; a_scale, b_scale their device tensor scales;
 *   bias device bf16 [N] or NULL), then the epilogue an FP4 layer uses:
 *     ESM_EPI_BIAS_F32  out device float32 [M, N] = v;
 *     ESM_EPI_RESIDUAL  out device float32 [M, N] += v;
 *     ESM_EPI_GELU      out device bf16 [M, N] = GELU(v);
 *     ESM_EPI_QKV_ROPE  out device bf16 [M, N] = v with RoPE on the q and k columns at the
 *                       row's position pos_id[row] (device int32 [M], clamped to the handle's
 *                       max_positions); N must equal 3 * hidden of the handle.
 *   pos_id is ignored by the other epilogues.  M % 128, N % 128, K % 256 all 0 (else
 *   ESM_ERR_INVALID_ARG).  tcgen05.mma kind::mxf4nvf4 with block scaling (the E4M3 block scales
 *   multiply on the tensor core).  Needs an ESM_BF16 or ESM_FP8_E4M3 handle (for its error word,
 *   tensor-map cache and RoPE table). */
ESM_API esm_status esm_op_quantize_nvfp4(esm_encoder_t* h, const void* x, int rows, int cols, uint8_t* codes,
                                         uint8_t* scales, float* amax, float* scale, esm_stream_t stream);
ESM_API esm_status esm_op_gemm_nvfp4(esm_encoder_t* h, esm_epilogue epi, const uint8_t* a_codes,
                                     const uint8_t* a_scales, const float* a_scale, const uint8_t* b_codes,
                                     const uint8_t* b_scales, const float* b_scale, const void* bias,
                                     const int32_t* pos_id, void* out, int M, int N, int K, esm_stream_t stream);

/* ---- FP8 delayed-scaling state (ESM_FP8_E4M3 handles) ----
 * Layout, float32: for each layer l and each of the 8 quantised tensors k in the order
 * {x_qkv, w_qkv, x_o, w_o, x_1, w_1, x_2, w_2}: scale[l][k] (num_layers*8 floats), then
 * amax_history[l][k][amax_history_len] (newest first).  n is the number of floats in
 * host_buf and must equal num_layers*8*(1 + amax_history_len).  Initial state: every
 * scale 1, every history entry 0.  get synchronises the device. */
ESM_API esm_status esm_encoder_get_fp8_state(const esm_encoder_t* h, float* host_buf, size_t n);
ESM_API esm_status esm_encoder_set_fp8_state(esm_encoder_t* h, const float* host_buf, size_t n);

/* ---- training: a forward that keeps its activations, and the backward pass ----
 * The hotelren.com guide trains the packed model over cu_seqlens (section 3.2, the packed
 * training loop; section 6, the training step with loss.backward()); the mlqm.cn walkthrough
 * describes the same layer stack under training.  The pages do not write the backward
 * out: it is the exact gradient of the forward above (chain rule through the final
 * LayerNorm, every layer in reverse, and the embedding), with bf16 GEMM and attention
 * operands and fp32 accumulation, reductions over tokens in a fixed order.
 * ESM_BF16 handles with hidden <= 4096 only (others: ESM_ERR_UNSUPPORTED).
 *
 * Gradient buffers: device float32, same shapes as the weights ([out, in] for linear
 * maps); the per-layer members point to HOST arrays of num_layers DEVICE pointers.
 * Every buffer is overwritten (not accumulated into); 16-byte aligned. */
typedef struct {
  float* emb;                 /* [vocab, hidden]                                 */
  float* const* ln1_g;
  float* const* ln1_b;
  float* const* w_qkv;        /* [3*hidden, hidden]                              */
  float* const* b_qkv;
  float* const* w_o;          /* [hidden, hidden]                                */
  float* const* b_o;
  float* const* ln2_g;
  float* const* ln2_b;
  float* const* w_1;          /* [ffn, hidden]                                   */
  float* const* b_1;
  float* const* w_2;          /* [hidden, ffn]                                   */
  float* const* b_2;
  float* lnf_g;               /* [hidden] (ignored if final_ln == 0)             */
  float* lnf_b;
} esm_grads;

/* Bytes of the training buffer for up to max_tokens tokens: per layer the layer input and
 * mid-layer residual (float32 [T, hidden]), the LayerNorm outputs, q|k|v after RoPE, the
 * attention output (bf16), the attention log-sum-exp (float32 [heads, T]), fc1's
 * pre-activation and GELU output (bf16 [T, ffn]); then the backward's scratch.  About
 * 46 KB per token per layer for ESM-2 650M. */
ESM_API esm_status esm_encoder_train_buffer_size(const esm_encoder_t* h, int max_tokens, size_t* bytes);

/* The packed forward of esm_encoder_forward (same arguments, same hidden_out in bf16) that
 * also keeps its activations in train_buf (device, 256-byte aligned, at least
 * esm_encoder_train_buffer_size bytes).  total_tokens > 0.  The workspace and train_buf
 * belong to the handle's next esm_encoder_backward: leave both untouched until then (another
 * call of this handle with the same workspace withdraws that backward, which then returns
 * ESM_ERR_INVALID_ARG).
 * Errors as esm_encoder_forward; ESM_ERR_WORKSPACE for a short train_buf. */
ESM_API esm_status esm_encoder_forward_train(esm_encoder_t* h, const esm_weights* w, const int32_t* token_ids,
                                             const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                                             int max_seqlen, void* hidden_out, void* train_buf, size_t train_bytes,
                                             void* workspace, size_t workspace_bytes, esm_stream_t stream);

/* Gradients of a loss L with respect to every parameter, given d_hidden_out = dL/d(hidden_out)
 * (device float32 [T, hidden], T of the last esm_encoder_forward_train on this handle).
 * train_buf and workspace must be the ones that forward used (ESM_ERR_INVALID_ARG
 * otherwise); weights as in that forward.  grads->emb receives emb_scale times the sum of
 * the embedded rows' gradients per token id. */
ESM_API esm_status esm_encoder_backward(esm_encoder_t* h, const esm_weights* w, const float* d_hidden_out,
                                        const esm_grads* grads, void* train_buf, size_t train_bytes,
                                        void* workspace, size_t workspace_bytes, esm_stream_t stream);

/* Backward hooks (the kernels the backward uses, exposed for parity); bf16 operands,
 * handles of precision ESM_BF16 or ESM_FP8_E4M3.
 * esm_op_gemm_dgrad: out[M, K] = dY[M, N] W with dY device bf16 [M, N] and W device bf16
 *   [N, K] (a weight, [out, in]); out device float32, or bf16 with out_bf16 != 0.
 *   N % 64 == 0, K % 256 == 0, 16-byte aligned pointers.
 * esm_op_gemm_wgrad: dW[N, K] = dY^T X summed over the M rows of dY (bf16 [M, N]) and X
 *   (bf16 [M, K]); dW device float32.  N % 256 == 0, K % 256 == 0, any M.  The workspace
 *   (esm_op_gemm_wgrad_workspace_size bytes, 256-byte aligned; NULL allowed, then the
 *   token reduction is not split) holds split partial products, added in a fixed order. */
ESM_API esm_status esm_op_gemm_dgrad(esm_encoder_t* h, const void* dY, const void* W, void* out, int out_bf16, int M,
                                     int N, int K, esm_stream_t stream);
ESM_API esm_status esm_op_gemm_wgrad_workspace_size(const esm_encoder_t* h, int N, int K, size_t* bytes);
ESM_API esm_status esm_op_gemm_wgrad(esm_encoder_t* h, const void* dY, const void* X, float* dW, int M, int N, int K,
                                     void* workspace, size_t workspace_bytes, esm_stream_t stream);

/* LayerNorm backward over rows of x (device float32 [rows, cols], cols % 4 == 0, cols <= 4096): with
 * dy = dL/dy (float32 [rows, cols]) and gamma in the parameter dtype,
 *   dx = dres + dL/dx (dres may be NULL or equal to dx), dgamma = sum_rows dy xhat,
 *   dbeta = sum_rows dy (float32 [cols]).  Workspace: the size query's bytes. */
ESM_API esm_status esm_op_layernorm_backward_workspace_size(const esm_encoder_t* h, int rows, int cols,
                                                            size_t* bytes);
ESM_API esm_status esm_op_layernorm_backward(esm_encoder_t* h, const float* x, const void* gamma, const float* dy,
                                             const float* dres, float* dx, float* dgamma, float* dbeta, int rows,
                                             int cols, void* workspace, size_t workspace_bytes,
                                             esm_stream_t stream);

/* esm_op_attention (bf16, head_dim 64) that also writes lse (device float32 [heads, T],
 * head-major): the natural-log softmax normaliser log sum_s exp(q_t . k_s / 8) of every query
 * row.
 * esm_op_attention_backward: from the same qkv (bf16 [T, 3*hidden], q | k | v as the
 * attention read them), its output o (bf16 [T, hidden]), lse and d_o = dL/do (bf16
 * [T, hidden]), writes dqkv = dL/d(q | k | v) (bf16 [T, 3*hidden]).  Workspace:
 * esm_op_attention_backward_workspace_size bytes (the forward's work list plus float32
 * scratch [heads, T] and [T, hidden]). */
ESM_API esm_status esm_op_attention_train(esm_encoder_t* h, const void* qkv, const int32_t* cu_seqlens, int num_seqs,
                                          int total_tokens, int max_seqlen, void* o, float* lse, void* workspace,
                                          size_t workspace_bytes, esm_stream_t stream);
ESM_API esm_status esm_op_attention_backward_workspace_size(const esm_encoder_t* h, int total_tokens, int num_seqs,
                                                            size_t* bytes);
ESM_API esm_status esm_op_attention_backward(esm_encoder_t* h, const void* qkv, const void* o, const float* lse,
                                             const void* d_o, const int32_t* cu_seqlens, int num_seqs,
                                             int total_tokens, int max_seqlen, void* dqkv, void* workspace,
                                             size_t workspace_bytes, esm_stream_t stream);

/* ---- measurement hooks ----
 * Kernel classes of the forward: 0 QKV GEMM (+bias, RoPE), 1 attention, 2 output-projection
 * GEMM (+bias, residual), 3 fc1 GEMM (+bias, GELU), 4 fc2 GEMM (+bias, residual),
 * 5 LayerNorm, 6 everything else (packing, work list, embedding, FP8 quantise/update),
 * 7 the backward's GEMMs (input and weight gradients, with their split-K sums). */
#define ESM_PROFILE_CLASSES 8
typedef struct {
  double ms[ESM_PROFILE_CLASSES];           /* summed device time per class (profiling on)  */
  long long launches[ESM_PROFILE_CLASSES];  /* kernel launches per class                     */
  long long total_launches;                 /* all kernel launches since the last reset      */
} esm_profile;

/* enable != 0: bracket every kernel launch with CUDA events recorded on the launch stream,
 * so per-class device times can be read back (adds a small per-launch cost).  Launches are
 * counted whether or not profiling is on. */
ESM_API esm_status esm_encoder_set_profiling(esm_encoder_t* h, int enable);

/* Synchronise the device, fill *out with the totals since the last reset and, if reset is
 * nonzero, start new totals. */
ESM_API esm_status esm_encoder_get_profile(esm_encoder_t* h, esm_profile* out, int reset);

/* Static string for a status code. */
ESM_API const char* esm_status_string(esm_status s);

#ifdef __cplusplus
}
#endif

#endif /* ESM_ENCODER_H_ */
