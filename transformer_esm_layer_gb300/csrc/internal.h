// Internal declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/esm_encoder.h"

namespace esm {

// Rows of one attention query tile (mma.sync kernel; the tcgen05 kernel uses 128).
constexpr int kAttnQTile = 64;
constexpr int kAttnQTileTc = 128;
// Columns per RoPE table row (head_dim / 2, head_dim <= 64).
constexpr int kRopeMaxHalf = 32;

enum class Act { F32, BF16, E4M3 };

struct PackBuffers {
  int32_t* pos_id;     // [T]
  int32_t* seg_id;     // [T]
  int32_t* seg_start;  // [B]
  int32_t* seg_qlen;   // [B]  query rows of the segment
  int32_t* seg_klen;   // [B]  visible keys of the segment
  int32_t* work;       // [4 * max_items]: (first query row, query rows, first key row, keys)
  int32_t* work_count; // [1]
};

// ---------------------------------------------------------------- launchers (pack.cu)
void launch_pack_index(const int32_t* cu, int B, int T, int max_seqlen, int max_positions,
                       const PackBuffers& pb, unsigned* err, cudaStream_t st);
void launch_pad_index(const int32_t* seq_lens, int B, int S, const PackBuffers& pb, unsigned* err,
                      cudaStream_t st);
// Work items (segment, first query row) in tiles of q_tile rows, longest segments first.
void launch_attn_worklist(int B, int max_items, int q_tile, const PackBuffers& pb, cudaStream_t st);
void launch_embed(const int32_t* tok, int T, const void* emb, bool emb_f32, int vocab, int d, float scale,
                  float* x, unsigned* err, cudaStream_t st);
void launch_rope_table(float2* tab, int max_pos, int half, float base, cudaStream_t st);
// A bounded wait that runs out (failure-detection hook).
void launch_wait_timeout(unsigned long long limit_ns, unsigned* err, cudaStream_t st);

// ---------------------------------------------------------------- layernorm.cu
// y = LN(x) * g + b. Params in f32 or bf16; output f32, bf16 or e4m3 (scaled by
// *q_scale); for e4m3 and bf16 outputs max|y| is folded into *amax when amax is non-null.  With valid_* set, rows whose position is not below the
// segment's visible length are written as zero.
void launch_layernorm(const float* x, const void* g, const void* b, bool param_f32, void* y, Act out,
                      int rows, int cols, float eps, const float* q_scale, float* amax,
                      const int32_t* valid_pos, const int32_t* valid_seg, const int32_t* valid_klen,
                      cudaStream_t st);
// out = x (converted), zeroing invalid rows the same way (final_ln == 0).
// LayerNorm of a bfloat16 input (same arithmetic; no FP8 output, no validity mask).
void launch_layernorm_bf16in(const void* x, const void* g, const void* b, bool param_f32, void* y, Act out, int rows,
                             int cols, float eps, cudaStream_t st);
// Masked-LM head output stage (lm_head.cu): logits against the tied embedding, per-token
// masked cross-entropy, and its deterministic sum / scored count.
size_t lm_logits_smem_bytes(int vocab, int hidden, bool bf16);
bool lm_logits_supported(int vocab, int hidden, bool bf16);
cudaError_t launch_lm_logits(const void* z, bool bf16, const void* emb, const void* bias, int T, int d, int V,
                             const int32_t* targets, float* logits, float* token_loss, float* loss_sum, int* count,
                             int num_sms, unsigned* err, cudaStream_t st);
void launch_copy_out(const float* x, void* out, Act out_t, int rows, int cols, const int32_t* valid_pos,
                     const int32_t* valid_seg, const int32_t* valid_klen, cudaStream_t st);

// ---------------------------------------------------------------- GEMMs
struct EpiArgs {
  const void* bias;       // [N] param dtype
  bool bias_f32;
  void* out;              // [M, N]
  const int32_t* pos_id;  // [M] (QKV)
  const float2* rope;     // [kRopeMaxHalf/2][max_pos][2] (cos, sin), see rope_table_kernel
  int rope_cols;          // columns < rope_cols get RoPE (2 * hidden)
  int head_dim;
  int max_pos;
  const float* a_scale;   // FP8: scale of A (device)
  const float* b_scale;   // FP8: scale of B (device)
  const float* o_scale;   // FP8 GELU output: quantisation scale (device)
  float* o_amax;          // FP8 GELU output: amax (device)
  const void* res_in;     // ESM_EPI_RESIDUAL: residual read from here instead of out (NULL: in place)
  void* aux;              // ESM_EPI_GELU: also store the pre-activation here (bf16 [M, N]; NULL: no);
                          // kEpiDgelu: the forward's pre-activation z to multiply by GELU'(z)
  // LayerNorm folded into the next GEMM (bf16 forward).  The residual epilogue writes, for
  // the updated rows, the statistics of every 64-column group (mean, sum of squared
  // deviations: float2 [M, N / 64]) and, with ln_a_out, the next GEMM's operand
  // bf16(x * gamma) ([M, N]).  The consumer (QKV / GELU epilogue) reads the statistics of
  // its A rows and applies LN(x) W^T + b = rstd (acc - mean c) + b' per row, with
  // c_n = sum_k gamma_k W_nk and b'_n = b_n + sum_k beta_k W_nk (fp32 [N]) in place of the bias.
  float2* ln_stats_out;   // ESM_EPI_RESIDUAL: statistics of the new residual rows (NULL: none)
  const void* ln_gamma;   // ESM_EPI_RESIDUAL: gamma (bf16 [N]) of the LayerNorm that follows
  void* ln_a_out;         // ESM_EPI_RESIDUAL: bf16(x * gamma) [M, N] (NULL: not written)
  const float2* ln_stats_in;  // QKV / GELU: statistics of the A rows [M, ln_groups] (NULL: no fold)
  const float* ln_c;      // [N] sum_k gamma_k W_nk
  const float* ln_b;      // [N] b_n + sum_k beta_k W_nk
  int ln_groups;          // K / 64
  float ln_eps;
};
// Epilogue of the input gradient through fc1's GELU: out = acc * GELU'(z) (bf16), z = aux.
constexpr int kEpiDgelu = 16;

// tcgen05 GEMM: A [M,K] bf16 (or e4m3), B [N,K] bf16 (or e4m3); K % 64 == 0 (bf16) or
// K % 128 == 0 (e4m3); N % 256 == 0.
int gemm_tc_smem_bytes();
// Box heights of the A and B tensor maps launch_gemm_tc expects (each CTA of a pair loads
// 128 rows of A and 128 rows of the 256-row B tile).
int gemm_tc_a_box_rows();
int gemm_tc_b_box_rows();
int gemm_tc_out_box_rows();
// tmO: the output [M, N] (fp32, bf16 or e4m3) with a 128-byte x gemm_tc_out_box_rows() box
// and the 128-byte swizzle; for ESM_EPI_RESIDUAL it is also read (the residual stream).
cudaError_t launch_gemm_tc(esm_epilogue epi, bool fp8, Act out_act, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, const CUtensorMap* tmO, int M, int N, int K, const EpiArgs& ea,
                           int num_sms, unsigned* err, cudaStream_t st);

// Backward products on the same kernel with MN-major operands (bf16):
//   DGRAD_F32 / DGRAD_BF16: out[M, N] = A[M, K] * B, B stored [K, N] (a weight [out, in]
//     read as its transpose): tmB is a [K rows, N cols] map with a 64 x 64 box
//     (gemm_tc_mn_box_rows()); output fp32 (bias / no epilogue) or bf16 (ea.rope_cols = 0);
//   WGRAD_F32: out[M, N] = A^T B with A stored [K, M] and B stored [K, N] (dY and X over the
//     K tokens), both 64 x 64-box maps; with ksplit > 1 the output map covers
//     [ksplit * M, N] partial sums (M % 256 == 0).
// N % 256 == 0; K any (the last K-slice is zero-filled by the maps).
//   DGRAD_GELU: as DGRAD_BF16, times GELU'(z) with z = ea.aux (bf16 [M, N]).
enum class GemmBwd { DGRAD_F32, DGRAD_BF16, DGRAD_GELU, WGRAD_F32 };
int gemm_tc_mn_box_rows();
int gemm_tc_max_clusters(int num_sms);
cudaError_t launch_gemm_tc_bwd(GemmBwd kind, const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmO,
                               int M, int N, int K, int ksplit, const EpiArgs& ea, int num_sms, unsigned* err,
                               cudaStream_t st);

// SIMT fp32 GEMM (the ESM_FP32 precision): any M, N, K.
void launch_gemm_f32(esm_epilogue epi, const float* A, const float* B, int M, int N, int K,
                     const EpiArgs& ea, cudaStream_t st);
// In-place RoPE on the q and k blocks of qkv [T, 3*d] (fp32).
void launch_rope_f32(float* qkv, int T, int d, int head_dim, const int32_t* pos_id, const float2* rope,
                     int max_pos, cudaStream_t st);

// Folded-LayerNorm constants of one linear map W [n, k] (bf16) that follows a LayerNorm
// (gamma, beta [k], bf16) with bias (bf16 [n]): c_out[i] = sum_j gamma_j W_ij and
// b_out[i] = bias_i + sum_j beta_j W_ij (fp32).
struct LnFoldJob {
  const void* w;
  const void* gamma;
  const void* beta;
  const void* bias;
  float* c_out;
  float* b_out;
  int n;
};
constexpr int kLnFoldMaxJobs = 96;
void launch_ln_fold(const LnFoldJob* jobs, int num_jobs, int k, cudaStream_t st);

// ---------------------------------------------------------------- fp4.cu
// NVFP4 operand of x [rows_valid, K] bf16, padded with zero rows to `rows` (rows % 128 == 0,
// K % 256 == 0): E2M1 codes [rows, K/2] bytes, E4M3 block scales in 512-byte atoms of 128 rows
// x 64 values, the tensor's amax and its scale S = 448 * 6 / amax (device scalars).  With
// amax_ready the amax was already accumulated (from zero) by the kernel that wrote x, and only
// the scale and the codes are computed here.
cudaError_t launch_nvfp4_quantize(const __nv_bfloat16* x, int rows, int rows_valid, int K, uint8_t* codes,
                                  uint8_t* sf, float* amax, float* scale, bool amax_ready, int num_sms,
                                  cudaStream_t st);
// Epilogues of the NVFP4 GEMM (v = acc / (S_A S_B) + bias on rows below rows_valid).
enum : int { kFp4F32 = 0, kFp4Residual = 1, kFp4Gelu = 2, kFp4QkvRope = 3 };
struct Fp4Epi {
  const void* bias;       // bf16 [N] or NULL
  void* out;              // fp32 (F32, RESIDUAL) or bf16 (GELU, QKV_ROPE) [rows_valid, N]
  int rows_valid;
  const int32_t* pos_id;  // QKV_ROPE: [rows_valid]
  const float2* rope;     // QKV_ROPE: the (cos, sin) table
  int rope_cols;          // QKV_ROPE: columns below get RoPE
  int max_pos;
  float* amax;            // GELU: max |bf16 out| is folded in here when non-null
};
// out = epilogue((A B^T) / (a_scale b_scale)) for NVFP4 operands A [M, K], B [N, K] (tensor
// maps over the code bytes [rows, K/2] with a 128-row x 128-byte box and the 128-byte swizzle);
// M % 128 == 0, N % 128 == 0, K % 256 == 0.  Persistent: min(128 x 256 tiles, num_sms) CTAs.
int gemm_nvfp4_smem_bytes();
cudaError_t launch_gemm_nvfp4(int epi, const CUtensorMap* tmA, const CUtensorMap* tmB, const uint8_t* sfa,
                              const uint8_t* sfb, const float* a_scale, const float* b_scale, const Fp4Epi& ea, int M,
                              int N, int K, int num_sms, unsigned* err, cudaStream_t st);

// ---------------------------------------------------------------- attention.cu
// tcgen05 attention (head_dim 64): tm_qkv is a tensor map over qkv [T, 3d] bf16 with a
// 64 x 128 box and the 128-byte swizzle; work items in tiles of kAttnQTileTc rows.
int attention_tc_smem_bytes();
// lse (optional, fp32 [heads, lse_stride], head-major): the natural-log softmax normaliser of
// every query row (scores scaled by 1/sqrt(head_dim)), kept by the training forward for the
// backward; lse_stride >= T.
// The tensor map launch_attention_tc expects over qkv [T, 3d] bf16, encoded on the host
// (no allocation); false if the CUDA tensor-map encoder is unavailable or rejects the layout.
bool encode_attention_qkv_map(const void* qkv, int total_tokens, int hidden, CUtensorMap* out);
cudaError_t launch_attention_tc(const CUtensorMap* tm_qkv, void* o, Act out, int d, int heads, int max_items,
                                const PackBuffers& pb, const float* q_scale, float* amax, unsigned* err,
                                cudaStream_t st, float* lse = nullptr, int lse_stride = 0);
void launch_attention_f32(const float* qkv, float* o, int d, int heads, int T, const PackBuffers& pb,
                          cudaStream_t st);

// tcgen05 attention backward (attention_bwd_tc.cu): dqkv (bf16 [T, 3d]) from the saved
// qkv (RoPE applied), O, the forward's lse ([heads, T]) and dO (bf16 [T, d], tm_do a
// 64 x 128-box map);
// with rope set the q and k gradients are turned back through RoPE (positions pb.pos_id).
// Scratch: dsum [heads, T], dq_acc [T, d] (fp32; tm_dq a map over it with a 32 x 32 box and
// the 128-byte swizzle, the target of the dQ reduce-adds).
cudaError_t launch_attention_bwd_tc(const CUtensorMap* tm_qkv, const CUtensorMap* tm_do, const CUtensorMap* tm_dq,
                                    const __nv_bfloat16* o,
                                    const __nv_bfloat16* dout, const float* lse, float* dsum, float* dq_acc,
                                    __nv_bfloat16* dqkv, int T, int d, int heads, int max_items, const PackBuffers& pb,
                                    const float2* rope, int max_pos, int num_sms, unsigned* err, cudaStream_t st);

// ---------------------------------------------------------------- backward.cu
// Scratch floats for the column reductions of rows x cols (LayerNorm: two sums per column).
size_t bwd_partial_floats(int rows, int cols);
size_t emb_bwd_partial_floats(int rows, int vocab, int d);
// LayerNorm backward: dx = dres + dLN/dx (dres may be NULL or alias dx), dgamma, dbeta
// (float32 [cols]); partial: bwd_partial_floats(rows, cols) floats of scratch.  cols % 4 == 0.
void launch_ln_bwd(const float* x, const void* gamma, bool gf32, const float* dy, const float* dres, float* dx,
                   float* dgamma, float* dbeta, float* partial, int rows, int cols, float eps, cudaStream_t st);
// out[c] = sum_r src[r][c] (fp32 or bf16 rows); copy (fp32 input only, may be NULL): the
// rows as bf16.  partial: bwd_partial_floats(rows, cols) / 2 floats.  cols % 4 == 0.
void launch_colsum(const void* src, bool bf16_in, int rows, int cols, float* out, float* partial, __nv_bfloat16* copy,
                   cudaStream_t st);
// out[i] = scale * sum_k partial[k * stride + i] over k = 0..chunks-1, in index order.
void reduce_chunks(const float* partial, int chunks, size_t stride, size_t n, float scale, float* out, cudaStream_t st);
// LayerNorm backward of a bf16 input x (no residual gradient added): dx, dgamma, dbeta.
void launch_ln_bwd_bf16in(const void* x, const void* gamma, bool gf32, const float* dy, float* dx, float* dgamma,
                          float* dbeta, float* partial, int rows, int cols, float eps, cudaStream_t st);
// dz = du * GELU'(a) (a: bf16 pre-activation; dz bf16); n % 4 == 0, buffers 16-byte aligned.
void launch_gelu_bwd(const float* du, const __nv_bfloat16* a, __nv_bfloat16* dz, size_t n, cudaStream_t st);
// Masked-LM head backward, output stage: dlogits of the mean masked cross-entropy (count =
// number of scored tokens, device), dz = dlogits * emb (fp32 [T, d]), the tied embedding's
// and the vocabulary bias's gradients (fp32, fixed-order sums over token chunks).  emb bf16,
// z (the LayerNorm output) bf16.  partial: lm_backward_partial_floats floats.
size_t lm_backward_partial_floats(int T, int V, int d);
cudaError_t launch_lm_backward_head(const float* logits, const int32_t* targets, const int* count, const void* emb,
                                    const __nv_bfloat16* z, int T, int d, int V, float* dl, float* dz, float* demb,
                                    float* dbias, float* partial, int num_sms, cudaStream_t st);
// out[i] = sum_s partial[s * n + i] (split-K partial products, in split order).
void launch_reduce_splits(const float* partial, int splits, size_t n, float* out, cudaStream_t st);
// demb[v] = scale * sum over tokens t with tok[t] == v of dx[t] (float32 [vocab, d]).
void launch_emb_bwd(const float* dx, const int32_t* tok, int T, int d, int vocab, float scale, float* partial,
                    float* demb, cudaStream_t st);

// ---------------------------------------------------------------- fp8.cu
// Quantise a bf16 tensor to e4m3 with *scale; record max|w| into *amax.
void launch_quantize_e4m3(const __nv_bfloat16* w, uint8_t* q, size_t n, const float* scale, float* amax,
                          cudaStream_t st);
// Delayed-scaling update of n tensors: push amax[i] into hist[i][0..len), scale[i] =
// 448 / max(hist[i]) (kept if the max is zero or not finite); amax[i] reset to 0.
void launch_fp8_update(float* scale, float* hist, float* amax, int n, int len, cudaStream_t st);

}  // namespace esm
