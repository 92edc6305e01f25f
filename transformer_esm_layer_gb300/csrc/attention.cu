// Variable-length bidirectional attention over packed sequences, fp32 (the ESM_FP32
// precision of the small fp32 configuration; bf16 and FP8 encoders use the tcgen05 kernel
// in attention_tc.cu).
//
// Section 3.2 of the hotelren.com guide ("生物大模型训练加速实战") runs every layer over
// cu_seqlens (thd format); the BioNeMo ESM-2 model card describes a bidirectional
// (BERT-style) encoder.  So each token attends to every token of its own sequence and to
// nothing else:
//
//   o_t = sum_s softmax_s(q_t . k_s / sqrt(dh)) v_s,   s over the sequence of t.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

// fp32 attention (the ESM_FP32 precision): one warp per (query row, head); lanes split
// the keys, each keeps a running max / sum / output, merged across lanes at the end.
__global__ void attention_f32_kernel(const float* __restrict__ qkv, float* __restrict__ o, int d, int heads, int T,
                                     PackBuffers pb) {
  const int warps = blockDim.x >> 5;
  const int gw = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= T * heads) return;
  const int t = gw / heads, h = gw - (gw / heads) * heads;
  const int dh = d / heads;
  const int seg = pb.seg_id[t];
  const int start = pb.seg_start[seg];
  const int klen = pb.seg_klen[seg];
  const int ld = 3 * d;
  float q[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) q[c] = c < dh ? qkv[(size_t)t * ld + h * dh + c] : 0.f;
  const float scale = 1.f / sqrtf((float)dh);
  float m = -INFINITY, l = 0.f, acc[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) acc[c] = 0.f;
  for (int j = lane; j < klen; j += 32) {
    const float* kr = qkv + (size_t)(start + j) * ld + d + h * dh;
    const float* vr = qkv + (size_t)(start + j) * ld + 2 * d + h * dh;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c < dh) s = fmaf(q[c], kr[c], s);
    s *= scale;
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn), p = expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c < dh) acc[c] = acc[c] * corr + p * vr[c];
    m = mn;
  }
  float M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float f = (m == -INFINITY) ? 0.f : expf(m - M);
  l *= f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    if (c >= dh) break;
    float v = acc[c] * f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) o[(size_t)t * d + h * dh + c] = v / l;
  }
}

}  // namespace

void launch_attention_f32(const float* qkv, float* o, int d, int heads, int T, const PackBuffers& pb,
                          cudaStream_t st) {
  if (T <= 0) return;
  const int warps = 4;
  const long long n = (long long)T * heads;
  attention_f32_kernel<<<(unsigned)((n + warps - 1) / warps), 32 * warps, 0, st>>>(qkv, o, d, heads, T, pb);
}

}  // namespace esm
