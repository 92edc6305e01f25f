// fp32 GEMM on the CUDA cores (FFMA) for the ESM_FP32 precision, with the same fused
// epilogues as the tensor-core GEMM, and the in-place RoPE pass that follows its QKV
// projection.  TF32 tensor cores keep only a 10-bit mantissa, too coarse for a 1e-4
// relative error budget, so this precision stays on true fp32 arithmetic.
//
// RoPE: rotary position embedding of size hidden // heads (mlqm.cn ESM-2 walkthrough,
// rotary section); pairs (j, j + dh/2) of q and k turn by pos * base^(-2j/dh).
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int TB = 64;   // output tile 64 x 64
constexpr int TK = 16;   // K slice

template <int EPI>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, const float* __restrict__ B, int M,
                                                       int N, int K, EpiArgs ea) {
  __shared__ float sA[TK][TB + 4];
  __shared__ float sB[TK][TB + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * TB, n0 = blockIdx.x * TB;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TB * TK; i += 256) {
      const int r = i / TK, k = i % TK;
      sA[k][r] = (m0 + r < M && k0 + k < K) ? A[(size_t)(m0 + r) * K + k0 + k] : 0.f;
      sB[k][r] = (n0 + r < N && k0 + k < K) ? B[(size_t)(n0 + r) * K + k0 + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < TK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = sA[k][ty * 4 + i]; b[i] = sB[k][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  const float* bias = static_cast<const float*>(ea.bias);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + ty * 4 + i;
    if (r >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c >= N) continue;
      float v = acc[i][j] + (bias ? bias[c] : 0.f);
      float* out = static_cast<float*>(ea.out) + (size_t)r * N + c;
      if (EPI == ESM_EPI_RESIDUAL) *out += v;
      else if (EPI == ESM_EPI_GELU) *out = gelu_erf(v);
      else *out = v;
    }
  }
}

__global__ void rope_f32_kernel(float* qkv, int T, int d, int dh, const int32_t* pos_id, const float2* rope,
                                int max_pos) {
  const int half = dh / 2;
  const long long n = (long long)T * 2 * (d / dh) * half;  // (token, q|k head, pair)
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(i % half);
    const long long th = i / half;
    const int hh = (int)(th % (2 * (d / dh)));  // 0 .. 2H-1 over the q and k blocks
    const int t = (int)(th / (2 * (d / dh)));
    int p = pos_id[t];
    p = p < 0 ? 0 : (p >= max_pos ? max_pos - 1 : p);
    const float2 cs = rope[((size_t)(j >> 1) * max_pos + p) * 2 + (j & 1)];
    float* u = qkv + (size_t)t * 3 * d + hh * dh;
    const float a = u[j], b = u[j + half];
    u[j] = a * cs.x - b * cs.y;
    u[j + half] = b * cs.x + a * cs.y;
  }
}

}  // namespace

void launch_gemm_f32(esm_epilogue epi, const float* A, const float* B, int M, int N, int K, const EpiArgs& ea,
                     cudaStream_t st) {
  if (M <= 0 || N <= 0) return;
  dim3 grid((N + TB - 1) / TB, (M + TB - 1) / TB);
  switch (epi) {
    case ESM_EPI_RESIDUAL: gemm_f32_kernel<ESM_EPI_RESIDUAL><<<grid, 256, 0, st>>>(A, B, M, N, K, ea); break;
    case ESM_EPI_GELU: gemm_f32_kernel<ESM_EPI_GELU><<<grid, 256, 0, st>>>(A, B, M, N, K, ea); break;
    default: gemm_f32_kernel<ESM_EPI_BIAS_F32><<<grid, 256, 0, st>>>(A, B, M, N, K, ea); break;
  }
  if (epi == ESM_EPI_QKV_ROPE)
    launch_rope_f32(static_cast<float*>(ea.out), M, N / 3, ea.head_dim, ea.pos_id, ea.rope, ea.max_pos, st);
}

void launch_rope_f32(float* qkv, int T, int d, int head_dim, const int32_t* pos_id, const float2* rope, int max_pos,
                     cudaStream_t st) {
  const long long n = (long long)T * 2 * (d / head_dim) * (head_dim / 2);
  if (n <= 0) return;
  int grid = (int)((n + 255) / 256);
  if (grid > 8192) grid = 8192;
  rope_f32_kernel<<<grid, 256, 0, st>>>(qkv, T, d, head_dim, pos_id, rope, max_pos);
}

}  // namespace esm
