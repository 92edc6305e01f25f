// FP8 E4M3 delayed scaling (aikraft.ru TransformerEngine summary, "Рецепт FP8: Delayed
// Scaling": E4M3 in the forward pass, a 16-entry amax history, the max algorithm; section
// 4.1 of the hotelren.com guide uses the same DelayedScaling recipe).
//
// Every quantised GEMM operand t has a scale s_t.  A forward quantises with the current
// s_t (q = E4M3(t * s_t), round to nearest even, saturating at +-448), records this
// call's max |t| and, once the call is done, pushes it into the history and sets
// s_t = 448 / max(history) for the next call.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

__global__ void quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ w, uint8_t* __restrict__ q, size_t n,
                                     const float* scale, float* amax_out) {
  const float s = __ldg(scale);
  float amax = 0.f;
  const size_t n8 = n / 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(w) + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 t = __bfloat1622float2(h[j]);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    __nv_fp8x4_e4m3 a(make_float4(f[0] * s, f[1] * s, f[2] * s, f[3] * s));
    __nv_fp8x4_e4m3 b(make_float4(f[4] * s, f[5] * s, f[6] * s, f[7] * s));
    reinterpret_cast<uint2*>(q)[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) atomic_max_nonneg(amax_out, amax);
}

__global__ void fp8_update_kernel(float* scale, float* hist, float* amax, int n, int len) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float* h = hist + (size_t)i * len;
  for (int j = len - 1; j > 0; --j) h[j] = h[j - 1];
  h[0] = amax[i];
  float m = 0.f;
  bool finite = true;
  for (int j = 0; j < len; ++j) {
    finite = finite && isfinite(h[j]);
    m = fmaxf(m, h[j]);
  }
  if (finite && m > 0.f) scale[i] = 448.0f / m;
  amax[i] = 0.f;
}

}  // namespace

void launch_quantize_e4m3(const __nv_bfloat16* w, uint8_t* q, size_t n, const float* scale, float* amax,
                          cudaStream_t st) {
  if (n == 0) return;
  const size_t n8 = n / 8;
  int grid = (int)((n8 + 255) / 256);
  if (grid > 4 * 152) grid = 4 * 152;
  quantize_e4m3_kernel<<<grid, 256, 0, st>>>(w, q, n, scale, amax);
}

void launch_fp8_update(float* scale, float* hist, float* amax, int n, int len, cudaStream_t st) {
  if (n <= 0) return;
  fp8_update_kernel<<<(n + 127) / 128, 128, 0, st>>>(scale, hist, amax, n, len);
}

}  // namespace esm
