// LayerNorm over the hidden dimension, one warp per row (hotelren.com guide section 3.1,
// the layer's LayerNorm; aikraft.ru te.LayerNorm / LayerNormLinear / LayerNormMLP).
//
//   y = (x - mean) / sqrt(var + eps) * gamma + beta,   var biased (divided by cols)
//
// The row stays in registers (16-byte loads, cols/128 float4 per lane); mean and variance
// are two exact passes over the registers, reduced with warp shuffles in fp32.  The output
// is the next GEMM's operand: fp32, bf16, or E4M3 scaled by the delayed-scaling factor; for
// E4M3 and bf16 outputs the rows' max |y| is folded into a tensor amax when one is given.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float4 load_param4(const void* p, int c, bool f32) {
  if (f32) return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + c));
  uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p) + c));
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.x));
  float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ bool row_valid(int row, const int32_t* vp, const int32_t* vs, const int32_t* vk) {
  if (vp == nullptr) return true;
  return vp[row] < vk[vs[row]];
}

// x is float32 (the residual stream) or bfloat16 (IN_BF16: an activation, e.g. the masked-LM
// head's dense output).
template <int N4, Act OUT, bool IN_BF16>
__global__ void layernorm_kernel(const void* __restrict__ x, const void* __restrict__ g, const void* __restrict__ b,
                                 bool param_f32, void* __restrict__ y, int rows, int cols, float eps,
                                 const float* q_scale, float* amax_out, const int32_t* vp, const int32_t* vs,
                                 const int32_t* vk) {
  const int warps = blockDim.x >> 5;
  const int row = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int n4 = cols >> 2;
  float4 v[N4];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < N4; ++i) {
    const int c = i * 32 + lane;
    if constexpr (IN_BF16) {
      v[i] = c < n4 ? load_param4(static_cast<const __nv_bfloat16*>(x) + (size_t)row * cols, 4 * c, false)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      const float4* xr = reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)row * cols);
      v[i] = c < n4 ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  }
  const float mean = warp_sum(s) / (float)cols;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < N4; ++i) {
    const int c = i * 32 + lane;
    if (c < n4) {
      const float a = v[i].x - mean, bb = v[i].y - mean, cc = v[i].z - mean, dd = v[i].w - mean;
      ss += (a * a + bb * bb) + (cc * cc + dd * dd);
    }
  }
  const float rstd = rsqrtf(warp_sum(ss) / (float)cols + eps);
  const bool valid = row_valid(row, vp, vs, vk);
  float amax = 0.f;
  const float qs = (OUT == Act::E4M3) ? __ldg(q_scale) : 1.f;
#pragma unroll
  for (int i = 0; i < N4; ++i) {
    const int c = i * 32 + lane;
    if (c >= n4) continue;
    const float4 gg = load_param4(g, 4 * c, param_f32);
    const float4 bb = load_param4(b, 4 * c, param_f32);
    float4 o;
    o.x = (v[i].x - mean) * rstd * gg.x + bb.x;
    o.y = (v[i].y - mean) * rstd * gg.y + bb.y;
    o.z = (v[i].z - mean) * rstd * gg.z + bb.z;
    o.w = (v[i].w - mean) * rstd * gg.w + bb.w;
    if (!valid) o = make_float4(0.f, 0.f, 0.f, 0.f);
    const size_t off = (size_t)row * cols + 4 * c;
    if constexpr (OUT == Act::F32) {
      reinterpret_cast<float4*>(static_cast<float*>(y) + off)[0] = o;
    } else if constexpr (OUT == Act::BF16) {
      uint2 w;
      w.x = pack_bf16x2(o.x, o.y);
      w.y = pack_bf16x2(o.z, o.w);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + off)[0] = w;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(o.x), fabsf(o.y)), fmaxf(fabsf(o.z), fabsf(o.w))));
    } else {
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(o.x), fabsf(o.y)), fmaxf(fabsf(o.z), fabsf(o.w))));
      __nv_fp8x4_e4m3 q(make_float4(o.x * qs, o.y * qs, o.z * qs, o.w * qs));
      reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(y) + off)[0] = *reinterpret_cast<uint32_t*>(&q);
    }
  }
  if constexpr (OUT == Act::E4M3 || OUT == Act::BF16) {
    if (amax_out) {
      // a bf16 output's amax is that of the rounded values: rounding is monotone, so round the max
      if constexpr (OUT == Act::BF16) amax = __bfloat162float(__float2bfloat16_rn(amax));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) atomic_max_nonneg(amax_out, amax);
    }
  }
}

template <Act OUT>
__global__ void copy_out_kernel(const float* __restrict__ x, void* __restrict__ out, int rows, int cols,
                                const int32_t* vp, const int32_t* vs, const int32_t* vk) {
  const size_t n4 = (size_t)rows * cols / 4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const int row = (int)(i * 4 / cols);
    float4 v = reinterpret_cast<const float4*>(x)[i];
    if (!row_valid(row, vp, vs, vk)) v = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (OUT == Act::F32) {
      reinterpret_cast<float4*>(out)[i] = v;
    } else {
      uint2 w;
      w.x = pack_bf16x2(v.x, v.y);
      w.y = pack_bf16x2(v.z, v.w);
      reinterpret_cast<uint2*>(out)[i] = w;
    }
  }
}

template <int N4, bool IN_BF16>
void ln_dispatch_out(const void* x, const void* g, const void* b, bool pf32, void* y, Act out, int rows, int cols,
                     float eps, const float* qs, float* amax, const int32_t* vp, const int32_t* vs, const int32_t* vk,
                     cudaStream_t st) {
  const int warps = 8;
  const int grid = (rows + warps - 1) / warps;
  if (out == Act::F32)
    layernorm_kernel<N4, Act::F32, IN_BF16>
        <<<grid, 32 * warps, 0, st>>>(x, g, b, pf32, y, rows, cols, eps, qs, amax, vp, vs, vk);
  else if (out == Act::BF16)
    layernorm_kernel<N4, Act::BF16, IN_BF16>
        <<<grid, 32 * warps, 0, st>>>(x, g, b, pf32, y, rows, cols, eps, qs, amax, vp, vs, vk);
  else
    layernorm_kernel<N4, Act::E4M3, IN_BF16>
        <<<grid, 32 * warps, 0, st>>>(x, g, b, pf32, y, rows, cols, eps, qs, amax, vp, vs, vk);
}

template <bool IN_BF16>
void ln_dispatch(const void* x, const void* g, const void* b, bool pf32, void* y, Act out, int rows, int cols,
                 float eps, const float* qs, float* amax, const int32_t* vp, const int32_t* vs, const int32_t* vk,
                 cudaStream_t st) {
  const int n4 = (cols / 4 + 31) / 32;  // float4 per lane
  if (n4 <= 1) ln_dispatch_out<1, IN_BF16>(x, g, b, pf32, y, out, rows, cols, eps, qs, amax, vp, vs, vk, st);
  else if (n4 <= 2) ln_dispatch_out<2, IN_BF16>(x, g, b, pf32, y, out, rows, cols, eps, qs, amax, vp, vs, vk, st);
  else if (n4 <= 4) ln_dispatch_out<4, IN_BF16>(x, g, b, pf32, y, out, rows, cols, eps, qs, amax, vp, vs, vk, st);
  else if (n4 <= 8) ln_dispatch_out<8, IN_BF16>(x, g, b, pf32, y, out, rows, cols, eps, qs, amax, vp, vs, vk, st);
  else if (n4 <= 10) ln_dispatch_out<10, IN_BF16>(x, g, b, pf32, y, out, rows, cols, eps, qs, amax, vp, vs, vk, st);
  else if (n4 <= 20) ln_dispatch_out<20, IN_BF16>(x, g, b, pf32, y, out, rows, cols, eps, qs, amax, vp, vs, vk, st);
  else ln_dispatch_out<32, IN_BF16>(x, g, b, pf32, y, out, rows, cols, eps, qs, amax, vp, vs, vk, st);
}

struct LnFoldJobs {
  LnFoldJob j[kLnFoldMaxJobs];
};

// One warp per output row i of job blockIdx.y: the dot products of W's row with gamma and
// with beta (fp32 accumulation of the bf16 products), 8 columns per lane per step.
__global__ void __launch_bounds__(256) ln_fold_kernel(const __grid_constant__ LnFoldJobs jobs, int k) {
  const LnFoldJob& jb = jobs.j[blockIdx.y];
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= jb.n) return;
  const uint4* wr = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(jb.w) + (size_t)i * k);
  const uint4* gr = reinterpret_cast<const uint4*>(jb.gamma);
  const uint4* br = reinterpret_cast<const uint4*>(jb.beta);
  float sc = 0.f, sb = 0.f;
  for (int u = lane; u < k / 8; u += 32) {
    const uint4 wv = __ldg(wr + u), gv = __ldg(gr + u), bv = __ldg(br + u);
    const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 w = __bfloat1622float2(w2[t]), g = __bfloat1622float2(g2[t]), b = __bfloat1622float2(b2[t]);
      sc = fmaf(w.x, g.x, fmaf(w.y, g.y, sc));
      sb = fmaf(w.x, b.x, fmaf(w.y, b.y, sb));
    }
  }
  sc = warp_sum(sc);
  sb = warp_sum(sb);
  if (lane == 0) {
    jb.c_out[i] = sc;
    jb.b_out[i] = sb + (jb.bias ? __bfloat162float(static_cast<const __nv_bfloat16*>(jb.bias)[i]) : 0.f);
  }
}

}  // namespace

void launch_ln_fold(const LnFoldJob* jobs, int num_jobs, int k, cudaStream_t st) {
  if (num_jobs <= 0) return;
  LnFoldJobs p{};
  int max_n = 0;
  for (int i = 0; i < num_jobs && i < kLnFoldMaxJobs; ++i) {
    p.j[i] = jobs[i];
    max_n = jobs[i].n > max_n ? jobs[i].n : max_n;
  }
  ln_fold_kernel<<<dim3((max_n + 7) / 8, num_jobs < kLnFoldMaxJobs ? num_jobs : kLnFoldMaxJobs), 256, 0, st>>>(p, k);
}

void launch_layernorm(const float* x, const void* g, const void* b, bool param_f32, void* y, Act out, int rows,
                      int cols, float eps, const float* q_scale, float* amax, const int32_t* vp, const int32_t* vs,
                      const int32_t* vk, cudaStream_t st) {
  if (rows <= 0) return;
  ln_dispatch<false>(x, g, b, param_f32, y, out, rows, cols, eps, q_scale, amax, vp, vs, vk, st);
}

void launch_layernorm_bf16in(const void* x, const void* g, const void* b, bool param_f32, void* y, Act out, int rows,
                             int cols, float eps, cudaStream_t st) {
  if (rows <= 0) return;
  ln_dispatch<true>(x, g, b, param_f32, y, out, rows, cols, eps, nullptr, nullptr, nullptr, nullptr, nullptr, st);
}

void launch_copy_out(const float* x, void* out, Act out_t, int rows, int cols, const int32_t* vp, const int32_t* vs,
                     const int32_t* vk, cudaStream_t st) {
  if (rows <= 0) return;
  const size_t n4 = (size_t)rows * cols / 4;
  int grid = (int)((n4 + 255) / 256);
  if (grid > 4096) grid = 4096;
  if (out_t == Act::F32)
    copy_out_kernel<Act::F32><<<grid, 256, 0, st>>>(x, out, rows, cols, vp, vs, vk);
  else
    copy_out_kernel<Act::BF16><<<grid, 256, 0, st>>>(x, out, rows, cols, vp, vs, vk);
}

}  // namespace esm
