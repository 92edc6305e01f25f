// Row, column and elementwise kernels of the training step (the backward of the packed
// layer stack that the hotelren.com guide trains over cu_seqlens, §3.2 and §6):
//   * LayerNorm backward, by rows (dx) and by columns (dgamma, dbeta);
//   * column sums (bias gradients) with an optional bfloat16 copy of the rows (the next
//     GEMM's operand);
//   * the exact GELU and its derivative (the training forward keeps the pre-activation);
//   * the embedding table's gradient (scatter-add of the embedded rows' gradient).
// Every reduction over rows runs in a fixed order: chunks of rows give partial sums, and
// one pass adds the chunks in index order, so results do not depend on scheduling.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float4 ld_param4(const void* p, int c, bool f32) {
  if (f32) return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + c));
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p) + c));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// One warp per row: mean, variance (two passes), then with g = dy * gamma and xhat the
// normalised row
//   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat))
// (dres may alias dx).  stats[row] = (mean, rstd) for the column pass.
__global__ void ln_bwd_rows_kernel(const float* __restrict__ x, const void* __restrict__ gamma, bool gf32,
                                   const float* __restrict__ dy, const float* dres, float* dx, float2* stats, int rows,
                                   int cols, float eps) {
  const int warps = blockDim.x >> 5;
  const int row = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int n4 = cols >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * cols);
  const float4* dr = reinterpret_cast<const float4*>(dy + (size_t)row * cols);
  float s = 0.f;
  for (int c = lane; c < n4; c += 32) {
    const float4 v = xr[c];
    s += (v.x + v.y) + (v.z + v.w);
  }
  const float mu = wsum(s) / (float)cols;
  float q = 0.f;
  for (int c = lane; c < n4; c += 32) {
    const float4 v = xr[c];
    const float a = v.x - mu, b = v.y - mu, e = v.z - mu, f = v.w - mu;
    q += (a * a + b * b) + (e * e + f * f);
  }
  const float rstd = rsqrtf(wsum(q) / (float)cols + eps);
  float sg = 0.f, sgx = 0.f;
  for (int c = lane; c < n4; c += 32) {
    const float4 v = xr[c], d = dr[c], g = ld_param4(gamma, 4 * c, gf32);
    const float g0 = d.x * g.x, g1 = d.y * g.y, g2 = d.z * g.z, g3 = d.w * g.w;
    sg += (g0 + g1) + (g2 + g3);
    sgx += (g0 * (v.x - mu) + g1 * (v.y - mu)) + (g2 * (v.z - mu) + g3 * (v.w - mu));
  }
  const float mg = wsum(sg) / (float)cols;
  const float mgx = wsum(sgx) * rstd / (float)cols;
  float4* out = reinterpret_cast<float4*>(dx + (size_t)row * cols);
  const float4* res = dres ? reinterpret_cast<const float4*>(dres + (size_t)row * cols) : nullptr;
  for (int c = lane; c < n4; c += 32) {
    const float4 v = xr[c], d = dr[c], g = ld_param4(gamma, 4 * c, gf32);
    float4 r = res ? res[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    r.x += rstd * (d.x * g.x - mg - (v.x - mu) * rstd * mgx);
    r.y += rstd * (d.y * g.y - mg - (v.y - mu) * rstd * mgx);
    r.z += rstd * (d.z * g.z - mg - (v.z - mu) * rstd * mgx);
    r.w += rstd * (d.w * g.w - mg - (v.w - mu) * rstd * mgx);
    out[c] = r;
  }
  if (lane == 0) stats[row] = make_float2(mu, rstd);
}

// Column partial sums of the LayerNorm parameter gradients over one chunk of rows:
// partial[chunk][0][c] = sum dy * xhat, partial[chunk][1][c] = sum dy.
__global__ void ln_bwd_cols_kernel(const float* __restrict__ x, const float* __restrict__ dy,
                                   const float2* __restrict__ stats, float* __restrict__ partial, int rows, int cols,
                                   int chunk_rows) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int chunk = blockIdx.y;
  if (c >= cols) return;
  const int r0 = chunk * chunk_rows, r1 = min(rows, r0 + chunk_rows);
  float a = 0.f, b = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float2 st = __ldg(stats + r);
    const float g = dy[(size_t)r * cols + c];
    a = fmaf(g, (x[(size_t)r * cols + c] - st.x) * st.y, a);
    b += g;
  }
  partial[((size_t)chunk * 2) * cols + c] = a;
  partial[((size_t)chunk * 2 + 1) * cols + c] = b;
}

// partial[chunk][c] = sum over the chunk's rows of src[r][c]; with copy (fp32 input) the
// rows are also written as bfloat16.
template <bool BF16IN>
__global__ void colsum_kernel(const void* __restrict__ src, int rows, int cols, int chunk_rows,
                              float* __restrict__ partial, __nv_bfloat16* __restrict__ copy) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int chunk = blockIdx.y;
  if (c >= cols) return;
  const int r0 = chunk * chunk_rows, r1 = min(rows, r0 + chunk_rows);
  float a = 0.f;
  for (int r = r0; r < r1; ++r) {
    const size_t i = (size_t)r * cols + c;
    float v;
    if (BF16IN) {
      v = __bfloat162float(static_cast<const __nv_bfloat16*>(src)[i]);
    } else {
      v = static_cast<const float*>(src)[i];
      if (copy) copy[i] = __float2bfloat16_rn(v);
    }
    a += v;
  }
  partial[(size_t)chunk * cols + c] = a;
}

// out[i] = scale * sum_k partial[k * stride + i], k in index order.
__global__ void reduce_chunks_kernel(const float* __restrict__ partial, int chunks, size_t stride, int n, float scale,
                                     float* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float a = 0.f;
  for (int k = 0; k < chunks; ++k) a += partial[(size_t)k * stride + i];
  out[i] = a * scale;
}

// u = GELU(z) = z Phi(z), exact (erf), bf16 -> bf16.
__global__ void gelu_fwd_kernel(const __nv_bfloat16* __restrict__ z, __nv_bfloat16* __restrict__ u, size_t n) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = __bfloat162float(z[i]);
  u[i] = __float2bfloat16_rn(0.5f * a * (1.f + erff(a * 0.70710678118654752f)));
}

// dz = du * GELU'(z), GELU'(z) = Phi(z) + z phi(z); du fp32, z bf16, dz bf16.
__global__ void gelu_bwd_kernel(const float* __restrict__ du, const __nv_bfloat16* __restrict__ z,
                                __nv_bfloat16* __restrict__ dz, size_t n) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = __bfloat162float(z[i]);
  const float d = 0.5f * (1.f + erff(a * 0.70710678118654752f)) + a * 0.3989422804014327f * expf(-0.5f * a * a);
  dz[i] = __float2bfloat16_rn(du[i] * d);
}

// partial[chunk][v][c] = sum of dx[t][c] over the chunk's tokens t with tok[t] == v (each
// thread owns one column, so the sums run in token order).
__global__ void emb_bwd_kernel(const float* __restrict__ dx, const int32_t* __restrict__ tok, int T, int d, int vocab,
                               int chunk_rows, float* __restrict__ partial) {
  extern __shared__ float acc[];  // [vocab][blockDim.x]
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int chunk = blockIdx.y;
  for (int v = 0; v < vocab; ++v) acc[v * blockDim.x + threadIdx.x] = 0.f;
  if (c < d) {
    const int t0 = chunk * chunk_rows, t1 = min(T, t0 + chunk_rows);
    for (int t = t0; t < t1; ++t) {
      int v = __ldg(tok + t);
      if (v < 0 || v >= vocab) continue;
      acc[v * blockDim.x + threadIdx.x] += dx[(size_t)t * d + c];
    }
    for (int v = 0; v < vocab; ++v) partial[((size_t)chunk * vocab + v) * d + c] = acc[v * blockDim.x + threadIdx.x];
  }
}

constexpr int kChunkRows = 128;

int chunks_for(int rows) { return rows <= 0 ? 1 : (rows + kChunkRows - 1) / kChunkRows; }

}  // namespace

size_t bwd_partial_floats(int rows, int cols) { return (size_t)chunks_for(rows) * 2 * cols; }
size_t emb_bwd_partial_floats(int rows, int vocab, int d) { return (size_t)chunks_for(rows) * vocab * d; }

void launch_ln_bwd(const float* x, const void* gamma, bool gf32, const float* dy, const float* dres, float* dx,
                   float2* stats, float* dgamma, float* dbeta, float* partial, int rows, int cols, float eps,
                   cudaStream_t st) {
  if (rows <= 0) {
    cudaMemsetAsync(dgamma, 0, sizeof(float) * cols, st);
    cudaMemsetAsync(dbeta, 0, sizeof(float) * cols, st);
    return;
  }
  ln_bwd_rows_kernel<<<(rows + 7) / 8, 256, 0, st>>>(x, gamma, gf32, dy, dres, dx, stats, rows, cols, eps);
  const int chunks = chunks_for(rows);
  ln_bwd_cols_kernel<<<dim3((cols + 255) / 256, chunks), 256, 0, st>>>(x, dy, stats, partial, rows, cols, kChunkRows);
  reduce_chunks_kernel<<<(cols + 255) / 256, 256, 0, st>>>(partial, chunks, (size_t)2 * cols, cols, 1.f, dgamma);
  reduce_chunks_kernel<<<(cols + 255) / 256, 256, 0, st>>>(partial + cols, chunks, (size_t)2 * cols, cols, 1.f, dbeta);
}

void launch_colsum(const void* src, bool bf16_in, int rows, int cols, float* out, float* partial, __nv_bfloat16* copy,
                   cudaStream_t st) {
  if (rows <= 0) {
    cudaMemsetAsync(out, 0, sizeof(float) * cols, st);
    return;
  }
  const int chunks = chunks_for(rows);
  const dim3 grid((cols + 255) / 256, chunks);
  if (bf16_in) colsum_kernel<true><<<grid, 256, 0, st>>>(src, rows, cols, kChunkRows, partial, nullptr);
  else colsum_kernel<false><<<grid, 256, 0, st>>>(src, rows, cols, kChunkRows, partial, copy);
  reduce_chunks_kernel<<<(cols + 255) / 256, 256, 0, st>>>(partial, chunks, (size_t)cols, cols, 1.f, out);
}

void launch_reduce_splits(const float* partial, int splits, size_t n, float* out, cudaStream_t st) {
  reduce_chunks_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(partial, splits, n, (int)n, 1.f, out);
}

void launch_gelu_fwd(const __nv_bfloat16* z, __nv_bfloat16* u, size_t n, cudaStream_t st) {
  if (n) gelu_fwd_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(z, u, n);
}

void launch_gelu_bwd(const float* du, const __nv_bfloat16* z, __nv_bfloat16* dz, size_t n, cudaStream_t st) {
  if (n) gelu_bwd_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(du, z, dz, n);
}

void launch_emb_bwd(const float* dx, const int32_t* tok, int T, int d, int vocab, float scale, float* partial,
                    float* demb, cudaStream_t st) {
  if (T <= 0) {
    cudaMemsetAsync(demb, 0, sizeof(float) * (size_t)vocab * d, st);
    return;
  }
  const int chunks = chunks_for(T);
  emb_bwd_kernel<<<dim3((d + 127) / 128, chunks), 128, sizeof(float) * 128 * vocab, st>>>(dx, tok, T, d, vocab,
                                                                                          kChunkRows, partial);
  reduce_chunks_kernel<<<(vocab * d + 255) / 256, 256, 0, st>>>(partial, chunks, (size_t)vocab * d, vocab * d, scale,
                                                                demb);
}

}  // namespace esm
