// Row, column and elementwise kernels of the training step (the backward of the packed
// layer stack that the hotelren.com guide trains over cu_seqlens, §3.2 and §6):
//   * LayerNorm backward (dx by rows, dgamma and dbeta as column sums in the same pass);
//   * column sums (bias gradients) with an optional bfloat16 copy of the rows (the next
//     GEMM's operand);
//   * the embedding table's gradient (scatter-add of the embedded rows' gradient).
// (GELU's derivative runs in the epilogue of the GEMM that produces its input gradient.)
// Every reduction over rows runs in a fixed order: chunks of rows give partial sums, and
// one pass adds the chunks in index order, so results do not depend on scheduling.
#include <algorithm>

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

// LayerNorm backward, one warp per row, the row held in registers (N4 float4 per lane):
// mean and variance (two passes), then with g = dy * gamma and xhat the normalised row
//   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat))
// (dres may alias dx).  The parameter gradients are column sums: each warp adds its rows'
// dy * xhat and dy into its own shared-memory slice, and at the end the block adds the
// slices in warp order into partial[block][0 | 1][cols].
template <int N4, bool XBF16 = false>
__global__ void __launch_bounds__(256, N4 <= 10 ? 2 : 1) ln_bwd_kernel(const void* __restrict__ xv, const void* __restrict__ gamma,
                                                     bool gf32, const float* __restrict__ dy, const float* dres,
                                                     float* dx, float* __restrict__ partial, int rows, int cols,
                                                     int rows_per_block, float eps) {
  extern __shared__ float4 slice4[];  // [warps][2][cols / 4]
  const int warps = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n4 = cols >> 2;
  float4* mine = slice4 + (size_t)warp * 2 * n4;
  for (int c = lane; c < 2 * n4; c += 32) mine[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int r0 = blockIdx.x * rows_per_block, r1 = min(rows, r0 + rows_per_block);
  for (int row = r0 + warp; row < r1; row += warps) {
    const float4* dr = reinterpret_cast<const float4*>(dy + (size_t)row * cols);
    // the residual gradient of this row is read last: start it towards L2 now, and the
    // next row of this warp as well (one 128-byte line per prefetch)
    if ((lane & 7) == 0) {
#pragma unroll
      for (int i = 0; i < N4; ++i) {
        const int c = i * 32 + lane;
        if (c < n4) {
          if (dres) prefetch_l2(dres + (size_t)row * cols + 4 * c);
          if (row + warps < r1) {
            if constexpr (!XBF16) prefetch_l2(static_cast<const float*>(xv) + (size_t)(row + warps) * cols + 4 * c);
            prefetch_l2(dy + (size_t)(row + warps) * cols + 4 * c);
          }
        }
      }
    }
    float4 v[N4], d[N4];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < N4; ++i) {
      const int c = i * 32 + lane;
      if constexpr (XBF16) {  // x is a bf16 activation (the masked-LM head's GELU output)
        v[i] = c < n4 ? ld_param4(static_cast<const __nv_bfloat16*>(xv) + (size_t)row * cols, 4 * c, false)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const float4* xr = reinterpret_cast<const float4*>(static_cast<const float*>(xv) + (size_t)row * cols);
        v[i] = c < n4 ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      d[i] = c < n4 ? dr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
    const float mu = wsum(s) / (float)cols;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < N4; ++i) {
      if (i * 32 + lane < n4) {
        v[i].x -= mu; v[i].y -= mu; v[i].z -= mu; v[i].w -= mu;
        q += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
      }
    }
    const float rstd = rsqrtf(wsum(q) / (float)cols + eps);
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int i = 0; i < N4; ++i) {  // v becomes xhat; gamma is re-read from L1 (5 KB per row)
      v[i].x *= rstd; v[i].y *= rstd; v[i].z *= rstd; v[i].w *= rstd;
      const float4 gm = i * 32 + lane < n4 ? ld_param4(gamma, 4 * (i * 32 + lane), gf32) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float g0 = d[i].x * gm.x, g1 = d[i].y * gm.y, g2 = d[i].z * gm.z, g3 = d[i].w * gm.w;
      sg += (g0 + g1) + (g2 + g3);
      sgx += (g0 * v[i].x + g1 * v[i].y) + (g2 * v[i].z + g3 * v[i].w);
    }
    const float mg = wsum(sg) / (float)cols, mgx = wsum(sgx) / (float)cols;
    float4* out = reinterpret_cast<float4*>(dx + (size_t)row * cols);
    if constexpr (N4 > 20) {
      // widest rows (1 block per SM, registers at the limit): one pass, the residual
      // gradient read element by element before the store that may overwrite it
      const float4* res = dres ? reinterpret_cast<const float4*>(dres + (size_t)row * cols) : nullptr;
#pragma unroll
      for (int i = 0; i < N4; ++i) {
        const int c = i * 32 + lane;
        if (c < n4) {
          const float4 gm = ld_param4(gamma, 4 * c, gf32);
          float4 o = res ? res[c] : make_float4(0.f, 0.f, 0.f, 0.f);
          o.x += rstd * (d[i].x * gm.x - mg - v[i].x * mgx);
          o.y += rstd * (d[i].y * gm.y - mg - v[i].y * mgx);
          o.z += rstd * (d[i].z * gm.z - mg - v[i].z * mgx);
          o.w += rstd * (d[i].w * gm.w - mg - v[i].w * mgx);
          out[c] = o;
          float4 a = mine[c], b = mine[n4 + c];
          a.x = fmaf(d[i].x, v[i].x, a.x); a.y = fmaf(d[i].y, v[i].y, a.y);
          a.z = fmaf(d[i].z, v[i].z, a.z); a.w = fmaf(d[i].w, v[i].w, a.w);
          b.x += d[i].x; b.y += d[i].y; b.z += d[i].z; b.w += d[i].w;
          mine[c] = a;
          mine[n4 + c] = b;
        }
      }
    } else {
      // dgamma/dbeta slices first; then d becomes this row's dx increment and v is free
#pragma unroll
      for (int i = 0; i < N4; ++i) {
        const int c = i * 32 + lane;
        if (c < n4) {
          const float4 gm = ld_param4(gamma, 4 * c, gf32);
          float4 a = mine[c], b = mine[n4 + c];
          a.x = fmaf(d[i].x, v[i].x, a.x); a.y = fmaf(d[i].y, v[i].y, a.y);
          a.z = fmaf(d[i].z, v[i].z, a.z); a.w = fmaf(d[i].w, v[i].w, a.w);
          b.x += d[i].x; b.y += d[i].y; b.z += d[i].z; b.w += d[i].w;
          mine[c] = a;
          mine[n4 + c] = b;
          d[i].x = rstd * (d[i].x * gm.x - mg - v[i].x * mgx);
          d[i].y = rstd * (d[i].y * gm.y - mg - v[i].y * mgx);
          d[i].z = rstd * (d[i].z * gm.z - mg - v[i].z * mgx);
          d[i].w = rstd * (d[i].w * gm.w - mg - v[i].w * mgx);
        }
      }
      if (dres) {
        // the residual gradient may alias dx: every load of the row is issued before its
        // first store, so the loads overlap instead of waiting one by one behind the stores
        const float4* res = reinterpret_cast<const float4*>(dres + (size_t)row * cols);
#pragma unroll
        for (int i = 0; i < N4; ++i) {
          const int c = i * 32 + lane;
          if (c < n4) v[i] = res[c];
        }
#pragma unroll
        for (int i = 0; i < N4; ++i) {
          const int c = i * 32 + lane;
          if (c < n4) out[c] = make_float4(v[i].x + d[i].x, v[i].y + d[i].y, v[i].z + d[i].z, v[i].w + d[i].w);
        }
      } else {
#pragma unroll
        for (int i = 0; i < N4; ++i) {
          const int c = i * 32 + lane;
          if (c < n4) out[c] = d[i];
        }
      }
    }
  }
  __syncthreads();
  float* sl = reinterpret_cast<float*>(slice4);
  for (int c = threadIdx.x; c < 2 * cols; c += blockDim.x) {
    float a = 0.f;
    for (int w = 0; w < warps; ++w) a += sl[(size_t)w * 2 * cols + c];
    partial[(size_t)blockIdx.x * 2 * cols + c] = a;
  }
}

// partial[chunk][c] = sum over the chunk's rows of src[r][c], four columns per thread; with
// copy (fp32 input) the rows are also written as bfloat16.
template <bool BF16IN>
__global__ void __launch_bounds__(128) colsum_kernel(const void* __restrict__ src, int rows, int cols, int chunk_rows,
                                                     float* __restrict__ partial, __nv_bfloat16* __restrict__ copy) {
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;  // columns 4 c4 .. 4 c4 + 3
  const int chunk = blockIdx.y;
  if (4 * c4 >= cols) return;
  const int r0 = chunk * chunk_rows, r1 = min(rows, r0 + chunk_rows);
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int r = r0; r < r1; ++r) {
    const size_t i = (size_t)r * cols + 4 * c4;
    float4 v;
    if (BF16IN) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(src) + i));
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      v = make_float4(lo.x, lo.y, hi.x, hi.y);
    } else {
      v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(src) + i));
      if (copy) *reinterpret_cast<uint2*>(copy + i) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
    a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
  }
  *reinterpret_cast<float4*>(partial + (size_t)chunk * cols + 4 * c4) = a;
}

// out[i] = scale * sum_k partial[k * stride + i] in a fixed order: a block owns 32
// consecutive i; warp w of kReduceWarps adds the chunks k = w, w + kReduceWarps, ... (lane =
// i, coalesced), then the warp sums are added in warp order.  The sums have few columns
// (a block per 32) and hundreds of chunks, so the block is wide: more loads in flight.
constexpr int kReduceWarps = 32;
__global__ void __launch_bounds__(32 * kReduceWarps) reduce_chunks_kernel(const float* __restrict__ partial, int chunks,
                                                                          size_t stride, int n, float scale,
                                                                          float* __restrict__ out) {
  __shared__ float part[kReduceWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 32 + lane;
  float a = 0.f;
  if (i < n) {
#pragma unroll 4
    for (int k = warp; k < chunks; k += kReduceWarps) a += __ldg(partial + (size_t)k * stride + i);
  }
  part[warp][lane] = a;
  __syncthreads();
  if (warp == 0 && i < n) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kReduceWarps; ++w) t += part[w][lane];
    out[i] = t * scale;
  }
}

// Few chunks over many elements (split-K partial products): one thread per element.
__global__ void reduce_few_chunks_kernel(const float* __restrict__ partial, int chunks, size_t stride, size_t n,
                                         float scale, float* __restrict__ out) {
  const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < chunks; ++k) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(partial + (size_t)k * stride + i));
    a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
  }
  *reinterpret_cast<float4*>(out + i) = make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale);
}


// dz = du * GELU'(a), GELU'(a) = Phi(a) + a phi(a); du fp32, a bf16 (the pre-activation),
// dz bf16.
// (four elements per thread: one 16-byte load of du, 8-byte load of a and store of dz; n % 4
// == 0, buffers 16-byte aligned)
__device__ __forceinline__ float gelu_grad(float x) {
  return 0.5f * (1.f + erff(x * 0.70710678118654752f)) + x * 0.3989422804014327f * expf(-0.5f * x * x);
}
__global__ void gelu_bwd_kernel(const float* __restrict__ du, const __nv_bfloat16* __restrict__ a,
                                __nv_bfloat16* __restrict__ dz, size_t n4) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 u = __ldg(reinterpret_cast<const float4*>(du) + i);
  const uint2 av = __ldg(reinterpret_cast<const uint2*>(a) + i);
  const float2 a01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av.x));
  const float2 a23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av.y));
  reinterpret_cast<uint2*>(dz)[i] = make_uint2(pack_bf16x2(u.x * gelu_grad(a01.x), u.y * gelu_grad(a01.y)),
                                               pack_bf16x2(u.z * gelu_grad(a23.x), u.w * gelu_grad(a23.y)));
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

constexpr int kChunkRows = 32;

int chunks_for(int rows) { return rows <= 0 ? 1 : (rows + kChunkRows - 1) / kChunkRows; }
constexpr int kEmbChunkRows = 256;  // tokens per embedding-gradient chunk
int emb_chunks_for(int rows) { return rows <= 0 ? 1 : (rows + kEmbChunkRows - 1) / kEmbChunkRows; }

}  // namespace

void reduce_chunks(const float* partial, int chunks, size_t stride, size_t n, float scale, float* out, cudaStream_t st) {
  if (n == 0) return;
  if (chunks <= 16 && n % 4 == 0 && stride % 4 == 0)
    reduce_few_chunks_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, st>>>(partial, chunks, stride, n, scale, out);
  else
    reduce_chunks_kernel<<<(unsigned)((n + 31) / 32), 32 * kReduceWarps, 0, st>>>(partial, chunks, stride, (int)n, scale,
                                                                                 out);
}

constexpr int kLnRowsPerBlock = 64;

size_t bwd_partial_floats(int rows, int cols) {
  const int blocks = rows <= 0 ? 1 : (rows + kLnRowsPerBlock - 1) / kLnRowsPerBlock;
  return std::max((size_t)chunks_for(rows), (size_t)blocks) * 2 * cols;
}
size_t emb_bwd_partial_floats(int rows, int vocab, int d) { return (size_t)emb_chunks_for(rows) * vocab * d; }

// LayerNorm backward grid: as many blocks as fit on the device at once (1 or 2 per SM, by
// the dgamma/dbeta slices in shared memory), the rows split evenly between them, so every
// SM streams the same number of rows; at most chunks_for(rows) blocks (the partial buffer's
// size) and at least 8 rows per block (one per warp).
struct LnBwdGrid {
  int blocks, rows_per_block;
};
LnBwdGrid ln_bwd_grid(int rows, int cols) {
  static int num_sms = 0;
  if (num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || num_sms <= 0)
      num_sms = 148;
  }
  const int warps = std::max(1, std::min(8, (int)(196608 / (8 * (size_t)cols))));
  const size_t smem = (size_t)warps * 2 * cols * sizeof(float);
  const int n4 = (cols / 4 + 31) / 32;
  const int per_sm = (n4 <= 10 && 2 * (smem + 1024) <= 227 * 1024) ? 2 : 1;  // the kernel's launch bounds
  int blocks = std::min(per_sm * num_sms, std::min(chunks_for(rows), std::max(1, (rows + 7) / 8)));
  blocks = std::max(blocks, 1);
  const int rpb = std::max(1, (rows + blocks - 1) / blocks);
  return {std::max(1, (rows + rpb - 1) / rpb), rpb};
}

template <int N4, bool XBF16>
cudaError_t ln_bwd_launch(const void* x, const void* gamma, bool gf32, const float* dy, const float* dres, float* dx,
                          float* partial, int rows, int cols, float eps, cudaStream_t st) {
  const int warps = std::max(1, std::min(8, (int)(196608 / (8 * (size_t)cols))));
  const size_t smem = (size_t)warps * 2 * cols * sizeof(float);
  static size_t configured = 0;
  if (smem > 48 * 1024 && smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(ln_bwd_kernel<N4, XBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const LnBwdGrid g = ln_bwd_grid(rows, cols);
  ln_bwd_kernel<N4, XBF16><<<g.blocks, 32 * warps, smem, st>>>(x, gamma, gf32, dy, dres, dx, partial, rows, cols,
                                                              g.rows_per_block, eps);
  return cudaGetLastError();
}

template <bool XBF16>
void ln_bwd_any(const void* x, const void* gamma, bool gf32, const float* dy, const float* dres, float* dx,
                float* dgamma, float* dbeta, float* partial, int rows, int cols, float eps, cudaStream_t st) {
  if (rows <= 0) {
    cudaMemsetAsync(dgamma, 0, sizeof(float) * cols, st);
    cudaMemsetAsync(dbeta, 0, sizeof(float) * cols, st);
    return;
  }
  const int n4 = (cols / 4 + 31) / 32;  // float4 per lane
  if (n4 <= 2) ln_bwd_launch<2, XBF16>(x, gamma, gf32, dy, dres, dx, partial, rows, cols, eps, st);
  else if (n4 <= 4) ln_bwd_launch<4, XBF16>(x, gamma, gf32, dy, dres, dx, partial, rows, cols, eps, st);
  else if (n4 <= 8) ln_bwd_launch<8, XBF16>(x, gamma, gf32, dy, dres, dx, partial, rows, cols, eps, st);
  else if (n4 <= 10) ln_bwd_launch<10, XBF16>(x, gamma, gf32, dy, dres, dx, partial, rows, cols, eps, st);
  else if (n4 <= 16) ln_bwd_launch<16, XBF16>(x, gamma, gf32, dy, dres, dx, partial, rows, cols, eps, st);
  else if (n4 <= 20) ln_bwd_launch<20, XBF16>(x, gamma, gf32, dy, dres, dx, partial, rows, cols, eps, st);
  else ln_bwd_launch<32, XBF16>(x, gamma, gf32, dy, dres, dx, partial, rows, cols, eps, st);
  const int blocks = ln_bwd_grid(rows, cols).blocks;
  reduce_chunks(partial, blocks, (size_t)2 * cols, cols, 1.f, dgamma, st);
  reduce_chunks(partial + cols, blocks, (size_t)2 * cols, cols, 1.f, dbeta, st);
}

void launch_ln_bwd(const float* x, const void* gamma, bool gf32, const float* dy, const float* dres, float* dx,
                   float* dgamma, float* dbeta, float* partial, int rows, int cols, float eps, cudaStream_t st) {
  ln_bwd_any<false>(x, gamma, gf32, dy, dres, dx, dgamma, dbeta, partial, rows, cols, eps, st);
}

void launch_ln_bwd_bf16in(const void* x, const void* gamma, bool gf32, const float* dy, float* dx, float* dgamma,
                          float* dbeta, float* partial, int rows, int cols, float eps, cudaStream_t st) {
  ln_bwd_any<true>(x, gamma, gf32, dy, nullptr, dx, dgamma, dbeta, partial, rows, cols, eps, st);
}

void launch_colsum(const void* src, bool bf16_in, int rows, int cols, float* out, float* partial, __nv_bfloat16* copy,
                   cudaStream_t st) {
  if (rows <= 0) {
    cudaMemsetAsync(out, 0, sizeof(float) * cols, st);
    return;
  }
  const int chunks = chunks_for(rows);
  const dim3 grid((cols / 4 + 127) / 128, chunks);
  if (bf16_in) colsum_kernel<true><<<grid, 128, 0, st>>>(src, rows, cols, kChunkRows, partial, nullptr);
  else colsum_kernel<false><<<grid, 128, 0, st>>>(src, rows, cols, kChunkRows, partial, copy);
  reduce_chunks(partial, chunks, (size_t)cols, cols, 1.f, out, st);
}

void launch_reduce_splits(const float* partial, int splits, size_t n, float* out, cudaStream_t st) {
  reduce_chunks(partial, splits, n, (int)n, 1.f, out, st);
}

void launch_gelu_bwd(const float* du, const __nv_bfloat16* a, __nv_bfloat16* dz, size_t n, cudaStream_t st) {
  if (n) gelu_bwd_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, st>>>(du, a, dz, n / 4);
}

void launch_emb_bwd(const float* dx, const int32_t* tok, int T, int d, int vocab, float scale, float* partial,
                    float* demb, cudaStream_t st) {
  if (T <= 0) {
    cudaMemsetAsync(demb, 0, sizeof(float) * (size_t)vocab * d, st);
    return;
  }
  const int chunks = emb_chunks_for(T);
  emb_bwd_kernel<<<dim3((d + 127) / 128, chunks), 128, sizeof(float) * 128 * vocab, st>>>(dx, tok, T, d, vocab,
                                                                                          kEmbChunkRows, partial);
  reduce_chunks(partial, chunks, (size_t)vocab * d, vocab * d, scale, demb, st);
}

}  // namespace esm
