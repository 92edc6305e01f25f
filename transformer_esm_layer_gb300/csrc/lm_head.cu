// Masked-LM head output stage: logits against the tied token embedding and the masked
// cross-entropy (the head the mlqm.cn walkthrough loads as AutoModelForMaskedLM; the BioNeMo
// ESM-2 model card scores it by perplexity).  The dense + GELU and the LayerNorm before it
// run on the encoder's own GEMM and LayerNorm kernels.
//
//   logits[t, v] = z[t] . emb[v] + bias[v]
//   loss[t]      = log(sum_v exp(logits[t, v])) - logits[t, target[t]]   (0 if target = -100)
//
// bf16 (hidden a multiple of 128): the logits are a [T, hidden] x [hidden, vocab] contraction
// on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), 16 tokens per warp, the
// table in shared memory.  fp32: one warp per token, persistent grid; the whole embedding
// (vocab x hidden) sits in shared memory, lane l holds the 16-byte units l, l + 32, ... of the
// token's row and each logit is a warp-wide sum, kept by lane v % 32.  The loss sum is a
// separate one-block reduction in a fixed order, so it is bitwise reproducible.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int kIgnore = -100;

__device__ __forceinline__ float warp_sum_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 16-byte unit of a row: 8 bf16 or 4 fp32 values
template <bool BF16>
__device__ __forceinline__ void unpack(const uint4& u, float* f) {
  if constexpr (BF16) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 p = __bfloat1622float2(h[k]);
      f[2 * k] = p.x;
      f[2 * k + 1] = p.y;
    }
  } else {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
}

// NU: 16-byte units of the row per lane (the row has d * es / 16 units, lane l holds units
// l, l + 32, ...).
template <bool BF16, int NU>
__global__ void __launch_bounds__(256) lm_logits_kernel(const void* __restrict__ z, const void* __restrict__ emb,
                                                        const void* __restrict__ bias, int T, int d, int V,
                                                        const int32_t* __restrict__ targets, float* logits,
                                                        float* token_loss, unsigned* err) {
  extern __shared__ __align__(16) uint8_t smem_e[];
  constexpr int kPer = BF16 ? 8 : 4;  // values per 16-byte unit
  const int units = d / kPer;         // per row
  {  // the embedding table into shared memory, 16 bytes per thread
    const uint4* src = static_cast<const uint4*>(emb);
    uint4* dst = reinterpret_cast<uint4*>(smem_e);
    const int n16 = V * units;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldg(src + i);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  auto bias_at = [&](int v) -> float {
    return BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(bias)[v]) : static_cast<const float*>(bias)[v];
  };
  const float b_lo = lane < V ? bias_at(lane) : 0.f;
  const float b_hi = lane + 32 < V ? bias_at(lane + 32) : 0.f;
  const uint4* e16 = reinterpret_cast<const uint4*>(smem_e);
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps) {
    const uint4* z16 = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(z) + (size_t)t * units * 16);
    uint4 row[NU];
#pragma unroll
    for (int i = 0; i < NU; ++i) {
      const int c = i * 32 + lane;
      row[i] = c < units ? __ldg(z16 + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    float lo = -INFINITY, hi = -INFINITY;  // logits v = lane and v = lane + 32
    for (int v = 0; v < V; ++v) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < NU; ++i) {
        const int c = i * 32 + lane;
        if (c < units) {
          float a[kPer], e[kPer];
          unpack<BF16>(row[i], a);
          unpack<BF16>(e16[v * units + c], e);
#pragma unroll
          for (int k = 0; k < kPer; ++k) acc = fmaf(a[k], e[k], acc);
        }
      }
      acc = warp_sum_all(acc);
      if (v == lane) lo = acc + b_lo;
      if (v == lane + 32) hi = acc + b_hi;
    }
    if (logits) {
      if (lane < V) logits[(size_t)t * V + lane] = lo;
      if (lane + 32 < V) logits[(size_t)t * V + lane + 32] = hi;
    }
    if (token_loss) {
      const float m = warp_max_all(fmaxf(lo, hi));
      const float se = warp_sum_all((lane < V ? expf(lo - m) : 0.f) + (lane + 32 < V ? expf(hi - m) : 0.f));
      int tg = targets ? targets[t] : kIgnore;
      if (tg != kIgnore && (tg < 0 || tg >= V)) {
        if (lane == 0) latch_error(err, ERRBIT_TOKEN);
        tg = kIgnore;
      }
      const int src = tg == kIgnore ? 0 : (tg & 31);
      const float l_src = __shfl_sync(0xffffffffu, tg >= 32 ? hi : lo, src);
      if (lane == 0) token_loss[t] = tg == kIgnore ? 0.f : (m + logf(se)) - l_src;
    }
  }
}

// D += A B for one m16n8k16 tile: A 16 x 16 bf16 (row-major fragment a0..a3), B 16 x 8 bf16
// (column-major fragment b0, b1), D 16 x 8 fp32.  Lane (g, t) = (lane / 4, lane % 4) holds
// A[g][2t, 2t+1], A[g+8][2t, 2t+1], A[g][2t+8, 2t+9], A[g+8][2t+8, 2t+9], B[2t, 2t+1][g],
// B[2t+8, 2t+9][g] and D[g][2t, 2t+1], D[g+8][2t, 2t+1] (lower column in the lower half).
__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16 logits and loss on the tensor cores.  A warp takes 16 tokens (rows r0 = 16 grp + g and
// r1 = r0 + 8 of its group); the vocabulary is padded with zero rows to NB blocks of 8.  In
// each 32-column slice of the hidden dimension lane (g, t) reads columns 8t..8t+7 of rows r0,
// r1 and of table rows 8 nb + g as one 16-byte unit each, and the slice's two k-steps give
// columns 8t + {0,1 | 2,3} and 8t + {4,5 | 6,7} the k positions {2t, 2t+1 | 2t+8, 2t+9} that
// the instruction assigns to lane t, in A and in B alike, so every column of the slice is
// summed exactly once.  Table rows lie row_bytes apart with row_bytes = 64 (mod 512), so the
// eight rows one instruction reads fall in distinct banks.  A logit of row r0 (r1) sits in
// D[g][.] (D[g+8][.]) of its block: the row's max, sum of exponentials and target logit
// reduce over the four lanes of a quad.  Rows past T load row T - 1 and are never written.
template <int NB>
__global__ void __launch_bounds__(128) lm_logits_mma_kernel(const __nv_bfloat16* __restrict__ z,
                                                            const __nv_bfloat16* __restrict__ emb,
                                                            const __nv_bfloat16* __restrict__ bias, int T, int d, int V,
                                                            int row_bytes, const int32_t* __restrict__ targets,
                                                            float* logits, float* token_loss, unsigned* err) {
  extern __shared__ __align__(16) uint8_t smem_e[];
  const int units = d / 8;  // 16-byte units per row
  for (int i = threadIdx.x; i < 8 * NB * units; i += blockDim.x) {
    const int r = i / units, u = i - r * units;
    const uint4 val = r < V ? __ldg(reinterpret_cast<const uint4*>(emb) + (size_t)r * units + u) : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(smem_e + (size_t)r * row_bytes + 16 * u) = val;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int warps = blockDim.x >> 5;
  float bv[NB][2];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int v = 8 * nb + 2 * t + j;
      bv[nb][j] = v < V ? __bfloat162float(bias[v]) : 0.f;
    }
  const uint8_t* eb = smem_e + (size_t)g * row_bytes + 16 * t;
  const int groups = (T + 15) / 16;
  for (int grp = blockIdx.x * warps + (threadIdx.x >> 5); grp < groups; grp += gridDim.x * warps) {
    const int r0 = 16 * grp + g, r1 = r0 + 8;
    const uint4* z0 = reinterpret_cast<const uint4*>(z + (size_t)min(r0, T - 1) * d) + t;
    const uint4* z1 = reinterpret_cast<const uint4*>(z + (size_t)min(r1, T - 1) * d) + t;
    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
#pragma unroll 1
    for (int kb = 0; kb < d / 32; kb += 4) {  // four slices per step: eight 16-byte loads in flight
      uint4 pa[4], pb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pa[j] = __ldg(z0 + 4 * (kb + j));
        pb[j] = __ldg(z1 + 4 * (kb + j));
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const uint4 q = *reinterpret_cast<const uint4*>(eb + (size_t)(8 * nb) * row_bytes + 64 * (kb + j));
          mma_16816_bf16(acc[nb], pa[j].x, pb[j].x, pa[j].y, pb[j].y, q.x, q.y);
          mma_16816_bf16(acc[nb], pa[j].z, pb[j].z, pa[j].w, pb[j].w, q.z, q.w);
        }
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        acc[nb][j] += bv[nb][j];
        acc[nb][2 + j] += bv[nb][j];
        if (8 * nb + 2 * t + j < V) {
          m0 = fmaxf(m0, acc[nb][j]);
          m1 = fmaxf(m1, acc[nb][2 + j]);
        }
      }
    if (logits) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int v = 8 * nb + 2 * t + j;
          if (v < V) {
            if (r0 < T) logits[(size_t)r0 * V + v] = acc[nb][j];
            if (r1 < T) logits[(size_t)r1 * V + v] = acc[nb][2 + j];
          }
        }
    }
    if (token_loss) {
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
      int tg0 = (targets && r0 < T) ? targets[r0] : kIgnore;
      int tg1 = (targets && r1 < T) ? targets[r1] : kIgnore;
      if (tg0 != kIgnore && (tg0 < 0 || tg0 >= V)) {
        if (t == 0) latch_error(err, ERRBIT_TOKEN);
        tg0 = kIgnore;
      }
      if (tg1 != kIgnore && (tg1 < 0 || tg1 >= V)) {
        if (t == 0) latch_error(err, ERRBIT_TOKEN);
        tg1 = kIgnore;
      }
      float s0 = 0.f, s1 = 0.f, own0 = 0.f, own1 = 0.f;  // own: the target's logit (one lane of the quad)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int v = 8 * nb + 2 * t + j;
          if (v < V) {
            s0 += expf(acc[nb][j] - m0);
            s1 += expf(acc[nb][2 + j] - m1);
          }
          if (v == tg0) own0 = acc[nb][j];
          if (v == tg1) own1 = acc[nb][2 + j];
        }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        own0 += __shfl_xor_sync(0xffffffffu, own0, o);
        own1 += __shfl_xor_sync(0xffffffffu, own1, o);
      }
      if (t == 0) {
        if (r0 < T) token_loss[r0] = tg0 == kIgnore ? 0.f : (m0 + logf(s0)) - own0;
        if (r1 < T) token_loss[r1] = tg1 == kIgnore ? 0.f : (m1 + logf(s1)) - own1;
      }
    }
  }
}

// Table row pitch of lm_logits_mma_kernel: 2 d bytes rounded up to 64 (mod 512).
int lm_mma_row_bytes(int d) { return 2 * d + (((64 - 2 * d) % 512) + 512) % 512; }

template <int NB>
void launch_mma_nb(int num_sms, const void* z, const void* emb, const void* bias, int T, int d, int V,
                   const int32_t* targets, float* logits, float* token_loss, unsigned* err, cudaStream_t st) {
  const int rb = lm_mma_row_bytes(d);
  const size_t smem = (size_t)8 * NB * rb;
  cudaFuncSetAttribute(lm_logits_mma_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const int per_sm = smem <= 110 * 1024 ? 2 : 1;
  const int warps = 4, groups = (T + 15) / 16;
  int grid = std::min(num_sms * per_sm, (groups + warps - 1) / warps);
  grid = std::max(grid, 1);
  lm_logits_mma_kernel<NB><<<grid, 32 * warps, smem, st>>>(
      static_cast<const __nv_bfloat16*>(z), static_cast<const __nv_bfloat16*>(emb),
      static_cast<const __nv_bfloat16*>(bias), T, d, V, rb, targets, logits, token_loss, err);
}

// Sum of the per-token losses and count of scored tokens: one block, fixed order.
__global__ void __launch_bounds__(1024) loss_reduce_kernel(const float* __restrict__ token_loss,
                                                           const int32_t* __restrict__ targets, int T, float* loss_sum,
                                                           int* count) {
  __shared__ float ss[1024];
  __shared__ int sc[1024];
  float s = 0.f;
  int n = 0;
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    s += token_loss[i];
    n += (targets && targets[i] != kIgnore) ? 1 : 0;
  }
  ss[threadIdx.x] = s;
  sc[threadIdx.x] = n;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) {
      ss[threadIdx.x] += ss[threadIdx.x + w];
      sc[threadIdx.x] += sc[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (loss_sum) *loss_sum = ss[0];
    if (count) *count = sc[0];
  }
}

// ---------------------------------------------------------------- backward of the mean loss
// dl[t, v] = (softmax(logits[t])[v] - [v == target[t]]) / count for scored tokens, 0 for the
// others (and everywhere when nothing is scored).  One warp per token, lanes v and v + 32.
__global__ void __launch_bounds__(256) lm_dlogits_kernel(const float* __restrict__ logits,
                                                         const int32_t* __restrict__ targets,
                                                         const int* __restrict__ count, int T, int V,
                                                         float* __restrict__ dl) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int n = *count;
  int tg = targets ? targets[t] : kIgnore;
  if (tg != kIgnore && (tg < 0 || tg >= V)) tg = kIgnore;  // latched by the forward pass
  const float* row = logits + (size_t)t * V;
  float* out = dl + (size_t)t * V;
  if (tg == kIgnore || n <= 0) {
    if (lane < V) out[lane] = 0.f;
    if (lane + 32 < V) out[lane + 32] = 0.f;
    return;
  }
  const float lo = lane < V ? row[lane] : -INFINITY, hi = lane + 32 < V ? row[lane + 32] : -INFINITY;
  const float m = warp_max_all(fmaxf(lo, hi));
  const float elo = lane < V ? expf(lo - m) : 0.f, ehi = lane + 32 < V ? expf(hi - m) : 0.f;
  const float inv = 1.f / warp_sum_all(elo + ehi);
  const float sc = 1.f / (float)n;
  if (lane < V) out[lane] = (elo * inv - (lane == tg ? 1.f : 0.f)) * sc;
  if (lane + 32 < V) out[lane + 32] = (ehi * inv - (lane + 32 == tg ? 1.f : 0.f)) * sc;
}

// dz[t, :] = sum_v dl[t, v] emb[v, :] (bf16 table, fp32 out).  A block owns 64 tokens x 128
// columns: the table's 128 columns (as fp32) and the 64 tokens' dl rows (transposed, so a
// thread's eight tokens are contiguous) sit in shared memory; thread (w, l) keeps tokens
// 8w..8w+7 x columns 4l..4l+3 in registers and adds the vocabulary rows in order v = 0, 1, ...
constexpr int kDzTok = 64, kDzCols = 128, kDzTStride = kDzTok + 4;
__global__ void __launch_bounds__(256) lm_dz_kernel(const float* __restrict__ dl, const __nv_bfloat16* __restrict__ emb,
                                                    int T, int d, int V, float* __restrict__ dz) {
  extern __shared__ __align__(16) float smem_f[];
  float* se = smem_f;                          // [V][kDzCols]
  float* sdt = smem_f + (size_t)V * kDzCols;   // [V][kDzTStride]: dl of token t0 + i at [v][i]
  const int c_base = blockIdx.x * kDzCols, t0 = blockIdx.y * kDzTok;
  const int nt = min(kDzTok, T - t0), nc = min(kDzCols, d - c_base);
  for (int i = threadIdx.x; i < V * kDzCols; i += blockDim.x) {
    const int v = i / kDzCols, c = i - v * kDzCols;
    se[i] = c < nc ? __bfloat162float(emb[(size_t)v * d + c_base + c]) : 0.f;
  }
  for (int i = threadIdx.x; i < kDzTok * V; i += blockDim.x) {
    const int t = i / V, v = i - t * V;
    sdt[v * kDzTStride + t] = t < nt ? dl[(size_t)(t0 + t) * V + v] : 0.f;
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  for (int v = 0; v < V; ++v) {
    const float4 e = *reinterpret_cast<const float4*>(se + v * kDzCols + 4 * l);
    const float4 g0 = *reinterpret_cast<const float4*>(sdt + v * kDzTStride + 8 * w);
    const float4 g1 = *reinterpret_cast<const float4*>(sdt + v * kDzTStride + 8 * w + 4);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc[i][0] = fmaf(g[i], e.x, acc[i][0]);
      acc[i][1] = fmaf(g[i], e.y, acc[i][1]);
      acc[i][2] = fmaf(g[i], e.z, acc[i][2]);
      acc[i][3] = fmaf(g[i], e.w, acc[i][3]);
    }
  }
  if (4 * l < nc) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = 8 * w + i;
      if (t < nt)
        *reinterpret_cast<float4*>(dz + (size_t)(t0 + t) * d + c_base + 4 * l) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
  }
}

// Partial sums over one chunk of tokens of the tied embedding's gradient
// demb[v, c] = sum_t dl[t, v] z[t, c] (z bf16) and, in the blocks of column tile 0, of the
// vocabulary bias's gradient dbias[v] = sum_t dl[t, v].  A block owns 128 columns of one
// chunk (the chunk's dl rows in shared memory); thread (w, l) keeps columns 4l..4l+3 of the
// vocabulary rows w, w + 8, ... (V <= 64) in registers and adds the chunk's tokens in order.
__global__ void __launch_bounds__(256) lm_demb_kernel(const float* __restrict__ dl, const __nv_bfloat16* __restrict__ z,
                                                      int T, int d, int V, int chunk_rows, float* __restrict__ pe,
                                                      float* __restrict__ pb) {
  extern __shared__ float sdl[];  // [chunk_rows][V]
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int c0 = blockIdx.x * 128 + 4 * l;
  const int chunk = blockIdx.y;
  const int t0 = chunk * chunk_rows, t1 = min(T, t0 + chunk_rows);
  for (int i = threadIdx.x; i < (t1 - t0) * V; i += blockDim.x) sdl[i] = dl[(size_t)t0 * V + i];
  __syncthreads();
  if (c0 < d) {  // d % 4 == 0: the thread's four columns are in the row
    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll 8
    for (int t = t0; t < t1; ++t) {
      const uint2 zz = __ldg(reinterpret_cast<const uint2*>(z + (size_t)t * d + c0));
      const float2 za = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zz.x));
      const float2 zb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zz.y));
      const float* g = sdl + (size_t)(t - t0) * V;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int v = w + 8 * j;
        if (v < V) {
          const float gv = g[v];
          acc[j][0] = fmaf(gv, za.x, acc[j][0]);
          acc[j][1] = fmaf(gv, za.y, acc[j][1]);
          acc[j][2] = fmaf(gv, zb.x, acc[j][2]);
          acc[j][3] = fmaf(gv, zb.y, acc[j][3]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int v = w + 8 * j;
      if (v < V)
        *reinterpret_cast<float4*>(pe + ((size_t)chunk * V + v) * d + c0) =
            make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
    }
  }
  if (blockIdx.x == 0 && (int)threadIdx.x < V) {
    float b = 0.f;
    for (int t = 0; t < t1 - t0; ++t) b += sdl[(size_t)t * V + threadIdx.x];
    pb[(size_t)chunk * V + threadIdx.x] = b;
  }
}

}  // namespace

constexpr int kLmChunkRows = 128;  // tokens per partial sum of the embedding's gradient

size_t lm_backward_partial_floats(int T, int V, int d) {
  const size_t chunks = T <= 0 ? 1 : (T + kLmChunkRows - 1) / kLmChunkRows;
  return chunks * V * (size_t)d + chunks * V;
}

cudaError_t launch_lm_backward_head(const float* logits, const int32_t* targets, const int* count, const void* emb,
                                    const __nv_bfloat16* z, int T, int d, int V, float* dl, float* dz, float* demb,
                                    float* dbias, float* partial, int num_sms, cudaStream_t st) {
  if (T <= 0) {
    cudaMemsetAsync(demb, 0, sizeof(float) * (size_t)V * d, st);
    cudaMemsetAsync(dbias, 0, sizeof(float) * V, st);
    return cudaGetLastError();
  }
  lm_dlogits_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits, targets, count, T, V, dl);
  const size_t smem = sizeof(float) * (size_t)V * (kDzCols + kDzTStride);
  cudaFuncSetAttribute(lm_dz_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  lm_dz_kernel<<<dim3((d + kDzCols - 1) / kDzCols, (T + kDzTok - 1) / kDzTok), 256, smem, st>>>(
      dl, static_cast<const __nv_bfloat16*>(emb), T, d, V, dz);
  const int chunks = (T + kLmChunkRows - 1) / kLmChunkRows;
  float* pe = partial;
  float* pb = partial + (size_t)chunks * V * d;
  const size_t smem2 = sizeof(float) * (size_t)kLmChunkRows * V;
  cudaFuncSetAttribute(lm_demb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
  lm_demb_kernel<<<dim3((d + 127) / 128, chunks), 256, smem2, st>>>(dl, z, T, d, V, kLmChunkRows, pe, pb);
  reduce_chunks(pe, chunks, (size_t)V * d, (size_t)V * d, 1.f, demb, st);
  reduce_chunks(pb, chunks, (size_t)V, (size_t)V, 1.f, dbias, st);
  return cudaGetLastError();
}

size_t lm_logits_smem_bytes(int vocab, int hidden, bool bf16) { return (size_t)vocab * hidden * (bf16 ? 2 : 4); }

template <bool BF16, int NU>
void launch_nu(int grid, size_t smem, const void* z, const void* emb, const void* bias, int T, int d, int V,
               const int32_t* targets, float* logits, float* token_loss, unsigned* err, cudaStream_t st) {
  cudaFuncSetAttribute(lm_logits_kernel<BF16, NU>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  lm_logits_kernel<BF16, NU><<<grid, 256, smem, st>>>(z, emb, bias, T, d, V, targets, logits, token_loss, err);
}

// false when the table does not fit shared memory or the row is too long for the register plan
bool lm_logits_supported(int vocab, int hidden, bool bf16) {
  const int per = bf16 ? 8 : 4;
  return vocab >= 1 && vocab <= 64 && hidden % per == 0 && hidden / per <= 16 * 32 &&
         lm_logits_smem_bytes(vocab, hidden, bf16) <= 200 * 1024;
}

cudaError_t launch_lm_logits(const void* z, bool bf16, const void* emb, const void* bias, int T, int d, int V,
                             const int32_t* targets, float* logits, float* token_loss, float* loss_sum, int* count,
                             int num_sms, unsigned* err, cudaStream_t st) {
  const size_t smem = lm_logits_smem_bytes(V, d, bf16);
  const int nb = (V + 7) / 8;
  if (T > 0 && bf16 && d % 128 == 0 && nb >= 1 && nb <= 8 &&
      (size_t)8 * nb * lm_mma_row_bytes(d) <= 227 * 1024) {
    switch (nb) {
      case 1: launch_mma_nb<1>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
      case 2: launch_mma_nb<2>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
      case 3: launch_mma_nb<3>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
      case 4: launch_mma_nb<4>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
      case 5: launch_mma_nb<5>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
      case 6: launch_mma_nb<6>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
      case 7: launch_mma_nb<7>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
      default: launch_mma_nb<8>(num_sms, z, emb, bias, T, d, V, targets, logits, token_loss, err, st); break;
    }
  } else if (T > 0) {
    const int per_sm = smem <= 100 * 1024 ? 2 : 1;
    int grid = num_sms * per_sm;
    const int need = (T + 7) / 8;
    if (grid > need) grid = need;
    const int units = d / (bf16 ? 8 : 4);
    const int nu = (units + 31) / 32;
    if (bf16) {
      if (nu <= 1) launch_nu<true, 1>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else if (nu <= 2) launch_nu<true, 2>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else if (nu <= 4) launch_nu<true, 4>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else if (nu <= 8) launch_nu<true, 8>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else launch_nu<true, 16>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
    } else {
      if (nu <= 1) launch_nu<false, 1>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else if (nu <= 2) launch_nu<false, 2>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else if (nu <= 4) launch_nu<false, 4>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else if (nu <= 8) launch_nu<false, 8>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
      else launch_nu<false, 16>(grid, smem, z, emb, bias, T, d, V, targets, logits, token_loss, err, st);
    }
  }
  if (loss_sum || count) loss_reduce_kernel<<<1, 1024, 0, st>>>(token_loss, targets, T, loss_sum, count);
  return cudaGetLastError();
}

}  // namespace esm
