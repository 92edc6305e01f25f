// Persistent warp-specialised tcgen05 GEMM with fused epilogues (sm_103a).
//
//   C[M, N] = A[M, K] * B[N, K]^T      A: activations, B: nn.Linear-style weights
//
// Clusters of two CTAs (one per SM) walk the 256 x 256 output tiles in a static stride;
// the pair multiplies with tcgen05.mma.cta_group::2 (M = 256: 128 rows per CTA, B split by
// N between the two CTAs, so each SM streams 32 KB per 64-wide K-slice).  Roles:
//   warp 0       TMA producer (each CTA): its A rows and its half of B, K-slices of 128
//                bytes with the 128-byte swizzle, into a 6-stage shared-memory ring; both
//                CTAs' copies complete on the leader CTA's "full" mbarrier;
//   warp 1       MMA issuer (leader CTA, one thread): tcgen05.mma (K=16 for bf16, K=32 for
//                e4m3) into one of two TMEM accumulators; tcgen05.commit multicasts to both
//                CTAs to free ring stages and to signal the finished accumulator;
//   warps 2..9   epilogue (each CTA): tcgen05.ld of its accumulator half (one TMEM lane =
//                one output row), fused bias / RoPE / GELU / residual add, global stores;
//                each warp then arrives on the leader's "accumulator free" mbarrier.
// Two accumulators (2 x 256 of the 512 TMEM columns) let the epilogue of one tile run
// while the tensor core works on the next.  Every mbarrier wait is bounded: on timeout
// the kernel latches an error bit, stops issuing work and still releases its TMEM.
//
// This is the dense contraction of the layer's four linear maps (QKV projection, output
// projection, fc1, fc2: the LayerNormLinear / Linear / LayerNormMLP modules of the
// aikraft.ru TransformerEngine summary and section 3.1 of the hotelren.com guide).
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int ROW_BYTES = 128;                 // one K-slice row: 64 bf16 or 128 e4m3
constexpr int A_STAGE = BM * ROW_BYTES;        // 16 KB
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int TMEM_COLS = 2 * BN;              // two accumulators

struct Smem {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort;
};

// Load 32 bias values starting at column c (param dtype bf16 or f32).
__device__ __forceinline__ void load_bias32(const EpiArgs& ea, int c, float (&b)[32]) {
  if (ea.bias == nullptr) {
#pragma unroll
    for (int i = 0; i < 32; ++i) b[i] = 0.f;
    return;
  }
  if (ea.bias_f32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(ea.bias) + c);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 v = __ldg(p + i);
      b[4 * i] = v.x; b[4 * i + 1] = v.y; b[4 * i + 2] = v.z; b[4 * i + 3] = v.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ea.bias) + c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 v = __ldg(p + i);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 f = __bfloat1622float2(h[j]);
        b[8 * i + 2 * j] = f.x;
        b[8 * i + 2 * j + 1] = f.y;
      }
    }
  }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    p[i] = w;
  }
}

__device__ __forceinline__ void store_e4m3x32(uint8_t* dst, const float (&v)[32], float s, float& amax) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* f = &v[16 * i + 4 * j];
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
      __nv_fp8x4_e4m3 q(make_float4(f[0] * s, f[1] * s, f[2] * s, f[3] * s));
      w[j] = *reinterpret_cast<uint32_t*>(&q);
    }
    p[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Epilogue of one 64-column group of one row: v0 = columns c..c+31, v1 = c+32..c+63.
template <int EPI, bool FP8, Act OUT>
__device__ __forceinline__ void epilogue_group(const EpiArgs& ea, int row, int N, int c, float (&v0)[32],
                                               float (&v1)[32], float acc_scale, float& amax) {
  float b[32];
  if (FP8) {
#pragma unroll
    for (int i = 0; i < 32; ++i) { v0[i] *= acc_scale; v1[i] *= acc_scale; }
  }
  load_bias32(ea, c, b);
#pragma unroll
  for (int i = 0; i < 32; ++i) v0[i] += b[i];
  load_bias32(ea, c + 32, b);
#pragma unroll
  for (int i = 0; i < 32; ++i) v1[i] += b[i];

  const size_t off = (size_t)row * N + c;
  if constexpr (EPI == ESM_EPI_BIAS_F32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(ea.out) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = make_float4(v0[4 * i], v0[4 * i + 1], v0[4 * i + 2], v0[4 * i + 3]);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[8 + i] = make_float4(v1[4 * i], v1[4 * i + 1], v1[4 * i + 2], v1[4 * i + 3]);
  } else if constexpr (EPI == ESM_EPI_RESIDUAL) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(ea.out) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 x = o[i];
      o[i] = make_float4(x.x + v0[4 * i], x.y + v0[4 * i + 1], x.z + v0[4 * i + 2], x.w + v0[4 * i + 3]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 x = o[8 + i];
      o[8 + i] = make_float4(x.x + v1[4 * i], x.y + v1[4 * i + 1], x.z + v1[4 * i + 2], x.w + v1[4 * i + 3]);
    }
  } else if constexpr (EPI == ESM_EPI_QKV_ROPE) {
    // head_dim 64: the group is exactly one head; pair (j, j + 32) = (v0[j], v1[j]).
    if (c < ea.rope_cols) {
      int p = ea.pos_id[row];
      p = p < 0 ? 0 : (p >= ea.max_pos ? ea.max_pos - 1 : p);
      const float4* tab = reinterpret_cast<const float4*>(ea.rope + (size_t)p * kRopeMaxHalf);
#pragma unroll
      for (int j2 = 0; j2 < 16; ++j2) {
        const float4 cs = __ldg(tab + j2);  // (cos_j, sin_j, cos_j+1, sin_j+1)
        const int j = 2 * j2;
        float a = v0[j], bb = v1[j];
        v0[j] = a * cs.x - bb * cs.y;
        v1[j] = bb * cs.x + a * cs.y;
        a = v0[j + 1]; bb = v1[j + 1];
        v0[j + 1] = a * cs.z - bb * cs.w;
        v1[j + 1] = bb * cs.z + a * cs.w;
      }
    }
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(ea.out) + off;
    store_bf16x32(o, v0);
    store_bf16x32(o + 32, v1);
  } else {  // GELU
#pragma unroll
    for (int i = 0; i < 32; ++i) { v0[i] = gelu_erf(v0[i]); v1[i] = gelu_erf(v1[i]); }
    if constexpr (OUT == Act::E4M3) {
      const float s = *ea.o_scale;
      uint8_t* o = static_cast<uint8_t*>(ea.out) + off;
      store_e4m3x32(o, v0, s, amax);
      store_e4m3x32(o + 32, v1, s, amax);
    } else {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(ea.out) + off;
      store_bf16x32(o, v0);
      store_bf16x32(o + 32, v1);
    }
  }
}

// PAIR = false: one CTA per 128 x 256 tile (tcgen05 cta_group::1, M = 128).
// PAIR = true:  a cluster of two CTAs per 256 x 256 tile (cta_group::2, M = 256): each CTA
//               loads its own 128 rows of A and its half (128 rows) of B, the leader CTA
//               issues the MMAs, each CTA's TMEM receives its 128 rows x 256 columns.
template <bool PAIR>
struct Geo {
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr int kBStage = (PAIR ? BN / 2 : BN) * ROW_BYTES;  // B rows this CTA loads
  static constexpr int kSmem = kStages * (A_STAGE + kBStage) + 1024 + 256;
};

template <int EPI, bool FP8, Act OUT, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M,
                   int N, int K, EpiArgs ea, unsigned* err) {
  constexpr int S = Geo<PAIR>::kStages;
  constexpr int B_ST = Geo<PAIR>::kBStage;
  constexpr int TILE_M = PAIR ? 2 * BM : BM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + S * A_STAGE;
  Smem* sm = reinterpret_cast<Smem*>(sB + S * B_ST);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // cluster (or CTA) index
  const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int m_tiles = (M + TILE_M - 1) / TILE_M;
  const int n_tiles = N / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int kb_count = K / (FP8 ? 128 : 64);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm->full[s], 1);
      mbar_init(&sm->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm->tfull[a], 1);
      mbar_init(&sm->tempty[a], NUM_EPI_WARPS * (PAIR ? 2 : 1));  // one arrival per epilogue warp
    }
    mbar_init(&sm->mma_done, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    if (PAIR) tmem_alloc_pair(&sm->tmem_base, TMEM_COLS);
    else tmem_alloc(&sm->tmem_base, TMEM_COLS);
  }
  tc_fence_before();
  if (PAIR) cluster_sync();  // the peer's barriers exist before anyone signals them
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issues = 0;
      for (int tile = unit; tile < num_tiles && !sm->abort; tile += units) {
        const int m0 = (tile / n_tiles) * TILE_M + (int)rank * BM;
        const int n0 = (tile % n_tiles) * BN + (PAIR ? (int)rank * (BN / 2) : 0);
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&sm->empty[stage], phase ^ 1)) {
            latch_error(err, ERRBIT_TIMEOUT);
            sm->abort = 1;
            break;
          }
          const int kx = kb * (FP8 ? 128 : 64);
          if (PAIR) {
            // Both CTAs' copies complete on the leader's barrier; the leader arms it with
            // the bytes of the whole pair.
            if (leader) mbar_arrive_expect_tx(&sm->full[stage], 2 * (A_STAGE + B_ST));
            const uint32_t bar = map_to_rank(&sm->full[stage], 0);
            tma_load_2d_pair(sA + stage * A_STAGE, &tmA, kx, m0, bar);
            tma_load_2d_pair(sB + stage * B_ST, &tmB, kx, n0, bar);
          } else {
            mbar_arrive_expect_tx(&sm->full[stage], A_STAGE + B_ST);
            tma_load_2d(sA + stage * A_STAGE, &tmA, kx, m0, &sm->full[stage]);
            tma_load_2d(sB + stage * B_ST, &tmB, kx, n0, &sm->full[stage]);
          }
          ++issues;
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      // The copies of the last S issues may still be in flight (only when a consumer gave
      // up early): wait, bounded, until they have landed (the leader sees the whole pair's
      // bytes; the peer waits for its stages to be released instead).
      for (int i = issues - 1; i >= 0 && i >= issues - S; --i) {
        const uint32_t ph = (uint32_t)(i / S) & 1u;
        if (!PAIR || leader) {
          if (!mbar_wait(&sm->full[i % S], ph)) break;
        } else {
          if (!mbar_wait(&sm->empty[i % S], ph)) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = FP8 ? idesc_e4m3(TILE_M, BN) : idesc_bf16(TILE_M, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = unit; tile < num_tiles && !sm->abort; tile += units) {
        if (!mbar_wait(&sm->tempty[acc], acc_phase ^ 1)) {
          latch_error(err, ERRBIT_TIMEOUT);
          sm->abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&sm->full[stage], phase)) {
            latch_error(err, ERRBIT_TIMEOUT);
            sm->abort = 1;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * A_STAGE);
          const uint32_t b0 = smem_u32(sB + stage * B_ST);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 4 x 32 bytes of K per 128-byte row
            const uint64_t ad = make_sw128_desc(a0 + 32 * k);
            const uint64_t bd = make_sw128_desc(b0 + 32 * k);
            if (PAIR) {
              if (FP8) mma_f8_pair(d_tmem, ad, bd, idesc, (kb | k) != 0);
              else mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0);
            } else {
              if (FP8) mma_f8_ss(d_tmem, ad, bd, idesc, (kb | k) != 0);
              else mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0);
            }
          }
          if (PAIR) mma_commit_pair(&sm->empty[stage]);
          else mma_commit(&sm->empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (sm->abort) break;
        if (PAIR) mma_commit_pair(&sm->tfull[acc]);
        else mma_commit(&sm->tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      // All MMAs of this thread complete before TMEM may be released.
      if (PAIR) mma_commit_pair(&sm->mma_done);
      else mma_commit(&sm->mma_done);
      mbar_wait(&sm->mma_done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;         // which 128-column half of the tile
    const uint32_t tempty_leader = PAIR ? map_to_rank(&sm->tempty[0], 0) : 0u;
    int acc = 0;
    uint32_t acc_phase = 0;
    float amax = 0.f;
    float acc_scale = 1.f;
    if (FP8) acc_scale = 1.f / (__ldg(ea.a_scale) * __ldg(ea.b_scale));
    for (int tile = unit; tile < num_tiles; tile += units) {
      if (!mbar_wait_warp(&sm->tfull[acc], acc_phase)) {
        latch_error(err, ERRBIT_TIMEOUT);
        sm->abort = 1;
        break;
      }
      tc_fence_after();
      const int row = (tile / n_tiles) * TILE_M + (int)rank * BM + q * 32 + lane;
      const int n0 = (tile % n_tiles) * BN + half * (BN / 2);
      const uint32_t tbase = tmem_base + acc * BN + half * (BN / 2) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int g = 0; g < BN / 2; g += 64) {
        float v0[32], v1[32];
        tmem_ld32(tbase + g, v0);
        tmem_ld32(tbase + g + 32, v1);
        if (row < M) epilogue_group<EPI, FP8, OUT>(ea, row, N, n0 + g, v0, v1, acc_scale, amax);
      }
      // This warp is done with the accumulator: one arrival per warp on the MMA issuer's
      // barrier (in the leader CTA for a pair).
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR) mbar_arrive_remote(tempty_leader + acc * (uint32_t)sizeof(uint64_t));
        else mbar_arrive(&sm->tempty[acc]);
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if constexpr (OUT == Act::E4M3) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0 && ea.o_amax) atomic_max_nonneg(ea.o_amax, amax);
    }
  }

  tc_fence_before();
  if (PAIR) cluster_sync();  // nobody leaves while the peer may still touch its shared memory
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int EPI, bool FP8, Act OUT>
cudaError_t launch_impl(const CUtensorMap* tmA, const CUtensorMap* tmB, int M, int N, int K, const EpiArgs& ea,
                        int num_sms, unsigned* err, cudaStream_t st) {
  constexpr bool PAIR = true;
  auto kern = gemm_tc_kernel<EPI, FP8, OUT, PAIR>;
  constexpr int smem = Geo<PAIR>::kSmem;
  static int max_clusters = 0;  // per instantiation: co-resident clusters of two on this device
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess || n <= 0) n = num_sms / 2;
    max_clusters = n;
  }
  const int tiles = ((M + 2 * BM - 1) / (2 * BM)) * (N / BN);
  const int clusters = tiles < max_clusters ? tiles : max_clusters;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *tmA, *tmB, M, N, K, ea, err);
}

}  // namespace

int gemm_tc_smem_bytes() { return Geo<true>::kSmem; }
// Rows of the TMA boxes the launched kernel expects: its own 128 rows of A, and its half of
// the 256-wide B tile.
int gemm_tc_a_box_rows() { return BM; }
int gemm_tc_b_box_rows() { return BN / 2; }

cudaError_t launch_gemm_tc(esm_epilogue epi, bool fp8, Act out_act, const CUtensorMap* tmA, const CUtensorMap* tmB,
                           int M, int N, int K, const EpiArgs& ea, int num_sms, unsigned* err, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (!fp8) {
    switch (epi) {
      case ESM_EPI_BIAS_F32: return launch_impl<ESM_EPI_BIAS_F32, false, Act::F32>(tmA, tmB, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_QKV_ROPE: return launch_impl<ESM_EPI_QKV_ROPE, false, Act::BF16>(tmA, tmB, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_RESIDUAL: return launch_impl<ESM_EPI_RESIDUAL, false, Act::F32>(tmA, tmB, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_GELU: return launch_impl<ESM_EPI_GELU, false, Act::BF16>(tmA, tmB, M, N, K, ea, num_sms, err, st);
    }
  } else {
    switch (epi) {
      case ESM_EPI_BIAS_F32: return launch_impl<ESM_EPI_BIAS_F32, true, Act::F32>(tmA, tmB, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_QKV_ROPE: return launch_impl<ESM_EPI_QKV_ROPE, true, Act::BF16>(tmA, tmB, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_RESIDUAL: return launch_impl<ESM_EPI_RESIDUAL, true, Act::F32>(tmA, tmB, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_GELU:
        if (out_act == Act::E4M3)
          return launch_impl<ESM_EPI_GELU, true, Act::E4M3>(tmA, tmB, M, N, K, ea, num_sms, err, st);
        return launch_impl<ESM_EPI_GELU, true, Act::BF16>(tmA, tmB, M, N, K, ea, num_sms, err, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace esm
