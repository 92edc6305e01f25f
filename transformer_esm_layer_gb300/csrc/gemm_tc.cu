// Persistent warp-specialised tcgen05 GEMM with fused epilogues (sm_103a).
//
//   C[M, N] = A[M, K] * B[N, K]^T      A: activations, B: nn.Linear-style weights
//
// Clusters of two CTAs (one per SM) walk the 256 x 256 output tiles in a static stride;
// the pair multiplies with tcgen05.mma.cta_group::2 (M = 256: 128 rows per CTA, B split by
// N between the two CTAs, so each SM streams 32 KB per 64-wide K-slice).  Roles:
//   warp 0       TMA producer (each CTA): its A rows and its half of B, K-slices of 128
//                bytes with the 128-byte swizzle, into a 5- or 6-stage shared-memory ring; both
//                CTAs' copies complete on the leader CTA's "full" mbarrier;
//   warp 1       MMA issuer (leader CTA, one thread): tcgen05.mma (K=16 for bf16, K=32 for
//                e4m3) into one of two TMEM accumulators; tcgen05.commit multicasts to both
//                CTAs to free ring stages and to signal the finished accumulator;
//   warps 2..9   epilogue (each CTA): warp w owns TMEM lanes 32*(w%4).. (rows) and one
//                128-column half of the tile.  Per chunk of 128 bytes per row it reads the
//                accumulator (tcgen05.ld), applies bias / RoPE / GELU / residual add, writes
//                the chunk into a swizzled shared-memory staging buffer and one thread stores
//                it with a TMA bulk-tensor store.  The fp32 residual (read and written in
//                place) instead moves through the load/store unit, each warp copying its
//                own rows, so it never queues behind the operand loads in the TMA engine
//                and needs no barrier between warps.  Each warp arrives on the
//                leader's "accumulator free" mbarrier as soon as it has read its last
//                accumulator columns, before finishing that chunk.
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

constexpr int BM = 128;                        // rows per CTA
constexpr int BN = 256;                        // columns per tile
constexpr int TILE_M = 2 * BM;                 // rows per CTA pair
constexpr int S_MAX = 6;                       // ring stages (at most)
constexpr int ROW_BYTES = 128;                 // one K-slice row: 64 bf16 or 128 e4m3
constexpr int A_STAGE = BM * ROW_BYTES;        // 16 KB
constexpr int B_STAGE = (BN / 2) * ROW_BYTES;  // 16 KB: this CTA's half of B
constexpr int E_BUF = 128 * 128;               // 16 KB epilogue staging chunk (128 rows x 128 B)
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int TMEM_COLS = 2 * BN;              // two accumulators

// Shared-memory plan per epilogue.  The bf16 / E4M3 outputs leave through TMA stores from
// two 16 KB staging chunks per column half (one being stored while the next is written),
// which leaves room for a 5-stage operand ring.  The residual epilogue moves its fp32
// chunks through the load/store unit one chunk per warp at a time, so one staging chunk
// per half suffices and the ring gets a 6th stage (its long-K launch streams A from HBM).
// The QKV and fc1 launches (K = hidden = 1280 at 650M) run as fast on a 4-stage ring as on 5
// (measured), so they keep 4.
template <int EPI>
struct Plan {
  static constexpr int kStages =
      (EPI == ESM_EPI_RESIDUAL) ? 6 : ((EPI == ESM_EPI_QKV_ROPE || EPI == ESM_EPI_GELU) ? 4 : 5);
  static constexpr int kEBufs = (EPI == ESM_EPI_RESIDUAL) ? 1 : 2;  // staging chunks per half
  static constexpr int kSmemBytes =
      kStages * (A_STAGE + B_STAGE) + 2 * kEBufs * E_BUF + 1024 /*align*/ + 256 /*barriers*/;
  static_assert(kStages <= S_MAX, "barrier arrays");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

struct Smem {
  uint64_t full[S_MAX];
  uint64_t empty[S_MAX];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort;
  volatile int fail[2];  // [half]: an epilogue warp of that half gave up waiting
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

// Scale the W accumulator values of columns c.. and add their bias, 8 bias values at a
// time (keeps few registers live next to the accumulators).
template <int W>
__device__ __forceinline__ void scale_add_bias(const EpiArgs& ea, int c, float scale, float (&v)[W]) {
#pragma unroll
  for (int i8 = 0; i8 < W / 8; ++i8) {
    float b[8];
    if (ea.bias == nullptr) {
#pragma unroll
      for (int k = 0; k < 8; ++k) b[k] = 0.f;
    } else if (ea.bias_f32) {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(ea.bias) + c + 8 * i8);
      const float4 x = __ldg(p), y = __ldg(p + 1);
      b[0] = x.x; b[1] = x.y; b[2] = x.z; b[3] = x.w; b[4] = y.x; b[5] = y.y; b[6] = y.z; b[7] = y.w;
    } else {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ea.bias) + c + 8 * i8));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        b[2 * k] = f.x;
        b[2 * k + 1] = f.y;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) v[8 * i8 + k] = v[8 * i8 + k] * scale + b[k];
  }
}

// Byte offset of 16-byte unit j of row r in a 128-row x 128-byte staging chunk laid out
// with the 128-byte swizzle (the layout the TMA maps of the outputs use).
__device__ __forceinline__ uint32_t swz_off(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

__device__ __forceinline__ void st_shared_v4(uint8_t* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}

// Residual rows of one epilogue warp (rows 32q .. 32q+31 of the CTA's 128, one 128-byte
// chunk of fp32 columns starting at col) between global memory and the swizzled staging
// buffer.  Lane l moves 16-byte unit (l & 7) of rows 4i + (l >> 3): every instruction covers
// four whole 128-byte rows.  Rows at or beyond M are zero-filled / not written.
__device__ __forceinline__ void residual_rows_async(const EpiArgs& ea, uint8_t* buf, int q, int lane, int row0,
                                                    int M, int N, int col) {
  const float* x = static_cast<const float*>(ea.res_in ? ea.res_in : ea.out);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = q * 32 + 4 * i + (lane >> 3);
    const int u = lane & 7;
    const int grow = row0 + rr;
    const bool in = grow < M;
    const float* src = x + (in ? (size_t)grow * N + col + 4 * u : 0);
    cp_async_16(buf + swz_off(rr, u), src, in ? 16u : 0u);
  }
}
__device__ __forceinline__ void residual_rows_store(const EpiArgs& ea, const uint8_t* buf, int q, int lane, int row0,
                                                    int M, int N, int col) {
  float* x = static_cast<float*>(ea.out);
  const int u = lane & 7;
  // folded LayerNorm: the next GEMM's operand bf16(x * gamma), 4 columns (8 bytes) per lane,
  // so each instruction writes 64 contiguous bytes of four rows
  float4 gm = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ea.ln_a_out != nullptr) {
    const uint2 g = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(ea.ln_gamma) + col + 4 * u));
    const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.x));
    const float2 g1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.y));
    gm = make_float4(g0.x, g0.y, g1.x, g1.y);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = q * 32 + 4 * i + (lane >> 3);
    const int grow = row0 + rr;
    const uint4 v = *reinterpret_cast<const uint4*>(buf + swz_off(rr, u));
    if (grow < M) {
      *reinterpret_cast<uint4*>(x + (size_t)grow * N + col + 4 * u) = v;
      if (ea.ln_a_out != nullptr) {
        const float4 f = *reinterpret_cast<const float4*>(&v);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(ea.ln_a_out) + (size_t)grow * N + col + 4 * u) =
            make_uint2(pack_bf16x2(f.x * gm.x, f.y * gm.y), pack_bf16x2(f.z * gm.z, f.w * gm.w));
      }
    }
  }
}

// Folded LayerNorm, consumer side: rstd and mean * rstd of row `row` from the (mean, sum of
// squared deviations) of its ln_groups groups of 64 columns (the parallel-variance
// combination: M2 = sum M2_g + 64 sum (mean_g - mean)^2, var = M2 / (64 groups)).  One pass
// over 16-byte loads (two groups each) issued together; the group means enter as deviations
// from the first one, so the between-group term has no cancellation.
__device__ __forceinline__ float2 ln_row_stats(const EpiArgs& ea, int row, int M) {
  if (row >= M) return make_float2(0.f, 0.f);
  const float4* st = reinterpret_cast<const float4*>(ea.ln_stats_in + (size_t)row * ea.ln_groups);
  const int pairs = ea.ln_groups >> 1;  // ln_groups is even (hidden % 128 == 0)
  const float m0 = __ldg(reinterpret_cast<const float*>(st));
  float sd = 0.f, sd2 = 0.f, sm2 = 0.f;
  constexpr int kMaxPairs = 32;  // hidden <= 4096
#pragma unroll
  for (int p = 0; p < kMaxPairs; ++p) {
    if (p < pairs) {
      const float4 v = __ldg(st + p);  // (mean, M2) of groups 2p and 2p + 1
      const float d0 = v.x - m0, d1 = v.z - m0;
      sd += d0 + d1;
      sd2 += d0 * d0 + d1 * d1;
      sm2 += v.y + v.w;
    }
  }
  const float G = (float)ea.ln_groups;
  const float dmean = sd / G;
  const float m2 = sm2 + 64.f * fmaxf(sd2 - sd * dmean, 0.f);
  const float rstd = rsqrtf(m2 / (64.f * G) + ea.ln_eps);
  return make_float2(rstd, (m0 + dmean) * rstd);
}

// Folded LayerNorm applied to W accumulator values of columns c..: v = rstd v - mr c_n + b'_n.
template <int W>
__device__ __forceinline__ void ln_fold_apply(const EpiArgs& ea, int c, float2 rs, float (&v)[W]) {
#pragma unroll
  for (int i4 = 0; i4 < W / 4; ++i4) {
    const float4 cc = __ldg(reinterpret_cast<const float4*>(ea.ln_c + c) + i4);
    const float4 bb = __ldg(reinterpret_cast<const float4*>(ea.ln_b + c) + i4);
    v[4 * i4 + 0] = fmaf(v[4 * i4 + 0], rs.x, fmaf(-rs.y, cc.x, bb.x));
    v[4 * i4 + 1] = fmaf(v[4 * i4 + 1], rs.x, fmaf(-rs.y, cc.y, bb.y));
    v[4 * i4 + 2] = fmaf(v[4 * i4 + 2], rs.x, fmaf(-rs.y, cc.z, bb.z));
    v[4 * i4 + 3] = fmaf(v[4 * i4 + 3], rs.x, fmaf(-rs.y, cc.w, bb.w));
  }
}

// 32 fp32 values (columns of this thread's row) as bf16 into 16-byte units u0..u0+3.
__device__ __forceinline__ void stage_bf16x32(uint8_t* buf, int r, int u0, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    st_shared_v4(buf, swz_off(r, u0 + i), w);
  }
}

// 16 fp32 values as bf16 into 16-byte units u0, u0+1.
__device__ __forceinline__ void stage_bf16x16(uint8_t* buf, int r, int u0, const float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    st_shared_v4(buf, swz_off(r, u0 + i), w);
  }
}

// 32 fp32 values as E4M3 (scaled by s) into 16-byte units u0, u0+1; max |v| into amax.
__device__ __forceinline__ void stage_e4m3x32(uint8_t* buf, int r, int u0, const float (&v)[32], float s,
                                              float& amax) {
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
    st_shared_v4(buf, swz_off(r, u0 + i), make_uint4(w[0], w[1], w[2], w[3]));
  }
}

// Tile t of the static schedule.  The first full_tiles are 256 x 256 (row band t / n_tiles,
// column tile t % n_tiles); the rest split the remaining full tiles, in order, into two
// 256 x 128 halves each, so that a partly filled last wave of full tiles becomes a wave of
// half-length tiles.
struct TileXY {
  int m, n0, bn;
};
__device__ __forceinline__ TileXY tile_xy(int t, int n_tiles, int full_tiles) {
  TileXY r;
  if (t < full_tiles) {
    r.m = t / n_tiles;
    r.n0 = (t % n_tiles) * BN;
    r.bn = BN;
  } else {
    const int h = t - full_tiles, orig = full_tiles + (h >> 1);
    r.m = orig / n_tiles;
    r.n0 = (orig % n_tiles) * BN + (h & 1) * (BN / 2);
    r.bn = BN / 2;
  }
  return r;
}

// Columns per staging chunk (128 bytes of one row) for each output type.
template <int EPI, Act OUT>
struct Chunk {
  static constexpr int kElemBytes = (EPI == ESM_EPI_BIAS_F32 || EPI == ESM_EPI_RESIDUAL) ? 4
                                    : (OUT == Act::E4M3)                                  ? 1
                                                                                          : 2;
  static constexpr int kCols = 128 / kElemBytes;     // 32, 64 or 128
  static constexpr int kPerHalf = (BN / 2) / kCols;  // 4, 2 or 1
};

// AMN / BMN: the operand is stored MN-major (its M or N index contiguous, the reduction
// index the row), as the backward products need: A = dY^T and B = X for a weight gradient
// (reduction over the tokens), B = W for an input gradient (reduction over the output
// features).  Each 128-row operand stage is then two 64 x 64 TMA boxes side by side.
// ksplit > 1 splits the K loop into ksplit ranges of kb_per K-slices; range s of tile t is
// work item s * num_tiles + t and writes output rows s * M.. (a [ksplit * M, N] partial
// buffer that the caller sums).
template <int EPI, bool FP8, Act OUT, bool AMN, bool BMN>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, int M, int N, int kb_total, int kb_per, int ksplit,
                   int full_tiles, int num_tiles, EpiArgs ea, unsigned* err) {
  static_assert(!(FP8 && (AMN || BMN)), "MN-major operands are bf16 only");
  using CH = Chunk<EPI, OUT>;
  constexpr int S = Plan<EPI>::kStages;
  constexpr int NB = Plan<EPI>::kEBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + S * A_STAGE;
  uint8_t* sE = sB + S * B_STAGE;  // [half][buffer] 16 KB each
  Smem* sm = reinterpret_cast<Smem*>(sE + 2 * NB * E_BUF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int unit = (int)(blockIdx.x >> 1);  // cluster index
  const int units = (int)(gridDim.x >> 1);
  const int n_tiles = N / BN;
  const int num_work = num_tiles * ksplit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm->full[s], 1);
      mbar_init(&sm->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm->tfull[a], 1);
      mbar_init(&sm->tempty[a], 2 * NUM_EPI_WARPS);  // one arrival per epilogue warp of the pair
    }
    mbar_init(&sm->mma_done, 1);
    sm->abort = 0;
    sm->fail[0] = 0;
    sm->fail[1] = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 1) tmem_alloc_pair(&sm->tmem_base, TMEM_COLS);
  tc_fence_before();
  cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issues = 0;
      for (int wk = unit; wk < num_work && !sm->abort; wk += units) {
        const int tile = wk % num_tiles, ks = wk / num_tiles;
        const int kb0 = ks * kb_per, kb1 = min(kb_total, kb0 + kb_per);
        const TileXY tx = tile_xy(tile, n_tiles, full_tiles);
        const int m0 = tx.m * TILE_M + (int)rank * BM;
        const int n0 = tx.n0 + (int)rank * (tx.bn / 2);  // a half-width tile loads 64 surplus rows
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&sm->empty[stage], phase ^ 1)) {
            latch_error(err, ERRBIT_TIMEOUT);
            sm->abort = 1;
            break;
          }
          const int kx = kb * (FP8 ? 128 : 64);
          // Both CTAs' copies complete on the leader's barrier; the leader arms it with the
          // bytes of the whole pair.
          if (leader) mbar_arrive_expect_tx(&sm->full[stage], 2 * (A_STAGE + B_STAGE));
          const uint32_t bar = map_to_rank(&sm->full[stage], 0);
          if (AMN) {
            tma_load_2d_pair(sA + stage * A_STAGE, &tmA, m0, kx, bar);
            tma_load_2d_pair(sA + stage * A_STAGE + A_STAGE / 2, &tmA, m0 + 64, kx, bar);
          } else {
            tma_load_2d_pair(sA + stage * A_STAGE, &tmA, kx, m0, bar);
          }
          if (BMN) {
            tma_load_2d_pair(sB + stage * B_STAGE, &tmB, n0, kx, bar);
            tma_load_2d_pair(sB + stage * B_STAGE + B_STAGE / 2, &tmB, n0 + 64, kx, bar);
          } else {
            tma_load_2d_pair(sB + stage * B_STAGE, &tmB, kx, n0, bar);
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
        if (leader) {
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
      constexpr uint32_t kMajor = (AMN ? kIdescAMn : 0u) | (BMN ? kIdescBMn : 0u);
      constexpr uint32_t idesc_full = (FP8 ? idesc_e4m3(TILE_M, BN) : idesc_bf16(TILE_M, BN)) | kMajor;
      constexpr uint32_t idesc_half = (FP8 ? idesc_e4m3(TILE_M, BN / 2) : idesc_bf16(TILE_M, BN / 2)) | kMajor;
      // K step of one MMA (32 bytes of K): +32 bytes inside a K-major row, two 1024-byte
      // atoms (+2048 bytes) in an MN-major tile; in descriptor units of 16 bytes.
      constexpr uint64_t kStepA = AMN ? 128 : 2, kStepB = BMN ? 128 : 2;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      // Descriptors of stage 0; a stage adds its byte offset >> 4 to the start-address field
      // (every shared address here is below 256 KB, so the 14-bit field cannot carry), and
      // each 32-byte step of K inside the 128-byte row adds 2.
      const uint64_t adesc0 = AMN ? make_sw128_mn_desc(smem_u32(sA), A_STAGE / 2) : make_sw128_desc(smem_u32(sA));
      const uint64_t bdesc0 = BMN ? make_sw128_mn_desc(smem_u32(sB), B_STAGE / 2) : make_sw128_desc(smem_u32(sB));
      for (int wk = unit; wk < num_work && !sm->abort; wk += units) {
        const int tile = wk % num_tiles, ks = wk / num_tiles;
        const int kb_count = min(kb_total, (ks + 1) * kb_per) - ks * kb_per;
        if (!mbar_wait(&sm->tempty[acc], acc_phase ^ 1)) {
          latch_error(err, ERRBIT_TIMEOUT);
          sm->abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const uint32_t idesc = tile < full_tiles ? idesc_full : idesc_half;
        // A stage whose operands have landed is issued; if the next one has landed too (a
        // non-blocking test), its four MMAs follow back to back.  The issuing thread blocks
        // while the tensor pipe's short queue is full, and the instructions between two
        // stages (barrier test, fence, descriptors) could otherwise let the queue run dry when
        // the epilogue warps on its scheduler are busy; a stage still in flight is not waited
        // for, so delivery-bound GEMMs lose nothing.
        for (int kb = 0; kb < kb_count;) {
          const int stage1 = stage + 1 == S ? 0 : stage + 1;
          const uint32_t phase1 = stage + 1 == S ? phase ^ 1u : phase;
          if (!mbar_wait(&sm->full[stage], phase)) {
            latch_error(err, ERRBIT_TIMEOUT);
            sm->abort = 1;
            break;
          }
          const bool two = kb + 1 < kb_count && mbar_test(&sm->full[stage1], phase1);
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h == 1 && !two) break;
            const int sg = h ? stage1 : stage;
            // descriptor arithmetic on the low word only (the start-address field cannot carry):
            // fewer instructions for the issuing thread between two MMAs
            const uint32_t alo = (uint32_t)adesc0 + (uint32_t)((sg * A_STAGE) >> 4);
            const uint32_t blo = (uint32_t)bdesc0 + (uint32_t)((sg * B_STAGE) >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // 4 x 32 bytes of K per 128-byte row
              const uint64_t ad = (adesc0 & 0xFFFFFFFF00000000ull) | (uint64_t)(alo + (uint32_t)kStepA * (uint32_t)k);
              const uint64_t bd = (bdesc0 & 0xFFFFFFFF00000000ull) | (uint64_t)(blo + (uint32_t)kStepB * (uint32_t)k);
              if (FP8) mma_f8_pair(d_tmem, ad, bd, idesc, (kb | h | k) != 0);
              else mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | h | k) != 0);
            }
            mma_commit_pair(&sm->empty[sg]);
          }
          if (two) {
            kb += 2;
            stage = stage1 + 1 == S ? 0 : stage1 + 1;
            phase = stage1 + 1 == S ? phase1 ^ 1u : phase1;
          } else {
            kb += 1;
            stage = stage1;
            phase = phase1;
          }
        }
        if (sm->abort) break;
        mma_commit_pair(&sm->tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      // All MMAs of this thread complete before TMEM may be released.
      mma_commit_pair(&sm->mma_done);
      mbar_wait(&sm->mma_done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                    // TMEM lane quarter: rows 32q .. 32q+31
    const int half = (warp - 2) >> 2;          // which 128-column half of the tile
    const int r = q * 32 + lane;               // this thread's row inside the CTA's 128
    const bool elect = (warp == 2 + 4 * half) && lane == 0;  // issues the half's bulk copies
    const uint32_t bar_id = 1 + (uint32_t)half;             // named barrier of the half's 4 warps
    uint8_t* const ebuf0 = sE + (NB * half) * E_BUF;  // buffer b of this half: ebuf0 + b * E_BUF
    const uint32_t tempty_leader = map_to_rank(&sm->tempty[0], 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    float amax = 0.f;
    float acc_scale = 1.f;
    if (FP8) acc_scale = 1.f / (__ldg(ea.a_scale) * __ldg(ea.b_scale));
    const float o_scale = (OUT == Act::E4M3) ? __ldg(ea.o_scale) : 1.f;

    for (int wk = unit; wk < num_work; wk += units) {
      const int tile = wk % num_tiles, ks = wk / num_tiles;
      const TileXY tx = tile_xy(tile, n_tiles, full_tiles);
      const int row0 = tx.m * TILE_M + (int)rank * BM;                 // first row of this CTA
      const int col0 = tx.n0 + half * (tx.bn / 2);                     // first column of this half
      const int nch = tx.bn == BN ? CH::kPerHalf : CH::kPerHalf / 2;  // chunks of this half
      const int row = row0 + r;
      // This warp has read the whole accumulator into registers: hand it back to the MMA
      // warp (one arrival per warp on the leader's barrier) before finishing the chunk.
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty_leader + acc * (uint32_t)sizeof(uint64_t));
      };
      if constexpr (EPI == ESM_EPI_RESIDUAL) {
        // The residual goes through the load/store unit, not the TMA engine (whose queue is
        // full of operand loads): each warp copies its own 32 rows of chunks 0 and 1 into
        // its rows of the two staging buffers (coalesced: 4 rows x 128 bytes per
        // instruction) and pulls its rows of the later chunks into L2.
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          residual_rows_async(ea, ebuf0 + b * E_BUF, q, lane, row0, M, N, col0 + b * CH::kCols);
          cp_async_commit();
        }
        if (row < M) {
          const float* xr = static_cast<const float*>(ea.res_in ? ea.res_in : ea.out) + (size_t)row * N + col0;
          for (int c = NB; c < nch; ++c) prefetch_l2(xr + c * CH::kCols);
        }
      }
      // RoPE: this row's (cos, sin) for the 32 pairs of a 64-wide head are the same for every
      // q and k head of the tile; fetch them once, before the accumulator is ready.
      float4 cs[EPI == ESM_EPI_QKV_ROPE ? 16 : 1];
      if constexpr (EPI == ESM_EPI_QKV_ROPE) {
        if (col0 < ea.rope_cols) {
          int p = row < M ? __ldg(ea.pos_id + row) : 0;
          p = p < 0 ? 0 : (p >= ea.max_pos ? ea.max_pos - 1 : p);
          const float4* tab = reinterpret_cast<const float4*>(ea.rope) + p;  // group g at g * max_pos
#pragma unroll
          for (int g = 0; g < 16; ++g) cs[g] = __ldg(tab + (size_t)g * ea.max_pos);
        }
      }
      // folded LayerNorm: this row's statistics (QKV / GELU epilogues of a bf16 forward)
      float2 ln_rs = make_float2(1.f, 0.f);
      if constexpr (!FP8 && (EPI == ESM_EPI_QKV_ROPE || EPI == ESM_EPI_GELU)) {
        if (ea.ln_stats_in != nullptr) ln_rs = ln_row_stats(ea, row, M);
      }
      const bool ok = mbar_wait_warp(&sm->tfull[acc], acc_phase);
      if (!ok && lane == 0) {
        latch_error(err, ERRBIT_TIMEOUT);
        sm->abort = 1;
        sm->fail[half] = 1;
      }
      // fail[half] is written only by this half's warps before this barrier and read by all
      // of them after it, so the whole half takes the same branch.
      named_bar_sync(bar_id, 128);
      if (sm->fail[half]) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + acc * BN + half * (tx.bn / 2) + ((uint32_t)(q * 32) << 16);
      float vlast[(EPI == ESM_EPI_BIAS_F32 || EPI == ESM_EPI_RESIDUAL) ? 32 : 1];
      float2 ln_pend = make_float2(0.f, 0.f);  // residual: statistics of the group's first chunk

#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        const int b = c % NB;
        uint8_t* buf = ebuf0 + b * E_BUF;
        const int col = col0 + c * CH::kCols;
        if constexpr (EPI != ESM_EPI_RESIDUAL) {
          // the store that last used this buffer must be done reading it
          if (elect) bulk_wait_read<1>();
          named_bar_sync(bar_id, 128);
        }
        if constexpr (EPI == ESM_EPI_BIAS_F32 || EPI == ESM_EPI_RESIDUAL) {
          // 32-column chunks: the last two are read from TMEM together, so the accumulator
          // is released one chunk early.
          float v[32], bb[32];
          if (c + 2 < nch) {
            tmem_ld32(tbase + c * CH::kCols, v);
          } else if (c + 2 == nch) {
            tmem_ld32(tbase + c * CH::kCols, v);
            tmem_ld32(tbase + (c + 1) * CH::kCols, vlast);
            release_acc();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = vlast[i];
          }
          if constexpr (EPI == ESM_EPI_RESIDUAL) {
            // this chunk's rows have landed (the next chunk's may still be in flight)
            if (NB == 2 && c + 1 < nch) cp_async_wait<1>();
            else cp_async_wait<0>();
            __syncwarp();
          }
          load_bias32(ea, col, bb);
          // folded LayerNorm statistics of the new residual: sums of deviations from the
          // chunk's first value (shifted sums keep the variance free of cancellation)
          float k0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t off = swz_off(r, j);
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (EPI == ESM_EPI_RESIDUAL) x = *reinterpret_cast<const float4*>(buf + off);
            float4 o;
            o.x = x.x + (v[4 * j + 0] * acc_scale + bb[4 * j + 0]);
            o.y = x.y + (v[4 * j + 1] * acc_scale + bb[4 * j + 1]);
            o.z = x.z + (v[4 * j + 2] * acc_scale + bb[4 * j + 2]);
            o.w = x.w + (v[4 * j + 3] * acc_scale + bb[4 * j + 3]);
            *reinterpret_cast<float4*>(buf + off) = o;
            if constexpr (EPI == ESM_EPI_RESIDUAL) {
              if (j == 0) k0 = o.x;
              const float a0 = o.x - k0, a1 = o.y - k0, a2 = o.z - k0, a3 = o.w - k0;
              s1 += (a0 + a1) + (a2 + a3);
              s2 += (a0 * a0 + a1 * a1) + (a2 * a2 + a3 * a3);
            }
          }
          if constexpr (EPI == ESM_EPI_RESIDUAL) {
            if (ea.ln_stats_out != nullptr) {
              // chunk statistics (32 columns), merged in pairs into 64-column groups
              const float cm = k0 + s1 * (1.f / 32.f);
              const float cm2 = fmaxf(s2 - s1 * s1 * (1.f / 32.f), 0.f);
              if ((c & 1) == 0) {
                ln_pend = make_float2(cm, cm2);
              } else if (row < M) {
                const float dm = ln_pend.x - cm;
                ea.ln_stats_out[(size_t)row * (N / 64) + (col - 32) / 64] =
                    make_float2(0.5f * (ln_pend.x + cm), ln_pend.y + cm2 + 16.f * dm * dm);
              }
            }
          }
          if constexpr (EPI == ESM_EPI_RESIDUAL) {
            // coalesced write-back of this warp's 32 rows, then refill the buffer with the
            // residual of chunk c + NB
            __syncwarp();
            residual_rows_store(ea, buf, q, lane, row0, M, N, col);
            __syncwarp();
            if (c + NB < nch) {
              residual_rows_async(ea, buf, q, lane, row0, M, N, col + NB * CH::kCols);
              cp_async_commit();
            }
            continue;
          }
        } else if constexpr (OUT == Act::E4M3) {  // fc1 + GELU -> E4M3, 128 columns
#pragma unroll 1
          for (int s4 = 0; s4 < 4; ++s4) {
            float v[32], bb[32];
            tmem_ld32(tbase + 32 * s4, v);
            if (s4 == 3) release_acc();
            load_bias32(ea, col + 32 * s4, bb);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = v[i] * acc_scale + bb[i];
#pragma unroll
            for (int i = 0; i < 32; i += 2) gelu2_as7126(v[i], v[i + 1]);
            stage_e4m3x32(buf, r, 2 * s4, v, o_scale, amax);
          }
        } else if constexpr (EPI == ESM_EPI_QKV_ROPE) {
          // bf16 output, 64 columns = one head.  RoPE pairs column j with j + 32; the head is
          // done in two passes of 16 pairs (columns 16h.. and 32 + 16h..).
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float a[16], bq[16];
            {  // both 16-column halves of the pass in one TMEM round trip
              uint32_t ra[16], rb[16];
              asm volatile(
                  "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                  "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
                  "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                  "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
                  "tcgen05.wait::ld.sync.aligned;"
                  : "=r"(ra[0]), "=r"(ra[1]), "=r"(ra[2]), "=r"(ra[3]), "=r"(ra[4]), "=r"(ra[5]), "=r"(ra[6]), "=r"(ra[7]),
                    "=r"(ra[8]), "=r"(ra[9]), "=r"(ra[10]), "=r"(ra[11]), "=r"(ra[12]), "=r"(ra[13]), "=r"(ra[14]), "=r"(ra[15]),
                    "=r"(rb[0]), "=r"(rb[1]), "=r"(rb[2]), "=r"(rb[3]), "=r"(rb[4]), "=r"(rb[5]), "=r"(rb[6]), "=r"(rb[7]),
                    "=r"(rb[8]), "=r"(rb[9]), "=r"(rb[10]), "=r"(rb[11]), "=r"(rb[12]), "=r"(rb[13]), "=r"(rb[14]), "=r"(rb[15])
                  : "r"(tbase + c * CH::kCols + 16 * h), "r"(tbase + c * CH::kCols + 32 + 16 * h)
                  : "memory");
#pragma unroll
              for (int i = 0; i < 16; ++i) { a[i] = __uint_as_float(ra[i]); bq[i] = __uint_as_float(rb[i]); }
            }
            if (h == 1 && c == nch - 1) release_acc();
            if (!FP8 && ea.ln_stats_in != nullptr) {
              ln_fold_apply<16>(ea, col + 16 * h, ln_rs, a);
              ln_fold_apply<16>(ea, col + 32 + 16 * h, ln_rs, bq);
            } else {
              scale_add_bias<16>(ea, col + 16 * h, acc_scale, a);
              scale_add_bias<16>(ea, col + 32 + 16 * h, acc_scale, bq);
            }
            if (col < ea.rope_cols) {
#pragma unroll
              for (int i = 0; i < 16; i += 2) {  // cs[g] = (cos, sin) of pairs 2g and 2g + 1
                const float4 t = cs[8 * h + i / 2];
                float x = a[i], y = bq[i];
                a[i] = x * t.x - y * t.y;
                bq[i] = y * t.x + x * t.y;
                x = a[i + 1]; y = bq[i + 1];
                a[i + 1] = x * t.z - y * t.w;
                bq[i + 1] = y * t.z + x * t.w;
              }
            }
            stage_bf16x16(buf, r, 2 * h, a);
            stage_bf16x16(buf, r, 4 + 2 * h, bq);
          }
        } else if constexpr (EPI == kEpiDgelu) {  // bf16 output, 64 columns: acc * GELU'(z)
          float v0[32], v1[32];
          tmem_ld32(tbase + c * CH::kCols, v0);
          tmem_ld32(tbase + c * CH::kCols + 32, v1);
          if (c == nch - 1) release_acc();
          uint4 zz[8];
          const uint4* zr = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ea.aux) +
                                                           (size_t)(row < M ? row : 0) * N + col);
#pragma unroll
          for (int u = 0; u < 8; ++u) zz[u] = __ldg(zr + u);
          const __nv_bfloat162* zh = reinterpret_cast<const __nv_bfloat162*>(zz);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 a = __bfloat1622float2(zh[i]), b = __bfloat1622float2(zh[16 + i]);
            v0[2 * i] *= gelu_grad_as7126(a.x);
            v0[2 * i + 1] *= gelu_grad_as7126(a.y);
            v1[2 * i] *= gelu_grad_as7126(b.x);
            v1[2 * i + 1] *= gelu_grad_as7126(b.y);
          }
          stage_bf16x32(buf, r, 0, v0);
          stage_bf16x32(buf, r, 4, v1);
        } else {  // bf16 output, 64 columns: GELU
          float v0[32], v1[32];
          tmem_ld32(tbase + c * CH::kCols, v0);
          tmem_ld32(tbase + c * CH::kCols + 32, v1);
          if (c == nch - 1) release_acc();
          if (!FP8 && ea.ln_stats_in != nullptr) {
            ln_fold_apply<32>(ea, col, ln_rs, v0);
            ln_fold_apply<32>(ea, col + 32, ln_rs, v1);
          } else {
            scale_add_bias<32>(ea, col, acc_scale, v0);
            scale_add_bias<32>(ea, col + 32, acc_scale, v1);
          }
          if (ea.aux != nullptr && row < M) {  // training forward: keep the pre-activation
            uint4* zr = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(ea.aux) + (size_t)row * N + col);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              zr[u] = make_uint4(pack_bf16x2(v0[8 * u], v0[8 * u + 1]), pack_bf16x2(v0[8 * u + 2], v0[8 * u + 3]),
                                 pack_bf16x2(v0[8 * u + 4], v0[8 * u + 5]), pack_bf16x2(v0[8 * u + 6], v0[8 * u + 7]));
              zr[4 + u] = make_uint4(pack_bf16x2(v1[8 * u], v1[8 * u + 1]), pack_bf16x2(v1[8 * u + 2], v1[8 * u + 3]),
                                     pack_bf16x2(v1[8 * u + 4], v1[8 * u + 5]), pack_bf16x2(v1[8 * u + 6], v1[8 * u + 7]));
            }
          }
#pragma unroll
          for (int i = 0; i < 32; i += 2) { gelu2_as7126(v0[i], v0[i + 1]); gelu2_as7126(v1[i], v1[i + 1]); }
          stage_bf16x32(buf, r, 0, v0);
          stage_bf16x32(buf, r, 4, v1);
        }
        // chunk complete in shared memory -> one TMA store for the 128 rows
        fence_async_smem();
        named_bar_sync(bar_id, 128);
        if (elect) {
          tma_store_2d(&tmO, col, row0 + ks * M, buf);
          bulk_commit();
        }
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (elect) bulk_wait_all();  // stores complete before the CTA may exit
    if constexpr (EPI == ESM_EPI_RESIDUAL) cp_async_wait<0>();  // (only after an early exit)
    if constexpr (OUT == Act::E4M3) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0 && ea.o_amax) atomic_max_nonneg(ea.o_amax, amax);
    }
  }

  tc_fence_before();
  cluster_sync();  // nobody leaves while the peer may still touch its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Number r of trailing full tiles to split into half-width tiles: the static stride gives
// cluster u the tiles u, u + clusters, ...; with full = 2 units of work and half = 1 the
// r minimising the busiest cluster's work is found by trial (remembered per shape).
int tail_split(int tiles, int clusters) {
  static int last_tiles = -1, last_clusters = -1, last_split = 0;
  if (tiles == last_tiles && clusters == last_clusters) return last_split;
  long best = -1;
  int split = 0;
  for (int r = 0; r <= tiles && r <= 2 * clusters; ++r) {
    const long f = tiles - r, total = f + 2l * r;
    long worst = 0;
    for (int u = 0; u < clusters; ++u) {
      const long nf = f > u ? (f - u + clusters - 1) / clusters : 0;
      const long all = total > u ? (total - u + clusters - 1) / clusters : 0;
      const long w = 2 * nf + (all - nf);
      if (w > worst) worst = w;
    }
    if (best < 0 || worst < best) {
      best = worst;
      split = r;
    }
  }
  last_tiles = tiles;
  last_clusters = clusters;
  last_split = split;
  return split;
}

template <int EPI, bool FP8, Act OUT, bool AMN = false, bool BMN = false>
cudaError_t launch_impl(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmO, int M, int N, int K,
                        const EpiArgs& ea, int num_sms, unsigned* err, cudaStream_t st, int ksplit = 1) {
  auto kern = gemm_tc_kernel<EPI, FP8, OUT, AMN, BMN>;
  static int max_clusters = 0;  // per instantiation: co-resident clusters of two on this device
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Plan<EPI>::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = Plan<EPI>::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess || n <= 0) n = num_sms / 2;
    max_clusters = n;
  }
  const int tiles = ((M + TILE_M - 1) / TILE_M) * (N / BN);
  const int clusters = tiles * ksplit < max_clusters ? tiles * ksplit : max_clusters;
  // Residual epilogue (fp32 chunks of 32 columns): split the last r full tiles into halves
  // when that shortens the longest cluster's work under the static stride.
  const int split = EPI == ESM_EPI_RESIDUAL && ksplit == 1 ? tail_split(tiles, clusters) : 0;
  const int full_tiles = tiles - split, num_tiles = tiles + split;
  const int kb_total = (K + (FP8 ? 127 : 63)) / (FP8 ? 128 : 64);
  const int kb_per = (kb_total + ksplit - 1) / ksplit;
  if (ksplit < 1 || kb_per * (ksplit - 1) >= kb_total) return cudaErrorInvalidValue;  // every split non-empty
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Plan<EPI>::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *tmA, *tmB, *tmO, M, N, kb_total, kb_per, ksplit, full_tiles, num_tiles, ea,
                            err);
}

}  // namespace

int gemm_tc_smem_bytes() { return Plan<ESM_EPI_QKV_ROPE>::kSmemBytes; }
// Rows of the TMA boxes the launched kernel expects: its own 128 rows of A, and its half of
// the 256-wide B tile; the output map's box is 128 bytes of columns by 128 rows.
int gemm_tc_a_box_rows() { return BM; }
int gemm_tc_b_box_rows() { return BN / 2; }
int gemm_tc_out_box_rows() { return 128; }
int gemm_tc_mn_box_rows() { return 64; }

int gemm_tc_max_clusters(int num_sms) { return num_sms / 2; }

cudaError_t launch_gemm_tc_bwd(GemmBwd kind, const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmO,
                               int M, int N, int K, int ksplit, const EpiArgs& ea, int num_sms, unsigned* err,
                               cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  switch (kind) {
    case GemmBwd::DGRAD_F32:
      return launch_impl<ESM_EPI_BIAS_F32, false, Act::F32, false, true>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
    case GemmBwd::DGRAD_BF16:
      return launch_impl<ESM_EPI_QKV_ROPE, false, Act::BF16, false, true>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
    case GemmBwd::DGRAD_GELU:
      return launch_impl<kEpiDgelu, false, Act::BF16, false, true>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
    case GemmBwd::WGRAD_F32:
      return launch_impl<ESM_EPI_BIAS_F32, false, Act::F32, true, true>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st,
                                                                       ksplit);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(esm_epilogue epi, bool fp8, Act out_act, const CUtensorMap* tmA, const CUtensorMap* tmB,
                           const CUtensorMap* tmO, int M, int N, int K, const EpiArgs& ea, int num_sms, unsigned* err,
                           cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (!fp8) {
    switch (epi) {
      case ESM_EPI_BIAS_F32: return launch_impl<ESM_EPI_BIAS_F32, false, Act::F32>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_QKV_ROPE: return launch_impl<ESM_EPI_QKV_ROPE, false, Act::BF16>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_RESIDUAL: return launch_impl<ESM_EPI_RESIDUAL, false, Act::F32>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_GELU: return launch_impl<ESM_EPI_GELU, false, Act::BF16>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
    }
  } else {
    switch (epi) {
      case ESM_EPI_BIAS_F32: return launch_impl<ESM_EPI_BIAS_F32, true, Act::F32>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_QKV_ROPE: return launch_impl<ESM_EPI_QKV_ROPE, true, Act::BF16>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_RESIDUAL: return launch_impl<ESM_EPI_RESIDUAL, true, Act::F32>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
      case ESM_EPI_GELU:
        if (out_act == Act::E4M3)
          return launch_impl<ESM_EPI_GELU, true, Act::E4M3>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
        return launch_impl<ESM_EPI_GELU, true, Act::BF16>(tmA, tmB, tmO, M, N, K, ea, num_sms, err, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace esm
