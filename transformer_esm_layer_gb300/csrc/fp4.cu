// NVFP4 (block-scaled E2M1) GEMM operands and their product on the 5th-generation tensor
// cores (tcgen05.mma kind::mxf4nvf4 with block scaling).
//
// The mlqm.cn walkthrough ("深入源码NVIDIA ESM-2 TransformerEngine优化的实现原理与技术细节",
// section FP8与FP4混合精度支持) gives NVEsmEncoder an fp4_recipe beside the FP8 one; the pages
// give no FP4 format.  Reading (the block-scaled FP4 of the tensor cores): every value is
// E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3,
// 4, 6), every block of 16 consecutive values along the reduction axis has one E4M3 scale,
// and the tensor has one fp32 scale S = 448 * 6 / amax chosen so that the largest block scale
// is representable:
//   sb = E4M3(max|block| / 6 * S),   q = E2M1(x * S / sb)   (0 for an all-zero block),
//   x ~ q * sb / S.
// The GEMM multiplies the E2M1 codes with their block scales on the tensor core (the E4M3
// block scales enter the MMA through tensor memory) and divides by S_A * S_B in the epilogue.
//
// Layouts (this library's):
//   codes  [rows, K / 2] bytes, value k of a row in the low nibble of byte k / 2 for even k;
//   scales one byte per 16 values, in 512-byte atoms of 128 rows x 64 values: atom
//          (row / 128, k / 64) at byte ((row / 128) * (K / 64) + k / 64) * 512, and inside it
//          row r (of the 128) and 16-value block b (of the 4) at (r % 32) * 16 + (r / 32) * 4 + b
//          -- the arrangement each TMEM lane quarter holds as the scale
//          factors of one M = 128 MMA (lane r % 32 of every lane quarter, column r / 32).
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int BM = 128, BN = 256;   // output tile
constexpr int STAGE_K = 256;        // E2M1 values per row per stage (128 bytes)
constexpr int STAGES = 4;
constexpr int ROW_BYTES = 128;
constexpr int A_TILE = BM * ROW_BYTES;       // 16 KB
constexpr int B_TILE = BN * ROW_BYTES;       // 32 KB (two 128-row halves)
constexpr int ATOM_BYTES = 512;              // scales of 128 rows x 64 values
constexpr int SF_ROWS_BYTES = 4 * ATOM_BYTES;   // one 128-row block, the 4 MMA k-steps of a stage
constexpr int EPI_WARPS = 8;                 // two per TMEM lane quarter, one 128-column half each
constexpr int SF_WARP0 = 4;                  // warps 4-7 (lane quarters 0-3) write the scale factors
constexpr int EPI_WARP0 = 8;                 // warps 8-15: epilogue
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
// Registers per thread at launch (65536 / 512) and after setmaxnreg: warpgroups 0 (producer,
// MMA, two idle warps) and 1 (scale-factor warps) give registers to the epilogue warpgroups.
constexpr int kRegsLaunch = 128, kRegsLow = 56, kRegsEpi = 200;
static_assert(2 * 128 * kRegsLow + 2 * 128 * kRegsEpi == THREADS * kRegsLaunch, "register split");
constexpr uint32_t TMEM_COLS = 512;          // accumulator 256 + scale-factor ring STAGES x 48
constexpr uint32_t COL_SF = BN;              // stage s: SFA at +48 s + 4 ks, SFB at +48 s + 16 + 8 ks + 4 h
constexpr uint32_t SF_COLS = 48;
static_assert(COL_SF + SF_COLS * STAGES <= TMEM_COLS, "tensor memory");

struct Fp4Smem {
  uint64_t full[STAGES], empty[STAGES], sf_full[STAGES], acc_full, acc_empty, done;
  uint32_t tmem_base;
  volatile int abort;
};
constexpr int A_OFF = 0, B_OFF = STAGES * A_TILE, SFA_OFF = B_OFF + STAGES * B_TILE,
              SFB_OFF = SFA_OFF + STAGES * SF_ROWS_BYTES, BAR_OFF = SFB_OFF + STAGES * 2 * SF_ROWS_BYTES;
constexpr int SMEM_BYTES = BAR_OFF + 1024 + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory per block");

__device__ __forceinline__ size_t sf_offset(int row, int k16, int K) {
  const int rb = row >> 7, r = row & 127, ks = k16 >> 2, b = k16 & 3;
  return ((size_t)rb * (K / 64) + ks) * ATOM_BYTES + (r & 31) * 16 + (r >> 5) * 4 + b;
}

__device__ __forceinline__ void bf16x8(uint4 u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// max |x| over a bf16 tensor of n8 16-byte units: a grid of a few blocks per SM, four loads in
// flight per thread, one atomic per block.
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const __nv_bfloat16* __restrict__ x, size_t n8,
                                                         float* amax) {
  const uint4* p = reinterpret_cast<const uint4*>(x);
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  float m = 0.f;
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = __ldg(p + i + k * stride);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float f[8];
      bf16x8(u[k], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
    }
  }
  for (; i < n8; i += stride) {
    float f[8];
    bf16x8(__ldg(p + i), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) atomic_max_nonneg(amax, m);
  }
}

// Eight values to E2M1 codes (round to nearest even, saturating at +-6), q[0] in bits 0-3 up
// to q[7] in bits 28-31.
__device__ __forceinline__ uint32_t e2m1x8(const float* q) {
  uint32_t r;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

// One lane per block of 16 values (32 contiguous bytes), one warp per 512 values of a row,
// QSEGS such segments per warp with their loads issued first.  The quotients x S / sb are
// the correctly rounded fp32 quotient of the correctly rounded fp32 product, as two steps:
// x S / sb often lands exactly on an E2M1 midpoint, and a product with the reciprocal alone
// would move it off.  The quotient is y r corrected once by the exact residual y - sb (y r)
// (Markstein's theorem on division through a correctly rounded reciprocal r = RN(1 / sb),
// round to nearest), two values per f32x2 instruction; its sign is that of y (a zero
// residual would otherwise turn -0 into +0).  Checked on GB300 against IEEE division over
// every finite E4M3 divisor sb and every fp32 |y| below 16 sb: identical E2M1 codes, and
// identical quotients for |y| >= sb / 16.  Lanes 4j gather the four scales of their 64-value
// group.  Rows from rows_valid on (the padding to a multiple of 128) quantise as zeros.
// grid (ceil(rows / 8), ceil(ceil(K / 512) / QSEGS)), 256 threads; K a multiple of 16.
template <int QSEGS>
__global__ void __launch_bounds__(256) nvfp4_quantize_kernel(const __nv_bfloat16* __restrict__ x, int rows,
                                                             int rows_valid, int K, const float* amax,
                                                             uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                             float* scale_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  const int nseg = (K + 511) / 512;
  const float a = __ldg(amax);
  const float S = a > 0.f ? (448.f * 6.f) / a : 1.f;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && scale_out) *scale_out = S;
  if (row >= rows) return;  // whole warps
  uint4 u[QSEGS][2];
#pragma unroll
  for (int j = 0; j < QSEGS; ++j) {
    const int k0 = (blockIdx.y * QSEGS + j) * 512 + lane * 16;
    u[j][0] = u[j][1] = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows_valid && k0 < K) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)row * K + k0);
      u[j][0] = __ldg(src);
      u[j][1] = __ldg(src + 1);
    }
  }
#pragma unroll
  for (int j = 0; j < QSEGS; ++j) {
    const int seg = blockIdx.y * QSEGS + j;
    if (seg >= nseg) break;  // the same for the whole warp
    const int k0 = seg * 512 + lane * 16;
    const uint32_t wd[8] = {u[j][0].x, u[j][0].y, u[j][0].z, u[j][0].w, u[j][1].x, u[j][1].y, u[j][1].z, u[j][1].w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(wd[i] << 16);
      v[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
    }
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
    const __nv_fp8_e4m3 sb8(bmax / 6.f * S);  // round to nearest even, saturating at 448
    const float sb = static_cast<float>(sb8);
    uint32_t w0 = 0u, w1 = 0u;
    if (sb > 0.f) {
      const float r = 1.f / sb;
      const uint64_t S2 = f2_pack(S, S), r2 = f2_pack(r, r), nb2 = f2_pack(-sb, -sb);
      float q[16];
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const uint64_t y = f2_mul(f2_pack(v[i], v[i + 1]), S2);
        const uint64_t q0 = f2_mul(y, r2);
        const uint64_t e = f2_fma(q0, nb2, y);
        const uint64_t qs = (f2_fma(e, r2, q0) & 0x7FFFFFFF7FFFFFFFull) | (y & 0x8000000080000000ull);
        f2_unpack(qs, q[i], q[i + 1]);
      }
      w0 = e2m1x8(q);
      w1 = e2m1x8(q + 8);
    }
    if (k0 < K) *reinterpret_cast<uint2*>(codes + (size_t)row * (K / 2) + k0 / 2) = make_uint2(w0, w1);
    const uint32_t s0 = sb8.__x;
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, s0, 1), s2 = __shfl_down_sync(0xffffffffu, s0, 2),
                   s3 = __shfl_down_sync(0xffffffffu, s0, 3);
    if ((lane & 3) == 0 && k0 < K)
      *reinterpret_cast<uint32_t*>(sf + sf_offset(row, k0 / 16, K)) = s0 | s1 << 8 | s2 << 16 | s3 << 24;
  }
}
constexpr int kQuantSegs = 2;

// 1-D bulk copy global -> shared completing `bytes` on the mbarrier (16-byte aligned, size a
// multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Warp-collective: 32 lanes x 16 consecutive 32-bit TMEM columns from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Instruction descriptor, kind::mxf4nvf4 with block scaling: D f32, A and B E2M1 (format 1),
// both K-major, scale factors UE4M3 (scale format 0), scale-factor data ids 0, M x N.
__host__ __device__ constexpr uint32_t idesc_nvfp4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Epilogue: v = acc / (S_A S_B) + bias for the rows below ea.rows_valid, then
//   F32      out fp32 [M, N] = v;          RESIDUAL  out fp32 [M, N] += v;
//   GELU     out bf16 [M, N] = GELU(v) (exact-erf, A&S 7.1.26), and max |out| into ea.amax
//            when given (the next operand's tensor amax);
//   QKV_ROPE out bf16 [M, N] = v, with RoPE on the 64-column heads below ea.rope_cols at the
//            row's position (the library's (cos, sin) table).
template <int EPI>
__device__ __forceinline__ void fp4_epilogue_store(float* v, int row, int col0, int N, const Fp4Epi& ea,
                                                   float& amax) {
  if constexpr (EPI == kFp4F32 || EPI == kFp4Residual) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(ea.out) + (size_t)row * N + col0);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      if constexpr (EPI == kFp4Residual) {
        const float4 x = dst[j];
        o.x += x.x; o.y += x.y; o.z += x.z; o.w += x.w;
      }
      dst[j] = o;
    }
  } else {
    if constexpr (EPI == kFp4Gelu) {
#pragma unroll
      for (int i = 0; i < 64; i += 2) gelu2_as7126(v[i], v[i + 1]);
#pragma unroll
      for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
    } else if (col0 < ea.rope_cols) {
      int p = __ldg(ea.pos_id + row);
      p = p < 0 ? 0 : (p >= ea.max_pos ? ea.max_pos - 1 : p);
      const float4* tab = reinterpret_cast<const float4*>(ea.rope) + p;  // group g at g * max_pos
#pragma unroll
      for (int g = 0; g < 16; ++g) {  // pairs (2g, 2g + 32) and (2g + 1, 2g + 33) turn by their angles
        const float4 t = __ldg(tab + (size_t)g * ea.max_pos);
        const float x0 = v[2 * g], y0 = v[2 * g + 32], x1 = v[2 * g + 1], y1 = v[2 * g + 33];
        v[2 * g] = x0 * t.x - y0 * t.y;
        v[2 * g + 32] = y0 * t.x + x0 * t.y;
        v[2 * g + 1] = x1 * t.z - y1 * t.w;
        v[2 * g + 33] = y1 * t.z + x1 * t.w;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(ea.out) + (size_t)row * N + col0);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      dst[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                          pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
  }
}

// Persistent block-scaled GEMM: one CTA per SM walks the 128 x 256 output tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... (column tiles fastest).  Warp 0 loads A (128 rows) and B (256
// rows) code tiles by TMA and their scale-factor atoms by bulk copy into a STAGES-deep ring.
// Warps 4-7, one per TMEM lane quarter, write each stage's scale factors into tensor memory
// with tcgen05.st (each lane quarter needs its own copy of the 32-row layout the MMA reads);
// a tcgen05.cp per 512-byte atom would occupy the tensor pipe about as long as the MMAs.
// Warp 1 issues the four MMAs of 64 values (M 128, N 256) of a stage once its codes and scale
// factors are in place.  Warps 8-15 (lane quarter warp % 4, 128-column half (warp - 8) / 4)
// load the finished accumulator into registers, hand it back at once, and run the epilogue
// from registers while the next tile accumulates.  A 256-column tile doubles the tensor work
// of a stage for 1.5x its bytes, so the ring holds enough work to cover the delivery latency.
// A half tile past N (N an odd multiple of 128) loads zero-filled codes and no scales and
// stores nothing.
template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const uint8_t* __restrict__ sfa, const uint8_t* __restrict__ sfb, const float* a_scale,
                      const float* b_scale, Fp4Epi ea, int M, int N, int K, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Fp4Smem* sm = reinterpret_cast<Fp4Smem*>(base + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb128 = N / 128;                    // 128-row blocks of B
  const int tiles_n = (nb128 + 1) / 2, tiles = (M / BM) * tiles_n;
  const int kb_total = K / STAGE_K;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm->full[s], 1);
      mbar_init(&sm->empty[s], 1);
      mbar_init(&sm->sf_full[s], 4);  // one arrival per scale-factor warp
    }
    mbar_init(&sm->acc_full, 1);
    mbar_init(&sm->acc_empty, EPI_WARPS);
    mbar_init(&sm->done, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(&sm->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  if (warp < EPI_WARP0) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));

  if (warp == 0) {
    if (lane == 0) {
      // ---- producer
      uint32_t it = 0;
      bool bad = false;
      for (int t = blockIdx.x; t < tiles && !bad; t += gridDim.x) {
        const int m0 = (t / tiles_n) * BM, nb0 = 2 * (t % tiles_n);
        const bool hi_in = nb0 + 1 < nb128;  // the tile's second 128-row block of B exists
        const uint8_t* sa = sfa + (size_t)(m0 / 128) * (K / 64) * ATOM_BYTES;
        const uint8_t* sb0 = sfb + (size_t)nb0 * (K / 64) * ATOM_BYTES;
        const uint32_t bytes = A_TILE + B_TILE + SF_ROWS_BYTES * (hi_in ? 3 : 2);
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          if (sm->abort || !mbar_wait(&sm->empty[s], ((it / STAGES) & 1u) ^ 1u)) {
            bad = true;
            break;
          }
          mbar_arrive_expect_tx(&sm->full[s], bytes);
          tma_load_2d(base + A_OFF + s * A_TILE, &tmA, kb * ROW_BYTES, m0, &sm->full[s]);
          tma_load_2d(base + B_OFF + s * B_TILE, &tmB, kb * ROW_BYTES, nb0 * 128, &sm->full[s]);
          tma_load_2d(base + B_OFF + s * B_TILE + B_TILE / 2, &tmB, kb * ROW_BYTES, nb0 * 128 + 128, &sm->full[s]);
          bulk_load(base + SFA_OFF + s * SF_ROWS_BYTES, sa + (size_t)4 * kb * ATOM_BYTES, SF_ROWS_BYTES,
                    &sm->full[s]);
          bulk_load(base + SFB_OFF + s * 2 * SF_ROWS_BYTES, sb0 + (size_t)4 * kb * ATOM_BYTES, SF_ROWS_BYTES,
                    &sm->full[s]);
          if (hi_in)
            bulk_load(base + SFB_OFF + s * 2 * SF_ROWS_BYTES + SF_ROWS_BYTES,
                      sb0 + ((size_t)(K / 64) + 4 * kb) * ATOM_BYTES, SF_ROWS_BYTES, &sm->full[s]);
        }
      }
      if (bad) {
        if (!sm->abort) latch_error(err, ERRBIT_TIMEOUT);
        sm->abort = 1;
        // copies in flight land before the CTA may exit (bounded): the last STAGES issued
        for (uint32_t k = it; k > 0 && k + STAGES > it; --k)
          if (!mbar_wait(&sm->full[(k - 1) % STAGES], ((k - 1) / STAGES) & 1u)) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idesc = idesc_nvfp4(BM, BN);
      const uint64_t adesc0 = make_sw128_desc(smem_u32(base + A_OFF));
      const uint64_t bdesc0 = make_sw128_desc(smem_u32(base + B_OFF));
      uint32_t it = 0, j = 0;
      bool bad = false;
      for (int t = blockIdx.x; t < tiles && !bad; t += gridDim.x, ++j) {
        if (sm->abort || !mbar_wait(&sm->acc_empty, (j & 1u) ^ 1u)) {
          bad = true;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          // the stage's codes have landed and its scale factors are in tensor memory
          if (sm->abort || !mbar_wait(&sm->full[s], (it / STAGES) & 1u) ||
              !mbar_wait(&sm->sf_full[s], (it / STAGES) & 1u)) {
            bad = true;
            break;
          }
          tc_fence_after();
          const uint32_t sf_col = tmem + COL_SF + SF_COLS * (uint32_t)s;
          const uint64_t ad = adesc0 + (uint64_t)((s * A_TILE) >> 4);
          const uint64_t bd = bdesc0 + (uint64_t)((s * B_TILE) >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {  // 64 values = 32 bytes of each 128-byte row
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.b32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
                "p;\n\t}" ::"r"(tmem),
                "l"(ad + (uint64_t)(2 * ks)), "l"(bd + (uint64_t)(2 * ks)), "r"(idesc), "r"(sf_col + 4 * ks),
                "r"(sf_col + 16 + 8 * ks), "r"((kb | ks) != 0 ? 1u : 0u)
                : "memory");
          }
          mma_commit(&sm->empty[s]);
        }
        if (bad) break;
        mma_commit(&sm->acc_full);
      }
      if (bad) {
        if (!sm->abort) latch_error(err, ERRBIT_TIMEOUT);
        sm->abort = 1;
      }
      mma_commit(&sm->done);  // completes once every MMA issued above has finished
    }
  } else if (warp >= SF_WARP0 && warp < EPI_WARP0) {
    // ---- scale-factor warps: lane quarter q = warp & 3.  TMEM columns of stage s (48): SFA
    // k-step ks at +4 ks, SFB rows 128 h.. of k-step ks at +16 + 8 ks + 4 h; in each, lane
    // 32 q + i holds the 16 bytes of row i of the 512-byte atom (the scales of rows i, 32 + i,
    // 64 + i, 96 + i, four per row), the same in every lane quarter.
    uint32_t it = 0;
    bool bad = false;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    for (int t = blockIdx.x; t < tiles && !bad; t += gridDim.x) {
      for (int kb = 0; kb < kb_total; ++kb, ++it) {
        const int s = (int)(it % STAGES);
        if (sm->abort || !mbar_wait_warp(&sm->full[s], (it / STAGES) & 1u)) {
          bad = true;
          break;
        }
        const uint8_t* sfa_s = base + SFA_OFF + s * SF_ROWS_BYTES + 16 * lane;
        const uint8_t* sfb_s = base + SFB_OFF + s * 2 * SF_ROWS_BYTES + 16 * lane;
        const uint32_t col = tmem + lane_off + COL_SF + SF_COLS * (uint32_t)s;
        uint32_t r[16];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {  // SFA: columns +0..15
          const uint4 u = *reinterpret_cast<const uint4*>(sfa_s + ks * ATOM_BYTES);
          r[4 * ks] = u.x; r[4 * ks + 1] = u.y; r[4 * ks + 2] = u.z; r[4 * ks + 3] = u.w;
        }
        tmem_st16(col, r);
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // SFB: columns +16..31 (ks 0, 1), +32..47 (ks 2, 3)
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 u =
                  *reinterpret_cast<const uint4*>(sfb_s + h * SF_ROWS_BYTES + (2 * part + k2) * ATOM_BYTES);
              const int o = 8 * k2 + 4 * h;
              r[o] = u.x; r[o + 1] = u.y; r[o + 2] = u.z; r[o + 3] = u.w;
            }
          tmem_st16(col + 16 + 16 * part, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->sf_full[s]);
      }
    }
    if (bad && lane == 0) {
      if (!sm->abort) latch_error(err, ERRBIT_TIMEOUT);
      sm->abort = 1;
    }
  } else if (warp >= EPI_WARP0) {
    // ---- epilogue warps: 32 rows x 128 columns each
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    const int quarter = warp & 3, half = (warp - EPI_WARP0) >> 2;
    const float inv = 1.f / (__ldg(a_scale) * __ldg(b_scale));
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float amax = 0.f;
    uint32_t j = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++j) {
      if constexpr (EPI == kFp4Residual) {  // this row's residual towards L2 while the tile accumulates
        const int prow = (t / tiles_n) * BM + quarter * 32 + lane, pcol = (t % tiles_n) * BN + 128 * half;
        if (prow < ea.rows_valid && pcol < N) {
          const float* xr = static_cast<const float*>(ea.out) + (size_t)prow * N + pcol;
#pragma unroll
          for (int c = 0; c < 4; ++c) prefetch_l2(xr + 32 * c);  // 4 x 128 bytes
        }
      }
      if (!mbar_wait_warp(&sm->acc_full, j & 1u)) {
        if (lane == 0) {
          if (!sm->abort) latch_error(err, ERRBIT_TIMEOUT);
          sm->abort = 1;
        }
        break;
      }
      tc_fence_after();
      float v[128];
      {
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tmem + lane_off + (uint32_t)(128 * half + 32 * c), r[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait_regs(r[c]);  // one wait; each array tied to it
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[c][i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->acc_empty);  // the accumulator is free for the next tile
      const int row = (t / tiles_n) * BM + quarter * 32 + lane;
      const int col_h = (t % tiles_n) * BN + 128 * half;
      if (col_h >= N || row >= ea.rows_valid) continue;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float* vh = v + 64 * hh;
        const int col0 = col_h + 64 * hh;
        if (ea.bias) {  // 16-byte aligned (checked on the host), eight bf16 per load
          const uint4* bp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ea.bias) + col0);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 u = __ldg(bp + g);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              vh[8 * g + 2 * k] = vh[8 * g + 2 * k] * inv + __uint_as_float(w[k] << 16);
              vh[8 * g + 2 * k + 1] = vh[8 * g + 2 * k + 1] * inv + __uint_as_float(w[k] & 0xFFFF0000u);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) vh[i] *= inv;
        }
        fp4_epilogue_store<EPI>(vh, row, col0, N, ea, amax);
      }
    }
    if constexpr (EPI == kFp4Gelu) {
      if (ea.amax) {  // of the bf16 outputs: rounding is monotone, so round the maximum
        amax = __bfloat162float(__float2bfloat16_rn(amax));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) atomic_max_nonneg(ea.amax, amax);
      }
    }
  }
  __syncwarp();
  if (warp == 1) {  // every MMA has finished before its tensor memory is released
    if (!mbar_wait_warp(&sm->done, 0) && lane == 0) latch_error(err, ERRBIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_nvfp4_quantize(const __nv_bfloat16* x, int rows, int rows_valid, int K, uint8_t* codes,
                                  uint8_t* sf, float* amax, float* scale, bool amax_ready, int num_sms,
                                  cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const size_t n8 = (size_t)rows_valid * K / 8;
  if (!amax_ready) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  if (!amax_ready && n8 > 0) {
    const size_t need = (n8 + 1023) / 1024;  // at least four units per thread
    const int grid = (int)(need < (size_t)num_sms * 8 ? need : (size_t)num_sms * 8);
    nvfp4_amax_kernel<<<grid, 256, 0, st>>>(x, n8, amax);
  }
  const int nseg = (K + 511) / 512;
  const dim3 grid((unsigned)((rows + 7) / 8), (unsigned)((nseg + kQuantSegs - 1) / kQuantSegs));
  nvfp4_quantize_kernel<kQuantSegs><<<grid, 256, 0, st>>>(x, rows, rows_valid, K, amax, codes, sf, scale);
  return cudaGetLastError();
}

int gemm_nvfp4_smem_bytes() { return SMEM_BYTES; }

template <int EPI>
static cudaError_t launch_epi(const CUtensorMap* tmA, const CUtensorMap* tmB, const uint8_t* sfa, const uint8_t* sfb,
                              const float* a_scale, const float* b_scale, const Fp4Epi& ea, int M, int N, int K,
                              int num_sms, unsigned* err, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_nvfp4_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long tiles = (long long)(M / BM) * ((N / 128 + 1) / 2);
  const unsigned grid = (unsigned)(tiles < num_sms ? tiles : num_sms);
  gemm_nvfp4_kernel<EPI><<<grid, THREADS, SMEM_BYTES, st>>>(*tmA, *tmB, sfa, sfb, a_scale, b_scale, ea, M, N, K, err);
  return cudaGetLastError();
}

cudaError_t launch_gemm_nvfp4(int epi, const CUtensorMap* tmA, const CUtensorMap* tmB, const uint8_t* sfa,
                              const uint8_t* sfb, const float* a_scale, const float* b_scale, const Fp4Epi& ea, int M,
                              int N, int K, int num_sms, unsigned* err, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (num_sms <= 0) return cudaErrorInvalidValue;
  switch (epi) {
    case kFp4F32: return launch_epi<kFp4F32>(tmA, tmB, sfa, sfb, a_scale, b_scale, ea, M, N, K, num_sms, err, st);
    case kFp4Residual:
      return launch_epi<kFp4Residual>(tmA, tmB, sfa, sfb, a_scale, b_scale, ea, M, N, K, num_sms, err, st);
    case kFp4Gelu: return launch_epi<kFp4Gelu>(tmA, tmB, sfa, sfb, a_scale, b_scale, ea, M, N, K, num_sms, err, st);
    case kFp4QkvRope:
      return launch_epi<kFp4QkvRope>(tmA, tmB, sfa, sfb, a_scale, b_scale, ea, M, N, K, num_sms, err, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace esm
