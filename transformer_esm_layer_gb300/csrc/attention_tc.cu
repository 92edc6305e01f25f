// Variable-length bidirectional attention on the 5th-generation tensor cores (tcgen05),
// head_dim 64, bf16 in, fp32 softmax and accumulation.
//
// Each token attends to every token of its own sequence (hotelren.com guide §3.2: layers
// run over cu_seqlens in thd format; BioNeMo ESM-2 model card: bidirectional encoder):
//   o_t = sum_s softmax_s(q_t . k_s / 8) v_s.
//
// One CTA = one (sequence, 128-query tile, head) work item of the length-ordered list.
//   warp 0      TMA: the Q tile once, then K and V tiles of 128 keys into a 2-stage ring
//               (128-byte rows with the 128-byte swizzle, straight from the packed qkv
//               buffer: x = column of the head, y = token row).
//   warp 1      one thread issues the MMAs:  S = Q K^T  (M=128, N=128, K=64) into TMEM, and
//               O += P V  (M=128, N=64, K=128) with P read from TMEM and V as an MN-major
//               shared-memory operand.  S of tile j+1 is issued before P V of tile j, so the
//               tensor core works while the softmax warps exponentiate.
//   warps 2..5  softmax: thread r owns query row r.  It loads its whole S row from TMEM,
//               masks keys past the sequence end, and keeps a running reference max m with
//               a lazy update: O and the running sum l are rescaled (in TMEM) only when a
//               tile's max exceeds m by more than 8 (in log2 units), so P stays <= 2^8 and
//               most tiles need no rescale.  P = 2^(s*log2e/8 - m) goes back to TMEM as
//               bf16; at the end O / l is written as bf16 (or E4M3 with the FP8 scale).
// Tensor memory: S 128 columns, P 64 (bf16 pairs), O 64 -> 256 columns, so two CTAs share
// an SM and one CTA's softmax overlaps the other's MMAs.  Every mbarrier wait is bounded.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int DH = 64;
constexpr int QT = 128;
constexpr int KT = 128;
constexpr int STG = 2;
constexpr int TILE_BYTES = 128 * 128;  // 128 rows x 128 bytes
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_S = 0, COL_P = 128, COL_O = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct AttnSmem {
  uint64_t q_full;
  uint64_t kv_full[STG];
  uint64_t kv_empty[STG];
  uint64_t s_full, s_free, p_full, pv_done, mma_done;
  uint32_t tmem_base;
  volatile int abort;
};
constexpr int SMEM_BYTES = TILE_BYTES * (1 + 2 * STG) + 1024 + 256;

// 2^x on the special-function unit (the hardware ex2 instruction, flushing subnormal
// results to zero; P values that small are below bf16 resolution of the row sum anyway).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <Act OUT>
__global__ void __launch_bounds__(THREADS, 2)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm, void* __restrict__ o, int d, int heads,
                        PackBuffers pb, const float* q_scale, float* amax_out, unsigned* err) {
  const int item = blockIdx.x / heads;
  const int h = blockIdx.x - item * heads;
  if (item >= *pb.work_count) return;  // whole CTA, before any barrier or TMEM use
  const int seg = pb.work[2 * item];
  const int q0 = pb.work[2 * item + 1];
  const int start = pb.seg_start[seg];
  const int qrows = min(QT, pb.seg_qlen[seg] - q0);
  const int klen = pb.seg_klen[seg];
  const int nkb = (klen + KT - 1) / KT;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = base + TILE_BYTES;                 // stage s: sK + 2*s*TILE_BYTES
  uint8_t* sV = base + 2 * TILE_BYTES;             // stage s: sV + 2*s*TILE_BYTES
  AttnSmem* sm = reinterpret_cast<AttnSmem*>(base + TILE_BYTES * (1 + 2 * STG));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&sm->q_full, 1);
    for (int s = 0; s < STG; ++s) {
      mbar_init(&sm->kv_full[s], 1);
      mbar_init(&sm->kv_empty[s], 1);
    }
    mbar_init(&sm->s_full, 1);
    mbar_init(&sm->s_free, 4);
    mbar_init(&sm->p_full, 4);
    mbar_init(&sm->pv_done, 1);
    mbar_init(&sm->mma_done, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tm);
  if (warp == 1) tmem_alloc(&sm->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(&sm->q_full, TILE_BYTES);
      tma_load_2d(sQ, &tm, h * DH, start + q0, &sm->q_full);
      int issued = 0;
      for (int j = 0; j < nkb && !sm->abort; ++j) {
        const int st = j % STG;
        const uint32_t ph = (uint32_t)(j / STG) & 1u;
        if (!mbar_wait(&sm->kv_empty[st], ph ^ 1u)) {
          latch_error(err, ERRBIT_TIMEOUT);
          sm->abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&sm->kv_full[st], 2 * TILE_BYTES);
        tma_load_2d(sK + 2 * st * TILE_BYTES, &tm, d + h * DH, start + j * KT, &sm->kv_full[st]);
        tma_load_2d(sV + 2 * st * TILE_BYTES, &tm, 2 * d + h * DH, start + j * KT, &sm->kv_full[st]);
        ++issued;
      }
      // wait (bounded) for copies that may still be in flight before the CTA can exit
      mbar_wait(&sm->q_full, 0);
      for (int j = issued - 1; j >= 0 && j >= issued - STG; --j)
        if (!mbar_wait(&sm->kv_full[j % STG], (uint32_t)(j / STG) & 1u)) break;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(QT, KT);
      constexpr uint32_t idesc_pv = idesc_bf16(QT, DH) | (1u << 16);  // B (= V) MN-major
      bool ok = mbar_wait(&sm->q_full, 0);
      auto issue_pv = [&](int i) -> bool {
        if (!mbar_wait(&sm->p_full, (uint32_t)i & 1u)) return false;
        tc_fence_after();
        const uint32_t v0 = smem_u32(sV + 2 * (i % STG) * TILE_BYTES);
#pragma unroll
        for (int k = 0; k < KT / 16; ++k)
          mma_bf16_ts(tmem + COL_O, tmem + COL_P + 8 * k, make_sw128_desc(v0 + 2048 * k), idesc_pv,
                      (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(&sm->pv_done);
        mma_commit(&sm->kv_empty[i % STG]);
        return true;
      };
      for (int j = 0; j < nkb && ok; ++j) {
        const int st = j % STG;
        if (!mbar_wait(&sm->kv_full[st], (uint32_t)(j / STG) & 1u)) { ok = false; break; }
        if (j > 0 && !mbar_wait(&sm->s_free, (uint32_t)(j - 1) & 1u)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sQ);
        const uint32_t b0 = smem_u32(sK + 2 * st * TILE_BYTES);
#pragma unroll
        for (int k = 0; k < DH / 16; ++k)
          mma_bf16_ss(tmem + COL_S, make_sw128_desc(a0 + 32 * k), make_sw128_desc(b0 + 32 * k), idesc_s,
                      k > 0 ? 1u : 0u);
        mma_commit(&sm->s_full);
        if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && nkb > 0) ok = issue_pv(nkb - 1);
      if (!ok) {
        latch_error(err, ERRBIT_TIMEOUT);
        sm->abort = 1;
      }
      mma_commit(&sm->mma_done);
      mbar_wait(&sm->mma_done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = (warp & 3) * 32 + lane;                 // query row of this thread
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float c = 1.4426950408889634f / sqrtf((float)DH);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      if (!mbar_wait_warp(&sm->s_full, (uint32_t)j & 1u)) { ok = false; break; }
      tc_fence_after();
      float s[KT];
#pragma unroll
      for (int ch = 0; ch < KT / 32; ++ch) {
        float v[32];
        tmem_ld32(tmem + lane_off + COL_S + 32 * ch, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * ch + i] = v[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->s_free);
      const int kvalid = klen - j * KT;  // keys >= kvalid lie past the sequence end
      // scale, mask (last tile only) and row max with 8 independent chains
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      if (kvalid >= KT) {
#pragma unroll
        for (int i = 0; i < KT; ++i) {
          s[i] *= c;
          mx[i & 7] = fmaxf(mx[i & 7], s[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < KT; ++i) {
          s[i] = i < kvalid ? s[i] * c : -INFINITY;
          mx[i & 7] = fmaxf(mx[i & 7], s[i]);
        }
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const bool need = mt > m_ref + kRescaleThreshold;
      const float m_new = need ? mt : m_ref;
      const float f = need ? fast_exp2(m_ref - m_new) : 1.f;  // 0 on the first tile
      if (j > 0) {
        if (!mbar_wait_warp(&sm->pv_done, (uint32_t)(j - 1) & 1u)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {  // warp-collective TMEM round trip of O
#pragma unroll
          for (int ch = 0; ch < DH / 32; ++ch) {
            float v[32];
            tmem_ld32(tmem + lane_off + COL_O + 32 * ch, v);
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i] * f);
            tmem_st32(tmem + lane_off + COL_O + 32 * ch, w);
          }
          tmem_st_wait();
        }
      }
      l *= f;
      m_ref = m_new;
      float ls[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ls[i] = 0.f;
#pragma unroll
      for (int ch = 0; ch < KT / 32; ++ch) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(s[32 * ch + 2 * i] - m_ref);
          const float p1 = fast_exp2(s[32 * ch + 2 * i + 1] - m_ref);
          ls[i & 7] += p0 + p1;
          w[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tmem + lane_off + COL_P + 16 * ch, w);
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->p_full);
    }
    if (ok && nkb > 0 && mbar_wait_warp(&sm->pv_done, (uint32_t)(nkb - 1) & 1u)) {
      tc_fence_after();
      float out[DH];
#pragma unroll
      for (int ch = 0; ch < DH / 32; ++ch) {
        float v[32];
        tmem_ld32(tmem + lane_off + COL_O + 32 * ch, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) out[32 * ch + i] = v[i];
      }
      const float inv = 1.f / l;
      if (r < qrows) {
        const size_t off = (size_t)(start + q0 + r) * d + h * DH;
        if constexpr (OUT == Act::BF16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + off);
#pragma unroll
          for (int i = 0; i < DH / 8; ++i) {
            uint4 w;
            w.x = pack_bf16x2(out[8 * i] * inv, out[8 * i + 1] * inv);
            w.y = pack_bf16x2(out[8 * i + 2] * inv, out[8 * i + 3] * inv);
            w.z = pack_bf16x2(out[8 * i + 4] * inv, out[8 * i + 5] * inv);
            w.w = pack_bf16x2(out[8 * i + 6] * inv, out[8 * i + 7] * inv);
            dst[i] = w;
          }
        } else {
          const float qs = __ldg(q_scale);
          float amax = 0.f;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(o) + off);
#pragma unroll
          for (int i = 0; i < DH / 16; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float* f4 = &out[16 * i + 4 * k];
              const float a0 = f4[0] * inv, a1 = f4[1] * inv, a2 = f4[2] * inv, a3 = f4[3] * inv;
              amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))));
              __nv_fp8x4_e4m3 qv(make_float4(a0 * qs, a1 * qs, a2 * qs, a3 * qs));
              w[k] = *reinterpret_cast<uint32_t*>(&qv);
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          atomic_max_nonneg(amax_out, amax);
        }
      }
    } else if (!ok) {
      latch_error(err, ERRBIT_TIMEOUT);
      sm->abort = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int attention_tc_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_attention_tc(const CUtensorMap* tm_qkv, void* o, Act out, int d, int heads, int max_items,
                                const PackBuffers& pb, const float* q_scale, float* amax, unsigned* err,
                                cudaStream_t st) {
  if (max_items <= 0) return cudaSuccess;
  static bool configured[2] = {false, false};
  const int which = out == Act::E4M3 ? 1 : 0;
  if (!configured[which]) {
    cudaError_t e = which ? cudaFuncSetAttribute(attention_tc_kernel<Act::E4M3>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)
                          : cudaFuncSetAttribute(attention_tc_kernel<Act::BF16>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[which] = true;
  }
  const unsigned grid = (unsigned)max_items * (unsigned)heads;
  if (which)
    attention_tc_kernel<Act::E4M3><<<grid, THREADS, SMEM_BYTES, st>>>(*tm_qkv, o, d, heads, pb, q_scale, amax, err);
  else
    attention_tc_kernel<Act::BF16><<<grid, THREADS, SMEM_BYTES, st>>>(*tm_qkv, o, d, heads, pb, q_scale, amax, err);
  return cudaGetLastError();
}

}  // namespace esm
