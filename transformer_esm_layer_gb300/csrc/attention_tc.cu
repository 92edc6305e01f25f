// Variable-length bidirectional attention on the 5th-generation tensor cores (tcgen05),
// head_dim 64, bf16 in, fp32 softmax and accumulation.
//
// Each token attends to every token of its own sequence (hotelren.com guide §3.2: layers
// run over cu_seqlens in thd format; BioNeMo ESM-2 model card: bidirectional encoder):
//   o_t = sum_s softmax_s(q_t . k_s / 8) v_s.
//
// Persistent: two CTAs per SM walk the (sequence, 128-query tile, head) work items of the
// length-ordered list in rounds of one item per CTA, in snake order; barrier phases run on
// across items.
//   warp 0      TMA: each item's Q tile (double-buffered, 128-byte swizzle) and its K tiles
//               of 128 keys into a 2-stage ring, straight from the packed qkv buffer
//               (x = column of the head, y = token row);
//   warp 2      TMA: the V tiles into their own 2-stage ring (a V stage frees only after its
//               P V, a K stage right after its S, so K runs ahead of V).
//   warp 1      one thread issues S(g) = Q K^T (M=128, N=128, K=64) into TMEM for the
//               global sequence of key tiles g, each as soon as its operands are ready;
//   warp 3      one thread issues O += P V (M=128, N=64, K=128; P read from TMEM, V an
//               MN-major shared-memory operand) for the same sequence.  Two issuers keep a
//               ready S from waiting behind the P V MMAs the pipe is still accepting.
//   warps 4..7  softmax (warpgroup 1, register budget raised with setmaxnreg): thread r owns
//               query row r.  It reads its whole S row (128 scores) from TMEM into registers
//               and immediately releases S, so the tensor core computes S(g+1) while this
//               tile is exponentiated.  Keys past the sequence end are masked; a running
//               reference max m is updated lazily: O and the running sum l are rescaled (in
//               TMEM) only when a tile's max exceeds m by more than 8 (log2 units), so
//               P <= 2^8.  P = 2^(s*log2e/8 - m) goes back to TMEM as bf16.  After an item's
//               last tile O / l is written (bf16, or E4M3 with the FP8 scale) into the
//               item's Q buffer, which the last S has finished reading, and each warp stores
//               its 32 rows with coalesced 16-byte stores; only then is the Q buffer handed
//               back to the TMA warp.
// Tensor memory: S 128 columns, P 64 (bf16 pairs), O 64 -> 256 columns per CTA.  Every
// mbarrier wait is bounded.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int DH = 64;
constexpr int QT = 128;
constexpr int KT = 128;
constexpr int STG = 2;
constexpr int TILE_BYTES = 128 * 128;  // 128 rows x 128 bytes
constexpr int THREADS = 256;
// Register budget per thread at launch (2 CTAs of 256 threads per SM) and after the
// warpgroup-wide setmaxnreg: warpgroup 0 (TMA, MMA) gives up registers to warpgroup 1
// (softmax), 128 * kRegsWg0 + 128 * kRegsWg1 = 256 * kRegsLaunch.
constexpr int kRegsLaunch = 128, kRegsWg0 = 56, kRegsWg1 = 200;
static_assert(128 * kRegsWg0 + 128 * kRegsWg1 == THREADS * kRegsLaunch, "register split");
constexpr int CTAS_PER_SM = 2;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_S = 0, COL_P = 128, COL_O = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct AttnSmem {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[STG], k_empty[STG];  // K tile landed / read by its S = Q K^T
  uint64_t v_full[STG], v_empty[STG];  // V tile landed / read by its O += P V
  uint64_t s_full, s_free, p_full, pv_done, mma_done, pv_fin;
  uint32_t tmem_base;
  volatile int abort;
};
// [Q0][Q1][K0][V0][K1][V1] then the barriers
constexpr int SMEM_BYTES = TILE_BYTES * (2 + 2 * STG) + 1024 + 256;

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

// 16-byte unit j of row r of a 128-row x 128-byte staging tile, XOR-swizzled by row so the
// row-per-thread writes and the rows-per-instruction reads are both conflict-free.
__device__ __forceinline__ uint32_t stage_off(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

// max of three (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

struct Item {
  int qrow0, qrows, krow0, klen, nkb, h;
};

// Work item `it` = (work-list entry it / heads, head it % heads); one 16-byte load.
__device__ __forceinline__ int4 load_item(const PackBuffers& pb, int it, int heads) {
  return __ldg(reinterpret_cast<const int4*>(pb.work) + it / heads);
}
__device__ __forceinline__ Item make_item(int4 w, int it, int heads) {
  Item x;
  x.h = it % heads;
  x.qrow0 = w.x;
  x.qrows = w.y;
  x.krow0 = w.z;
  x.klen = w.w;
  x.nkb = (x.klen + KT - 1) / KT;
  return x;
}

// AMAX: a bf16 output also records its max |value| into amax_out (compiled only into the
// instantiation that needs it, so the others keep their registers).
template <Act OUT, bool AMAX = false>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm, void* __restrict__ o, int d, int heads,
                        PackBuffers pb, const float* q_scale, float* amax_out, float* __restrict__ lse,
                        int lse_stride, unsigned* err) {
  const int n_items = *pb.work_count * heads;
  if ((int)blockIdx.x >= n_items) return;  // whole CTA, before any barrier or TMEM use

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                       // buffer b: sQ + b * TILE_BYTES
  uint8_t* sK = base + 2 * TILE_BYTES;      // stage s: sK + 2 * s * TILE_BYTES
  uint8_t* sV = base + 3 * TILE_BYTES;      // stage s: sV + 2 * s * TILE_BYTES
  AttnSmem* sm = reinterpret_cast<AttnSmem*>(base + TILE_BYTES * (2 + 2 * STG));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Items in rounds of gridDim.x, snake order: even rounds give CTA c item c of the round,
  // odd rounds item gridDim.x - 1 - c (the list is longest first, so this evens out loads).
  auto item_at = [&](int rnd) -> int {
    return rnd * (int)gridDim.x + ((rnd & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
  };
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->q_full[b], 1);
      mbar_init(&sm->q_empty[b], 4);  // one arrival per softmax warp after its O rows are out
    }
    for (int s = 0; s < STG; ++s) {
      mbar_init(&sm->k_full[s], 1);
      mbar_init(&sm->k_empty[s], 1);
      mbar_init(&sm->v_full[s], 1);
      mbar_init(&sm->v_empty[s], 1);
    }
    mbar_init(&sm->s_full, 1);
    mbar_init(&sm->s_free, 4);
    mbar_init(&sm->p_full, 4);
    mbar_init(&sm->pv_done, 1);
    mbar_init(&sm->mma_done, 1);
    mbar_init(&sm->pv_fin, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tm);
  if (warp == 1) tmem_alloc(&sm->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWg0));

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers
    // Warp 0 loads each item's Q and its K tiles, warp 2 its V tiles: a K stage is free as
    // soon as its S is done, a V stage only after its P V, so K never waits behind V.
    if (lane == 0) {
      const bool kq = warp == 0;
      int g = 0, qi = 0;
      int4 nxt = load_item(pb, item_at(0), heads);
      for (int rnd = 0, it = item_at(0); it < n_items && !sm->abort; it = item_at(++rnd), ++qi) {
        const Item x = make_item(nxt, it, heads);
        if (item_at(rnd + 1) < n_items) nxt = load_item(pb, item_at(rnd + 1), heads);  // prefetch
        if (kq) {
          const int qb = qi & 1;
          if (!mbar_wait(&sm->q_empty[qb], ((uint32_t)(qi >> 1) & 1u) ^ 1u)) {
            latch_error(err, ERRBIT_TIMEOUT);
            sm->abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&sm->q_full[qb], TILE_BYTES);
          tma_load_2d(sQ + qb * TILE_BYTES, &tm, x.h * DH, x.qrow0, &sm->q_full[qb]);
        }
        uint64_t* empty = kq ? sm->k_empty : sm->v_empty;
        uint64_t* full = kq ? sm->k_full : sm->v_full;
        uint8_t* dst0 = kq ? sK : sV;
        const int xcol = (kq ? d : 2 * d) + x.h * DH;
        for (int j = 0; j < x.nkb; ++j, ++g) {
          const int st = g % STG;
          if (!mbar_wait(&empty[st], ((uint32_t)(g / STG) & 1u) ^ 1u)) {
            latch_error(err, ERRBIT_TIMEOUT);
            sm->abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[st], TILE_BYTES);
          tma_load_2d(dst0 + 2 * st * TILE_BYTES, &tm, xcol, x.krow0 + j * KT, &full[st]);
        }
      }
      // Copies still in flight can only exist if a consumer gave up early: then the last
      // STG stages are waited for (bounded) before the CTA exits.
      if (sm->abort) {
        uint64_t* full = kq ? sm->k_full : sm->v_full;
        for (int k = g - 1; k >= 0 && k >= g - STG; --k)
          if (!mbar_wait(&full[k % STG], (uint32_t)(k / STG) & 1u)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads issue to the one tensor pipe: warp 1 every S = Q K^T, warp 3 every
    // O += P V, each in tile order and each blocking only on its own operands.  An issuing
    // thread is held until the pipe accepts its MMA, so with one issuer an S that was ready
    // waited behind the eight P V MMAs before it (and a ready P V behind an S).
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(QT, KT);
      constexpr uint32_t idesc_pv = idesc_bf16(QT, DH) | (1u << 16);  // B (= V) MN-major
      const bool is_s = warp == 1;
      const uint64_t qdesc0 = make_sw128_desc(smem_u32(sQ));  // buffer b: + b * (TILE_BYTES >> 4)
      const uint64_t kdesc0 = make_sw128_desc(smem_u32(sK));  // stage s: + 2 s (TILE_BYTES >> 4)
      const uint64_t vdesc0 = make_sw128_desc(smem_u32(sV));
      bool ok = true;
      int g = 0, qi = 0;
      int4 nxt = load_item(pb, item_at(0), heads);
      for (int rnd = 0, it = item_at(0); it < n_items && ok && !sm->abort; it = item_at(++rnd), ++qi) {
        const Item x = make_item(nxt, it, heads);
        if (item_at(rnd + 1) < n_items) nxt = load_item(pb, item_at(rnd + 1), heads);  // prefetch
        const int qb = qi & 1;
        for (int j = 0; j < x.nkb; ++j, ++g) {
          const int st = g % STG;
          if (is_s) {
            // the K tile has landed, the previous S has been read, the item's Q has landed
            if (!mbar_wait(&sm->k_full[st], (uint32_t)(g / STG) & 1u) ||
                (g > 0 && !mbar_wait(&sm->s_free, (uint32_t)(g - 1) & 1u)) ||
                (j == 0 && !mbar_wait(&sm->q_full[qb], (uint32_t)(qi >> 1) & 1u))) {
              ok = false;
              break;
            }
            tc_fence_after();
            // descriptor arithmetic on the low word (the start-address field cannot carry)
            const uint32_t alo = (uint32_t)qdesc0 + (uint32_t)((qb * TILE_BYTES) >> 4);
            const uint32_t blo = (uint32_t)kdesc0 + (uint32_t)((2 * st * TILE_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < DH / 16; ++k)  // 16 dims = 32 bytes of each 128-byte row
              mma_bf16_ss(tmem + COL_S, (qdesc0 & 0xFFFFFFFF00000000ull) | (uint64_t)(alo + 2u * (uint32_t)k),
                          (kdesc0 & 0xFFFFFFFF00000000ull) | (uint64_t)(blo + 2u * (uint32_t)k), idesc_s,
                          k > 0 ? 1u : 0u);
            mma_commit(&sm->s_full);
            mma_commit(&sm->k_empty[st]);
          } else {
            // P of this tile is in tensor memory and its V tile has landed
            if (!mbar_wait(&sm->p_full, (uint32_t)g & 1u) || !mbar_wait(&sm->v_full[st], (uint32_t)(g / STG) & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t vlo = (uint32_t)vdesc0 + (uint32_t)((2 * st * TILE_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < KT / 16; ++k)  // 16 keys = 16 rows of V = 2048 bytes
              mma_bf16_ts(tmem + COL_O, tmem + COL_P + 8 * k,
                          (vdesc0 & 0xFFFFFFFF00000000ull) | (uint64_t)(vlo + 128u * (uint32_t)k), idesc_pv,
                          (j > 0 || k > 0) ? 1u : 0u);
            mma_commit(&sm->pv_done);
            mma_commit(&sm->v_empty[st]);
          }
        }
      }
      if (!ok) {
        latch_error(err, ERRBIT_TIMEOUT);
        sm->abort = 1;
      }
      // every MMA of this thread has completed before tensor memory may be released
      uint64_t* fin = is_s ? &sm->mma_done : &sm->pv_fin;
      mma_commit(fin);
      mbar_wait(fin, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWg1));
    const int wq = warp & 3;                                // TMEM lane quarter
    const int r = wq * 32 + lane;                           // query row of this thread
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = 1.4426950408889634f / sqrtf((float)DH);
    const float qs = (OUT == Act::E4M3) ? __ldg(q_scale) : 1.f;
    float amax = 0.f;
    bool ok = true;
    int g = 0, qi = 0;
    int4 nxt = load_item(pb, item_at(0), heads);
    for (int rnd = 0, it = item_at(0); it < n_items && ok; it = item_at(++rnd), ++qi) {
      const Item x = make_item(nxt, it, heads);
      if (item_at(rnd + 1) < n_items) nxt = load_item(pb, item_at(rnd + 1), heads);  // prefetch
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < x.nkb; ++j, ++g) {
        if (!mbar_wait_warp(&sm->s_full, (uint32_t)g & 1u)) { ok = false; break; }
        tc_fence_after();
        // the whole S row into registers; S is then free for the next tile's Q K^T
        float sv[KT];
        {
          uint32_t su[KT / 32][32];
#pragma unroll
          for (int ch = 0; ch < KT / 32; ++ch) tmem_ld32_nowait(tmem + lane_off + COL_S + 32 * ch, su[ch]);
#pragma unroll
          for (int ch = 0; ch < KT / 32; ++ch) tmem_ld_wait_regs(su[ch]);
#pragma unroll
          for (int i = 0; i < KT; ++i) sv[i] = __uint_as_float(su[i >> 5][i & 31]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->s_free);
        const int kvalid = x.klen - j * KT;  // keys >= kvalid lie past the sequence end
        if (kvalid < KT) {
#pragma unroll
          for (int i = 0; i < KT; ++i) sv[i] = i < kvalid ? sv[i] : -INFINITY;
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < KT; i += 8) {
          mx[0] = fmax3(mx[0], sv[i], sv[i + 1]);
          mx[1] = fmax3(mx[1], sv[i + 2], sv[i + 3]);
          mx[2] = fmax3(mx[2], sv[i + 4], sv[i + 5]);
          mx[3] = fmax3(mx[3], sv[i + 6], sv[i + 7]);
        }
        const float mt = c * fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
        const bool need = mt > m_ref + kRescaleThreshold;
        const float m_new = need ? mt : m_ref;
        const float f = need ? fast_exp2(m_ref - m_new) : 1.f;  // 0 on the first tile
        l *= f;
        m_ref = m_new;
        // P = 2^(s*c - m) (hardware ex2) as bf16 pairs, computed while the previous P V may
        // still be reading the P columns
        // (scale-subtract and row sums two scores per f32x2 instruction)
        const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_ref, -m_ref);
        uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
        uint32_t w[KT / 32][16];
#pragma unroll
        for (int ch = 0; ch < KT / 32; ++ch) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float p0, p1;
            f2_unpack(f2_fma(f2_pack(sv[32 * ch + 2 * i], sv[32 * ch + 2 * i + 1]), c2, nm2), p0, p1);
            p0 = fast_exp2(p0);
            p1 = fast_exp2(p1);
            ls2[i & 1] = f2_add(ls2[i & 1], f2_pack(p0, p1));
            w[ch][i] = pack_bf16x2(p0, p1);
          }
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(ls2[0], a0, a1);
          f2_unpack(ls2[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        // P (and, within an item, O) may be rewritten once the previous P V is done
        if (g > 0) {
          if (!mbar_wait_warp(&sm->pv_done, (uint32_t)(g - 1) & 1u)) { ok = false; break; }
          tc_fence_after();
        }
#pragma unroll
        for (int ch = 0; ch < KT / 32; ++ch) tmem_st16(tmem + lane_off + COL_P + 16 * ch, w[ch]);
        if (j > 0 && __any_sync(0xffffffffu, need)) {  // warp-collective TMEM round trip of O
#pragma unroll
          for (int ch = 0; ch < DH / 16; ++ch) {
            float v[16];
            tmem_ld16(tmem + lane_off + COL_O + 16 * ch, v);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i] * f);
            tmem_st16(tmem + lane_off + COL_O + 16 * ch, w);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->p_full);
      }
      if (!ok) break;
      // ---- item epilogue: O / l through this item's Q buffer (the last S has read it) to
      // global memory, 16 bytes per lane covering whole output rows per instruction
      if (!mbar_wait_warp(&sm->pv_done, (uint32_t)(g - 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      uint32_t u[2][32];
      tmem_ld32_nowait(tmem + lane_off + COL_O, u[0]);
      tmem_ld32_nowait(tmem + lane_off + COL_O + 32, u[1]);
      tmem_ld_wait_regs(u[0]);
      tmem_ld_wait_regs(u[1]);
      tc_fence_before();
      const float inv = 1.f / l;
      // training forward: the natural-log softmax normaliser of this row and head (scores
      // scaled by 1/sqrt(dh)), ln 2 * (m + log2 l) in the base-2 units used above
      if (lse != nullptr && r < x.qrows) lse[(size_t)x.h * lse_stride + x.qrow0 + r] = 0.6931471805599453f * (m_ref + log2f(l));
      uint8_t* stage = sQ + (qi & 1) * TILE_BYTES;
      constexpr int kUnits = (OUT == Act::BF16) ? 8 : 4;  // 16-byte units per output row
      if constexpr (OUT == Act::BF16) {
        if (AMAX && r < x.qrows) {  // max |O| of this row: max |acc| / l
          float m = 0.f;
#pragma unroll
          for (int i = 0; i < DH; ++i) m = fmaxf(m, fabsf(__uint_as_float(u[i >> 5][i & 31])));
          amax = fmaxf(amax, m * inv);
        }
#pragma unroll
        for (int i = 0; i < DH / 8; ++i) {
          const uint32_t* w = &u[i >> 2][(i & 3) * 8];
          uint4 q;
          q.x = pack_bf16x2(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv);
          q.y = pack_bf16x2(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv);
          q.z = pack_bf16x2(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv);
          q.w = pack_bf16x2(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv);
          *reinterpret_cast<uint4*>(stage + stage_off(r, i)) = q;
        }
      } else {
#pragma unroll
        for (int i = 0; i < DH / 16; ++i) {
          uint32_t w4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t* w = &u[i >> 1][(i & 1) * 16 + 4 * k];
            const float a0 = __uint_as_float(w[0]) * inv, a1 = __uint_as_float(w[1]) * inv;
            const float a2 = __uint_as_float(w[2]) * inv, a3 = __uint_as_float(w[3]) * inv;
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))));
            __nv_fp8x4_e4m3 qv(make_float4(a0 * qs, a1 * qs, a2 * qs, a3 * qs));
            w4[k] = *reinterpret_cast<uint32_t*>(&qv);
          }
          *reinterpret_cast<uint4*>(stage + stage_off(r, i)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      __syncwarp();
      {
        constexpr int kRowsPerInst = 32 / kUnits;
        constexpr size_t kElem = (OUT == Act::BF16) ? 2 : 1;
        uint8_t* ob = static_cast<uint8_t*>(o);
#pragma unroll
        for (int i = 0; i < 32 / kRowsPerInst; ++i) {
          const int rr = wq * 32 + i * kRowsPerInst + lane / kUnits;
          const int un = lane % kUnits;
          const uint4 v = *reinterpret_cast<const uint4*>(stage + stage_off(rr, un));
          if (rr < x.qrows)
            *reinterpret_cast<uint4*>(ob + ((size_t)(x.qrow0 + rr) * d + (size_t)x.h * DH) * kElem + 16 * un) = v;
        }
      }
      // generic-proxy accesses of the Q buffer are ordered before the next TMA write to it
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->q_empty[qi & 1]);
    }
    if (!ok) {
      latch_error(err, ERRBIT_TIMEOUT);
      sm->abort = 1;
    }
    if constexpr (OUT == Act::E4M3 || AMAX) {
      // a bf16 output's amax is that of the rounded values: rounding is monotone, so round the max
      if constexpr (OUT == Act::BF16) amax = __bfloat162float(__float2bfloat16_rn(amax));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      if (lane == 0) atomic_max_nonneg(amax_out, amax);
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
                                cudaStream_t st, float* lse, int lse_stride) {
  if (max_items <= 0) return cudaSuccess;
  static int num_sms = 0;
  static bool configured[3] = {false, false, false};
  const int which = out == Act::E4M3 ? 1 : (amax != nullptr ? 2 : 0);
  if (!configured[which]) {
    cudaError_t e = which == 1 ? cudaFuncSetAttribute(attention_tc_kernel<Act::E4M3>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)
                    : which == 2 ? cudaFuncSetAttribute(attention_tc_kernel<Act::BF16, true>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)
                                 : cudaFuncSetAttribute(attention_tc_kernel<Act::BF16>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[which] = true;
  }
  if (num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || num_sms <= 0)
      num_sms = 148;
  }
  // persistent: at most CTAS_PER_SM CTAs per SM; CTAs past the (device-side) item count exit
  const long long items = (long long)max_items * heads;
  const long long cap = (long long)CTAS_PER_SM * num_sms;
  const unsigned grid = (unsigned)(items < cap ? items : cap);
  if (which == 1)
    attention_tc_kernel<Act::E4M3><<<grid, THREADS, SMEM_BYTES, st>>>(*tm_qkv, o, d, heads, pb, q_scale, amax, lse,
                                                                      lse_stride, err);
  else if (which == 2)
    attention_tc_kernel<Act::BF16, true><<<grid, THREADS, SMEM_BYTES, st>>>(*tm_qkv, o, d, heads, pb, q_scale, amax,
                                                                            lse, lse_stride, err);
  else
    attention_tc_kernel<Act::BF16><<<grid, THREADS, SMEM_BYTES, st>>>(*tm_qkv, o, d, heads, pb, q_scale, amax, lse,
                                                                      lse_stride, err);
  return cudaGetLastError();
}

}  // namespace esm
