// Backward of the variable-length bidirectional attention on the tcgen05 tensor cores
// (head_dim 64, bf16 operands, fp32 accumulation): the gradient step of the packed layer
// stack that the hotelren.com guide trains over cu_seqlens (§3.2, §6).
//
// With S = Q K^T / 8, P = softmax(S) (rows: queries), O = P V and dO given, per head:
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D) with D_i = sum_c dO_ic O_ic,
//   dK = dS^T Q / 8,  dQ = dS K / 8.
// P is rebuilt from the forward's log-sum-exp (no softmax pass over the keys here).
//
// One CTA per SM walks the work items (sequence, 128-key tile, head) of the forward's work
// list (a forward query tile is, in packed self-attention, also a key tile: its rows, and
// the sequence's row range).  For each item it holds K and V in shared memory and loops
// over the sequence's 128-query tiles; TMEM lanes are keys throughout:
//   S^T  = K Q^T        (M=128 keys, N=128 queries, K=64)        TMEM cols [0,128)
//   dP^T = V dO^T       (M=128, N=128, K=64)                       cols [128,256)
//   dV  += P^T dO       (M=128, N=64, K=128; dO MN-major)          cols [384,448)
//   dK  += dS^T Q       (M=128, N=64, K=128; Q MN-major)           cols [320,384)
//   dQ_i = dS K         (M=128 queries, N=64, K=128 keys; dS and K MN-major)  cols [256,320)
// Roles (512 threads; registers rebalanced per warpgroup with setmaxnreg):
//   warp 0       TMA: the item's K and V tiles, then Q and dO tiles of each query tile into
//                a 2-stage ring (straight from the packed qkv and dO buffers);
//   warp 1       one thread issues the MMAs: S^T and dP^T of tile i, then the three
//                gradient products of tile i-1 (whose P^T and dS^T are in shared memory);
//   warps 2, 3   no role (they complete warpgroup 0);
//   warps 4..11  two warpgroups, one per 64 queries of the tile; thread r owns key r: reads
//                its S^T and dP^T row segment, forms P^T = 2^(S^T c - lse) and
//                dS^T = P^T (dP^T - D) for the valid (key, query) pairs in registers (f32x2
//                pairs), hands S^T back, then (once the previous tile's gradient products have
//                read them) writes both as bf16 into shared memory (K-major, 128-byte swizzle);
//                at the end of the item they scale dK, turn it back through RoPE and store it,
//                and store dV (bf16), 32 values per key and pass;
//   warps 12..15 thread r owns query r of the tile: reads dQ_i from TMEM, stages it in shared
//                memory and adds it into an fp32 accumulator in global memory with TMA
//                reduce-add (several key tiles contribute to each query row).
// Every mbarrier wait is bounded; on timeout the kernel latches an error bit and stops.
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int DH = 64;
constexpr int TB = 128;                 // rows of a key or query tile
constexpr int TILE = 128 * 128;         // 128 rows x 128 bytes (64 bf16)
constexpr int kComputeWgs = 2;                      // P^T / dS^T warpgroups
constexpr int QPW = 128 / kComputeWgs;               // queries of a tile per compute warpgroup
constexpr int NSUB = QPW / 16;                       // 16-query sub-chunks per thread
// Warpgroups: 0 = TMA (warp 0), MMA (warp 1), two idle warps; 1..kComputeWgs = compute;
// the last = dQ.  Warp w reaches the TMEM lanes 32 (w % 4) .. + 31.
constexpr int kWarpCompute = 4, kWarpDq = 4 + 4 * kComputeWgs;
constexpr int THREADS = 32 * (kWarpDq + 4);
// Registers per thread at launch and after the warpgroup-wide setmaxnreg: the dQ warpgroup
// gives registers to the compute warpgroups (their P^T / dS^T pairs stay in registers until
// the shared buffers are free); warpgroup 0 (TMA, MMA) keeps its launch count.  The compute
// warpgroups' increase equals what the dQ warpgroup releases, so it never waits long.
constexpr int kRegsLaunch = 65536 / THREADS / 8 * 8, kRegsWg0 = kRegsLaunch, kRegsDq = 80;
constexpr int kRegsCompute = (THREADS * kRegsLaunch - 128 * (kRegsWg0 + kRegsDq)) / (128 * kComputeWgs) / 8 * 8;
static_assert(128 * (kRegsWg0 + kRegsDq) + 128 * kComputeWgs * kRegsCompute <= THREADS * kRegsLaunch,
              "register split");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 256, COL_DK = 320, COL_DV = 384;

struct BwdSmem {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, s_free, p_full, p_free, dq_full, dq_free, acc_full, acc_free, mma_done;
  uint32_t tmem_base;
  volatile int abort;
  // per compute warp: -(log2-sum-exp2 of the scaled scores) and -D of its warpgroup's QPW
  // queries of the current tile
  alignas(16) float wstat[4 * kComputeWgs][2][QPW];
};
// [dS^T 32K][P^T 32K][Q0][Q1][dO0][dO1][K][V][dQ staging 4 x 8K] then BwdSmem
constexpr int OFF_DS = 0, OFF_P = 2 * TILE, OFF_Q = 4 * TILE, OFF_DO = 6 * TILE, OFF_K = 8 * TILE,
              OFF_V = 9 * TILE, OFF_DQ = 10 * TILE, OFF_BAR = 12 * TILE;
constexpr int DQ_WARP_BYTES = 32 * 256;  // one dQ warp's 32 rows x 64 fp32, as two 32 x 128-byte boxes
constexpr int SMEM_BYTES = OFF_BAR + (int)sizeof(BwdSmem) + 1024;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte unit j of row r of a 128-row x 128-byte tile with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

// Two 32-lane x 16-column TMEM loads (S^T and dP^T of the same queries) and one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&a)[16], float (&b)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[16 + i]);
  }
}

// Read-only global load issued exactly where it stands in the program (a prefetch whose
// value is consumed one tile later must not be scheduled next to its use).
__device__ __forceinline__ float ld_nc_early(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

struct BItem {
  int k0, krows, s0, slen, h, nq;
};
__device__ __forceinline__ BItem bitem(const PackBuffers& pb, int it, int heads) {
  const int4 w = __ldg(reinterpret_cast<const int4*>(pb.work) + it / heads);
  BItem x;
  x.h = it % heads;
  x.k0 = w.x;
  x.krows = w.y;
  x.s0 = w.z;
  x.slen = w.w;
  x.nq = (w.w + TB - 1) / TB;
  return x;
}

__global__ void __launch_bounds__(THREADS, 1)
    attention_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                            const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse,
                            const float* __restrict__ dsum, __nv_bfloat16* __restrict__ dqkv, int T, int d, int heads,
                            PackBuffers pb, const float2* __restrict__ rope, int max_pos, unsigned* err) {
  const int n_items = *pb.work_count * heads;
  if ((int)blockIdx.x >= n_items) return;  // whole CTA, before any barrier or TMEM use

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdSmem* sm = reinterpret_cast<BwdSmem*>(base + OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&sm->kv_full, 1);
    mbar_init(&sm->kv_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->q_full[b], 1);
      mbar_init(&sm->q_empty[b], 1);
    }
    mbar_init(&sm->s_full, 1);
    mbar_init(&sm->s_free, 4 * kComputeWgs);
    mbar_init(&sm->p_full, 4 * kComputeWgs);
    mbar_init(&sm->p_free, 1);
    mbar_init(&sm->dq_full, 1);
    mbar_init(&sm->dq_free, 4);
    mbar_init(&sm->acc_full, 1);
    mbar_init(&sm->acc_free, 4 * kComputeWgs);
    mbar_init(&sm->mma_done, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sm->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  if constexpr (kRegsWg0 < kRegsLaunch) {
    if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWg0));
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_qkv);
      tma_prefetch_desc(&tm_do);
      int g = 0, n = 0;
      for (int it = blockIdx.x; it < n_items && !sm->abort; it += gridDim.x, ++n) {
        const BItem x = bitem(pb, it, heads);
        if (!mbar_wait(&sm->kv_empty, (uint32_t)(n & 1) ^ 1u)) { latch_error(err, ERRBIT_TIMEOUT); sm->abort = 1; break; }
        mbar_arrive_expect_tx(&sm->kv_full, 2 * TILE);
        tma_load_2d(base + OFF_K, &tm_qkv, d + x.h * DH, x.k0, &sm->kv_full);
        tma_load_2d(base + OFF_V, &tm_qkv, 2 * d + x.h * DH, x.k0, &sm->kv_full);
        for (int i = 0; i < x.nq; ++i, ++g) {
          const int st = g & 1;
          if (!mbar_wait(&sm->q_empty[st], (uint32_t)((g >> 1) & 1) ^ 1u)) {
            latch_error(err, ERRBIT_TIMEOUT);
            sm->abort = 1;
            break;
          }
          mbar_arrive_expect_tx(&sm->q_full[st], 2 * TILE);
          tma_load_2d(base + OFF_Q + st * TILE, &tm_qkv, x.h * DH, x.s0 + i * TB, &sm->q_full[st]);
          tma_load_2d(base + OFF_DO + st * TILE, &tm_do, x.h * DH, x.s0 + i * TB, &sm->q_full[st]);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(TB, TB);                                   // S^T, dP^T
      constexpr uint32_t idesc_kv = idesc_bf16(TB, DH) | kIdescBMn;                      // dV, dK
      constexpr uint32_t idesc_q = idesc_bf16(TB, DH) | kIdescAMn | kIdescBMn;           // dQ
      const uint32_t sb = smem_u32(base);
      const uint64_t k_kmaj = make_sw128_desc(sb + OFF_K);
      const uint64_t v_kmaj = make_sw128_desc(sb + OFF_V);
      const uint64_t k_mn = make_sw128_mn_desc(sb + OFF_K, TILE);
      const uint64_t p_kmaj = make_sw128_desc(sb + OFF_P);
      const uint64_t ds_kmaj = make_sw128_desc(sb + OFF_DS);
      const uint64_t ds_mn = make_sw128_mn_desc(sb + OFF_DS, TILE);  // queries 64.. one tile further
      bool ok = true;
      int g = 0, n = 0;
      // gradient products of global tile gb (item-local index i) from stage gb & 1
      auto back = [&](int gb, int i, int item_n) -> bool {
        if (!mbar_wait(&sm->p_full, (uint32_t)gb & 1u)) return false;
        if (!mbar_wait(&sm->dq_free, (uint32_t)(gb & 1) ^ 1u)) return false;
        if (i == 0 && !mbar_wait(&sm->acc_free, (uint32_t)(item_n & 1) ^ 1u)) return false;
        tc_fence_after();
        const int st = gb & 1;
        const uint64_t q_mn = make_sw128_mn_desc(sb + OFF_Q + st * TILE, TILE);
        const uint64_t do_mn = make_sw128_mn_desc(sb + OFF_DO + st * TILE, TILE);
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // K = 128 queries in steps of 16
          // K-major P^T / dS^T: queries 64k.. live in the second 16 KB block
          const uint64_t koff = (uint64_t)(((k >> 2) * TILE) >> 4) + 2u * (uint64_t)(k & 3);
          const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
          mma_bf16_ss(tmem + COL_DV, p_kmaj + koff, do_mn + 128u * (uint64_t)k, idesc_kv, acc);
          mma_bf16_ss(tmem + COL_DK, ds_kmaj + koff, q_mn + 128u * (uint64_t)k, idesc_kv, acc);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)  // K = 128 keys in steps of 16
          mma_bf16_ss(tmem + COL_DQ, ds_mn + 128u * (uint64_t)k, k_mn + 128u * (uint64_t)k, idesc_q, k > 0 ? 1u : 0u);
        mma_commit(&sm->p_free);
        mma_commit(&sm->dq_full);
        mma_commit(&sm->q_empty[st]);
        return true;
      };
      for (int it = blockIdx.x; it < n_items && ok && !sm->abort; it += gridDim.x, ++n) {
        const BItem x = bitem(pb, it, heads);
        if (!mbar_wait(&sm->kv_full, (uint32_t)n & 1u)) { ok = false; break; }
        for (int i = 0; i < x.nq; ++i, ++g) {
          const int st = g & 1;
          if (!mbar_wait(&sm->q_full[st], (uint32_t)(g >> 1) & 1u) ||
              !mbar_wait(&sm->s_free, (uint32_t)(g & 1) ^ 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t q_kmaj = make_sw128_desc(sb + OFF_Q + st * TILE);
          const uint64_t do_kmaj = make_sw128_desc(sb + OFF_DO + st * TILE);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(tmem + COL_S, k_kmaj + 2u * k, q_kmaj + 2u * k, idesc_s, k > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(tmem + COL_DP, v_kmaj + 2u * k, do_kmaj + 2u * k, idesc_s, k > 0 ? 1u : 0u);
          mma_commit(&sm->s_full);
          if (i > 0 && !back(g - 1, i - 1, n)) { ok = false; break; }
        }
        if (!ok || !back(g - 1, x.nq - 1, n)) { ok = false; break; }
        mma_commit(&sm->acc_full);
        mma_commit(&sm->kv_empty);
      }
      if (!ok) {
        latch_error(err, ERRBIT_TIMEOUT);
        sm->abort = 1;
      }
      mma_commit(&sm->mma_done);
      mbar_wait(&sm->mma_done, 0);
    }
    __syncwarp();
  } else if (warp >= kWarpCompute && warp < kWarpDq) {
    // ------------------------------------------------------------ P^T / dS^T, dK / dV
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCompute));
    const int wg = (warp - kWarpCompute) >> 2;  // warpgroup: queries QPW wg .. QPW wg + QPW - 1 of each tile
    const int wq = warp & 3;
    const int r = wq * 32 + lane;    // key row of the tile (and index of the lse / D slot)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    constexpr float kLog2e = 1.4426950408889634f;
    const float c = kLog2e / 8.f;  // scores scaled by 1/sqrt(64), in log2 units
    const uint64_t c2 = f2_pack(c, c);
    // this warpgroup's QPW queries of P^T / dS^T: 16-byte units unit0 .. of 64-query block
    uint8_t* sP = base + OFF_P + ((QPW * wg) >> 6) * TILE;
    uint8_t* sDS = base + OFF_DS + ((QPW * wg) >> 6) * TILE;
    const int unit0 = ((QPW * wg) & 63) >> 3;
    bool ok = true;
    int g = 0, n = 0;
    // -lse (log2 units) and -D of queries QPW wg + 32 k + lane of a tile (lse and D are
    // head-major [heads, T], so a warp reads 128 contiguous bytes of each per k); loaded one
    // tile ahead so the load latency overlaps the previous tile, then shared with the warp
    // through its slot
    constexpr int KS = QPW / 32;
    float* slot = &sm->wstat[warp - kWarpCompute][0][0];
    auto stat = [&](const BItem& y, int i, float (&nl)[KS], float (&nd)[KS]) {
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        const int q = QPW * wg + 32 * k + lane;
        nl[k] = 0.f;
        nd[k] = 0.f;
        if (q < min(TB, y.slen - i * TB)) {
          const size_t at = (size_t)y.h * T + y.s0 + i * TB + q;
          nl[k] = ld_nc_early(lse + at);
          nd[k] = ld_nc_early(dsum + at);
        }
      }
    };
    float nl_next[KS], nd_next[KS];
#pragma unroll
    for (int k = 0; k < KS; ++k) nl_next[k] = nd_next[k] = 0.f;
    if ((int)blockIdx.x < n_items) stat(bitem(pb, blockIdx.x, heads), 0, nl_next, nd_next);
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++n) {
      const BItem x = bitem(pb, it, heads);
      const bool kval = r < x.krows;
      for (int i = 0; i < x.nq; ++i, ++g) {
        const int qvalid = min(TB, x.slen - i * TB);
        __syncwarp();  // the warp is done reading the previous tile's slot
#pragma unroll
        for (int k = 0; k < KS; ++k) {  // (the loads return lse and D; stored negated, lse in log2 units)
          slot[32 * k + lane] = -nl_next[k] * kLog2e;
          slot[QPW + 32 * k + lane] = -nd_next[k];
        }
        __syncwarp();
        if (i + 1 < x.nq) stat(x, i + 1, nl_next, nd_next);
        else if (it + (int)gridDim.x < n_items) stat(bitem(pb, it + gridDim.x, heads), 0, nl_next, nd_next);
        if (!mbar_wait_warp(&sm->s_full, (uint32_t)g & 1u)) { ok = false; break; }
        tc_fence_after();
        // P^T and dS^T of this thread's key and QPW queries, as bf16 pairs, 16 queries at a time:
        // t = s c - lse (log2 units), p = 2^t, ds = p (dp - D), in f32x2 pairs
        const bool full = kval && qvalid == TB;
        uint32_t pw[NSUB][8], dw[NSUB][8];
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
          const int cq = QPW * wg + 16 * sub;  // first query (column) of the sub-chunk
          float sv[16], dp[16];
          tmem_ld16x2(tmem + lane_off + COL_S + cq, tmem + lane_off + COL_DP + cq, sv, dp);
          const float4* nl4 = reinterpret_cast<const float4*>(slot + 16 * sub);
          const float4* nd4 = reinterpret_cast<const float4*>(slot + QPW + 16 * sub);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 nl = nl4[j4], nd = nd4[j4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int j = 2 * j4 + h2;  // pair j: queries cq + 2j, cq + 2j + 1
              const uint64_t t = f2_fma(f2_pack(sv[2 * j], sv[2 * j + 1]), c2,
                                        h2 ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y));
              float t0, t1;
              f2_unpack(t, t0, t1);
              float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
              if (!full) {
                const int q = cq + 2 * j;
                p0 = (kval && q < qvalid) ? p0 : 0.f;
                p1 = (kval && q + 1 < qvalid) ? p1 : 0.f;
              }
              const uint64_t pp = f2_pack(p0, p1);
              const uint64_t dd = f2_mul(pp, f2_add(f2_pack(dp[2 * j], dp[2 * j + 1]),
                                                    h2 ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y)));
              float d0, d1;
              f2_unpack(dd, d0, d1);
              pw[sub][j] = pack_bf16x2(p0, p1);
              dw[sub][j] = pack_bf16x2(d0, d1);
            }
          }
        }
        // S^T / dP^T are read: the tensor core may compute the next tile's
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->s_free);
        // P^T / dS^T may be overwritten once the previous tile's gradient MMAs have read them
        if (!mbar_wait_warp(&sm->p_free, (uint32_t)(g & 1) ^ 1u)) { ok = false; break; }
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint32_t off = swz(r, unit0 + 2 * sub + h2);
            *reinterpret_cast<uint4*>(sP + off) =
                make_uint4(pw[sub][4 * h2], pw[sub][4 * h2 + 1], pw[sub][4 * h2 + 2], pw[sub][4 * h2 + 3]);
            *reinterpret_cast<uint4*>(sDS + off) =
                make_uint4(dw[sub][4 * h2], dw[sub][4 * h2 + 1], dw[sub][4 * h2 + 2], dw[sub][4 * h2 + 3]);
          }
        }
        fence_async_smem();  // generic-proxy writes of P^T / dS^T before the tensor core reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->p_full);
      }
      if (!ok) break;
      // ---- item epilogue, in four parts of 32 gradient values per key: part v = 0, 2 store dK
      // (scaled, RoPE undone) for the pairs (j, j + 32), j in 16 (v / 2) .. + 15; part v = 1, 3
      // store dV columns 32 (v / 2) .. + 31.  Warpgroup wg takes parts wg, wg + kComputeWgs, ...
      if (!mbar_wait_warp(&sm->acc_full, (uint32_t)n & 1u)) { ok = false; break; }
      tc_fence_after();
      const int key = x.k0 + r;
      int p = key - x.s0;
      p = p < 0 ? 0 : (p >= max_pos ? max_pos - 1 : p);
      __nv_bfloat16* row = dqkv + (size_t)key * 3 * d + x.h * DH;
#pragma unroll
      for (int v = wg; v < 4; v += kComputeWgs) {
        const bool is_k = (v & 1) == 0;
        const int c0 = is_k ? 16 * (v >> 1) : 32 * (v >> 1);  // dK: first pair j0; dV: first column
        float a[16], b[16];
        if (is_k) tmem_ld16x2(tmem + lane_off + COL_DK + c0, tmem + lane_off + COL_DK + 32 + c0, a, b);
        else tmem_ld16x2(tmem + lane_off + COL_DV + c0, tmem + lane_off + COL_DV + c0 + 16, a, b);
        if (v + kComputeWgs >= 4) {  // this warp's last TMEM read of the item
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm->acc_free);
        }
        if (!kval) continue;
        if (is_k) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {  // pair (c0 + j, c0 + j + 32) turned back by its angle
            const float u = a[j] * 0.125f, w = b[j] * 0.125f;
            if (rope != nullptr) {
              const int jj = c0 + j;
              const float2 cs = __ldg(rope + ((size_t)(jj >> 1) * max_pos + p) * 2 + (jj & 1));
              a[j] = u * cs.x + w * cs.y;
              b[j] = w * cs.x - u * cs.y;
            } else {
              a[j] = u;
              b[j] = w;
            }
          }
          uint4* lo = reinterpret_cast<uint4*>(row + d + c0);
          uint4* hi = reinterpret_cast<uint4*>(row + d + c0 + 32);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            lo[u] = make_uint4(pack_bf16x2(a[8 * u], a[8 * u + 1]), pack_bf16x2(a[8 * u + 2], a[8 * u + 3]),
                               pack_bf16x2(a[8 * u + 4], a[8 * u + 5]), pack_bf16x2(a[8 * u + 6], a[8 * u + 7]));
            hi[u] = make_uint4(pack_bf16x2(b[8 * u], b[8 * u + 1]), pack_bf16x2(b[8 * u + 2], b[8 * u + 3]),
                               pack_bf16x2(b[8 * u + 4], b[8 * u + 5]), pack_bf16x2(b[8 * u + 6], b[8 * u + 7]));
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(row + 2 * d + c0);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            dst[u] = make_uint4(pack_bf16x2(a[8 * u], a[8 * u + 1]), pack_bf16x2(a[8 * u + 2], a[8 * u + 3]),
                                pack_bf16x2(a[8 * u + 4], a[8 * u + 5]), pack_bf16x2(a[8 * u + 6], a[8 * u + 7]));
            dst[2 + u] = make_uint4(pack_bf16x2(b[8 * u], b[8 * u + 1]), pack_bf16x2(b[8 * u + 2], b[8 * u + 3]),
                                    pack_bf16x2(b[8 * u + 4], b[8 * u + 5]), pack_bf16x2(b[8 * u + 6], b[8 * u + 7]));
          }
        }
      }
    }
    if (!ok) {
      latch_error(err, ERRBIT_TIMEOUT);
      sm->abort = 1;
    }
  } else if (warp >= kWarpDq) {
    // ------------------------------------------------------------ dQ accumulation
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDq));
    // Each warp stages its 32 rows of dQ_i (fp32, 128-byte swizzle, two 32-column boxes) and
    // adds them into the global accumulator with TMA reduce-add; rows of queries past the
    // sequence end hold exact zeros (their dS columns are zero), so adding them is harmless.
    const int wq = warp & 3;  // lane l owns query row 32 wq + l of the tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    uint8_t* stage = base + OFF_DQ + wq * DQ_WARP_BYTES;
    if (lane == 0) tma_prefetch_desc(&tm_dq);
    bool ok = true;
    int g = 0;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const BItem x = bitem(pb, it, heads);
      for (int i = 0; i < x.nq; ++i, ++g) {
        if (!mbar_wait_warp(&sm->dq_full, (uint32_t)g & 1u)) { ok = false; break; }
        tc_fence_after();
        // the previous tile's reduce must have finished reading the staging rows
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {  // 16 columns at a time: box ch >> 1, units 4 (ch & 1) ..
          float a[16];
          tmem_ld16(tmem + lane_off + COL_DQ + 16 * ch, a);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int unit = 4 * (ch & 1) + u;
            const uint32_t off = (uint32_t)((ch >> 1) * 4096 + lane * 128 + ((unit ^ (lane & 7)) << 4));
            *reinterpret_cast<float4*>(stage + off) = make_float4(a[4 * u], a[4 * u + 1], a[4 * u + 2], a[4 * u + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->dq_free);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int row = x.s0 + i * TB + wq * 32;
          tma_reduce_add_2d(&tm_dq, x.h * DH, row, stage);
          tma_reduce_add_2d(&tm_dq, x.h * DH + 32, row, stage + 4096);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // reduces complete before the CTA may exit
    __syncwarp();
    if (!ok) {
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

// D[h, t] = sum_c dO[t, h*64 + c] * O[t, h*64 + c] (head-major).  Eight lanes per (token,
// head): lane p dots columns 8p..8p+7 (one 16-byte load of each operand, so the eight lanes
// read the head's 128 contiguous bytes together), then three shuffle steps add the eight
// partial sums.  Every lane reaches the shuffles (no early return).
static_assert(DH == 64, "eight 16-byte pieces per head row");
__global__ void attention_bwd_dsum_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                          float* __restrict__ dsum, int T, int d, int heads) {
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long i = g >> 3;
  const int p = (int)(g & 7);
  const bool ok = i < (long long)T * heads;
  const long long t = ok ? i / heads : 0;
  const int h = ok ? (int)(i % heads) : 0;
  float acc = 0.f;
  if (ok) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(o + t * d + h * DH) + p);
    const uint4 y = __ldg(reinterpret_cast<const uint4*>(dout + t * d + h * DH) + p);
    const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* yh = reinterpret_cast<const __nv_bfloat162*>(&y);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 xf = __bfloat1622float2(xh[k]), yf = __bfloat1622float2(yh[k]);
      acc = fmaf(xf.x, yf.x, acc);
      acc = fmaf(xf.y, yf.y, acc);
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  if (ok && p == 0) dsum[(size_t)h * T + t] = acc;
}

// dq = dq_acc / 8 with RoPE undone (pairs (j, j + 32) turned back by their angle) -> the q
// block of dqkv (bf16).  One thread per (token, head, 8 consecutive pairs): 16-byte loads
// of columns j0..j0+7 and j0+32..j0+39, two 16-byte stores.
__global__ void attention_bwd_dq_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dqkv,
                                        const int32_t* __restrict__ pos_id, const float2* __restrict__ rope,
                                        int max_pos, int T, int d) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_tok = d / 16;  // (heads) x (4 groups of 8 pairs)
  if (i >= (long long)T * per_tok) return;
  const long long t = i / per_tok;
  const int rem = (int)(i % per_tok);
  const int h = rem >> 2, j0 = (rem & 3) * 8;
  const float* src = dq_acc + t * d + h * DH;
  float a[8], b[8];
  *reinterpret_cast<float4*>(a) = __ldg(reinterpret_cast<const float4*>(src + j0));
  *reinterpret_cast<float4*>(a + 4) = __ldg(reinterpret_cast<const float4*>(src + j0 + 4));
  *reinterpret_cast<float4*>(b) = __ldg(reinterpret_cast<const float4*>(src + j0 + 32));
  *reinterpret_cast<float4*>(b + 4) = __ldg(reinterpret_cast<const float4*>(src + j0 + 36));
  int p = 0;
  if (rope != nullptr) {
    p = __ldg(pos_id + t);
    p = p < 0 ? 0 : (p >= max_pos ? max_pos - 1 : p);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float u = a[k] * 0.125f, v = b[k] * 0.125f;
    if (rope != nullptr) {
      const int j = j0 + k;
      const float2 cs = __ldg(rope + ((size_t)(j >> 1) * max_pos + p) * 2 + (j & 1));
      a[k] = u * cs.x + v * cs.y;
      b[k] = v * cs.x - u * cs.y;
    } else {
      a[k] = u;
      b[k] = v;
    }
  }
  __nv_bfloat16* dst = dqkv + t * 3 * d + h * DH;
  *reinterpret_cast<uint4*>(dst + j0) =
      make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
  *reinterpret_cast<uint4*>(dst + j0 + 32) =
      make_uint4(pack_bf16x2(b[0], b[1]), pack_bf16x2(b[2], b[3]), pack_bf16x2(b[4], b[5]), pack_bf16x2(b[6], b[7]));
}

}  // namespace

cudaError_t launch_attention_bwd_tc(const CUtensorMap* tm_qkv, const CUtensorMap* tm_do, const CUtensorMap* tm_dq,
                                    const __nv_bfloat16* o,
                                    const __nv_bfloat16* dout, const float* lse, float* dsum, float* dq_acc,
                                    __nv_bfloat16* dqkv, int T, int d, int heads, int max_items, const PackBuffers& pb,
                                    const float2* rope, int max_pos, int num_sms, unsigned* err, cudaStream_t st) {
  if (T <= 0 || max_items <= 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attention_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long th = (long long)T * heads;
  attention_bwd_dsum_kernel<<<(unsigned)((8 * th + 255) / 256), 256, 0, st>>>(o, dout, dsum, T, d, heads);
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)T * d, st);
  if (e != cudaSuccess) return e;
  const long long items = (long long)max_items * heads;
  const unsigned grid = (unsigned)(items < num_sms ? items : num_sms);
  attention_bwd_tc_kernel<<<grid, THREADS, SMEM_BYTES, st>>>(*tm_qkv, *tm_do, *tm_dq, lse, dsum, dqkv, T, d, heads, pb,
                                                             rope, max_pos, err);
  const long long tq = (long long)T * (d / 16);
  attention_bwd_dq_kernel<<<(unsigned)((tq + 255) / 256), 256, 0, st>>>(dq_acc, dqkv, pb.pos_id, rope, max_pos, T, d);
  return cudaGetLastError();
}

}  // namespace esm
