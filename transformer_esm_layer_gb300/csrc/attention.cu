// Variable-length bidirectional attention over packed sequences.
//
// Section 3.2 of the hotelren.com guide ("生物大模型训练加速实战") runs every layer over
// cu_seqlens (thd format); section 2.1 names TE's attention kernels for variable-length
// batches; the BioNeMo ESM-2 model card describes a bidirectional (BERT-style) encoder.
// So each token attends to every token of its own sequence and to nothing else:
//
//   o_t = sum_s softmax_s(q_t . k_s / sqrt(dh)) v_s,   s over the sequence of t.
//
// bf16 kernel (head_dim 64): one CTA = one (sequence, 64-query tile, head) work item from
// the length-ordered work list; 4 warps x 16 query rows.  K/V tiles of 64 keys are
// double-buffered in shared memory (cp.async, 128-byte XOR swizzle), S = Q K^T and
// O += P V run on the tensor cores (bf16 in, fp32 accumulate), softmax is the online
// (running max / running sum) form in fp32 with exp2, so the L x L score matrix never
// exists anywhere.  Keys past the sequence end are masked; query rows past it are not
// stored.  The padded layout uses the same kernel with klen < qlen (key padding mask).
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int DH = 64;
constexpr int QT = kAttnQTile;  // 64 query rows
constexpr int KT = 64;          // keys per tile
constexpr int ATT_THREADS = 128;

__device__ __forceinline__ int swz(int r, int c) {  // element offset in a [64][64] bf16 tile
  return r * DH + ((((c >> 3) ^ (r & 7))) << 3) + (c & 7);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const uint32_t s = smem_u32(smem);
  const int n = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Load `rows` valid rows (of 64) of a [64 x 64] bf16 tile with row stride ld (elements);
// the rest is zero-filled.
__device__ __forceinline__ void load_tile(__nv_bfloat16* s, const __nv_bfloat16* g, int ld, int rows) {
#pragma unroll
  for (int i = 0; i < (64 * 8) / ATT_THREADS; ++i) {
    const int id = threadIdx.x + i * ATT_THREADS;
    const int r = id >> 3, ch = id & 7;
    const bool ok = r < rows;
    const __nv_bfloat16* src = g + (size_t)(ok ? r : 0) * ld + ch * 8;
    cp_async16(s + swz(r, ch * 8), src, ok);
  }
}

template <Act OUT>
__global__ void __launch_bounds__(ATT_THREADS)
    attention_bf16_kernel(const __nv_bfloat16* __restrict__ qkv, void* __restrict__ o, int d, int heads,
                          PackBuffers pb, const float* q_scale, float* amax_out) {
  __shared__ __align__(128) __nv_bfloat16 sQ[QT * DH];
  __shared__ __align__(128) __nv_bfloat16 sK[2][KT * DH];
  __shared__ __align__(128) __nv_bfloat16 sV[2][KT * DH];

  const int item = blockIdx.x / heads;
  const int h = blockIdx.x - item * heads;
  if (item >= *pb.work_count) return;
  const int4 wi = reinterpret_cast<const int4*>(pb.work)[item];
  const int qrow0 = wi.x;
  const int start = wi.z;
  const int klen = wi.w;
  const int qrows = wi.y;
  const int ld = 3 * d;
  const __nv_bfloat16* gq = qkv + (size_t)qrow0 * ld + h * DH;
  const __nv_bfloat16* gk = qkv + (size_t)start * ld + d + h * DH;
  const __nv_bfloat16* gv = qkv + (size_t)start * ld + 2 * d + h * DH;
  const int nkb = (klen + KT - 1) / KT;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float sl2 = 1.4426950408889634f / sqrtf((float)DH);  // log2(e) / sqrt(dh)

  load_tile(sQ, gq, ld, qrows);
  load_tile(sK[0], gk, ld, min(KT, klen));
  load_tile(sV[0], gv, ld, min(KT, klen));
  cp_async_commit();

  uint32_t qa[4][4];
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int kb = 0; kb < nkb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nkb) {
      const int k1 = (kb + 1) * KT;
      load_tile(sK[buf ^ 1], gk + (size_t)k1 * ld, ld, min(KT, klen - k1));
      load_tile(sV[buf ^ 1], gv + (size_t)k1 * ld, ld, min(KT, klen - k1));
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int r = warp * 16 + (lane & 15);
        const int c = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(smem_u32(sQ + swz(r, c)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    // ---- S = Q K^T (16 rows x 64 keys per warp)
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    const __nv_bfloat16* k_s = sK[buf];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = kk * 16 + ((lane >> 3) & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(k_s + swz(key, c)), b0, b1, b2, b3);
        mma16816(s[2 * np], qa[kk], b0, b1);
        mma16816(s[2 * np + 1], qa[kk], b2, b3);
      }
    }
    // ---- mask keys past the sequence end, online softmax
    const int kbase = kb * KT;
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int kc = kbase + j * 8 + (lane & 3) * 2;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok = kc + e < klen;
        s[j][e] = ok ? s[j][e] * sl2 : -INFINITY;
        s[j][2 + e] = ok ? s[j][2 + e] * sl2 : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
      mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float corr0 = exp2f(m0 - mx0), corr1 = exp2f(m1 - mx1);
    m0 = mx0;
    m1 = mx1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pa[4][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p0 = exp2f(s[j][0] - m0), p1 = exp2f(s[j][1] - m0);
      const float p2 = exp2f(s[j][2] - m1), p3 = exp2f(s[j][3] - m1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      // C fragment of n-tile j -> A fragment of k-step j/2 (keys 16*(j/2) .. +15)
      pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
      pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[j][0] *= corr0; acc[j][1] *= corr0;
      acc[j][2] *= corr1; acc[j][3] *= corr1;
    }
    // ---- O += P V
    const __nv_bfloat16* v_s = sV[buf];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = dp * 16 + (lane >> 4) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(v_s + swz(key, c)), b0, b1, b2, b3);
        mma16816(acc[2 * dp], pa[kk], b0, b1);
        mma16816(acc[2 * dp + 1], pa[kk], b2, b3);
      }
    }
    __syncthreads();
  }

  // ---- normalise and store (row sums are quad-partial: reduce them first)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int r0 = warp * 16 + (lane >> 2);
  const int r1 = r0 + 8;
  float amax = 0.f;
  const float qs = (OUT == Act::E4M3) ? __ldg(q_scale) : 1.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = h * DH + j * 8 + (lane & 3) * 2;
    const float a0 = acc[j][0] * inv0, a1 = acc[j][1] * inv0;
    const float a2 = acc[j][2] * inv1, a3 = acc[j][3] * inv1;
    if constexpr (OUT == Act::BF16) {
      __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
      if (r0 < qrows) *reinterpret_cast<uint32_t*>(ob + (size_t)(qrow0 + r0) * d + c) = pack_bf16x2(a0, a1);
      if (r1 < qrows) *reinterpret_cast<uint32_t*>(ob + (size_t)(qrow0 + r1) * d + c) = pack_bf16x2(a2, a3);
    } else {
      uint8_t* ob = static_cast<uint8_t*>(o);
      if (r0 < qrows) {
        amax = fmaxf(amax, fmaxf(fabsf(a0), fabsf(a1)));
        __nv_fp8x2_e4m3 v(make_float2(a0 * qs, a1 * qs));
        *reinterpret_cast<uint16_t*>(ob + (size_t)(qrow0 + r0) * d + c) = *reinterpret_cast<uint16_t*>(&v);
      }
      if (r1 < qrows) {
        amax = fmaxf(amax, fmaxf(fabsf(a2), fabsf(a3)));
        __nv_fp8x2_e4m3 v(make_float2(a2 * qs, a3 * qs));
        *reinterpret_cast<uint16_t*>(ob + (size_t)(qrow0 + r1) * d + c) = *reinterpret_cast<uint16_t*>(&v);
      }
    }
  }
  if constexpr (OUT == Act::E4M3) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0 && amax_out) atomic_max_nonneg(amax_out, amax);
  }
}

// fp32 attention (the ESM_FP32 precision): one warp per (query row, head); lanes split
// the keys, each keeps a running max / sum / output, merged across lanes at the end.
__global__ void attention_f32_kernel(const float* __restrict__ qkv, float* __restrict__ o, int d, int heads, int T,
                                     PackBuffers pb) {
  const int warps = blockDim.x >> 5;
  const int gw = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= T * heads) return;
  const int t = gw / heads, h = gw - (gw / heads) * heads;
  const int dh = d / heads;
  const int seg = pb.seg_id[t];
  const int start = pb.seg_start[seg];
  const int klen = pb.seg_klen[seg];
  const int ld = 3 * d;
  float q[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) q[c] = c < dh ? qkv[(size_t)t * ld + h * dh + c] : 0.f;
  const float scale = 1.f / sqrtf((float)dh);
  float m = -INFINITY, l = 0.f, acc[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) acc[c] = 0.f;
  for (int j = lane; j < klen; j += 32) {
    const float* kr = qkv + (size_t)(start + j) * ld + d + h * dh;
    const float* vr = qkv + (size_t)(start + j) * ld + 2 * d + h * dh;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c < dh) s = fmaf(q[c], kr[c], s);
    s *= scale;
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn), p = expf(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c < dh) acc[c] = acc[c] * corr + p * vr[c];
    m = mn;
  }
  float M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float f = (m == -INFINITY) ? 0.f : expf(m - M);
  l *= f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    if (c >= dh) break;
    float v = acc[c] * f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) o[(size_t)t * d + h * dh + c] = v / l;
  }
}

}  // namespace

void launch_attention_bf16(const __nv_bfloat16* qkv, __nv_bfloat16* o, int d, int heads, int max_items,
                           const PackBuffers& pb, cudaStream_t st) {
  if (max_items <= 0) return;
  attention_bf16_kernel<Act::BF16><<<max_items * heads, ATT_THREADS, 0, st>>>(qkv, o, d, heads, pb, nullptr, nullptr);
}

void launch_attention_bf16_to_e4m3(const __nv_bfloat16* qkv, uint8_t* o, int d, int heads, int max_items,
                                   const PackBuffers& pb, const float* q_scale, float* amax, cudaStream_t st) {
  if (max_items <= 0) return;
  attention_bf16_kernel<Act::E4M3><<<max_items * heads, ATT_THREADS, 0, st>>>(qkv, o, d, heads, pb, q_scale, amax);
}

void launch_attention_f32(const float* qkv, float* o, int d, int heads, int T, const PackBuffers& pb,
                          cudaStream_t st) {
  if (T <= 0) return;
  const int warps = 4;
  const long long n = (long long)T * heads;
  attention_f32_kernel<<<(unsigned)((n + warps - 1) / warps), 32 * warps, 0, st>>>(qkv, o, d, heads, T, pb);
}

}  // namespace esm
