// Packing indices, the attention work list, the token embedding gather and the RoPE
// table.
//
// Packing follows section 3.2 of the hotelren.com guide ("生物大模型训练加速实战"): the
// batch is the concatenation of its sequences plus cu_seqlens = cumsum([0] + lengths);
// the packed forward consumes (input_ids, cu_seqlens, max_seqlen).  The padded layout
// with a key padding mask is the bshd / padding-mask configuration of the mlqm.cn
// ESM-2 TransformerEngine walkthrough (attention-mask section).
#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

// One CTA per sequence: validate its bounds, write pos_id / seg_id for its tokens and
// the sanitised segment table.  Malformed input latches ERRBIT_CU_SEQLENS; the table
// is clamped so that every later access stays inside [0, T).
__global__ void pack_index_kernel(const int32_t* __restrict__ cu, int B, int T, int max_seqlen, int max_positions,
                                  PackBuffers pb, unsigned* err) {
  const int i = blockIdx.x;
  int c0 = cu[i], c1 = cu[i + 1];
  bool bad = false;
  if (i == 0 && c0 != 0) bad = true;
  if (i == B - 1 && c1 != T) bad = true;
  if (c1 < c0 || c1 - c0 > max_seqlen || c1 - c0 > max_positions) bad = true;
  if (c0 < 0 || c1 > T) bad = true;
  if (bad) {
    if (threadIdx.x == 0) latch_error(err, ERRBIT_CU_SEQLENS);
    c0 = min(max(c0, 0), T);
    c1 = min(max(c1, c0), T);
    c1 = min(c1, c0 + max_positions);
  }
  const int L = c1 - c0;
  if (threadIdx.x == 0) {
    pb.seg_start[i] = c0;
    pb.seg_qlen[i] = L;
    pb.seg_klen[i] = L;
  }
  for (int p = threadIdx.x; p < L; p += blockDim.x) {
    pb.pos_id[c0 + p] = p;
    pb.seg_id[c0 + p] = i;
  }
}

// Padded [B, S] batch: segment b covers rows b*S .. b*S+S-1 (all of them are queries)
// and its first len_b rows are the visible keys.
__global__ void pad_index_kernel(const int32_t* __restrict__ seq_lens, int B, int S, PackBuffers pb,
                                 unsigned* err) {
  const int b = blockIdx.x;
  int len = seq_lens[b];
  if (len < 1 || len > S) {
    if (threadIdx.x == 0) latch_error(err, ERRBIT_CU_SEQLENS);
    len = min(max(len, 1), S);
  }
  if (threadIdx.x == 0) {
    pb.seg_start[b] = b * S;
    pb.seg_qlen[b] = S;
    pb.seg_klen[b] = len;
  }
  for (int p = threadIdx.x; p < S; p += blockDim.x) {
    pb.pos_id[b * S + p] = p;
    pb.seg_id[b * S + p] = b;
  }
}

constexpr int WL_THREADS = 1024;
constexpr int WL_SORT_MAX = 4096;

// Single CTA: list the (segment, query-tile) work items of the attention kernel, each as
// (first query row, query rows, first key row, visible keys), longest segments first so that the costliest tiles start in the first wave (when B is small
// enough to rank in shared memory; otherwise in segment order).
__global__ void __launch_bounds__(WL_THREADS) attn_worklist_kernel(int B, int max_items, int q_tile, PackBuffers pb) {
  __shared__ int s_len[WL_SORT_MAX];
  __shared__ int s_order[WL_SORT_MAX];
  __shared__ int s_warp[WL_THREADS / 32];
  __shared__ int s_base;
  const int tid = threadIdx.x;
  const bool sorted = B <= WL_SORT_MAX;
  if (sorted) {
    for (int i = tid; i < B; i += WL_THREADS) s_len[i] = pb.seg_klen[i] * 4096 + min(pb.seg_qlen[i], 4095);
    __syncthreads();
    for (int i = tid; i < B; i += WL_THREADS) {
      const int li = s_len[i];
      int rank = 0;
      for (int j = 0; j < B; ++j) {
        const int lj = s_len[j];
        rank += (lj > li) || (lj == li && j < i);
      }
      s_order[rank] = i;
    }
  }
  if (tid == 0) s_base = 0;
  __syncthreads();
  for (int chunk = 0; chunk < B; chunk += WL_THREADS) {
    const int r = chunk + tid;
    int seg = -1, tiles = 0;
    if (r < B) {
      seg = sorted ? s_order[r] : r;
      tiles = (pb.seg_qlen[seg] + q_tile - 1) / q_tile;
    }
    // block exclusive scan of `tiles`
    int v = tiles;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) s_warp[wid] = v;
    __syncthreads();
    if (wid == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int excl = s_base + (wid > 0 ? s_warp[wid - 1] : 0) + v - tiles;
    if (tiles > 0) {
      const int start = pb.seg_start[seg], qlen = pb.seg_qlen[seg], klen = pb.seg_klen[seg];
      for (int t = 0; t < tiles; ++t) {
        const int k = excl + t;
        if (k < max_items)
          reinterpret_cast<int4*>(pb.work)[k] = make_int4(start + t * q_tile, min(q_tile, qlen - t * q_tile), start, klen);
      }
    }
    __syncthreads();
    if (tid == WL_THREADS - 1) s_base = excl + tiles;
    __syncthreads();
  }
  if (tid == 0) pb.work_count[0] = min(s_base, max_items);
}

// x[t, :] = scale * E[tok[t], :] into the fp32 residual stream; one warp per token,
// 16-byte loads and stores.  Ids outside [0, vocab) latch ERRBIT_TOKEN and read row 0.
template <bool F32>
__global__ void embed_kernel(const int32_t* __restrict__ tok, int T, const void* __restrict__ emb, int vocab, int d,
                             float scale, float* __restrict__ x, unsigned* err) {
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int id = tok[t];
  if (id < 0 || id >= vocab) {
    if (lane == 0) latch_error(err, ERRBIT_TOKEN);
    id = 0;
  }
  float4* dst = reinterpret_cast<float4*>(x + (size_t)t * d);
  if (F32) {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(emb) + (size_t)id * d);
    for (int c = lane; c < d / 4; c += 32) {
      float4 v = __ldg(src + c);
      dst[c] = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
    }
  } else {
    const uint2* src = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(emb) + (size_t)id * d);
    for (int c = lane; c < d / 4; c += 32) {
      uint2 v = __ldg(src + c);
      float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.x));
      float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.y));
      dst[c] = make_float4(a.x * scale, a.y * scale, b.x * scale, b.y * scale);
    }
  }
}

// (cos, sin)(p * base^(-2j/dh)) for j < dh/2, computed in double precision and rounded once
// to float.  Layout [kRopeMaxHalf/2][max_pos][2] of float2: the pairs j = 2g and 2g+1 of
// position p form one 16-byte group at index g * max_pos + p, so the 32 consecutive
// positions of a warp read 512 contiguous bytes per group.
__global__ void rope_table_kernel(float2* tab, int max_pos, int half, double base) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= max_pos * kRopeMaxHalf) return;
  const int g = i / (2 * max_pos), p = (i / 2) % max_pos, j = 2 * g + (i & 1);
  if (j >= half) {
    tab[i] = make_float2(1.f, 0.f);
    return;
  }
  const double theta = pow(base, -2.0 * (double)j / (double)(2 * half));
  double s, c;
  sincos((double)p * theta, &s, &c);
  tab[i] = make_float2((float)c, (float)s);
}

// One warp waits on an mbarrier that nothing will ever arrive at, through the same bounded
// wait every kernel uses (here with a short limit): the wait gives up, the error bit is
// latched and the kernel returns normally.
__global__ void wait_timeout_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (!mbar_wait_limit(&bar, 0, limit_ns) && threadIdx.x == 0) latch_error(err, ERRBIT_TIMEOUT);
}

}  // namespace

void launch_wait_timeout(unsigned long long limit_ns, unsigned* err, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, err);
}

void launch_pack_index(const int32_t* cu, int B, int T, int max_seqlen, int max_positions, const PackBuffers& pb,
                       unsigned* err, cudaStream_t st) {
  if (B <= 0) return;
  pack_index_kernel<<<B, 256, 0, st>>>(cu, B, T, max_seqlen, max_positions, pb, err);
}

void launch_pad_index(const int32_t* seq_lens, int B, int S, const PackBuffers& pb, unsigned* err, cudaStream_t st) {
  if (B <= 0) return;
  pad_index_kernel<<<B, 256, 0, st>>>(seq_lens, B, S, pb, err);
}

void launch_attn_worklist(int B, int max_items, int q_tile, const PackBuffers& pb, cudaStream_t st) {
  attn_worklist_kernel<<<1, WL_THREADS, 0, st>>>(B, max_items, q_tile, pb);
}

void launch_embed(const int32_t* tok, int T, const void* emb, bool emb_f32, int vocab, int d, float scale, float* x,
                  unsigned* err, cudaStream_t st) {
  if (T <= 0) return;
  const int warps = 8;
  const int grid = (T + warps - 1) / warps;
  if (emb_f32)
    embed_kernel<true><<<grid, 32 * warps, 0, st>>>(tok, T, emb, vocab, d, scale, x, err);
  else
    embed_kernel<false><<<grid, 32 * warps, 0, st>>>(tok, T, emb, vocab, d, scale, x, err);
}

void launch_rope_table(float2* tab, int max_pos, int half, float base, cudaStream_t st) {
  const int n = max_pos * kRopeMaxHalf;
  rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(tab, max_pos, half, (double)base);
}

}  // namespace esm
