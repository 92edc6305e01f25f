// Host side of the C ABI declared in include/esm_encoder.h: handle, workspace layout,
// TMA descriptor cache and the per-layer launch sequence of the packed ESM-2 forward
// (section 3.2 of the hotelren.com guide: embedding, then every layer over cu_seqlens).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <unordered_map>
#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace esm;

namespace {

constexpr int kNumFp8Tensors = 8;  // x_qkv, w_qkv, x_o, w_o, x_1, w_1, x_2, w_2
enum Fp8Slot { X_QKV = 0, W_QKV, X_O, W_O, X_1, W_1, X_2, W_2 };

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

struct MapKey {
  uintptr_t ptr;
  uint64_t rows, cols;
  uint32_t box_rows, elem;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && box_rows == o.box_rows && elem == o.elem;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = std::hash<uintptr_t>()(k.ptr);
    h ^= std::hash<uint64_t>()(k.rows * 1000003ull + k.cols) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    h ^= std::hash<uint64_t>()((uint64_t)k.box_rows << 8 | k.elem) + (h << 6) + (h >> 2);
    return h;
  }
};

struct WsLayout {
  size_t pos, seg, seg_start, seg_qlen, seg_klen, work, work_count, x, y, qkv, o, u, wq, fp4, ln_stats, ln_fold,
      stage_tok, stage_cu, total;
  int max_items;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

struct esm_encoder {
  esm_config cfg;
  int device = 0;
  int num_sms = 0;
  unsigned* d_err = nullptr;     // device error word
  float2* d_rope = nullptr;      // [16][max_positions][2] (cos, sin)
  std::vector<uint8_t> layer_fp8;  // per layer: 1 = E4M3 GEMMs, 2 = NVFP4 GEMMs (FP8 handles only)
  float* d_fp8 = nullptr;        // scales [L*8] | history [L*8*len] | amax [L*8]
  float* d_fp4 = nullptr;        // NVFP4 tensor scales of the last forward [L*8] | amax [L*8]
  size_t fp8_floats = 0;
  // Tensor-map cache.  When it grows past its cap the current generation is retired, not
  // freed: maps handed out earlier in the same call stay valid until the next turnover.
  std::unordered_map<MapKey, CUtensorMap, MapKeyHash> maps, retired_maps;
  // the last training forward: its sizes and buffers, which the backward must be given
  int train_T = 0, train_B = 0, train_items = 0;
  const void* train_buf = nullptr;
  const void* train_ws = nullptr;
  // esm_encoder_forward_host with pinned host buffers: CUDA graphs of whole calls, keyed by
  // everything they bake in (host and device pointers, sizes, per-layer precision); a key is
  // captured at its second call (the first, eager, does the one-time kernel configuration)
  struct HostGraph {
    std::vector<uintptr_t> key;
    cudaGraphExec_t exec;
  };
  std::vector<HostGraph> host_graphs;              // oldest first, at most kHostGraphs
  std::vector<std::vector<uintptr_t>> host_seen;   // keys called once, at most kHostGraphs
  cudaStream_t cap_stream = nullptr;
  // measurement hooks
  bool profiling = false;
  long long launches[ESM_PROFILE_CLASSES] = {};
  long long total_launches = 0;
  struct Pending { int cls; cudaEvent_t e0, e1; };
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> event_pool;
  double ms[ESM_PROFILE_CLASSES] = {};

  cudaEvent_t take_event() {
    if (!event_pool.empty()) {
      cudaEvent_t e = event_pool.back();
      event_pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  // Fold finished event pairs into ms[] (synchronises on each pair's end event).
  void drain_events() {
    for (auto& p : pending) {
      float t = 0.f;
      if (cudaEventSynchronize(p.e1) == cudaSuccess && cudaEventElapsedTime(&t, p.e0, p.e1) == cudaSuccess)
        ms[p.cls] += t;
      event_pool.push_back(p.e0);
      event_pool.push_back(p.e1);
    }
    pending.clear();
  }

  bool bf16_params() const { return cfg.precision != ESM_FP32; }
  Act act() const { return cfg.precision == ESM_FP32 ? Act::F32 : Act::BF16; }
  size_t act_bytes() const { return cfg.precision == ESM_FP32 ? 4 : 2; }
  float* fp8_scale() const { return d_fp8; }
  float* fp8_hist() const { return d_fp8 + (size_t)cfg.num_layers * kNumFp8Tensors; }
  float* fp8_amax() const {
    return d_fp8 + (size_t)cfg.num_layers * kNumFp8Tensors * (1 + cfg.amax_history_len);
  }

  WsLayout layout(int Tm, int Bm) const {
    WsLayout L{};
    const size_t d = cfg.hidden, f = cfg.ffn, T = Tm > 0 ? Tm : 1, B = Bm > 0 ? Bm : 1;
    L.max_items = (int)((T + kAttnQTile - 1) / kAttnQTile + B);
    size_t off = 0;
    auto take = [&](size_t bytes) {
      size_t o = off;
      off += align256(bytes);
      return o;
    };
    L.pos = take(4 * T);
    L.seg = take(4 * T);
    L.seg_start = take(4 * B);
    L.seg_qlen = take(4 * B);
    L.seg_klen = take(4 * B);
    L.work = take(16 * (size_t)L.max_items);
    L.work_count = take(16);
    L.x = take(4 * T * d);
    L.y = take(act_bytes() * T * d);
    L.qkv = take(act_bytes() * T * 3 * d);
    L.o = take(act_bytes() * T * d);
    L.u = take(act_bytes() * T * f);
    L.wq = cfg.precision == ESM_FP8_E4M3 ? take(3 * d * d + d * d + 2 * d * f) : take(0);
    // NVFP4 layers (FP8 handles): one activation operand of up to [T rounded up to 128, ffn]
    // (codes and block scales); its weights reuse the E4M3 weight region
    const size_t tp = (T + 127) / 128 * 128;
    L.fp4 = cfg.precision == ESM_FP8_E4M3 ? take(tp * f / 2 + 256 + tp * f / 16) : take(0);
    // folded LayerNorm (bf16 forward): row statistics per 64-column group, and per layer the
    // QKV and fc1 constants c and b' (fp32 [3d] + [3d] + [f] + [f])
    L.ln_stats = cfg.precision == ESM_BF16 ? take(8 * T * (d / 64)) : take(0);
    L.ln_fold = cfg.precision == ESM_BF16 ? take(4 * (6 * d + 2 * f) * (size_t)cfg.num_layers) : take(0);
    L.stage_tok = take(4 * T);
    L.stage_cu = take(4 * (B + 1));
    L.total = off;
    return L;
  }

  // Cached 2-D tensor map over a row-major [rows, cols] matrix; the box is 128 bytes of
  // columns by box_rows rows with the 128-byte swizzle (one tcgen05 K-slice).
  const CUtensorMap* map(const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t elem) {
    MapKey k{reinterpret_cast<uintptr_t>(ptr), rows, cols, box_rows, elem};
    auto it = maps.find(k);
    if (it != maps.end()) return &it->second;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return nullptr;
    if (maps.size() > 4096) {
      retired_maps = std::move(maps);
      maps = std::unordered_map<MapKey, CUtensorMap, MapKeyHash>();
    }
    CUtensorMap m;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * elem};
    cuuint32_t box[2] = {128u / elem, box_rows};
    cuuint32_t es[2] = {1, 1};
    const CUtensorMapDataType dt = elem == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = fn(&m, dt, 2,
                    const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return nullptr;
    return &maps.emplace(k, m).first->second;
  }
};

namespace {

enum ProfClass { P_QKV = 0, P_ATTN = 1, P_OPROJ = 2, P_FC1 = 3, P_FC2 = 4, P_LN = 5, P_OTHER = 6, P_BWD_GEMM = 7 };

// Counts the launches of one call site and, with profiling on, brackets them with events
// recorded on the launch stream.
struct ProfScope {
  esm_encoder* h;
  int cls;
  cudaStream_t st;
  cudaEvent_t e0 = nullptr;
  ProfScope(esm_encoder* h_, int cls_, cudaStream_t st_, int n) : h(h_), cls(cls_), st(st_) {
    h->launches[cls] += n;
    h->total_launches += n;
    if (h->profiling) {
      e0 = h->take_event();
      cudaEventRecord(e0, st);
    }
  }
  ~ProfScope() {
    if (h->profiling && e0) {
      cudaEvent_t e1 = h->take_event();
      cudaEventRecord(e1, st);
      h->pending.push_back({cls, e0, e1});
      if (h->pending.size() > 20000) h->drain_events();
    }
  }
};
#define PROF(h, cls, st, n, expr) \
  do {                             \
    ProfScope _ps(h, cls, st, n);  \
    expr;                          \
  } while (0)

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

PackBuffers pack_buffers(void* ws, const WsLayout& L) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  PackBuffers pb;
  pb.pos_id = reinterpret_cast<int32_t*>(b + L.pos);
  pb.seg_id = reinterpret_cast<int32_t*>(b + L.seg);
  pb.seg_start = reinterpret_cast<int32_t*>(b + L.seg_start);
  pb.seg_qlen = reinterpret_cast<int32_t*>(b + L.seg_qlen);
  pb.seg_klen = reinterpret_cast<int32_t*>(b + L.seg_klen);
  pb.work = reinterpret_cast<int32_t*>(b + L.work);
  pb.work_count = reinterpret_cast<int32_t*>(b + L.work_count);
  return pb;
}

// Every call that indexes a batch into a workspace goes through here: one that reuses the
// workspace of the last training forward overwrites its pack buffers, so the pending
// backward of that forward is withdrawn (esm_encoder_backward then returns
// ESM_ERR_INVALID_ARG); a training forward re-arms it once it is fully enqueued.
esm_status check_ws(esm_encoder* h, int T, int B, void* ws, size_t bytes, WsLayout* out) {
  if (ws != nullptr && ws == h->train_ws) h->train_buf = nullptr;
  if (ws == nullptr || !aligned(ws, 256)) return ESM_ERR_WORKSPACE;
  *out = h->layout(T, B);
  if (bytes < out->total) return ESM_ERR_WORKSPACE;
  return ESM_OK;
}

esm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ESM_OK : ESM_ERR_CUDA; }

bool weights_ok(const esm_encoder* h, const esm_weights* w) {
  if (!w || !w->emb) return false;
  const void* const* arrs[] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o,
                               w->ln2_g, w->ln2_b, w->w_1,   w->b_1,   w->w_2, w->b_2};
  for (auto a : arrs) {
    if (!a) return false;
    for (int l = 0; l < h->cfg.num_layers; ++l)
      if (!a[l] || !aligned(a[l], 16)) return false;
  }
  if (h->cfg.final_ln && (!w->lnf_g || !w->lnf_b)) return false;
  return true;
}

// The folded-LayerNorm side of a GEMM launch (see EpiArgs).
struct LnFoldArgs {
  float2* stats_out = nullptr;
  const void* gamma = nullptr;
  void* a_out = nullptr;
  const float2* stats_in = nullptr;
  const float* c = nullptr;
  const float* b = nullptr;
};

// One GEMM of a layer.  A: activation [M, K]; B: weight [N, K].
// rope_cols >= 0 overrides the RoPE column range of ESM_EPI_QKV_ROPE (0: plain bias, bf16
// out); res_in != NULL makes ESM_EPI_RESIDUAL read its residual there instead of from out;
// ln != NULL adds the folded-LayerNorm outputs (residual) or inputs (QKV / GELU).
esm_status run_gemm(esm_encoder* h, int cls, esm_epilogue epi, const void* A, const void* B, const void* bias, void* out,
                    const int32_t* pos_id, int M, int N, int K, bool fp8, Act out_act, const float* a_scale,
                    const float* b_scale, const float* o_scale, float* o_amax, cudaStream_t st, int rope_cols = -1,
                    const void* res_in = nullptr, void* aux = nullptr, const LnFoldArgs* ln = nullptr) {
  EpiArgs ea{};
  if (ln != nullptr) {
    ea.ln_stats_out = ln->stats_out;
    ea.ln_gamma = ln->gamma;
    ea.ln_a_out = ln->a_out;
    ea.ln_stats_in = ln->stats_in;
    ea.ln_c = ln->c;
    ea.ln_b = ln->b;
    ea.ln_groups = K / 64;
    ea.ln_eps = h->cfg.ln_eps;
  }
  ea.bias = bias;
  ea.bias_f32 = !h->bf16_params();
  ea.out = out;
  ea.pos_id = pos_id;
  ea.rope = h->d_rope;
  ea.rope_cols = 2 * h->cfg.hidden;
  ea.head_dim = h->cfg.hidden / h->cfg.heads;
  ea.max_pos = h->cfg.max_positions;
  ea.a_scale = a_scale;
  ea.b_scale = b_scale;
  ea.o_scale = o_scale;
  ea.o_amax = o_amax;
  ea.res_in = res_in;
  ea.aux = aux;
  if (rope_cols >= 0) ea.rope_cols = rope_cols;
  if (M <= 0) return ESM_OK;
  if (h->cfg.precision == ESM_FP32) {
    PROF(h, cls, st, epi == ESM_EPI_QKV_ROPE ? 2 : 1,
         launch_gemm_f32(epi, static_cast<const float*>(A), static_cast<const float*>(B), M, N, K, ea, st));
    return cuda_status(cudaGetLastError());
  }
  const uint32_t elem = fp8 ? 1 : 2;
  const CUtensorMap* ma = h->map(A, (uint64_t)M, (uint64_t)K, (uint32_t)gemm_tc_a_box_rows(), elem);
  const CUtensorMap* mb = h->map(B, (uint64_t)N, (uint64_t)K, (uint32_t)gemm_tc_b_box_rows(), elem);
  const uint32_t out_elem = out_act == Act::F32 ? 4u : out_act == Act::BF16 ? 2u : 1u;
  const CUtensorMap* mo = h->map(out, (uint64_t)M, (uint64_t)N, (uint32_t)gemm_tc_out_box_rows(), out_elem);
  if (!ma || !mb || !mo) return ESM_ERR_CUDA;
  cudaError_t e;
  PROF(h, cls, st, 1, e = launch_gemm_tc(epi, fp8, out_act, ma, mb, mo, M, N, K, ea, h->num_sms, h->d_err, st));
  return cuda_status(e);
}

// One layer with NVFP4 GEMMs (an FP8 handle's per-layer precision): LayerNorm -> bf16, then
// every GEMM quantises its bf16 activation and its weight to NVFP4 (current scaling: S from
// the tensor's amax in this call) and runs the block-scaled tensor-core GEMM with the layer's
// epilogue; attention stays bf16.  The tensor scales are kept in the handle (get_fp4_scales).
esm_status run_fp4_layer(esm_encoder* h, const esm_weights* w, int l, int T, const WsLayout& L, void* ws,
                         const PackBuffers& pb, cudaStream_t st) {
  const esm_config& c = h->cfg;
  uint8_t* b = static_cast<uint8_t*>(ws);
  float* x = reinterpret_cast<float*>(b + L.x);
  void* y = b + L.y;
  void* qkv = b + L.qkv;
  void* o = b + L.o;
  void* u = b + L.u;
  const int d = c.hidden, f = c.ffn, H = c.heads;
  const int tp = (T + 127) / 128 * 128;
  const size_t nf = (size_t)c.num_layers * kNumFp8Tensors;
  float* sc = h->d_fp4 + (size_t)l * kNumFp8Tensors;
  float* am = h->d_fp4 + nf + (size_t)l * kNumFp8Tensors;
  uint8_t* a_codes = b + L.fp4;
  uint8_t* a_sf = a_codes + align256((size_t)tp * f / 2);
  uint8_t* w_codes = b + L.wq;
  // act_ready: the kernel that wrote `act` accumulated its amax (from the zero set below)
  auto gemm = [&](int cls, int epi, const void* act, bool act_ready, int K, const void* wt, int N, int sx, int sw,
                  const void* bias, void* out, float* out_amax) -> esm_status {
    uint8_t* w_sf = w_codes + align256((size_t)N * K / 2);
    {
      ProfScope _ps(h, P_OTHER, st, 4);
      if (launch_nvfp4_quantize(static_cast<const __nv_bfloat16*>(act), tp, T, K, a_codes, a_sf, am + sx, sc + sx,
                                act_ready, h->num_sms, st) != cudaSuccess ||
          launch_nvfp4_quantize(static_cast<const __nv_bfloat16*>(wt), N, N, K, w_codes, w_sf, am + sw, sc + sw,
                                false, h->num_sms, st) != cudaSuccess)
        return ESM_ERR_CUDA;
    }
    const CUtensorMap* ma = h->map(a_codes, (uint64_t)tp, (uint64_t)K / 2, 128, 1);
    const CUtensorMap* mb = h->map(w_codes, (uint64_t)N, (uint64_t)K / 2, 128, 1);
    if (!ma || !mb) return ESM_ERR_CUDA;
    Fp4Epi ea{};
    ea.bias = bias;
    ea.out = out;
    ea.rows_valid = T;
    ea.pos_id = pb.pos_id;
    ea.rope = h->d_rope;
    ea.rope_cols = 2 * d;
    ea.max_pos = c.max_positions;
    ea.amax = out_amax;
    cudaError_t e;
    PROF(h, cls, st, 1,
         e = launch_gemm_nvfp4(epi, ma, mb, a_sf, w_sf, sc + sx, sc + sw, ea, tp, N, K, h->num_sms, h->d_err, st));
    return cuda_status(e);
  };
  esm_status s;
  // the layer's amaxes start from zero; LN1, LN2, the attention and fc1's GELU epilogue fold theirs in
  if (cudaMemsetAsync(am, 0, kNumFp8Tensors * sizeof(float), st) != cudaSuccess) return ESM_ERR_CUDA;
  PROF(h, P_LN, st, 1,
       launch_layernorm(x, w->ln1_g[l], w->ln1_b[l], false, y, Act::BF16, T, d, c.ln_eps, nullptr, am + X_QKV,
                        nullptr, nullptr, nullptr, st));
  if ((s = gemm(P_QKV, kFp4QkvRope, y, true, d, w->w_qkv[l], 3 * d, X_QKV, W_QKV, w->b_qkv[l], qkv, nullptr)) !=
      ESM_OK)
    return s;
  {
    ProfScope _ps(h, P_ATTN, st, 1);
    const CUtensorMap* tq = h->map(qkv, (uint64_t)T, (uint64_t)3 * d, 128, 2);
    if (!tq) return ESM_ERR_CUDA;
    // the attention output's amax comes from the attention kernel (so its quantisation is one pass)
    if (launch_attention_tc(tq, o, Act::BF16, d, H, L.max_items, pb, nullptr, am + X_O, h->d_err, st) != cudaSuccess)
      return ESM_ERR_CUDA;
  }
  if ((s = gemm(P_OPROJ, kFp4Residual, o, true, d, w->w_o[l], d, X_O, W_O, w->b_o[l], x, nullptr)) != ESM_OK)
    return s;
  PROF(h, P_LN, st, 1,
       launch_layernorm(x, w->ln2_g[l], w->ln2_b[l], false, y, Act::BF16, T, d, c.ln_eps, nullptr, am + X_1, nullptr,
                        nullptr, nullptr, st));
  if ((s = gemm(P_FC1, kFp4Gelu, y, true, d, w->w_1[l], f, X_1, W_1, w->b_1[l], u, am + X_2)) != ESM_OK) return s;
  return gemm(P_FC2, kFp4Residual, u, true, f, w->w_2[l], d, X_2, W_2, w->b_2[l], x, nullptr);
}

// The layer stack over an already indexed batch (pack buffers filled, x = embedding).
esm_status run_layers(esm_encoder* h, const esm_weights* w, int T, int max_items, const WsLayout& L, void* ws,
                      void* out, bool padded, cudaStream_t st) {
  const esm_config& c = h->cfg;
  uint8_t* b = static_cast<uint8_t*>(ws);
  PackBuffers pb = pack_buffers(ws, L);
  float* x = reinterpret_cast<float*>(b + L.x);
  void* y = b + L.y;
  void* qkv = b + L.qkv;
  void* o = b + L.o;
  void* u = b + L.u;
  const int d = c.hidden, f = c.ffn, H = c.heads;
  const bool pf32 = !h->bf16_params();
  const Act act = h->act();
  esm_status s;
  // bf16 forward: every LayerNorm but the first and the final one is folded into the GEMMs
  // around it.  The residual epilogue of the out-projection (fc2) leaves the row statistics
  // and bf16(x * gamma2) (bf16(x * gamma1) of the next layer); fc1 (the next QKV projection)
  // applies rstd (acc - mean c) + b' with the per-layer constants computed here.
  const bool fold = c.precision == ESM_BF16 && d <= 4096;
  float2* ln_stats = reinterpret_cast<float2*>(b + L.ln_stats);
  float* ln_fold = reinterpret_cast<float*>(b + L.ln_fold);
  auto fold_c = [&](int l, int which) -> float* {  // which: 0 c_qkv, 1 b'_qkv, 2 c_1, 3 b'_1
    float* base = ln_fold + (size_t)l * (6 * d + 2 * f);
    return which < 2 ? base + (size_t)which * 3 * d : base + 6 * (size_t)d + (size_t)(which - 2) * f;
  };
  if (fold) {
    ProfScope _ps(h, P_OTHER, st, (2 * c.num_layers + kLnFoldMaxJobs - 1) / kLnFoldMaxJobs);
    LnFoldJob jobs[kLnFoldMaxJobs];
    int n = 0;
    for (int l = 0; l < c.num_layers; ++l) {
      jobs[n++] = LnFoldJob{w->w_qkv[l], w->ln1_g[l], w->ln1_b[l], w->b_qkv[l], fold_c(l, 0), fold_c(l, 1), 3 * d};
      jobs[n++] = LnFoldJob{w->w_1[l], w->ln2_g[l], w->ln2_b[l], w->b_1[l], fold_c(l, 2), fold_c(l, 3), f};
      if (n + 2 > kLnFoldMaxJobs || l + 1 == c.num_layers) {
        launch_ln_fold(jobs, n, d, st);
        n = 0;
      }
    }
  }
  for (int l = 0; l < c.num_layers; ++l) {
    const bool fp8 = c.precision == ESM_FP8_E4M3 && h->layer_fp8[l] == 1;
    if (c.precision == ESM_FP8_E4M3 && h->layer_fp8[l] == 2) {
      if ((s = run_fp4_layer(h, w, l, T, L, ws, pb, st)) != ESM_OK) return s;
      continue;
    }
    float* sc = h->fp8_scale() + (size_t)l * kNumFp8Tensors;
    float* am = h->fp8_amax() + (size_t)l * kNumFp8Tensors;
    uint8_t* wq_qkv = b + L.wq;
    uint8_t* wq_o = wq_qkv + (size_t)3 * d * d;
    uint8_t* wq_1 = wq_o + (size_t)d * d;
    uint8_t* wq_2 = wq_1 + (size_t)f * d;
    if (fp8) {
      ProfScope _ps(h, P_OTHER, st, 4);
      launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(w->w_qkv[l]), wq_qkv, (size_t)3 * d * d, sc + W_QKV,
                           am + W_QKV, st);
      launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(w->w_o[l]), wq_o, (size_t)d * d, sc + W_O, am + W_O, st);
      launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(w->w_1[l]), wq_1, (size_t)f * d, sc + W_1, am + W_1, st);
      launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(w->w_2[l]), wq_2, (size_t)d * f, sc + W_2, am + W_2, st);
    }
    // ---- attention block
    LnFoldArgs ln_qkv;
    if (fold && l > 0) {  // y = bf16(x * gamma1) and the row statistics from the last fc2
      ln_qkv.stats_in = ln_stats;
      ln_qkv.c = fold_c(l, 0);
      ln_qkv.b = fold_c(l, 1);
    } else {
      PROF(h, P_LN, st, 1,
           launch_layernorm(x, w->ln1_g[l], w->ln1_b[l], pf32, y, fp8 ? Act::E4M3 : act, T, d, c.ln_eps, sc + X_QKV,
                            fp8 ? am + X_QKV : nullptr, nullptr, nullptr, nullptr, st));
    }
    s = run_gemm(h, P_QKV, ESM_EPI_QKV_ROPE, y, fp8 ? (const void*)wq_qkv : w->w_qkv[l], w->b_qkv[l], qkv, pb.pos_id, T,
                 3 * d, d, fp8, act, sc + X_QKV, sc + W_QKV, nullptr, nullptr, st, -1, nullptr, nullptr,
                 fold && l > 0 ? &ln_qkv : nullptr);
    if (s != ESM_OK) return s;
    {
      ProfScope _ps(h, P_ATTN, st, 1);
      if (c.precision == ESM_FP32)
        launch_attention_f32(static_cast<const float*>(qkv), static_cast<float*>(o), d, H, T, pb, st);
      else {
        const CUtensorMap* tq = h->map(qkv, (uint64_t)T, (uint64_t)3 * d, 128, 2);
        if (!tq) return ESM_ERR_CUDA;
        if (launch_attention_tc(tq, o, fp8 ? Act::E4M3 : Act::BF16, d, H, max_items, pb, sc + X_O,
                                fp8 ? am + X_O : nullptr, h->d_err, st) != cudaSuccess)
          return ESM_ERR_CUDA;
      }
    }
    LnFoldArgs ln_out;  // out-projection: statistics and bf16(x * gamma2) for fc1
    if (fold) {
      ln_out.stats_out = ln_stats;
      ln_out.gamma = w->ln2_g[l];
      ln_out.a_out = y;
    }
    s = run_gemm(h, P_OPROJ, ESM_EPI_RESIDUAL, o, fp8 ? (const void*)wq_o : w->w_o[l], w->b_o[l], x, nullptr, T, d, d, fp8,
                 Act::F32, sc + X_O, sc + W_O, nullptr, nullptr, st, -1, nullptr, nullptr, fold ? &ln_out : nullptr);
    if (s != ESM_OK) return s;
    // ---- MLP block
    LnFoldArgs ln_fc1;
    if (fold) {
      ln_fc1.stats_in = ln_stats;
      ln_fc1.c = fold_c(l, 2);
      ln_fc1.b = fold_c(l, 3);
    } else {
      PROF(h, P_LN, st, 1,
           launch_layernorm(x, w->ln2_g[l], w->ln2_b[l], pf32, y, fp8 ? Act::E4M3 : act, T, d, c.ln_eps, sc + X_1,
                            fp8 ? am + X_1 : nullptr, nullptr, nullptr, nullptr, st));
    }
    s = run_gemm(h, P_FC1, ESM_EPI_GELU, y, fp8 ? (const void*)wq_1 : w->w_1[l], w->b_1[l], u, nullptr, T, f, d, fp8,
                 fp8 ? Act::E4M3 : act, sc + X_1, sc + W_1, sc + X_2, am + X_2, st, -1, nullptr, nullptr,
                 fold ? &ln_fc1 : nullptr);
    if (s != ESM_OK) return s;
    LnFoldArgs ln_fc2;  // fc2: statistics and bf16(x * gamma1) for the next layer's QKV
    const bool fold_next = fold && l + 1 < c.num_layers;
    if (fold_next) {
      ln_fc2.stats_out = ln_stats;
      ln_fc2.gamma = w->ln1_g[l + 1];
      ln_fc2.a_out = y;
    }
    s = run_gemm(h, P_FC2, ESM_EPI_RESIDUAL, u, fp8 ? (const void*)wq_2 : w->w_2[l], w->b_2[l], x, nullptr, T, d, f, fp8,
                 Act::F32, sc + X_2, sc + W_2, nullptr, nullptr, st, -1, nullptr, nullptr, fold_next ? &ln_fc2 : nullptr);
    if (s != ESM_OK) return s;
  }
  const int32_t* vp = padded ? pb.pos_id : nullptr;
  const int32_t* vs = padded ? pb.seg_id : nullptr;
  const int32_t* vk = padded ? pb.seg_klen : nullptr;
  if (c.final_ln)
    PROF(h, P_LN, st, 1,
         launch_layernorm(x, w->lnf_g, w->lnf_b, pf32, out, act, T, d, c.ln_eps, nullptr, nullptr, vp, vs, vk, st));
  else
    PROF(h, P_OTHER, st, 1, launch_copy_out(x, out, act, T, d, vp, vs, vk, st));
  if (c.precision == ESM_FP8_E4M3)
    PROF(h, P_OTHER, st, 1, launch_fp8_update(h->fp8_scale(), h->fp8_hist(), h->fp8_amax(), c.num_layers * kNumFp8Tensors,
                      c.amax_history_len, st));
  return cuda_status(cudaGetLastError());
}

esm_status forward_impl(esm_encoder* h, const esm_weights* w, const int32_t* tok, const int32_t* cu, int B, int T,
                        int max_seqlen, void* out, void* ws, size_t ws_bytes, cudaStream_t st) {
  WsLayout L;
  esm_status s = check_ws(h, T, B, ws, ws_bytes, &L);
  if (s != ESM_OK) return s;
  PackBuffers pb = pack_buffers(ws, L);
  uint8_t* b = static_cast<uint8_t*>(ws);
  if (cudaMemsetAsync(pb.pos_id, 0, 4 * (size_t)T, st) != cudaSuccess) return ESM_ERR_CUDA;
  if (cudaMemsetAsync(pb.seg_id, 0, 4 * (size_t)T, st) != cudaSuccess) return ESM_ERR_CUDA;
  {
    ProfScope _ps(h, P_OTHER, st, h->cfg.precision != ESM_FP32 ? 3 : 2);
    launch_pack_index(cu, B, T, max_seqlen, h->cfg.max_positions, pb, h->d_err, st);
    if (h->cfg.precision != ESM_FP32) launch_attn_worklist(B, L.max_items, kAttnQTileTc, pb, st);
    launch_embed(tok, T, w->emb, !h->bf16_params(), h->cfg.vocab, h->cfg.hidden, h->cfg.emb_scale,
                 reinterpret_cast<float*>(b + L.x), h->d_err, st);
  }
  return run_layers(h, w, T, L.max_items, L, ws, out, false, st);
}

bool config_ok(const esm_config* c) {
  if (!c) return false;
  if (c->num_layers < 0 || c->hidden <= 0 || c->heads <= 0 || c->ffn <= 0 || c->vocab <= 0) return false;
  if (c->hidden % c->heads) return false;
  if (c->max_positions <= 0 || c->max_positions > 65536) return false;
  if (!(c->ln_eps >= 0.f) || !(c->rope_base > 0.f)) return false;
  if (c->amax_history_len < 1 || c->amax_history_len > 1024) return false;
  const int dh = c->hidden / c->heads;
  if (c->precision == ESM_FP32) {
    return dh % 2 == 0 && dh <= 64 && c->hidden % 4 == 0 && c->hidden <= 4096;
  }
  if (c->precision == ESM_BF16 || c->precision == ESM_FP8_E4M3) {
    if (dh != 64 || c->hidden % 256 || c->ffn % 256) return false;
    if (c->precision == ESM_FP8_E4M3 && (c->hidden % 128 || c->ffn % 128)) return false;
    return c->hidden <= 4096 * 4;
  }
  return false;
}

// ------------------------------------------------------------------ training (backward)
// Buffer of a training forward: every activation the backward reads, per layer, plus the
// backward's scratch.  Per-layer tensors are slabs of layers (x: layers + 1) of one size.
struct TrainLayout {
  size_t tok, x, xmid, y1, qkv, o, lse, y2, z, u;                        // bases
  size_t sx, sy, sqkv, slse, sz;                                         // slab strides
  size_t dx, dxb, dy, dz, dob, dqkv, dqacc, dsum, partial, split, embp;  // scratch
  size_t split_floats, total;
};

constexpr int kMaxKSplit = 8;

TrainLayout train_layout(const esm_config& c, int Tm) {
  TrainLayout L{};
  const size_t T = Tm > 0 ? Tm : 1, d = c.hidden, f = c.ffn, H = c.heads, nl = c.num_layers > 0 ? c.num_layers : 0;
  L.sx = align256(4 * T * d);
  L.sy = align256(2 * T * d);
  L.sqkv = align256(2 * T * 3 * d);
  L.slse = align256(4 * T * H);
  L.sz = align256(2 * T * f);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.tok = take(4 * T);
  L.x = take(L.sx * (nl + 1));
  L.xmid = take(L.sx * nl);
  L.y1 = take(L.sy * nl);
  L.qkv = take(L.sqkv * nl);
  L.o = take(L.sy * nl);
  L.lse = take(L.slse * nl);
  L.y2 = take(L.sy * nl);
  L.z = take(L.sz * nl);
  L.u = take(L.sz * nl);
  L.dx = take(4 * T * d);
  L.dxb = take(2 * T * d);
  L.dy = take(4 * T * d);
  L.dz = take(2 * T * f);
  L.dob = take(2 * T * d);
  L.dqkv = take(2 * T * 3 * d);
  L.dqacc = take(4 * T * d);
  L.dsum = take(4 * T * H);
  const size_t widest = std::max(3 * d, f);
  L.partial = take(4 * bwd_partial_floats((int)T, (int)widest));
  L.split_floats = (size_t)kMaxKSplit * std::max(f * d, 3 * d * d);
  L.split = take(4 * L.split_floats);
  L.embp = take(4 * emb_bwd_partial_floats((int)T, c.vocab, (int)d));
  L.total = off;
  return L;
}

// Split of the token reduction of a weight gradient: tiles x splits work items over the
// clusters, fewest rounds per unit of work (ties to fewer splits).
int choose_ksplit(int tiles, int kb_total, int clusters) {
  int best = 1;
  double best_cost = 1e30;
  for (int ks = 1; ks <= kMaxKSplit && ks <= kb_total; ++ks) {
    const double rounds = (double)((tiles * ks + clusters - 1) / clusters);
    const double cost = rounds / ks + 0.02 * ks;  // small charge for the partial-sum pass
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = ks;
    }
  }
  return best;
}

// out[M, K] = dY[M, N] W with W stored [N, K] (bf16); fp32 or bf16 out; with gelu_z
// (bf16 [M, K], the forward's fc1 pre-activation) the bf16 out is multiplied by GELU'(z).
esm_status run_dgrad(esm_encoder* h, const void* dY, const void* W, void* out, bool out_bf16, int M, int N, int K,
                     cudaStream_t st, const void* gelu_z = nullptr) {
  if (M <= 0) return ESM_OK;
  const CUtensorMap* ma = h->map(dY, (uint64_t)M, (uint64_t)N, (uint32_t)gemm_tc_a_box_rows(), 2);
  const CUtensorMap* mb = h->map(W, (uint64_t)N, (uint64_t)K, (uint32_t)gemm_tc_mn_box_rows(), 2);
  const CUtensorMap* mo = h->map(out, (uint64_t)M, (uint64_t)K, (uint32_t)gemm_tc_out_box_rows(), out_bf16 ? 2u : 4u);
  if (!ma || !mb || !mo) return ESM_ERR_CUDA;
  EpiArgs ea{};
  ea.out = out;
  ea.rope_cols = 0;
  ea.aux = const_cast<void*>(gelu_z);
  const GemmBwd kind = gelu_z ? GemmBwd::DGRAD_GELU : out_bf16 ? GemmBwd::DGRAD_BF16 : GemmBwd::DGRAD_F32;
  cudaError_t e;
  PROF(h, P_BWD_GEMM, st, 1, e = launch_gemm_tc_bwd(kind, ma, mb, mo, M, K, N, 1, ea, h->num_sms, h->d_err, st));
  return cuda_status(e);
}

// dW[N, K] = dY^T X over M rows: dY [M, N], X [M, K] (bf16); fp32 out.  split: scratch of
// split_floats floats for the split-K partial products.
esm_status run_wgrad(esm_encoder* h, const void* dY, const void* X, float* dW, int M, int N, int K, float* split,
                     size_t split_floats, cudaStream_t st) {
  if (M <= 0) return cuda_status(cudaMemsetAsync(dW, 0, sizeof(float) * (size_t)N * K, st));
  const int tiles = (N / 256) * (K / 256);
  const int kb_total = (M + 63) / 64;
  int ks = choose_ksplit(tiles, kb_total, gemm_tc_max_clusters(h->num_sms));
  while (ks > 1 && (size_t)ks * N * K > split_floats) --ks;
  ks = (kb_total + (kb_total + ks - 1) / ks - 1) / ((kb_total + ks - 1) / ks);  // no empty split
  float* out = ks > 1 ? split : dW;
  const CUtensorMap* ma = h->map(dY, (uint64_t)M, (uint64_t)N, (uint32_t)gemm_tc_mn_box_rows(), 2);
  const CUtensorMap* mb = h->map(X, (uint64_t)M, (uint64_t)K, (uint32_t)gemm_tc_mn_box_rows(), 2);
  const CUtensorMap* mo = h->map(out, (uint64_t)ks * N, (uint64_t)K, (uint32_t)gemm_tc_out_box_rows(), 4);
  if (!ma || !mb || !mo) return ESM_ERR_CUDA;
  EpiArgs ea{};
  ea.out = out;
  ea.rope_cols = 0;
  cudaError_t e;
  PROF(h, P_BWD_GEMM, st, 1,
       e = launch_gemm_tc_bwd(GemmBwd::WGRAD_F32, ma, mb, mo, N, K, M, ks, ea, h->num_sms, h->d_err, st));
  if (e != cudaSuccess) return ESM_ERR_CUDA;
  if (ks > 1) PROF(h, P_BWD_GEMM, st, 1, launch_reduce_splits(split, ks, (size_t)N * K, dW, st));
  return cuda_status(cudaGetLastError());
}

bool grads_ok(const esm_encoder* h, const esm_grads* g) {
  if (!g || !g->emb || !aligned(g->emb, 16)) return false;
  float* const* arrs[] = {g->ln1_g, g->ln1_b, g->w_qkv, g->b_qkv, g->w_o, g->b_o,
                          g->ln2_g, g->ln2_b, g->w_1,   g->b_1,   g->w_2, g->b_2};
  for (auto a : arrs) {
    if (!a) return false;
    for (int l = 0; l < h->cfg.num_layers; ++l)
      if (!a[l] || !aligned(a[l], 16)) return false;
  }
  if (h->cfg.final_ln && (!g->lnf_g || !g->lnf_b)) return false;
  return true;
}

esm_status train_forward_impl(esm_encoder* h, const esm_weights* w, const int32_t* tok, const int32_t* cu, int B, int T,
                              int max_seqlen, void* out, void* train, void* ws, size_t ws_bytes, cudaStream_t st) {
  WsLayout L;
  esm_status s = check_ws(h, T, B, ws, ws_bytes, &L);
  if (s != ESM_OK) return s;
  const esm_config& c = h->cfg;
  const TrainLayout R = train_layout(c, T);
  uint8_t* tb = static_cast<uint8_t*>(train);
  PackBuffers pb = pack_buffers(ws, L);
  if (cudaMemsetAsync(pb.pos_id, 0, 4 * (size_t)T, st) != cudaSuccess) return ESM_ERR_CUDA;
  if (cudaMemsetAsync(pb.seg_id, 0, 4 * (size_t)T, st) != cudaSuccess) return ESM_ERR_CUDA;
  if (cudaMemcpyAsync(tb + R.tok, tok, 4 * (size_t)T, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return ESM_ERR_CUDA;
  const int d = c.hidden, f = c.ffn, H = c.heads;
  {
    ProfScope _ps(h, P_OTHER, st, 3);
    launch_pack_index(cu, B, T, max_seqlen, c.max_positions, pb, h->d_err, st);
    launch_attn_worklist(B, L.max_items, kAttnQTileTc, pb, st);
    launch_embed(tok, T, w->emb, false, c.vocab, d, c.emb_scale, reinterpret_cast<float*>(tb + R.x), h->d_err, st);
  }
  for (int l = 0; l < c.num_layers; ++l) {
    float* x = reinterpret_cast<float*>(tb + R.x + R.sx * l);
    float* xmid = reinterpret_cast<float*>(tb + R.xmid + R.sx * l);
    float* xnext = reinterpret_cast<float*>(tb + R.x + R.sx * (l + 1));
    void* y1 = tb + R.y1 + R.sy * l;
    void* qkv = tb + R.qkv + R.sqkv * l;
    void* o = tb + R.o + R.sy * l;
    float* lse = reinterpret_cast<float*>(tb + R.lse + R.slse * l);
    void* y2 = tb + R.y2 + R.sy * l;
    void* z = tb + R.z + R.sz * l;
    void* u = tb + R.u + R.sz * l;
    PROF(h, P_LN, st, 1,
         launch_layernorm(x, w->ln1_g[l], w->ln1_b[l], false, y1, Act::BF16, T, d, c.ln_eps, nullptr, nullptr, nullptr,
                          nullptr, nullptr, st));
    s = run_gemm(h, P_QKV, ESM_EPI_QKV_ROPE, y1, w->w_qkv[l], w->b_qkv[l], qkv, pb.pos_id, T, 3 * d, d, false,
                 Act::BF16, nullptr, nullptr, nullptr, nullptr, st);
    if (s != ESM_OK) return s;
    {
      ProfScope _ps(h, P_ATTN, st, 1);
      const CUtensorMap* tq = h->map(qkv, (uint64_t)T, (uint64_t)3 * d, 128, 2);
      if (!tq) return ESM_ERR_CUDA;
      if (launch_attention_tc(tq, o, Act::BF16, d, H, L.max_items, pb, nullptr, nullptr, h->d_err, st, lse, T) !=
          cudaSuccess)
        return ESM_ERR_CUDA;
    }
    s = run_gemm(h, P_OPROJ, ESM_EPI_RESIDUAL, o, w->w_o[l], w->b_o[l], xmid, nullptr, T, d, d, false, Act::F32,
                 nullptr, nullptr, nullptr, nullptr, st, -1, x);
    if (s != ESM_OK) return s;
    PROF(h, P_LN, st, 1,
         launch_layernorm(xmid, w->ln2_g[l], w->ln2_b[l], false, y2, Act::BF16, T, d, c.ln_eps, nullptr, nullptr,
                          nullptr, nullptr, nullptr, st));
    // fc1: u = GELU(z) feeds fc2; the epilogue also keeps the pre-activation z for GELU'(z)
    s = run_gemm(h, P_FC1, ESM_EPI_GELU, y2, w->w_1[l], w->b_1[l], u, nullptr, T, f, d, false, Act::BF16, nullptr,
                 nullptr, nullptr, nullptr, st, -1, nullptr, z);
    if (s != ESM_OK) return s;
    s = run_gemm(h, P_FC2, ESM_EPI_RESIDUAL, u, w->w_2[l], w->b_2[l], xnext, nullptr, T, d, f, false, Act::F32, nullptr,
                 nullptr, nullptr, nullptr, st, -1, xmid);
    if (s != ESM_OK) return s;
  }
  const float* xl = reinterpret_cast<const float*>(tb + R.x + R.sx * c.num_layers);
  if (c.final_ln)
    PROF(h, P_LN, st, 1,
         launch_layernorm(xl, w->lnf_g, w->lnf_b, false, out, Act::BF16, T, d, c.ln_eps, nullptr, nullptr, nullptr,
                          nullptr, nullptr, st));
  else
    PROF(h, P_OTHER, st, 1, launch_copy_out(xl, out, Act::BF16, T, d, nullptr, nullptr, nullptr, st));
  h->train_T = T;
  h->train_B = B;
  h->train_items = L.max_items;
  h->train_buf = train;
  h->train_ws = ws;
  return cuda_status(cudaGetLastError());
}

esm_status backward_impl(esm_encoder* h, const esm_weights* w, const float* d_out, const esm_grads* g, void* train,
                         void* ws, cudaStream_t st) {
  const esm_config& c = h->cfg;
  const int T = h->train_T, d = c.hidden, f = c.ffn, H = c.heads;
  const TrainLayout R = train_layout(c, T);
  const WsLayout L = h->layout(T, h->train_B);
  PackBuffers pb = pack_buffers(ws, L);
  uint8_t* tb = static_cast<uint8_t*>(train);
  float* dx = reinterpret_cast<float*>(tb + R.dx);
  __nv_bfloat16* dxb = reinterpret_cast<__nv_bfloat16*>(tb + R.dxb);
  float* dy = reinterpret_cast<float*>(tb + R.dy);
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(tb + R.dz);
  __nv_bfloat16* dob = reinterpret_cast<__nv_bfloat16*>(tb + R.dob);
  __nv_bfloat16* dqkv = reinterpret_cast<__nv_bfloat16*>(tb + R.dqkv);
  float* dqacc = reinterpret_cast<float*>(tb + R.dqacc);
  float* dsum = reinterpret_cast<float*>(tb + R.dsum);
  float* partial = reinterpret_cast<float*>(tb + R.partial);
  float* split = reinterpret_cast<float*>(tb + R.split);
  float* embp = reinterpret_cast<float*>(tb + R.embp);
  esm_status s;
  // final LayerNorm (or the identity)
  const float* xl = reinterpret_cast<const float*>(tb + R.x + R.sx * c.num_layers);
  if (c.final_ln) {
    PROF(h, P_LN, st, 4,
         launch_ln_bwd(xl, w->lnf_g, false, d_out, nullptr, dx, g->lnf_g, g->lnf_b, partial, T, d, c.ln_eps, st));
  } else if (cudaMemcpyAsync(dx, d_out, 4 * (size_t)T * d, cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
    return ESM_ERR_CUDA;
  }
  for (int l = c.num_layers - 1; l >= 0; --l) {
    const float* x = reinterpret_cast<const float*>(tb + R.x + R.sx * l);
    const float* xmid = reinterpret_cast<const float*>(tb + R.xmid + R.sx * l);
    const void* y1 = tb + R.y1 + R.sy * l;
    const void* qkv = tb + R.qkv + R.sqkv * l;
    const void* o = tb + R.o + R.sy * l;
    const float* lse = reinterpret_cast<const float*>(tb + R.lse + R.slse * l);
    const void* y2 = tb + R.y2 + R.sy * l;
    const void* z = tb + R.z + R.sz * l;
    const void* u = tb + R.u + R.sz * l;
    // ---- MLP block: x_{l+1} = xmid + GELU(LN2(xmid) W1^T + b1) W2^T + b2
    PROF(h, P_OTHER, st, 2, launch_colsum(dx, false, T, d, g->b_2[l], partial, dxb, st));
    if ((s = run_wgrad(h, dxb, u, g->w_2[l], T, d, f, split, R.split_floats, st)) != ESM_OK) return s;
    // dz = (dx W2) * GELU'(z), in the input-gradient GEMM's epilogue
    if ((s = run_dgrad(h, dxb, w->w_2[l], dz, true, T, d, f, st, z)) != ESM_OK) return s;
    PROF(h, P_OTHER, st, 2, launch_colsum(dz, true, T, f, g->b_1[l], partial, nullptr, st));
    if ((s = run_wgrad(h, dz, y2, g->w_1[l], T, f, d, split, R.split_floats, st)) != ESM_OK) return s;
    if ((s = run_dgrad(h, dz, w->w_1[l], dy, false, T, f, d, st)) != ESM_OK) return s;
    PROF(h, P_LN, st, 4,
         launch_ln_bwd(xmid, w->ln2_g[l], false, dy, dx, dx, g->ln2_g[l], g->ln2_b[l], partial, T, d, c.ln_eps,
                       st));
    // ---- attention block: xmid = x + Attn(LN1(x)) Wo^T + bo
    PROF(h, P_OTHER, st, 2, launch_colsum(dx, false, T, d, g->b_o[l], partial, dxb, st));
    if ((s = run_wgrad(h, dxb, o, g->w_o[l], T, d, d, split, R.split_floats, st)) != ESM_OK) return s;
    if ((s = run_dgrad(h, dxb, w->w_o[l], dob, true, T, d, d, st)) != ESM_OK) return s;
    {
      ProfScope _ps(h, P_ATTN, st, 4);
      const CUtensorMap* tq = h->map(qkv, (uint64_t)T, (uint64_t)3 * d, 128, 2);
      const CUtensorMap* td = h->map(dob, (uint64_t)T, (uint64_t)d, 128, 2);
      const CUtensorMap* tdq = h->map(dqacc, (uint64_t)T, (uint64_t)d, 32, 4);
      if (!tq || !td || !tdq) return ESM_ERR_CUDA;
      if (launch_attention_bwd_tc(tq, td, tdq, static_cast<const __nv_bfloat16*>(o), dob, lse, dsum, dqacc, dqkv, T, d, H,
                                  h->train_items, pb, h->d_rope, c.max_positions, h->num_sms, h->d_err,
                                  st) != cudaSuccess)
        return ESM_ERR_CUDA;
    }
    PROF(h, P_OTHER, st, 2, launch_colsum(dqkv, true, T, 3 * d, g->b_qkv[l], partial, nullptr, st));
    if ((s = run_wgrad(h, dqkv, y1, g->w_qkv[l], T, 3 * d, d, split, R.split_floats, st)) != ESM_OK) return s;
    if ((s = run_dgrad(h, dqkv, w->w_qkv[l], dy, false, T, 3 * d, d, st)) != ESM_OK) return s;
    PROF(h, P_LN, st, 4,
         launch_ln_bwd(x, w->ln1_g[l], false, dy, dx, dx, g->ln1_g[l], g->ln1_b[l], partial, T, d, c.ln_eps, st));
  }
  PROF(h, P_OTHER, st, 2,
       launch_emb_bwd(dx, reinterpret_cast<const int32_t*>(tb + R.tok), T, d, c.vocab, c.emb_scale, embp, g->emb, st));
  return cuda_status(cudaGetLastError());
}

}  // namespace

bool esm::encode_attention_qkv_map(const void* qkv, int total_tokens, int hidden, CUtensorMap* out) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !qkv || !out || total_tokens <= 0 || hidden <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)3 * hidden, (cuuint64_t)total_tokens};
  cuuint64_t strides[1] = {(cuuint64_t)3 * hidden * 2};
  cuuint32_t box[2] = {64u, 128u};
  cuuint32_t es[2] = {1, 1};
  return fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

extern "C" {

const char* esm_status_string(esm_status s) {
  switch (s) {
    case ESM_OK: return "ok";
    case ESM_ERR_INVALID_ARG: return "invalid argument";
    case ESM_ERR_UNSUPPORTED: return "unsupported device or geometry";
    case ESM_ERR_BAD_CU_SEQLENS: return "malformed cu_seqlens / sequence lengths";
    case ESM_ERR_TOKEN_RANGE: return "token id out of range";
    case ESM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ESM_ERR_CUDA: return "CUDA runtime error";
    case ESM_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

esm_status esm_encoder_create(const esm_config* cfg, esm_encoder_t** out) {
  if (!out) return ESM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return ESM_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ESM_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ESM_ERR_CUDA;
  if (major != 10 || minor != 3) return ESM_ERR_UNSUPPORTED;
  if (!config_ok(cfg)) {
    if (cfg->precision == ESM_FP4_E2M1) return ESM_ERR_UNSUPPORTED;  // named on the pages, no kernels here
    if (cfg->precision != ESM_FP32 && cfg->precision != ESM_BF16 && cfg->precision != ESM_FP8_E4M3)
      return ESM_ERR_INVALID_ARG;
    return (cfg->hidden > 0 && cfg->heads > 0 && cfg->num_layers >= 0) ? ESM_ERR_UNSUPPORTED : ESM_ERR_INVALID_ARG;
  }
  esm_encoder* h = new esm_encoder();
  h->cfg = *cfg;
  h->layer_fp8.assign((size_t)(cfg->num_layers > 0 ? cfg->num_layers : 0), cfg->precision == ESM_FP8_E4M3 ? 1 : 0);
  h->device = dev;
  h->num_sms = sms;
  const size_t nf = (size_t)cfg->num_layers * kNumFp8Tensors;
  h->fp8_floats = nf * (1 + cfg->amax_history_len);
  bool ok = cudaMalloc(&h->d_err, sizeof(unsigned)) == cudaSuccess &&
            cudaMalloc(&h->d_rope, sizeof(float2) * (size_t)cfg->max_positions * kRopeMaxHalf) == cudaSuccess &&
            cudaMalloc(&h->d_fp8, sizeof(float) * (h->fp8_floats + nf + 1)) == cudaSuccess &&
            cudaMalloc(&h->d_fp4, sizeof(float) * (2 * nf + 1)) == cudaSuccess;
  if (ok) {
    ok = cudaMemset(h->d_err, 0, sizeof(unsigned)) == cudaSuccess &&
         cudaMemset(h->d_fp8, 0, sizeof(float) * (h->fp8_floats + nf + 1)) == cudaSuccess &&
         cudaMemset(h->d_fp4, 0, sizeof(float) * (2 * nf + 1)) == cudaSuccess;
    std::vector<float> ones(nf, 1.0f);
    if (ok && nf) ok = cudaMemcpy(h->d_fp8, ones.data(), nf * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess;
    if (ok) {
      launch_rope_table(h->d_rope, cfg->max_positions, (cfg->hidden / cfg->heads) / 2, cfg->rope_base, 0);
      ok = cudaGetLastError() == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess;
    }
  }
  if (!ok) {
    esm_encoder_destroy(h);
    return ESM_ERR_CUDA;
  }
  *out = h;
  return ESM_OK;
}

void esm_encoder_destroy(esm_encoder_t* h) {
  if (!h) return;
  for (auto& g : h->host_graphs) cudaGraphExecDestroy(g.exec);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->d_err) cudaFree(h->d_err);
  if (h->d_rope) cudaFree(h->d_rope);
  if (h->d_fp8) cudaFree(h->d_fp8);
  if (h->d_fp4) cudaFree(h->d_fp4);
  h->drain_events();
  for (cudaEvent_t e : h->event_pool) cudaEventDestroy(e);
  delete h;
}

esm_status esm_encoder_workspace_size(const esm_encoder_t* h, int max_tokens, int max_seqs, size_t* bytes) {
  if (!h || !bytes || max_tokens < 0 || max_seqs < 0) return ESM_ERR_INVALID_ARG;
  *bytes = h->layout(max_tokens, max_seqs).total;
  return ESM_OK;
}

esm_status esm_encoder_forward(esm_encoder_t* h, const esm_weights* w, const int32_t* token_ids,
                               const int32_t* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                               void* hidden_out, void* workspace, size_t workspace_bytes, esm_stream_t stream) {
  if (!h || total_tokens < 0 || num_seqs < 0) return ESM_ERR_INVALID_ARG;
  if (total_tokens == 0) return ESM_OK;
  if (num_seqs == 0 || !token_ids || !cu_seqlens || !hidden_out || !aligned(hidden_out, 16)) return ESM_ERR_INVALID_ARG;
  if (max_seqlen <= 0 || max_seqlen > h->cfg.max_positions) return ESM_ERR_INVALID_ARG;
  if (!weights_ok(h, w)) return ESM_ERR_INVALID_ARG;
  return forward_impl(h, w, token_ids, cu_seqlens, num_seqs, total_tokens, max_seqlen, hidden_out, workspace,
                      workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

static size_t lm_head_bytes(const esm_encoder* h, int T, size_t* off_z2, size_t* off_loss) {
  const size_t es = h->cfg.precision == ESM_FP32 ? 4 : 2;
  const size_t act = ((size_t)T * h->cfg.hidden * es + 255) & ~size_t(255);
  *off_z2 = act;
  *off_loss = 2 * act;
  return 2 * act + (((size_t)T * 4 + 255) & ~size_t(255));
}

esm_status esm_encoder_get_fp4_scales(const esm_encoder_t* h, float* host_buf, size_t n) {
  if (!h || !host_buf || n != (size_t)h->cfg.num_layers * kNumFp8Tensors) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_FP8_E4M3) return ESM_ERR_UNSUPPORTED;
  if (cudaDeviceSynchronize() != cudaSuccess) return ESM_ERR_CUDA;
  return cuda_status(cudaMemcpy(host_buf, h->d_fp4, n * sizeof(float), cudaMemcpyDeviceToHost));
}

esm_status esm_encoder_set_layer_precision(esm_encoder_t* h, const esm_precision* per_layer, int num_layers) {
  if (!h || !per_layer || num_layers != h->cfg.num_layers) return ESM_ERR_INVALID_ARG;
  std::vector<uint8_t> v((size_t)num_layers);
  for (int l = 0; l < num_layers; ++l) {
    const esm_precision p = per_layer[l];
    if (h->cfg.precision == ESM_FP8_E4M3) {
      if (p != ESM_FP8_E4M3 && p != ESM_BF16 && p != ESM_FP4_E2M1) return ESM_ERR_UNSUPPORTED;
    } else if (p != h->cfg.precision) {
      return ESM_ERR_UNSUPPORTED;
    }
    v[l] = p == ESM_FP8_E4M3 ? 1 : p == ESM_FP4_E2M1 ? 2 : 0;
  }
  h->layer_fp8 = v;
  return ESM_OK;
}

esm_status esm_encoder_lm_head_workspace_size(const esm_encoder_t* h, int total_tokens, size_t* bytes) {
  if (!h || !bytes || total_tokens < 0) return ESM_ERR_INVALID_ARG;
  size_t a, b;
  *bytes = lm_head_bytes(h, total_tokens, &a, &b);
  return ESM_OK;
}

esm_status esm_encoder_lm_head(esm_encoder_t* h, const esm_lm_head* head, const void* hidden, int total_tokens,
                               const int32_t* targets, float* logits, float* token_loss, float* loss_sum, int* count,
                               void* workspace, size_t workspace_bytes, esm_stream_t stream) {
  if (!h || !head || total_tokens < 0) return ESM_ERR_INVALID_ARG;
  const void* p[6] = {head->dense_w, head->dense_b, head->ln_g, head->ln_b, head->emb, head->bias};
  for (const void* q : p)
    if (!q || !aligned(q, 16)) return ESM_ERR_INVALID_ARG;
  const bool bf16 = h->bf16_params();
  const int d = h->cfg.hidden, V = h->cfg.vocab, T = total_tokens;
  if (!lm_logits_supported(V, d, bf16) || (bf16 && d % 256)) return ESM_ERR_UNSUPPORTED;
  size_t off_z2, off_loss;
  const size_t need = lm_head_bytes(h, T, &off_z2, &off_loss);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (loss_sum || count)
      return cuda_status(launch_lm_logits(nullptr, bf16, head->emb, head->bias, 0, d, V, nullptr, nullptr, nullptr,
                                          loss_sum, count, h->num_sms, h->d_err, st));
    return ESM_OK;
  }
  if (!hidden || !aligned(hidden, 16) || (logits && !aligned(logits, 4))) return ESM_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return ESM_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* z1 = ws;
  void* z2 = ws + off_z2;
  float* tl = token_loss ? token_loss : reinterpret_cast<float*>(ws + off_loss);
  // dense + exact GELU on the encoder's GEMM (tensor cores for bf16), then LayerNorm
  esm_status s = run_gemm(h, P_OTHER, ESM_EPI_GELU, hidden, head->dense_w, head->dense_b, z1, nullptr, T, d, d, false,
                          h->act(), nullptr, nullptr, nullptr, nullptr, st);
  if (s != ESM_OK) return s;
  if (bf16)
    launch_layernorm_bf16in(z1, head->ln_g, head->ln_b, false, z2, Act::BF16, T, d, h->cfg.ln_eps, st);
  else
    launch_layernorm(static_cast<const float*>(z1), head->ln_g, head->ln_b, true, z2, Act::F32, T, d, h->cfg.ln_eps,
                     nullptr, nullptr, nullptr, nullptr, nullptr, st);
  const bool want_loss = token_loss || loss_sum || count;
  return cuda_status(launch_lm_logits(z2, bf16, head->emb, head->bias, T, d, V, targets, logits,
                                      want_loss ? tl : nullptr, loss_sum, count, h->num_sms, h->d_err, st));
}

// Workspace of esm_encoder_lm_head_backward: the recomputed forward (pre-activation a,
// GELU output u, LayerNorm output z: bf16 [T, d]; logits fp32 [T, V]; per-token loss; loss
// sum and count) and the backward's scratch (dlogits, dz and du fp32 [T, d], da bf16, partial
// sums, split-K partial products).
struct LmBwdLayout {
  size_t a, u, z, logits, tl, scal, dl, dz, du, da, partial, split, split_floats, total;
};
static LmBwdLayout lm_bwd_layout(const esm_config& c, int Tm) {
  LmBwdLayout L{};
  const size_t T = Tm > 0 ? Tm : 1, d = c.hidden, V = c.vocab;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.a = take(2 * T * d);
  L.u = take(2 * T * d);
  L.z = take(2 * T * d);
  L.logits = take(4 * T * V);
  L.tl = take(4 * T);
  L.scal = take(8);
  L.dl = take(4 * T * V);
  L.dz = take(4 * T * d);
  L.du = take(4 * T * d);
  L.da = take(2 * T * d);
  L.partial = take(4 * std::max(lm_backward_partial_floats((int)T, (int)V, (int)d), bwd_partial_floats((int)T, (int)d)));
  L.split_floats = (size_t)kMaxKSplit * d * d;
  L.split = take(4 * L.split_floats);
  L.total = off;
  return L;
}

esm_status esm_encoder_lm_head_backward_workspace_size(const esm_encoder_t* h, int total_tokens, size_t* bytes) {
  if (!h || !bytes || total_tokens < 0) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_BF16) return ESM_ERR_UNSUPPORTED;
  *bytes = lm_bwd_layout(h->cfg, total_tokens).total;
  return ESM_OK;
}

esm_status esm_encoder_lm_head_backward(esm_encoder_t* h, const esm_lm_head* head, const void* hidden,
                                        int total_tokens, const int32_t* targets, float* d_hidden,
                                        const esm_lm_head_grads* grads, float* loss_sum, int* count,
                                        const int* loss_count, void* workspace, size_t workspace_bytes,
                                        esm_stream_t stream) {
  if (!h || !head || !grads || total_tokens <= 0 || !hidden || !d_hidden) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_BF16) return ESM_ERR_UNSUPPORTED;
  const void* p[6] = {head->dense_w, head->dense_b, head->ln_g, head->ln_b, head->emb, head->bias};
  for (const void* q : p)
    if (!q || !aligned(q, 16)) return ESM_ERR_INVALID_ARG;
  float* gp[6] = {grads->dense_w, grads->dense_b, grads->ln_g, grads->ln_b, grads->emb, grads->bias};
  for (float* q : gp)
    if (!q || !aligned(q, 16)) return ESM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(d_hidden, 16)) return ESM_ERR_INVALID_ARG;
  const int d = h->cfg.hidden, V = h->cfg.vocab, T = total_tokens;
  if (!lm_logits_supported(V, d, true) || d % 256) return ESM_ERR_UNSUPPORTED;
  const LmBwdLayout L = lm_bwd_layout(h->cfg, T);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return ESM_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(ws + L.a);
  __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(ws + L.u);
  __nv_bfloat16* z = reinterpret_cast<__nv_bfloat16*>(ws + L.z);
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  float* tl = reinterpret_cast<float*>(ws + L.tl);
  float* lsum = reinterpret_cast<float*>(ws + L.scal);
  int* cnt = reinterpret_cast<int*>(ws + L.scal + 4);
  float* dl = reinterpret_cast<float*>(ws + L.dl);
  float* dz = reinterpret_cast<float*>(ws + L.dz);
  float* du = reinterpret_cast<float*>(ws + L.du);
  __nv_bfloat16* da = reinterpret_cast<__nv_bfloat16*>(ws + L.da);
  float* partial = reinterpret_cast<float*>(ws + L.partial);
  float* split = reinterpret_cast<float*>(ws + L.split);
  // forward, keeping the pre-activation: u = GELU(a), a = hidden Wd^T + bd; z = LN(u); logits
  esm_status s = run_gemm(h, P_OTHER, ESM_EPI_GELU, hidden, head->dense_w, head->dense_b, u, nullptr, T, d, d, false,
                          Act::BF16, nullptr, nullptr, nullptr, nullptr, st, -1, nullptr, a);
  if (s != ESM_OK) return s;
  launch_layernorm_bf16in(u, head->ln_g, head->ln_b, false, z, Act::BF16, T, d, h->cfg.ln_eps, st);
  if (launch_lm_logits(z, true, head->emb, head->bias, T, d, V, targets, logits, tl, lsum, cnt, h->num_sms, h->d_err,
                       st) != cudaSuccess)
    return ESM_ERR_CUDA;
  if (loss_sum && cudaMemcpyAsync(loss_sum, lsum, 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return ESM_ERR_CUDA;
  if (count && cudaMemcpyAsync(count, cnt, 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return ESM_ERR_CUDA;
  // backward of the mean masked cross-entropy (over this call's scored tokens, or over the
  // caller's global count)
  if (loss_count && !aligned(loss_count, 4)) return ESM_ERR_INVALID_ARG;
  if (launch_lm_backward_head(logits, targets, loss_count ? loss_count : cnt, head->emb, z, T, d, V, dl, dz, grads->emb, grads->bias, partial,
                              h->num_sms, st) != cudaSuccess)
    return ESM_ERR_CUDA;
  launch_ln_bwd_bf16in(u, head->ln_g, false, dz, du, grads->ln_g, grads->ln_b, partial, T, d, h->cfg.ln_eps, st);
  launch_gelu_bwd(du, a, da, (size_t)T * d, st);
  launch_colsum(da, true, T, d, grads->dense_b, partial, nullptr, st);
  if ((s = run_wgrad(h, da, hidden, grads->dense_w, T, d, d, split, L.split_floats, st)) != ESM_OK) return s;
  if ((s = run_dgrad(h, da, head->dense_w, d_hidden, false, T, d, d, st)) != ESM_OK) return s;
  return cuda_status(cudaGetLastError());
}

namespace {

constexpr size_t kHostGraphs = 8;

bool host_pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

std::vector<uintptr_t> host_graph_key(const esm_encoder* h, const esm_weights* w, const void* tok, const void* cu,
                                      int B, int T, int max_seqlen, const void* out, const void* ws, size_t ws_bytes) {
  std::vector<uintptr_t> k = {(uintptr_t)tok,  (uintptr_t)cu,       (uintptr_t)out,      (uintptr_t)B,
                              (uintptr_t)T,    (uintptr_t)max_seqlen, (uintptr_t)ws,     (uintptr_t)ws_bytes,
                              (uintptr_t)w->emb, (uintptr_t)w->lnf_g, (uintptr_t)w->lnf_b};
  const void* const* arrs[] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o,
                               w->ln2_g, w->ln2_b, w->w_1,   w->b_1,   w->w_2, w->b_2};
  for (const void* const* a : arrs)
    for (int l = 0; l < h->cfg.num_layers; ++l) k.push_back((uintptr_t)a[l]);
  for (uint8_t p : h->layer_fp8) k.push_back(p);
  return k;
}

// The work of one forward_host call, enqueued on st: inputs in, the forward, the output out.
esm_status enqueue_host_call(esm_encoder* h, const esm_weights* w, const int32_t* tok_host, const int32_t* cu_host,
                             int B, int T, int max_seqlen, void* out_host, void* workspace, size_t workspace_bytes,
                             const WsLayout& L, cudaStream_t st) {
  // the output staging lives in the qkv region, which is free once the last layer ran
  const size_t out_bytes = (size_t)T * h->cfg.hidden * (h->cfg.precision == ESM_FP32 ? 4 : 2);
  uint8_t* b = static_cast<uint8_t*>(workspace);
  int32_t* dtok = reinterpret_cast<int32_t*>(b + L.stage_tok);
  int32_t* dcu = reinterpret_cast<int32_t*>(b + L.stage_cu);
  void* dout = b + L.qkv;
  if (cudaMemcpyAsync(dtok, tok_host, 4 * (size_t)T, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(dcu, cu_host, 4 * (size_t)(B + 1), cudaMemcpyHostToDevice, st) != cudaSuccess)
    return ESM_ERR_CUDA;
  esm_status s = forward_impl(h, w, dtok, dcu, B, T, max_seqlen, dout, workspace, workspace_bytes, st);
  if (s != ESM_OK) return s;
  if (cudaMemcpyAsync(out_host, dout, out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return ESM_ERR_CUDA;
  return ESM_OK;
}

}  // namespace

esm_status esm_encoder_forward_host(esm_encoder_t* h, const esm_weights* w, const int32_t* token_ids_host,
                                    const int32_t* cu_seqlens_host, int num_seqs, int total_tokens, int max_seqlen,
                                    void* hidden_out_host, void* workspace, size_t workspace_bytes,
                                    esm_stream_t stream) {
  if (!h || total_tokens < 0 || num_seqs < 0) return ESM_ERR_INVALID_ARG;
  if (total_tokens == 0) return ESM_OK;
  if (num_seqs == 0 || !token_ids_host || !cu_seqlens_host || !hidden_out_host) return ESM_ERR_INVALID_ARG;
  if (max_seqlen <= 0 || max_seqlen > h->cfg.max_positions) return ESM_ERR_INVALID_ARG;
  if (!weights_ok(h, w)) return ESM_ERR_INVALID_ARG;
  WsLayout L;
  esm_status s = check_ws(h, total_tokens, num_seqs, workspace, workspace_bytes, &L);
  if (s != ESM_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // Pinned host buffers: replay a graph of the whole call (the ~170 kernel launches of a
  // forward cost more eagerly than as one graph).  Pageable buffers stay on the eager path.
  if (!h->profiling && host_pinned(token_ids_host) && host_pinned(cu_seqlens_host) && host_pinned(hidden_out_host)) {
    std::vector<uintptr_t> key = host_graph_key(h, w, token_ids_host, cu_seqlens_host, num_seqs, total_tokens,
                                                max_seqlen, hidden_out_host, workspace, workspace_bytes);
    for (const auto& g : h->host_graphs)
      if (g.key == key) {
        if (cudaGraphLaunch(g.exec, st) != cudaSuccess) return ESM_ERR_CUDA;
        return cuda_status(cudaStreamSynchronize(st));
      }
    auto seen = std::find(h->host_seen.begin(), h->host_seen.end(), key);
    if (seen != h->host_seen.end()) {  // second call of this key: capture it
      h->host_seen.erase(seen);
      bool ok = h->cap_stream || cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) == cudaSuccess;
      cudaGraph_t graph = nullptr;
      cudaGraphExec_t exec = nullptr;
      if (ok && cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
        const esm_status cs = enqueue_host_call(h, w, token_ids_host, cu_seqlens_host, num_seqs, total_tokens,
                                                max_seqlen, hidden_out_host, workspace, workspace_bytes, L,
                                                h->cap_stream);
        const cudaError_t ce = cudaStreamEndCapture(h->cap_stream, &graph);
        ok = cs == ESM_OK && ce == cudaSuccess && graph != nullptr &&
             cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
      } else {
        ok = false;
      }
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();  // a capture that failed falls back to eager launches below
      if (ok) {
        if (h->host_graphs.size() >= kHostGraphs) {
          cudaGraphExecDestroy(h->host_graphs.front().exec);
          h->host_graphs.erase(h->host_graphs.begin());
        }
        h->host_graphs.push_back({std::move(key), exec});
        if (cudaGraphLaunch(exec, st) != cudaSuccess) return ESM_ERR_CUDA;
        return cuda_status(cudaStreamSynchronize(st));
      }
    } else {
      if (h->host_seen.size() >= kHostGraphs) h->host_seen.erase(h->host_seen.begin());
      h->host_seen.push_back(std::move(key));
    }
  }
  s = enqueue_host_call(h, w, token_ids_host, cu_seqlens_host, num_seqs, total_tokens, max_seqlen, hidden_out_host,
                        workspace, workspace_bytes, L, st);
  if (s != ESM_OK) return s;
  return cuda_status(cudaStreamSynchronize(st));
}

esm_status esm_encoder_forward_padded(esm_encoder_t* h, const esm_weights* w, const int32_t* token_ids,
                                      const int32_t* seq_lens, int B, int S, void* hidden_out, void* workspace,
                                      size_t workspace_bytes, esm_stream_t stream) {
  if (!h || B < 0 || S < 0) return ESM_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return ESM_OK;
  if (!token_ids || !seq_lens || !hidden_out || !aligned(hidden_out, 16)) return ESM_ERR_INVALID_ARG;
  if (S > h->cfg.max_positions || (long long)B * S > (1ll << 31) - 1) return ESM_ERR_INVALID_ARG;
  if (!weights_ok(h, w)) return ESM_ERR_INVALID_ARG;
  const int T = B * S;
  WsLayout L;
  esm_status s = check_ws(h, T, B, workspace, workspace_bytes, &L);
  if (s != ESM_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  PackBuffers pb = pack_buffers(workspace, L);
  uint8_t* b = static_cast<uint8_t*>(workspace);
  {
    ProfScope _ps(h, P_OTHER, st, h->cfg.precision != ESM_FP32 ? 3 : 2);
    launch_pad_index(seq_lens, B, S, pb, h->d_err, st);
    if (h->cfg.precision != ESM_FP32) launch_attn_worklist(B, L.max_items, kAttnQTileTc, pb, st);
    launch_embed(token_ids, T, w->emb, !h->bf16_params(), h->cfg.vocab, h->cfg.hidden, h->cfg.emb_scale,
                 reinterpret_cast<float*>(b + L.x), h->d_err, st);
  }
  return run_layers(h, w, T, L.max_items, L, workspace, hidden_out, true, st);
}

esm_status esm_encoder_check(esm_encoder_t* h, esm_stream_t stream) {
  if (!h) return ESM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ESM_ERR_CUDA;
  unsigned e = 0;
  if (cudaMemcpy(&e, h->d_err, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return ESM_ERR_CUDA;
  if (e && cudaMemset(h->d_err, 0, sizeof(unsigned)) != cudaSuccess) return ESM_ERR_CUDA;
  if (e & ERRBIT_CU_SEQLENS) return ESM_ERR_BAD_CU_SEQLENS;
  if (e & ERRBIT_TOKEN) return ESM_ERR_TOKEN_RANGE;
  if (e & ERRBIT_TIMEOUT) return ESM_ERR_TIMEOUT;
  return ESM_OK;
}

esm_status esm_encoder_debug_pack_index(esm_encoder_t* h, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                                        int max_seqlen, int32_t* pos_id, int32_t* seg_id, void* workspace,
                                        size_t workspace_bytes, esm_stream_t stream) {
  if (!h || num_seqs <= 0 || total_tokens < 0 || !cu_seqlens || !pos_id || !seg_id) return ESM_ERR_INVALID_ARG;
  if (max_seqlen <= 0 || max_seqlen > h->cfg.max_positions) return ESM_ERR_INVALID_ARG;
  WsLayout L;
  esm_status s = check_ws(h, total_tokens, num_seqs, workspace, workspace_bytes, &L);
  if (s != ESM_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  PackBuffers pb = pack_buffers(workspace, L);
  if (total_tokens > 0) {
    if (cudaMemsetAsync(pb.pos_id, 0, 4 * (size_t)total_tokens, st) != cudaSuccess ||
        cudaMemsetAsync(pb.seg_id, 0, 4 * (size_t)total_tokens, st) != cudaSuccess)
      return ESM_ERR_CUDA;
  }
  launch_pack_index(cu_seqlens, num_seqs, total_tokens, max_seqlen, h->cfg.max_positions, pb, h->d_err, st);
  if (total_tokens > 0) {
    if (cudaMemcpyAsync(pos_id, pb.pos_id, 4 * (size_t)total_tokens, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(seg_id, pb.seg_id, 4 * (size_t)total_tokens, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return ESM_ERR_CUDA;
  }
  return cuda_status(cudaGetLastError());
}

esm_status esm_encoder_debug_wait_timeout(esm_encoder_t* h, int timeout_us, esm_stream_t stream) {
  if (!h || timeout_us < 1 || timeout_us > 1000000) return ESM_ERR_INVALID_ARG;
  launch_wait_timeout(1000ull * (unsigned long long)timeout_us, h->d_err, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

esm_status esm_op_layernorm(esm_encoder_t* h, const float* x, const void* gamma, const void* beta, void* y, int rows,
                            int cols, esm_stream_t stream) {
  if (!h || !x || !gamma || !beta || !y || rows < 0 || cols <= 0 || cols % 4 || cols > 4096)
    return ESM_ERR_INVALID_ARG;
  launch_layernorm(x, gamma, beta, !h->bf16_params(), y, h->act(), rows, cols, h->cfg.ln_eps, nullptr, nullptr,
                   nullptr, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

esm_status esm_op_gemm(esm_encoder_t* h, esm_epilogue epi, const void* A, const void* B, const void* bias, void* out,
                       const int32_t* pos_id, int M, int N, int K, esm_stream_t stream) {
  if (!h || !A || !B || !out || M < 0 || N <= 0 || K <= 0) return ESM_ERR_INVALID_ARG;
  if (epi < ESM_EPI_BIAS_F32 || epi > ESM_EPI_GELU) return ESM_ERR_INVALID_ARG;
  if (epi == ESM_EPI_QKV_ROPE && (!pos_id || N != 3 * h->cfg.hidden)) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_FP32) {
    if (K % 64 || N % 256 || !aligned(A, 16) || !aligned(B, 16) || !aligned(out, 16)) return ESM_ERR_INVALID_ARG;
    if (bias && !aligned(bias, 16)) return ESM_ERR_INVALID_ARG;
  }
  const Act out_act = (epi == ESM_EPI_BIAS_F32 || epi == ESM_EPI_RESIDUAL) ? Act::F32 : h->act();
  return run_gemm(h, P_OTHER, epi, A, B, bias, out, pos_id, M, N, K, false, out_act, nullptr, nullptr, nullptr, nullptr,
                  reinterpret_cast<cudaStream_t>(stream));
}

esm_status esm_op_layernorm_e4m3(esm_encoder_t* h, const float* x, const void* gamma, const void* beta, uint8_t* y,
                                 int rows, int cols, const float* scale, float* amax, esm_stream_t stream) {
  if (!h || !x || !gamma || !beta || !y || !scale || !amax || rows < 0 || cols <= 0 || cols % 4 || cols > 4096)
    return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_FP8_E4M3) return ESM_ERR_UNSUPPORTED;
  launch_layernorm(x, gamma, beta, false, y, Act::E4M3, rows, cols, h->cfg.ln_eps, scale, amax, nullptr, nullptr,
                   nullptr, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

esm_status esm_op_gemm_fp8(esm_encoder_t* h, esm_epilogue epi, const uint8_t* A, const uint8_t* B, const float* a_scale,
                           const float* b_scale, const void* bias, void* out, const int32_t* pos_id, int M, int N,
                           int K, esm_stream_t stream) {
  if (!h || !A || !B || !a_scale || !b_scale || !out || M < 0 || N <= 0 || K <= 0) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_FP8_E4M3) return ESM_ERR_UNSUPPORTED;
  if (epi < ESM_EPI_BIAS_F32 || epi > ESM_EPI_GELU) return ESM_ERR_INVALID_ARG;
  if (epi == ESM_EPI_QKV_ROPE && (!pos_id || N != 3 * h->cfg.hidden)) return ESM_ERR_INVALID_ARG;
  if (K % 128 || N % 256 || !aligned(A, 16) || !aligned(B, 16) || !aligned(out, 16)) return ESM_ERR_INVALID_ARG;
  if (bias && !aligned(bias, 16)) return ESM_ERR_INVALID_ARG;
  const Act out_act = (epi == ESM_EPI_BIAS_F32 || epi == ESM_EPI_RESIDUAL) ? Act::F32 : Act::BF16;
  return run_gemm(h, P_OTHER, epi, A, B, bias, out, pos_id, M, N, K, true, out_act, a_scale, b_scale, nullptr,
                  nullptr, reinterpret_cast<cudaStream_t>(stream));
}

esm_status esm_op_quantize_nvfp4(esm_encoder_t* h, const void* x, int rows, int cols, uint8_t* codes,
                                 uint8_t* scales, float* amax, float* scale, esm_stream_t stream) {
  if (!h || !x || !codes || !scales || !amax || !scale || rows < 0 || cols <= 0) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision == ESM_FP32) return ESM_ERR_UNSUPPORTED;
  if (rows % 128 || cols % 256 || !aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 16) ||
      !aligned(amax, 4) || !aligned(scale, 4))
    return ESM_ERR_INVALID_ARG;
  if (rows == 0) return ESM_OK;
  return cuda_status(launch_nvfp4_quantize(static_cast<const __nv_bfloat16*>(x), rows, rows, cols, codes, scales, amax,
                                           scale, false, h->num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

esm_status esm_op_gemm_nvfp4(esm_encoder_t* h, esm_epilogue epi, const uint8_t* a_codes, const uint8_t* a_scales,
                             const float* a_scale, const uint8_t* b_codes, const uint8_t* b_scales,
                             const float* b_scale, const void* bias, const int32_t* pos_id, void* out, int M, int N,
                             int K, esm_stream_t stream) {
  if (!h || !a_codes || !a_scales || !a_scale || !b_codes || !b_scales || !b_scale || !out) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision == ESM_FP32) return ESM_ERR_UNSUPPORTED;
  if (M < 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 256) return ESM_ERR_INVALID_ARG;
  int mode;
  switch (epi) {
    case ESM_EPI_BIAS_F32: mode = kFp4F32; break;
    case ESM_EPI_RESIDUAL: mode = kFp4Residual; break;
    case ESM_EPI_GELU: mode = kFp4Gelu; break;
    case ESM_EPI_QKV_ROPE: mode = kFp4QkvRope; break;
    default: return ESM_ERR_INVALID_ARG;
  }
  if (mode == kFp4QkvRope && (!pos_id || N != 3 * h->cfg.hidden)) return ESM_ERR_INVALID_ARG;
  if (!aligned(a_codes, 16) || !aligned(b_codes, 16) || !aligned(a_scales, 16) || !aligned(b_scales, 16) ||
      !aligned(out, 16) || (bias && !aligned(bias, 16)))
    return ESM_ERR_INVALID_ARG;
  if (M == 0) return ESM_OK;
  const CUtensorMap* ma = h->map(a_codes, (uint64_t)M, (uint64_t)K / 2, 128, 1);
  const CUtensorMap* mb = h->map(b_codes, (uint64_t)N, (uint64_t)K / 2, 128, 1);
  if (!ma || !mb) return ESM_ERR_CUDA;
  Fp4Epi ea{};
  ea.bias = bias;
  ea.out = out;
  ea.rows_valid = M;
  ea.pos_id = pos_id;
  ea.rope = h->d_rope;
  ea.rope_cols = 2 * h->cfg.hidden;
  ea.max_pos = h->cfg.max_positions;
  return cuda_status(launch_gemm_nvfp4(mode, ma, mb, a_scales, b_scales, a_scale, b_scale, ea, M, N, K, h->num_sms,
                                       h->d_err, reinterpret_cast<cudaStream_t>(stream)));
}

esm_status esm_op_attention(esm_encoder_t* h, const void* qkv, const int32_t* cu_seqlens, int num_seqs,
                            int total_tokens, int max_seqlen, void* o, void* workspace, size_t workspace_bytes,
                            esm_stream_t stream) {
  if (!h || !qkv || !cu_seqlens || !o || num_seqs <= 0 || total_tokens < 0) return ESM_ERR_INVALID_ARG;
  if (max_seqlen <= 0 || max_seqlen > h->cfg.max_positions) return ESM_ERR_INVALID_ARG;
  if (total_tokens == 0) return ESM_OK;
  WsLayout L;
  esm_status s = check_ws(h, total_tokens, num_seqs, workspace, workspace_bytes, &L);
  if (s != ESM_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  PackBuffers pb = pack_buffers(workspace, L);
  if (cudaMemsetAsync(pb.pos_id, 0, 4 * (size_t)total_tokens, st) != cudaSuccess ||
      cudaMemsetAsync(pb.seg_id, 0, 4 * (size_t)total_tokens, st) != cudaSuccess)
    return ESM_ERR_CUDA;
  launch_pack_index(cu_seqlens, num_seqs, total_tokens, max_seqlen, h->cfg.max_positions, pb, h->d_err, st);
  const int d = h->cfg.hidden, H = h->cfg.heads;
  if (h->cfg.precision == ESM_FP32) {
    launch_attention_f32(static_cast<const float*>(qkv), static_cast<float*>(o), d, H, total_tokens, pb, st);
  } else {
    launch_attn_worklist(num_seqs, L.max_items, kAttnQTileTc, pb, st);
    const CUtensorMap* tq = h->map(qkv, (uint64_t)total_tokens, (uint64_t)3 * d, 128, 2);
    if (!tq) return ESM_ERR_CUDA;
    if (launch_attention_tc(tq, o, Act::BF16, d, H, L.max_items, pb, nullptr, nullptr, h->d_err, st) != cudaSuccess)
      return ESM_ERR_CUDA;
  }
  return cuda_status(cudaGetLastError());
}

// ------------------------------------------------------------------ training
esm_status esm_encoder_train_buffer_size(const esm_encoder_t* h, int max_tokens, size_t* bytes) {
  if (!h || !bytes || max_tokens < 0) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_BF16 || h->cfg.hidden > 4096) return ESM_ERR_UNSUPPORTED;
  *bytes = train_layout(h->cfg, max_tokens).total;
  return ESM_OK;
}

esm_status esm_encoder_forward_train(esm_encoder_t* h, const esm_weights* w, const int32_t* token_ids,
                                     const int32_t* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen,
                                     void* hidden_out, void* train_buf, size_t train_bytes, void* workspace,
                                     size_t workspace_bytes, esm_stream_t stream) {
  if (!h || total_tokens <= 0 || num_seqs <= 0) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_BF16 || h->cfg.hidden > 4096) return ESM_ERR_UNSUPPORTED;
  if (!token_ids || !cu_seqlens || !hidden_out || !aligned(hidden_out, 16)) return ESM_ERR_INVALID_ARG;
  if (max_seqlen <= 0 || max_seqlen > h->cfg.max_positions) return ESM_ERR_INVALID_ARG;
  if (!weights_ok(h, w)) return ESM_ERR_INVALID_ARG;
  if (!train_buf || !aligned(train_buf, 256) || train_bytes < train_layout(h->cfg, total_tokens).total)
    return ESM_ERR_WORKSPACE;
  h->train_buf = nullptr;  // valid again only once this forward is fully enqueued
  return train_forward_impl(h, w, token_ids, cu_seqlens, num_seqs, total_tokens, max_seqlen, hidden_out, train_buf,
                            workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

esm_status esm_encoder_backward(esm_encoder_t* h, const esm_weights* w, const float* d_hidden_out,
                                const esm_grads* grads, void* train_buf, size_t train_bytes, void* workspace,
                                size_t workspace_bytes, esm_stream_t stream) {
  if (!h || !d_hidden_out || !aligned(d_hidden_out, 16)) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision != ESM_BF16) return ESM_ERR_UNSUPPORTED;
  if (!weights_ok(h, w) || !grads_ok(h, grads)) return ESM_ERR_INVALID_ARG;
  if (h->train_T <= 0 || train_buf != h->train_buf || workspace != h->train_ws) return ESM_ERR_INVALID_ARG;
  if (train_bytes < train_layout(h->cfg, h->train_T).total) return ESM_ERR_WORKSPACE;
  if (workspace_bytes < h->layout(h->train_T, h->train_B).total) return ESM_ERR_WORKSPACE;
  return backward_impl(h, w, d_hidden_out, grads, train_buf, workspace, reinterpret_cast<cudaStream_t>(stream));
}

esm_status esm_op_gemm_dgrad(esm_encoder_t* h, const void* dY, const void* W, void* out, int out_bf16, int M, int N,
                             int K, esm_stream_t stream) {
  if (!h || !dY || !W || !out || M < 0 || N <= 0 || K <= 0) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision == ESM_FP32) return ESM_ERR_UNSUPPORTED;
  if (N % 64 || K % 256 || !aligned(dY, 16) || !aligned(W, 16) || !aligned(out, 16)) return ESM_ERR_INVALID_ARG;
  return run_dgrad(h, dY, W, out, out_bf16 != 0, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

esm_status esm_op_gemm_wgrad_workspace_size(const esm_encoder_t* h, int N, int K, size_t* bytes) {
  if (!h || !bytes || N <= 0 || K <= 0) return ESM_ERR_INVALID_ARG;
  *bytes = sizeof(float) * (size_t)kMaxKSplit * N * K;
  return ESM_OK;
}

esm_status esm_op_gemm_wgrad(esm_encoder_t* h, const void* dY, const void* X, float* dW, int M, int N, int K,
                             void* workspace, size_t workspace_bytes, esm_stream_t stream) {
  if (!h || !dW || M < 0 || N <= 0 || K <= 0 || (M > 0 && (!dY || !X))) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision == ESM_FP32) return ESM_ERR_UNSUPPORTED;
  if (N % 256 || K % 256 || !aligned(dY, 16) || !aligned(X, 16) || !aligned(dW, 16)) return ESM_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return ESM_ERR_WORKSPACE;
  return run_wgrad(h, dY, X, dW, M, N, K, static_cast<float*>(workspace), workspace ? workspace_bytes / 4 : 0,
                   reinterpret_cast<cudaStream_t>(stream));
}

static size_t ln_bwd_ws_bytes(int rows, int cols, size_t* off_partial) {
  *off_partial = 0;
  return align256(4 * bwd_partial_floats(rows, cols));
}

esm_status esm_op_layernorm_backward_workspace_size(const esm_encoder_t* h, int rows, int cols, size_t* bytes) {
  if (!h || !bytes || rows < 0 || cols <= 0) return ESM_ERR_INVALID_ARG;
  size_t off;
  *bytes = ln_bwd_ws_bytes(rows, cols, &off);
  return ESM_OK;
}

esm_status esm_op_layernorm_backward(esm_encoder_t* h, const float* x, const void* gamma, const float* dy,
                                     const float* dres, float* dx, float* dgamma, float* dbeta, int rows, int cols,
                                     void* workspace, size_t workspace_bytes, esm_stream_t stream) {
  if (!h || !x || !gamma || !dy || !dx || !dgamma || !dbeta || rows < 0 || cols <= 0 || cols % 4 || cols > 4096)
    return ESM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(dy, 16) || !aligned(dx, 16) || (dres && !aligned(dres, 16)) || !aligned(gamma, 16))
    return ESM_ERR_INVALID_ARG;
  size_t off;
  const size_t need = ln_bwd_ws_bytes(rows, cols, &off);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return ESM_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  launch_ln_bwd(x, gamma, !h->bf16_params(), dy, dres, dx, dgamma, dbeta, reinterpret_cast<float*>(ws + off), rows,
                cols, h->cfg.ln_eps, reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

static size_t attn_bwd_ws_bytes(const esm_encoder* h, int T, int B, WsLayout* L, size_t* off_dsum, size_t* off_dq) {
  *L = h->layout(T, B);
  *off_dsum = L->total;
  *off_dq = *off_dsum + align256(4 * (size_t)(T > 0 ? T : 1) * h->cfg.heads);
  return *off_dq + align256(4 * (size_t)(T > 0 ? T : 1) * h->cfg.hidden);
}

esm_status esm_op_attention_backward_workspace_size(const esm_encoder_t* h, int total_tokens, int num_seqs,
                                                    size_t* bytes) {
  if (!h || !bytes || total_tokens < 0 || num_seqs < 0) return ESM_ERR_INVALID_ARG;
  WsLayout L;
  size_t a, b;
  *bytes = attn_bwd_ws_bytes(h, total_tokens, num_seqs, &L, &a, &b);
  return ESM_OK;
}

// Index the batch into the workspace's pack buffers (positions, segments, work list).
static esm_status index_batch(esm_encoder* h, const int32_t* cu, int B, int T, int max_seqlen, const WsLayout& L,
                              void* ws, cudaStream_t st) {
  PackBuffers pb = pack_buffers(ws, L);
  if (cudaMemsetAsync(pb.pos_id, 0, 4 * (size_t)T, st) != cudaSuccess ||
      cudaMemsetAsync(pb.seg_id, 0, 4 * (size_t)T, st) != cudaSuccess)
    return ESM_ERR_CUDA;
  launch_pack_index(cu, B, T, max_seqlen, h->cfg.max_positions, pb, h->d_err, st);
  launch_attn_worklist(B, L.max_items, kAttnQTileTc, pb, st);
  return cuda_status(cudaGetLastError());
}

esm_status esm_op_attention_train(esm_encoder_t* h, const void* qkv, const int32_t* cu_seqlens, int num_seqs,
                                  int total_tokens, int max_seqlen, void* o, float* lse, void* workspace,
                                  size_t workspace_bytes, esm_stream_t stream) {
  if (!h || !qkv || !cu_seqlens || !o || !lse || num_seqs <= 0 || total_tokens < 0) return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision == ESM_FP32) return ESM_ERR_UNSUPPORTED;
  if (max_seqlen <= 0 || max_seqlen > h->cfg.max_positions) return ESM_ERR_INVALID_ARG;
  if (total_tokens == 0) return ESM_OK;
  WsLayout L;
  esm_status s = check_ws(h, total_tokens, num_seqs, workspace, workspace_bytes, &L);
  if (s != ESM_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((s = index_batch(h, cu_seqlens, num_seqs, total_tokens, max_seqlen, L, workspace, st)) != ESM_OK) return s;
  const int d = h->cfg.hidden;
  const CUtensorMap* tq = h->map(qkv, (uint64_t)total_tokens, (uint64_t)3 * d, 128, 2);
  if (!tq) return ESM_ERR_CUDA;
  if (launch_attention_tc(tq, o, Act::BF16, d, h->cfg.heads, L.max_items, pack_buffers(workspace, L), nullptr, nullptr,
                          h->d_err, st, lse, total_tokens) != cudaSuccess)
    return ESM_ERR_CUDA;
  return cuda_status(cudaGetLastError());
}

esm_status esm_op_attention_backward(esm_encoder_t* h, const void* qkv, const void* o, const float* lse,
                                     const void* d_o, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                                     int max_seqlen, void* dqkv, void* workspace, size_t workspace_bytes,
                                     esm_stream_t stream) {
  if (!h || !qkv || !o || !lse || !d_o || !cu_seqlens || !dqkv || num_seqs <= 0 || total_tokens < 0)
    return ESM_ERR_INVALID_ARG;
  if (h->cfg.precision == ESM_FP32) return ESM_ERR_UNSUPPORTED;
  if (max_seqlen <= 0 || max_seqlen > h->cfg.max_positions) return ESM_ERR_INVALID_ARG;
  if (!aligned(qkv, 16) || !aligned(o, 16) || !aligned(d_o, 16) || !aligned(dqkv, 16)) return ESM_ERR_INVALID_ARG;
  if (total_tokens == 0) return ESM_OK;
  WsLayout L;
  size_t off_dsum, off_dq;
  const size_t need = attn_bwd_ws_bytes(h, total_tokens, num_seqs, &L, &off_dsum, &off_dq);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return ESM_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  esm_status s = index_batch(h, cu_seqlens, num_seqs, total_tokens, max_seqlen, L, workspace, st);
  if (s != ESM_OK) return s;
  const int d = h->cfg.hidden, T = total_tokens;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const CUtensorMap* tq = h->map(qkv, (uint64_t)T, (uint64_t)3 * d, 128, 2);
  const CUtensorMap* td = h->map(d_o, (uint64_t)T, (uint64_t)d, 128, 2);
  const CUtensorMap* tdq = h->map(ws + off_dq, (uint64_t)T, (uint64_t)d, 32, 4);
  if (!tq || !td || !tdq) return ESM_ERR_CUDA;
  if (launch_attention_bwd_tc(tq, td, tdq, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), lse,
                              reinterpret_cast<float*>(ws + off_dsum), reinterpret_cast<float*>(ws + off_dq),
                              static_cast<__nv_bfloat16*>(dqkv), T, d, h->cfg.heads, L.max_items,
                              pack_buffers(workspace, L), nullptr, h->cfg.max_positions, h->num_sms, h->d_err,
                              st) != cudaSuccess)
    return ESM_ERR_CUDA;
  return cuda_status(cudaGetLastError());
}

esm_status esm_encoder_set_profiling(esm_encoder_t* h, int enable) {
  if (!h) return ESM_ERR_INVALID_ARG;
  h->profiling = enable != 0;
  return ESM_OK;
}

esm_status esm_encoder_get_profile(esm_encoder_t* h, esm_profile* out, int reset) {
  if (!h || !out) return ESM_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return ESM_ERR_CUDA;
  h->drain_events();
  for (int i = 0; i < ESM_PROFILE_CLASSES; ++i) {
    out->ms[i] = h->ms[i];
    out->launches[i] = h->launches[i];
  }
  out->total_launches = h->total_launches;
  if (reset) {
    for (int i = 0; i < ESM_PROFILE_CLASSES; ++i) {
      h->ms[i] = 0;
      h->launches[i] = 0;
    }
    h->total_launches = 0;
  }
  return ESM_OK;
}

esm_status esm_encoder_get_fp8_state(const esm_encoder_t* h, float* host_buf, size_t n) {
  if (!h || !host_buf || n != h->fp8_floats) return ESM_ERR_INVALID_ARG;
  if (n == 0) return ESM_OK;
  return cuda_status(cudaMemcpy(host_buf, h->d_fp8, n * sizeof(float), cudaMemcpyDeviceToHost));
}

esm_status esm_encoder_set_fp8_state(esm_encoder_t* h, const float* host_buf, size_t n) {
  if (!h || !host_buf || n != h->fp8_floats) return ESM_ERR_INVALID_ARG;
  if (n == 0) return ESM_OK;
  return cuda_status(cudaMemcpy(h->d_fp8, host_buf, n * sizeof(float), cudaMemcpyHostToDevice));
}

}  // extern "C"
