// Host side of the C ABI declared in include/esm_encoder.h: handle, workspace layout,
// TMA descriptor cache and the per-layer launch sequence of the packed ESM-2 forward
// (section 3.2 of the hotelren.com guide: embedding, then every layer over cu_seqlens).
#include <cuda.h>
#include <cuda_runtime.h>

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
  size_t pos, seg, seg_start, seg_qlen, seg_klen, work, work_count, x, y, qkv, o, u, wq, stage_tok, stage_cu, total;
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
  std::vector<uint8_t> layer_fp8;  // per layer: 1 = E4M3 GEMMs (FP8 handles only)
  float* d_fp8 = nullptr;        // scales [L*8] | history [L*8*len] | amax [L*8]
  size_t fp8_floats = 0;
  std::unordered_map<MapKey, CUtensorMap, MapKeyHash> maps;
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
    if (maps.size() > 4096) maps.clear();
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

enum ProfClass { P_QKV = 0, P_ATTN = 1, P_OPROJ = 2, P_FC1 = 3, P_FC2 = 4, P_LN = 5, P_OTHER = 6 };

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

esm_status check_ws(const esm_encoder* h, int T, int B, void* ws, size_t bytes, WsLayout* out) {
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

// One GEMM of a layer.  A: activation [M, K]; B: weight [N, K].
esm_status run_gemm(esm_encoder* h, int cls, esm_epilogue epi, const void* A, const void* B, const void* bias, void* out,
                    const int32_t* pos_id, int M, int N, int K, bool fp8, Act out_act, const float* a_scale,
                    const float* b_scale, const float* o_scale, float* o_amax, cudaStream_t st) {
  EpiArgs ea{};
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
  for (int l = 0; l < c.num_layers; ++l) {
    const bool fp8 = c.precision == ESM_FP8_E4M3 && h->layer_fp8[l];
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
    PROF(h, P_LN, st, 1,
         launch_layernorm(x, w->ln1_g[l], w->ln1_b[l], pf32, y, fp8 ? Act::E4M3 : act, T, d, c.ln_eps, sc + X_QKV,
                          am + X_QKV, nullptr, nullptr, nullptr, st));
    s = run_gemm(h, P_QKV, ESM_EPI_QKV_ROPE, y, fp8 ? (const void*)wq_qkv : w->w_qkv[l], w->b_qkv[l], qkv, pb.pos_id, T,
                 3 * d, d, fp8, act, sc + X_QKV, sc + W_QKV, nullptr, nullptr, st);
    if (s != ESM_OK) return s;
    {
      ProfScope _ps(h, P_ATTN, st, 1);
      if (c.precision == ESM_FP32)
        launch_attention_f32(static_cast<const float*>(qkv), static_cast<float*>(o), d, H, T, pb, st);
      else {
        const CUtensorMap* tq = h->map(qkv, (uint64_t)T, (uint64_t)3 * d, 128, 2);
        if (!tq) return ESM_ERR_CUDA;
        if (launch_attention_tc(tq, o, fp8 ? Act::E4M3 : Act::BF16, d, H, max_items, pb, sc + X_O, am + X_O,
                                h->d_err, st) != cudaSuccess)
          return ESM_ERR_CUDA;
      }
    }
    s = run_gemm(h, P_OPROJ, ESM_EPI_RESIDUAL, o, fp8 ? (const void*)wq_o : w->w_o[l], w->b_o[l], x, nullptr, T, d, d, fp8,
                 Act::F32, sc + X_O, sc + W_O, nullptr, nullptr, st);
    if (s != ESM_OK) return s;
    // ---- MLP block
    PROF(h, P_LN, st, 1,
         launch_layernorm(x, w->ln2_g[l], w->ln2_b[l], pf32, y, fp8 ? Act::E4M3 : act, T, d, c.ln_eps, sc + X_1,
                          am + X_1, nullptr, nullptr, nullptr, st));
    s = run_gemm(h, P_FC1, ESM_EPI_GELU, y, fp8 ? (const void*)wq_1 : w->w_1[l], w->b_1[l], u, nullptr, T, f, d, fp8,
                 fp8 ? Act::E4M3 : act, sc + X_1, sc + W_1, sc + X_2, am + X_2, st);
    if (s != ESM_OK) return s;
    s = run_gemm(h, P_FC2, ESM_EPI_RESIDUAL, u, fp8 ? (const void*)wq_2 : w->w_2[l], w->b_2[l], x, nullptr, T, d, f, fp8,
                 Act::F32, sc + X_2, sc + W_2, nullptr, nullptr, st);
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

}  // namespace

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
            cudaMalloc(&h->d_fp8, sizeof(float) * (h->fp8_floats + nf + 1)) == cudaSuccess;
  if (ok) {
    ok = cudaMemset(h->d_err, 0, sizeof(unsigned)) == cudaSuccess &&
         cudaMemset(h->d_fp8, 0, sizeof(float) * (h->fp8_floats + nf + 1)) == cudaSuccess;
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
  if (h->d_err) cudaFree(h->d_err);
  if (h->d_rope) cudaFree(h->d_rope);
  if (h->d_fp8) cudaFree(h->d_fp8);
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

esm_status esm_encoder_set_layer_precision(esm_encoder_t* h, const esm_precision* per_layer, int num_layers) {
  if (!h || !per_layer || num_layers != h->cfg.num_layers) return ESM_ERR_INVALID_ARG;
  std::vector<uint8_t> v((size_t)num_layers);
  for (int l = 0; l < num_layers; ++l) {
    const esm_precision p = per_layer[l];
    if (p == ESM_FP4_E2M1) return ESM_ERR_UNSUPPORTED;
    if (h->cfg.precision == ESM_FP8_E4M3) {
      if (p != ESM_FP8_E4M3 && p != ESM_BF16) return ESM_ERR_UNSUPPORTED;
    } else if (p != h->cfg.precision) {
      return ESM_ERR_UNSUPPORTED;
    }
    v[l] = p == ESM_FP8_E4M3 ? 1 : 0;
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
  // the output staging lives in the qkv region, which is free once the last layer ran
  const size_t out_bytes = (size_t)total_tokens * h->cfg.hidden * (h->cfg.precision == ESM_FP32 ? 4 : 2);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(workspace);
  int32_t* dtok = reinterpret_cast<int32_t*>(b + L.stage_tok);
  int32_t* dcu = reinterpret_cast<int32_t*>(b + L.stage_cu);
  void* dout = b + L.qkv;
  if (cudaMemcpyAsync(dtok, token_ids_host, 4 * (size_t)total_tokens, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(dcu, cu_seqlens_host, 4 * (size_t)(num_seqs + 1), cudaMemcpyHostToDevice, st) != cudaSuccess)
    return ESM_ERR_CUDA;
  s = forward_impl(h, w, dtok, dcu, num_seqs, total_tokens, max_seqlen, dout, workspace, workspace_bytes, st);
  if (s != ESM_OK) return s;
  if (cudaMemcpyAsync(hidden_out_host, dout, out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return ESM_ERR_CUDA;
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
