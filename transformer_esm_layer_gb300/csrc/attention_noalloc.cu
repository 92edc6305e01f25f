// Variable-length attention entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory pool or
// allocator that owns the whole device, plugin hosts that hand out only input/output
// buffers, or runtimes that forbid allocation after start-up.  For them this file keeps
// the attention kernel's scratch (packing indices, segment table, work list, error word)
// in one file-scope device array of fixed size.  Every GPU that loads the library holds
// the array until the process exits.
//
// The attention itself is the library's tcgen05 kernel (attention_tc.cu), the same one the
// workspace-based esm_op_attention runs; its TMA descriptor is encoded on the host for
// every call and passed as a kernel parameter, so nothing is allocated for it either.
//
// The host never dereferences the array's name: in host code it is only a stand-in for
// the symbol.  The device address comes from cudaGetSymbolAddress, taken once per device
// (on the first call made with that device current) and cached.  That first call should
// therefore happen before any stream capture.  The array is shared by every call and
// keeps the previous call's contents, so each call clears what must start at zero, and
// calls that overlap on the GPU (on different streams) race on it.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace esm {
namespace {

constexpr int kMaxTokens = ESM_NOALLOC_MAX_TOKENS;
constexpr int kMaxSeqs = ESM_NOALLOC_MAX_SEQS;
constexpr int kMaxItems = kMaxTokens / kAttnQTileTc + kMaxSeqs;

// int32 word offsets inside the scratch array
constexpr size_t kOffPos = 0;
constexpr size_t kOffSeg = kOffPos + kMaxTokens;
constexpr size_t kOffStart = kOffSeg + kMaxTokens;
constexpr size_t kOffQlen = kOffStart + kMaxSeqs;
constexpr size_t kOffKlen = kOffQlen + kMaxSeqs;
constexpr size_t kOffWork = kOffKlen + kMaxSeqs;
constexpr size_t kOffCount = kOffWork + 4 * (size_t)kMaxItems;
constexpr size_t kOffErr = kOffCount + 4;
constexpr size_t kWords = kOffErr + 60;  // about 650 KB in total

__device__ __align__(256) int32_t g_attention_scratch[kWords];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
esm_status scratch_on_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ESM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ESM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attention_scratch) != cudaSuccess || p == nullptr) return ESM_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return ESM_OK;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The call's outcome as an esm_status code, from the error word the kernels latched.
__global__ void noalloc_status_kernel(const unsigned* err, int32_t* status) {
  const unsigned e = *err;
  *status = (e & ERRBIT_CU_SEQLENS) ? ESM_ERR_BAD_CU_SEQLENS : (e & ERRBIT_TIMEOUT) ? ESM_ERR_TIMEOUT : ESM_OK;
}

}  // namespace
}  // namespace esm

using namespace esm;

extern "C" esm_status esm_op_attention_noalloc(const void* qkv, const int32_t* cu_seqlens, int num_seqs,
                                               int total_tokens, int max_seqlen, int hidden, int heads, void* o,
                                               int32_t* status, esm_stream_t stream) {
  if (!qkv || !cu_seqlens || !o) return ESM_ERR_INVALID_ARG;
  if (num_seqs <= 0 || total_tokens < 0 || max_seqlen <= 0) return ESM_ERR_INVALID_ARG;
  if (num_seqs > kMaxSeqs || total_tokens > kMaxTokens || max_seqlen > kMaxTokens) return ESM_ERR_INVALID_ARG;
  if (heads <= 0 || hidden != 64 * heads) return ESM_ERR_UNSUPPORTED;
  if (!aligned_to(qkv, 16) || !aligned_to(o, 16) || (status && !aligned_to(status, 4))) return ESM_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ESM_ERR_CUDA;
  if (major != 10 || minor != 3) return ESM_ERR_UNSUPPORTED;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (total_tokens == 0) {
    if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), cs) != cudaSuccess) return ESM_ERR_CUDA;
    return ESM_OK;
  }
  CUtensorMap tm;
  if (!encode_attention_qkv_map(qkv, total_tokens, hidden, &tm)) return ESM_ERR_CUDA;
  int32_t* s = nullptr;
  esm_status st = scratch_on_current_device(&s);
  if (st != ESM_OK) return st;
  PackBuffers pb;
  pb.pos_id = s + kOffPos;
  pb.seg_id = s + kOffSeg;
  pb.seg_start = s + kOffStart;
  pb.seg_qlen = s + kOffQlen;
  pb.seg_klen = s + kOffKlen;
  pb.work = s + kOffWork;
  pb.work_count = s + kOffCount;
  unsigned* err = reinterpret_cast<unsigned*>(s + kOffErr);
  // Indices of tokens that no (malformed) segment covers must not keep an earlier call's
  // values, and the error word starts clear.
  if (cudaMemsetAsync(pb.pos_id, 0, sizeof(int32_t) * (size_t)total_tokens, cs) != cudaSuccess ||
      cudaMemsetAsync(pb.seg_id, 0, sizeof(int32_t) * (size_t)total_tokens, cs) != cudaSuccess ||
      cudaMemsetAsync(err, 0, sizeof(unsigned), cs) != cudaSuccess)
    return ESM_ERR_CUDA;
  const int max_items = (total_tokens + kAttnQTileTc - 1) / kAttnQTileTc + num_seqs;
  launch_pack_index(cu_seqlens, num_seqs, total_tokens, max_seqlen, kMaxTokens, pb, err, cs);
  launch_attn_worklist(num_seqs, max_items, kAttnQTileTc, pb, cs);
  if (launch_attention_tc(&tm, o, Act::BF16, hidden, heads, max_items, pb, nullptr, nullptr, err, cs) != cudaSuccess)
    return ESM_ERR_CUDA;
  if (status) noalloc_status_kernel<<<1, 1, 0, cs>>>(err, status);
  return cudaGetLastError() == cudaSuccess ? ESM_OK : ESM_ERR_CUDA;
}
