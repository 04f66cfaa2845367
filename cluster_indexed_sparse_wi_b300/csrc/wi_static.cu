// Decode entry point for callers that cannot allocate device memory.
//
// Some hosts of this library have no allocator to give it: an inference
// runtime that hands a plugin only pre-planned buffers, code running where
// cudaMalloc is forbidden or would break a memory budget fixed up front.  For
// them wi_decode_attention_static runs the same decode as wi_decode_attention
// but takes no workspace: it uses a fixed scratch array that lives in this
// file as a static device variable, so every GPU that loads the library holds
// WI_STATIC_SCRATCH_BYTES for it until the process exits.
#include <mutex>

#include "wi.h"
#include "wi_internal.h"

namespace {

constexpr size_t kScratchBytes = WI_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_lock;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WI_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return WI_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return WI_ERR_LAUNCH;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return WI_OK;
}

}  // namespace

extern "C" int wi_decode_attention_static(const wi_decode_params* p, const void* q, const void* K,
                                          const void* V, const wi_index* index, float* out,
                                          float* lse, int32_t* topk_ids, wi_stream_t stream) {
  // every host check first: a rejected call queues nothing on the stream and
  // leaves the scratch (and its status word) untouched
  int st = wi::decode_precheck(p, q, K, V, index, out);
  if (st != WI_OK) return st;
  wi_decode_layout lay;
  if ((st = wi_decode_workspace_layout(p, index->n_clusters, &lay)) != WI_OK) return st;
  if (lay.total > kScratchBytes) return WI_ERR_WORKSPACE;  // beyond the fixed scratch
  void* ws = nullptr;
  if ((st = scratch_address(&ws)) != WI_OK) return st;
  const cudaStream_t s = (cudaStream_t)stream;
  // The scratch keeps the previous call's contents (another caller may have
  // stopped mid-call): the per-call progress counters must start at zero.
  // The status word is left alone, so that an error of an earlier call stays
  // readable through wi_decode_static_status until it is read.
  char* base = static_cast<char*>(ws);
  if (cudaMemsetAsync(base + lay.counters, 0, (size_t)lay.counter_bytes, s) != cudaSuccess)
    return WI_ERR_LAUNCH;
  return wi_decode_attention(p, q, K, V, index, out, lse, topk_ids, ws, kScratchBytes, stream);
}

extern "C" int wi_decode_static_status(wi_stream_t stream, int* device_status) {
  if (device_status == nullptr) return WI_ERR_INVALID_ARG;
  void* ws = nullptr;
  const int st = scratch_address(&ws);
  if (st != WI_OK) return st;
  return wi_sync_status(ws, stream, device_status);
}
