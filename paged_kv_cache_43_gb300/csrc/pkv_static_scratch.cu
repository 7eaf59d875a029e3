// pkv_static_scratch.cu -- pkv_attention for callers that cannot allocate
// device memory.
//
// pkv_attention needs a caller-provided split-K workspace.  Some callers have
// no way to provide one: a plugin running inside a host framework that owns
// every device allocation through its own pool (a stray cudaMalloc there can
// synchronise the whole device and escapes the pool's accounting), or a
// latency-critical decode loop that is not allowed to enter the allocator at
// all.  This entry point serves them from a fixed-size array that lives in the
// library itself: a file-scope __device__ array, created when the library's
// device code is loaded on a GPU and held until the process exits.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  Nothing in it needs to start at zero: the split-K kernels
// write every partial they later read within the same call.  Two calls whose
// work overlaps on the GPU (for example on two streams) race on the array, so
// callers must order them (same stream, or an event between them).
#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// The scratch itself.  Host code must not take its address with `&`: on the
// host this name is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_E_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return PKV_E_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_attention_static_scratch(void* out, const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_tables,
                                            const int32_t* context_lens,
                                            const int32_t* query_start_loc, float scale,
                                            const pkv_cache_desc* cache,
                                            const pkv_attn_meta* meta, void* stream) {
  const size_t need = pkv_attention_workspace_size(cache, meta);
  if (need == static_cast<size_t>(-1)) {
    // Invalid description: let pkv_attention report the precise status.
    return pkv_attention(out, q, k_cache, v_cache, block_tables, context_lens,
                         query_start_loc, scale, cache, meta, nullptr, 0, stream);
  }
  if (need > PKV_STATIC_SCRATCH_BYTES) return PKV_E_WORKSPACE;
  void* scratch = nullptr;
  if (int st = pkv::scratch_address(&scratch)) return st;
  return pkv_attention(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                       scale, cache, meta, scratch, PKV_STATIC_SCRATCH_BYTES, stream);
}
