// pkv_write.cu -- KV-cache write: scatter this step's K/V rows into the paged
// cache through slot_mapping.
//
// Follows "Implémentation du cœur du moteur d'inférence haute performance
// vLLM", ch. 6 "Écriture du KV cache" (the write is a scatter through
// slot_mapping, whose length gives the token count) and ch. 5 "slot_mapping et
// la block table" (unused tail entries are -1 and must be skipped).
//
// A token row (num_kv_heads * head_size elements) is contiguous in both the
// input and the cache ([num_blocks, 16, Hkv, D] makes cache row `slot` the
// slot-th run of Hkv*D elements), so the copy is a plain 16-byte vector move:
// one thread per 16-byte vector of K and the same vector of V, consecutive
// threads on consecutive vectors of a row (coalesced reads and writes).
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

__global__ void __launch_bounds__(256) pkv_write_kernel(const WriteArgs a) {
  const uint4* __restrict__ k = static_cast<const uint4*>(a.k);
  const uint4* __restrict__ v = static_cast<const uint4*>(a.v);
  uint4* __restrict__ kc = static_cast<uint4*>(a.k_cache);
  uint4* __restrict__ vc = static_cast<uint4*>(a.v_cache);
  const int64_t total = static_cast<int64_t>(a.num_tokens) * a.row_vecs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / a.row_vecs;
    const int64_t c = i - t * a.row_vecs;
    const int64_t slot = __ldg(a.slot_mapping + t);
    if (slot < 0) continue;  // padding
    if (slot >= a.num_slots) {
      if (c == 0) raise_error(a.err, PKV_ERR_SLOT);
      continue;
    }
    const uint4 kv = __ldg(k + i);
    const uint4 vv = __ldg(v + i);
    kc[slot * a.row_vecs + c] = kv;
    vc[slot * a.row_vecs + c] = vv;
  }
}

cudaError_t launch_write(const WriteArgs& a, cudaStream_t stream, int num_sms) {
  const int64_t total = static_cast<int64_t>(a.num_tokens) * a.row_vecs;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  pkv_write_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv
