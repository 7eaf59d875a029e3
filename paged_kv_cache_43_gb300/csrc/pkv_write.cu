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
#include <cuda_fp8.h>

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

// FP8 (e4m3) cache: each thread turns 16 bf16 inputs (32 bytes) of K and of V
// into 16 codes (16 bytes): an IEEE fp32 division by the kv head's scale, then
// round-to-nearest-even to e4m3 with clamping to the largest finite value.
// row_vecs counts 16-byte vectors of the *cache* row (num_kv_heads * head_size
// codes / 16).
__device__ __forceinline__ uint4 quantise16(const uint4 lo, const uint4 hi, float scale) {
  const uint32_t in[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = make_float2(__fdiv_rn(bf16_lo(in[2 * i]), scale),
                                 __fdiv_rn(bf16_hi(in[2 * i]), scale));
    const float2 b = make_float2(__fdiv_rn(bf16_lo(in[2 * i + 1]), scale),
                                 __fdiv_rn(bf16_hi(in[2 * i + 1]), scale));
    const uint32_t pa = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
    const uint32_t pb = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
    out[i] = (pa & 0xFFFFu) | (pb << 16);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(256) pkv_write_fp8_kernel(const WriteArgs a) {
  const uint4* __restrict__ k = static_cast<const uint4*>(a.k);   // bf16: 2 vectors per cache vector
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
    const int h = static_cast<int>((c * 16) / a.head_size);  // kv head of these 16 elements
    kc[slot * a.row_vecs + c] = quantise16(__ldg(k + 2 * i), __ldg(k + 2 * i + 1), __ldg(a.k_scale + h));
    vc[slot * a.row_vecs + c] = quantise16(__ldg(v + 2 * i), __ldg(v + 2 * i + 1), __ldg(a.v_scale + h));
  }
}

cudaError_t launch_write_fp8(const WriteArgs& a, cudaStream_t stream, int num_sms) {
  const int64_t total = static_cast<int64_t>(a.num_tokens) * a.row_vecs;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  pkv_write_fp8_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
  return cudaGetLastError();
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
