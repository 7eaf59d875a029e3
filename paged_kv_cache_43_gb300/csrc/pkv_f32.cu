// pkv_f32.cu -- paged attention with fp32 I/O and fp32 arithmetic (decode and
// chunked prefill alike).
//
// Same definition as the bf16 path ("Implémentation du cœur du moteur
// d'inférence haute performance vLLM", ch. 6 "Flux des paramètres du chemin
// non-cascadé" and "Branche de masque"): query row j of a chunk of q_s rows of
// sequence s sits at position L - q_s + j and attends keys 0..L - q_s + j read
// through block_tables.  fp32 scores cannot go through bf16 tensor cores
// without losing the 1e-5 accuracy this dtype is held to, so this path uses
// CUDA-core FMAs: one CTA per (query row, q head), 4 warps taking every 4th
// key, a warp-wide dot product per key (coalesced 128/256-byte K and V rows),
// online softmax per warp, and a shared-memory merge of the warps.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kF32Warps = 4;

template <int D>
__global__ void __launch_bounds__(kF32Warps * 32) pkv_attention_f32_kernel(const F32Args a) {
  constexpr int PER = D / 32;
  __shared__ float sm_m[kF32Warps], sm_l[kF32Warps];
  __shared__ float sm_o[kF32Warps][D];
  const int t = blockIdx.x;
  const int hq = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Sequence owning row t: the last s with query_start_loc[s] <= t.
  if (t >= __ldg(a.query_start_loc + a.num_seqs)) return;  // row of no sequence
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.query_start_loc + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int q0 = __ldg(a.query_start_loc + s);
  const int qn = __ldg(a.query_start_loc + s + 1) - q0;
  const int j = t - q0;
  const int L = __ldg(a.context_lens + s);
  float* out = a.out + (static_cast<int64_t>(t) * a.num_q_heads + hq) * D;
  if (j < 0 || j >= qn) return;  // not a row of s (malformed query_start_loc)
  if (L < 1 || static_cast<int64_t>(L) > a.bt_stride * kBlock || qn > L) {
    if (threadIdx.x == 0 && hq == 0 && j == 0)
      raise_error(a.err, qn > L && L >= 1 ? PKV_ERR_QUERY_LEN : PKV_ERR_CONTEXT_LEN);
    for (int d = threadIdx.x; d < D; d += blockDim.x) out[d] = 0.f;
    return;
  }
  const int G = a.num_q_heads / a.num_kv_heads;
  const int kvh = hq / G;
  const int pos = L - qn + j;
  const float* qrow = a.q + (static_cast<int64_t>(t) * a.num_q_heads + hq) * D;
  float qv[PER], acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    qv[e] = __ldg(qrow + lane + 32 * e);
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int32_t* bt = a.block_tables + static_cast<int64_t>(s) * a.bt_stride;
  const int kfirst = (a.window > 0 && pos + 1 > a.window) ? pos + 1 - a.window : 0;
  for (int p = kfirst + warp; p <= pos; p += kF32Warps) {
    const int bid = __ldg(bt + p / kBlock);
    if (bid < 0 || bid >= a.num_blocks) {
      if (lane == 0) raise_error(a.err, PKV_ERR_BLOCK_ID);
      continue;
    }
    const int64_t row = ((static_cast<int64_t>(bid) * kBlock + p % kBlock) * a.num_kv_heads + kvh) * D;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) dot = fmaf(qv[e], __ldg(a.k_cache + row + lane + 32 * e), dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float x = dot * a.scale;
    const float mn = fmaxf(m, x);
    const float alpha = expf(m - mn);  // m = -inf on the first key: alpha = 0
    const float w = expf(x - mn);
    l = l * alpha + w;
#pragma unroll
    for (int e = 0; e < PER; ++e)
      acc[e] = fmaf(w, __ldg(a.v_cache + row + lane + 32 * e), acc[e] * alpha);
    m = mn;
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) sm_o[warp][lane + 32 * e] = acc[e];
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kF32Warps; ++w) M = fmaxf(M, sm_m[w]);
  float den = 0.f, f[kF32Warps];
#pragma unroll
  for (int w = 0; w < kF32Warps; ++w) {
    f[w] = (sm_m[w] == -INFINITY) ? 0.f : expf(sm_m[w] - M);
    den += f[w] * sm_l[w];
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < kF32Warps; ++w) r += f[w] * sm_o[w][d];
    out[d] = den > 0.f ? r / den : 0.f;
  }
}

}  // namespace

cudaError_t launch_attention_f32(const F32Args& a, cudaStream_t stream) {
  if (a.num_tokens == 0 || a.num_seqs == 0) return cudaSuccess;
  dim3 grid(a.num_tokens, a.num_q_heads);
  if (a.head_size == 128)
    pkv_attention_f32_kernel<128><<<grid, kF32Warps * 32, 0, stream>>>(a);
  else
    pkv_attention_f32_kernel<64><<<grid, kF32Warps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pkv
