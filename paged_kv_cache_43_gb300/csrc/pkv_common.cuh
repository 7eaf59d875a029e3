// pkv_common.cuh -- inline-PTX helpers shared by the libpkv kernels (sm_103a).
//
// mbarrier, TMA (cp.async.bulk.tensor), ldmatrix, movmatrix and the bf16
// mma.sync tile, plus the bounded wait every spin in this library goes through.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Longest any on-chip wait may spin before giving up with PKV_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ void raise_error(int32_t* err, int32_t bits) {
  if (err != nullptr && bits != 0) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same bytes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking probe: has the phase of `bar` with this parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// after `limit_ns` (kWaitLimitNs unless a launch was made with the test hook
// of pkv_debug_wait_test) and returns false (the caller raises
// PKV_ERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// The main-loop wait limit of a launch: kWaitLimitNs, or the short one the
// test hook of pkv_debug_wait_test sets.
__device__ __forceinline__ uint64_t wait_limit(uint64_t requested_ns) {
  return requested_ns != 0 ? requested_ns : kWaitLimitNs;
}

// The sequence holding query row `tok`: the s with qsl[s] <= tok < qsl[s + 1]
// (binary search over the num_seqs + 1 ascending entries; -1 if none).
__device__ __forceinline__ int seq_of_row(const int32_t* qsl, int num_seqs, int tok) {
  int lo = 0, hi = num_seqs;   // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(qsl + mid) <= tok) lo = mid;
    else hi = mid;
  }
  return (num_seqs > 0 && __ldg(qsl + lo) <= tok && tok < __ldg(qsl + lo + 1)) ? lo : -1;
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policy for data read exactly once (the KV stream).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data other CTAs will read again soon.
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 3-D tiled TMA load into this CTA's shared memory; completion is signalled on
// `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// 3-D tiled TMA store from this CTA's shared memory (bulk-group completion);
// elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Named barrier over `nthreads` threads returning whether `pred` held in all.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, %3, q;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------- warp MMA
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Transposes the warp's 8x8 b16 fragment (row lane/4, columns 2*(lane%4)+{0,1}).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col).  A pure register
// operation (not volatile): the compiler may interleave it with other work.
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ---- fp16 operands (the FP8-cache kernels: every e4m3 value is exact in fp16)

// D (16x8 fp32) += A (16x16 f16, row) * B (16x8 f16, col).
__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float f16_lo(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16)));
}

// Four e4m3 codes (byte i = code i) -> four fp16 values, exactly: .x holds
// codes 0, 1 and .y codes 2, 3 (low half first).  A NaN code gives a NaN.
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t codes) {
  uint32_t lo, hi;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(codes));
  return make_uint2(lo, hi);
}

// Byte offset of 16-byte chunk `c` of row `r` in a 16-row x D e4m3 tile that
// TMA wrote with the D-byte swizzle (128 B: chunk ^= r % 8; 64 B: chunk ^=
// (r / 2) % 4, i.e. address bits 4-5 XOR bits 7-8).
template <int D>
__device__ __forceinline__ uint32_t swz8(int r, int c) {
  if constexpr (D == 128) return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
  else return static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Operand-type switch of the mma.sync kernels: bf16 (bf16 caches) or fp16
// (FP8 caches).
template <bool F16>
__device__ __forceinline__ void mma_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (F16) mma_f16_16816(d, a0, a1, a2, a3, b0, b1);
  else mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) return pack_f16(lo, hi);
  else return pack_bf16(lo, hi);
}
template <bool F16>
__device__ __forceinline__ float lo2(uint32_t x) {
  if constexpr (F16) return f16_lo(x);
  else return bf16_lo(x);
}
template <bool F16>
__device__ __forceinline__ float hi2(uint32_t x) {
  if constexpr (F16) return f16_hi(x);
  else return bf16_hi(x);
}

// bf16 query values -> fp16 for the FP8 kernels.  A row whose largest
// magnitude exceeds 2^14 is first scaled by a power of two 2^-e (exact) so
// that it stays inside the fp16 range; the caller multiplies that row's
// scores by 2^e.  Returns e (0 for rows in range, or non-finite ones).
__device__ __forceinline__ int f16_row_exponent(float amax) {
  if (!(amax > 16384.f) || !(amax <= 3.402823466e38f)) return 0;
  return ((__float_as_int(amax) >> 23) & 0xFF) - 127 + 1 - 14;  // amax * 2^-e < 2^14
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float mul) {
  return pack_f16(bf16_lo(w) * mul, bf16_hi(w) * mul);
}

// Byte offset of element (row, d) inside one 16-row x head_size bf16 tile that
// TMA wrote as head_size/64 boxes of 16 rows x 128 B with the 128-byte
// swizzle: box h = d / 64 sits at h * 2048, row r at r * 128, and the 16-byte
// chunk index (d % 64) / 8 is XOR-ed with r % 8.  `d` must be a multiple of 8.
__device__ __forceinline__ uint32_t swz_offset(int row, int d) {
  return static_cast<uint32_t>((d >> 6) * 2048 + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4));
}

}  // namespace pkv
