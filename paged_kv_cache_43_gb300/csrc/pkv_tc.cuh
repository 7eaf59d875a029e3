// pkv_tc.cuh -- tcgen05 (5th-generation tensor core) and TMEM helpers for
// sm_103a: shared-memory matrix descriptors, instruction descriptors, MMA
// issue/commit, TMEM allocation and 32x32b loads/stores.
#pragma once

#include <stdint.h>

namespace pkv {
namespace tc {

// Shared-memory matrix descriptor (tcgen05 format, version 1) for a
// 128-byte-swizzled operand.  K-major: rows of 128 B (64 bf16 of K), 8-row
// groups `sbo` bytes apart (lbo unused).  MN-major: 128-B rows along MN, one
// row per K index, 8-K groups `sbo` apart, 64-element MN groups `lbo` apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, MxN tile;
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// The same with fp16 A and B (type fields 0).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Eight K-steps of one tile product in one instruction group:
//   D (+)= sum over k < 8 of A_k * B_k,  A_k / B_k = the base descriptors
//   advanced by OA_k / OB_k (16-byte units, immediates; address fields never
//   carry out of the low word).  Only the first step reads `accumulate`; the
//   others always accumulate.  One MMA costs a single tcgen05.mma plus two
//   32-bit adds on the issuing thread: its instructions share the SM
//   sub-partition's issue slots with busy softmax warps, so fewer of them
//   keep the tensor core fed.
template <int OA1, int OA2, int OA3, int OA4, int OA5, int OA6, int OA7, int OB1, int OB2, int OB3,
          int OB4, int OB5, int OB6, int OB7>
__device__ __forceinline__ void mma_ss_x8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b32 al, ah, bl, bh, x, y;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.eq.u32 t, 1, 1;\n\t"
      "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.u32 x, al, %5;\n\tadd.u32 y, bl, %12;\n\tmov.b64 a, {x, ah};\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.u32 x, al, %6;\n\tadd.u32 y, bl, %13;\n\tmov.b64 a, {x, ah};\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.u32 x, al, %7;\n\tadd.u32 y, bl, %14;\n\tmov.b64 a, {x, ah};\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.u32 x, al, %8;\n\tadd.u32 y, bl, %15;\n\tmov.b64 a, {x, ah};\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.u32 x, al, %9;\n\tadd.u32 y, bl, %16;\n\tmov.b64 a, {x, ah};\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.u32 x, al, %10;\n\tadd.u32 y, bl, %17;\n\tmov.b64 a, {x, ah};\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t"
      "add.u32 x, al, %11;\n\tadd.u32 y, bl, %18;\n\tmov.b64 a, {x, ah};\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(OA1), "n"(OA2), "n"(OA3),
      "n"(OA4), "n"(OA5), "n"(OA6), "n"(OA7), "n"(OB1), "n"(OB2), "n"(OB3), "n"(OB4), "n"(OB5),
      "n"(OB6), "n"(OB7)
      : "memory");
}

// The same with A in TMEM (columns a_tmem + 8k for step k) and B advanced by
// 128 (2048 bytes) per step: the P V product of one 128-key tile.
__device__ __forceinline__ void mma_ts_x8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b32 bl, bh, x, y;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.eq.u32 t, 1, 1;\n\t"
      "mov.b64 {bl, bh}, %2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 x, %1, 8;\n\tadd.u32 y, bl, 128;\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
      "add.u32 x, %1, 16;\n\tadd.u32 y, bl, 256;\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
      "add.u32 x, %1, 24;\n\tadd.u32 y, bl, 384;\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
      "add.u32 x, %1, 32;\n\tadd.u32 y, bl, 512;\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
      "add.u32 x, %1, 40;\n\tadd.u32 y, bl, 640;\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
      "add.u32 x, %1, 48;\n\tadd.u32 y, bl, 768;\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t"
      "add.u32 x, %1, 56;\n\tadd.u32 y, bl, 896;\n\tmov.b64 b, {y, bh};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %3, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole-warp TMEM allocation; the column base is written to `dst` (shared).
__device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// ---------------------------------------------------------------- softmax math
// Three-input maximum (one instruction on sm_100+).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two lanes of fp32 in one 64-bit register pair.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

// (y0, y1) = (x0, x1) * m + b, lane-wise (packed f32x2 FMA).
__device__ __forceinline__ void fma_f32x2(float x0, float x1, uint64_t m, uint64_t b, float& y0,
                                          float& y1) {
  asm("{\n\t.reg .b64 a, r;\n\tmov.b64 a, {%2, %3};\n\t"
      "fma.rn.f32x2 r, a, %4, %5;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "l"(m), "l"(b));
}

// acc += (x0, x1), lane-wise (packed f32x2 add).
__device__ __forceinline__ void add_f32x2(uint64_t& acc, float x0, float x1) {
  asm("{\n\t.reg .b64 a;\n\tmov.b64 a, {%1, %2};\n\tadd.rn.f32x2 %0, %0, a;\n\t}"
      : "+l"(acc)
      : "f"(x0), "f"(x1));
}

__device__ __forceinline__ float sum_f32x2(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}

}  // namespace tc
}  // namespace pkv
