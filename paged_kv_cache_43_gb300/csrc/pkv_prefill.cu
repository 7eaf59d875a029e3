// pkv_prefill.cu -- paged varlen attention for chunked prefill (any query
// length >= 1, causal inside the chunk), bf16 in, fp32 accumulate.
//
// What it computes: query j of a chunk of q_s new tokens of sequence s (L keys
// in total) sits at absolute position L - q_s + j ("Implémentation du cœur du
// moteur d'inférence haute performance vLLM", ch. 6 "Branche de masque":
// q_abs = q_idx + seqlen_k - seqlen_q) and attends keys 0..L - q_s + j, read
// through the block table (ch. 6 "Flux des paramètres du chemin non-cascadé").
// Sequences of a mixed batch are independent rows of one flattened batch
// ("Khám phá vLLM: Giải phẫu hệ thống suy luận LLM thông lượng cao",
// "Chạy forward pass").
//
// GB300 design:
//  * CTA = 64 query rows x one kv head of one sequence; rows are (token j,
//    q head g) pairs with g fastest, so the G heads sharing a kv head share
//    every K/V tile (GQA grouping on the MMA's M dimension).
//  * one producer warp streams 64-key tiles (4 cache blocks) of K and V with
//    TMA (64-column boxes, 128-byte swizzle) into an NS-deep ring guarded by
//    full/empty mbarriers; four consumer warps (16 rows each) compute
//    S = Q K^T and O += P V with bf16 m16n8k16 tensor-core MMAs, the
//    probabilities staying in registers between the two products.
//  * causal trimming: a CTA only loads the tiles its last row can see, and
//    masks only the tiles that straddle its rows' limits.
//  * tiles are visited heaviest-row-tile first (grid.x reversed).
//  * FP8 (e4m3) cache: the producer lands the codes (one box per block, half
//    the bytes, swizzled at the head row's width); the consumers widen each tile into one of two
//    fp16 tiles in the swizzled layout above (e4m3 -> fp16 is exact), release
//    the code stage at once, and run the same MMAs on fp16 operands (Q
//    converted once, a row whose values exceed 2^14 scaled by a power of two).
//    K's per-(sequence, kv head) descale folds into the score scale, V's into
//    the output.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kTileKeys = 64;  // 4 cache blocks per stage

template <int D, bool FP8>
struct PrefillTile {
  static constexpr int kBlkBytes = D * 2 * kBlock;            // one 16-bit block of K (or V)
  static constexpr int kKBytes = kBlkBytes * (kTileKeys / kBlock);
  // what TMA lands: bf16 tiles, or e4m3 codes (row r of the tile at r * D)
  static constexpr int kLoadBlk = FP8 ? D * kBlock : kBlkBytes;
  static constexpr int kLoadK = kLoadBlk * (kTileKeys / kBlock);
  static constexpr int kStageBytes = 2 * kLoadK;
  static constexpr int kConvBytes = FP8 ? 2 * kKBytes : 0;  // one widened K+V tile
};

template <int D, int NS, bool FP8>
constexpr int prefill_smem_bytes() {
  using T = PrefillTile<D, FP8>;
  return 1024 + NS * T::kStageBytes + 2 * T::kConvBytes + 2 * NS * 8;
}

// 16 codes -> 16 fp16 values (two 16-byte vectors), or zeros.
__device__ __forceinline__ void widen16(uint8_t* dst_lo, uint8_t* dst_hi, const uint8_t* src,
                                        bool zero) {
  uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
  if (!zero) {
    const uint4 c = *reinterpret_cast<const uint4*>(src);
    const uint2 x = e4m3x4_to_f16x4(c.x), y = e4m3x4_to_f16x4(c.y);
    const uint2 z = e4m3x4_to_f16x4(c.z), w = e4m3x4_to_f16x4(c.w);
    lo = make_uint4(x.x, x.y, y.x, y.y);
    hi = make_uint4(z.x, z.y, w.x, w.y);
  }
  *reinterpret_cast<uint4*>(dst_lo) = lo;
  *reinterpret_cast<uint4*>(dst_hi) = hi;
}

template <int D, int NS, bool FP8>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32)
    pkv_prefill_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using T = PrefillTile<D, FP8>;
  constexpr int NWC = kConsumerWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* conv0 = smem + NS * T::kStageBytes;  // FP8: two widened tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(conv0 + 2 * T::kConvBytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + NS);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int s = a.seq_begin + blockIdx.z;
  const int kvh = blockIdx.y;
  const int mtile = a.num_mtiles - 1 - blockIdx.x;  // heaviest first
  const int G = a.group;
  const int Hq = a.num_q_heads;

  const int L = __ldg(a.context_lens + s);
  const int q0 = __ldg(a.query_start_loc + s);
  const int qn = __ldg(a.query_start_loc + s + 1) - q0;
  const int nrows = qn * G;
  const int row0 = mtile * kPrefillRows;
  const bool bad_rows = qn < 0 || q0 < 0 || static_cast<int64_t>(q0) + qn > a.num_tokens;
  if (bad_rows || qn == 0 || row0 >= nrows) {
    if (bad_rows && blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0)
      raise_error(a.err, PKV_ERR_QUERY_LEN);
    return;
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  const bool bad_len = (L < 1 || static_cast<int64_t>(L) > a.bt_stride * kBlock);
  if (bad_len || qn > L || qn > a.max_query_len) {
    if (threadIdx.x == 0 && mtile == 0 && kvh == 0)
      raise_error(a.err, bad_len ? PKV_ERR_CONTEXT_LEN : PKV_ERR_QUERY_LEN);
    const int nr = min(kPrefillRows, nrows - row0);
    for (int i = threadIdx.x; i < nr * D; i += blockDim.x) {
      const int r = row0 + i / D;
      out[(static_cast<int64_t>(q0 + r / G) * Hq + kvh * G + r % G) * D + i % D] =
          __float2bfloat16(0.f);
    }
    return;
  }
  const int row_last = min(row0 + kPrefillRows, nrows) - 1;
  const int pos_max = L - qn + row_last / G;          // last key any row of this CTA sees
  const int ntiles = (pos_max + kTileKeys) / kTileKeys;
  const int nblk = (pos_max + kBlock) / kBlock;       // cache blocks to load
  // With a sliding window, tiles wholly before the lowest row's window are
  // never loaded (their block-table entries may hold the null block).
  const int pos_min = L - qn + row0 / G;
  const int j0 = (a.window > 0 && pos_min - a.window + 1 > 0)
                     ? (pos_min - a.window + 1) / kTileKeys : 0;
  // First cache block holding a key some row can see: earlier blocks of tile
  // j0 are not loaded (their entries may be null); their V rows are zeroed.
  const int b_lo = (a.window > 0 && pos_min - a.window + 1 > 0)
                       ? (pos_min - a.window + 1) / kBlock : 0;

  if (threadIdx.x == 0) {
    prefetch_tensor_map(&kmap);
    prefetch_tensor_map(&vmap);
#pragma unroll
    for (int st = 0; st < NS; ++st) {
      mbar_init(full0 + 8 * st, 1);
      mbar_init(empty0 + 8 * st, NWC);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == NWC) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = policy_evict_first();
    const int32_t* bt = a.block_tables + static_cast<int64_t>(s) * a.bt_stride;
    int my_bid = -1;
    for (int it = j0; it < ntiles; ++it) {
      const int rel = it - j0;  // ring position
      const int st = rel % NS;
      if (rel >= NS && !mbar_wait(empty0 + 8 * st, ((rel / NS) - 1) & 1)) {
        if (lane == 0) raise_error(a.err, PKV_ERR_TIMEOUT);
        break;
      }
      if ((rel & 7) == 0) {  // block ids for the next 8 tiles, one per lane
        const int b = it * 4 + lane;
        my_bid = b < nblk ? __ldg(bt + b) : -1;
      }
      bool ok[4];
      int bid[4];
      uint32_t bytes = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        bid[b] = __shfl_sync(0xffffffffu, my_bid, (rel & 7) * 4 + b);
        const bool in_range = it * 4 + b < nblk && it * 4 + b >= b_lo;
        ok[b] = in_range && bid[b] >= 0 && bid[b] < a.num_blocks;
        if (in_range && !ok[b] && lane == 0) raise_error(a.err, PKV_ERR_BLOCK_ID);
        bytes += ok[b] ? 2u * T::kLoadBlk : 0u;
      }
      if (lane == 0) {
        const uint32_t full = full0 + 8 * st;
        const uint32_t dst = smem_u32(smem + st * T::kStageBytes);
        if (bytes == 0) {
          mbar_arrive(full);
        } else {
          fence_proxy_async();
          mbar_arrive_expect_tx(full, bytes);
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            if (!ok[b]) continue;
            if constexpr (FP8) {
              tma_load_3d(dst + b * T::kLoadBlk, &kmap, full, 0, kvh, bid[b] * kBlock, policy);
              tma_load_3d(dst + T::kLoadK + b * T::kLoadBlk, &vmap, full, 0, kvh,
                          bid[b] * kBlock, policy);
            } else {
#pragma unroll
              for (int h = 0; h < D / 64; ++h) {
                tma_load_3d(dst + b * T::kBlkBytes + h * 2048, &kmap, full, h * 64, kvh,
                            bid[b] * kBlock, policy);
                tma_load_3d(dst + T::kKBytes + b * T::kBlkBytes + h * 2048, &vmap, full, h * 64,
                            kvh, bid[b] * kBlock, policy);
              }
            }
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int wrow0 = row0 + warp * 16;            // first row of this warp
  const int rA = wrow0 + (lane >> 2);            // the two rows this lane holds
  const int rB = rA + 8;
  const bool vA = rA < nrows, vB = rB < nrows;
  const int jA = vA ? rA / G : qn - 1, jB = vB ? rB / G : qn - 1;
  const int posA = L - qn + jA, posB = L - qn + jB;
  const int wpos_min = L - qn + min(wrow0, nrows - 1) / G;
  const int wpos_max = L - qn + min(wrow0 + 15, nrows - 1) / G;
  const int W = a.window;
  const int loA = W > 0 ? posA - W + 1 : 0, loB = W > 0 ? posB - W + 1 : 0;  // window starts

  // Q as the A operand: a0 = (rA, k), a1 = (rB, k), a2 = (rA, k+8), a3 = (rB, k+8)
  uint32_t qa[D / 16][4];
  {
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(a.q);
    const uint32_t* qrA = reinterpret_cast<const uint32_t*>(
        qbase + (static_cast<int64_t>(q0 + jA) * Hq + kvh * G + (vA ? rA % G : 0)) * D);
    const uint32_t* qrB = reinterpret_cast<const uint32_t*>(
        qbase + (static_cast<int64_t>(q0 + jB) * Hq + kvh * G + (vB ? rB % G : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = vA ? __ldg(qrA + kk * 8 + (lane & 3)) : 0u;
      qa[kk][1] = vB ? __ldg(qrB + kk * 8 + (lane & 3)) : 0u;
      qa[kk][2] = vA ? __ldg(qrA + kk * 8 + 4 + (lane & 3)) : 0u;
      qa[kk][3] = vB ? __ldg(qrB + kk * 8 + 4 + (lane & 3)) : 0u;
    }
  }

  float scale_log2 = a.scale_log2, out_scale = 1.f;
  float sclA = scale_log2, sclB = scale_log2;  // score scales of rows rA, rB
  if constexpr (FP8) {
    scale_log2 *= __ldg(a.k_descale + static_cast<int64_t>(s) * a.num_kv_heads + kvh);
    out_scale = __ldg(a.v_descale + static_cast<int64_t>(s) * a.num_kv_heads + kvh);
    // Q to fp16; a row held by the 4 lanes of lane/4 is scaled by 2^-e if its
    // values exceed 2^14, and its scores by 2^e.
    float mA_ = 0.f, mB_ = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      mA_ = fmaxf(mA_, fmaxf(fmaxf(fabsf(bf16_lo(qa[kk][0])), fabsf(bf16_hi(qa[kk][0]))),
                             fmaxf(fabsf(bf16_lo(qa[kk][2])), fabsf(bf16_hi(qa[kk][2])))));
      mB_ = fmaxf(mB_, fmaxf(fmaxf(fabsf(bf16_lo(qa[kk][1])), fabsf(bf16_hi(qa[kk][1]))),
                             fmaxf(fabsf(bf16_lo(qa[kk][3])), fabsf(bf16_hi(qa[kk][3])))));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mA_ = fmaxf(mA_, __shfl_xor_sync(0xffffffffu, mA_, off));
      mB_ = fmaxf(mB_, __shfl_xor_sync(0xffffffffu, mB_, off));
    }
    const int eA = f16_row_exponent(mA_), eB = f16_row_exponent(mB_);
    const float dA = pow2f(-eA), dB = pow2f(-eB);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = bf16x2_to_f16x2(qa[kk][0], dA);
      qa[kk][2] = bf16x2_to_f16x2(qa[kk][2], dA);
      qa[kk][1] = bf16x2_to_f16x2(qa[kk][1], dB);
      qa[kk][3] = bf16x2_to_f16x2(qa[kk][3], dB);
    }
    sclA = scale_log2 * pow2f(eA);
    sclB = scale_log2 * pow2f(eB);
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  const int kb_key = lane & 7;                          // K (B operand) ldmatrix rows
  const int kb_d = (lane >> 3) * 8;
  const int vb_key = (lane & 7) + ((lane >> 3) & 1) * 8;  // V (B operand, .trans)
  const int vb_d = (lane >> 4) * 8;

  // A warp whose wait ran out keeps joining the consumers' named barriers (so
  // the others cannot block on it) but does no more work; the error is set.
  bool dead = false;
  for (int it = j0; it < ntiles; ++it) {
    const int st = (it - j0) % NS;
    if (!dead && !mbar_wait(full0 + 8 * st, ((it - j0) / NS) & 1)) {
      if (lane == 0) raise_error(a.err, PKV_ERR_TIMEOUT);
      dead = true;
    }
    uint32_t kst = smem_u32(smem + st * T::kStageBytes);
    const int tile0 = it * kTileKeys;
    const int lead = min(kTileKeys, b_lo * kBlock - tile0);      // keys not loaded (> 0 only at j0)
    const int tail = (it == ntiles - 1) ? pos_max + 1 - tile0 : kTileKeys;  // first unseen key
    if constexpr (FP8) {
      // Widen the codes into conv tile (it - j0) & 1, V rows outside
      // [lead, tail) as zeros; the code stage is free once every warp is done.
      // The other conv tile was last read in the previous iteration, which
      // every warp finished before the barrier below.
      uint8_t* conv = conv0 + ((it - j0) & 1) * T::kConvBytes;
      const uint8_t* codes = smem + st * T::kStageBytes;
      constexpr int per_row = D / 16;  // 16-code chunks per key row
      for (int e = threadIdx.x; !dead && e < kTileKeys * per_row; e += NWC * 32) {
        const int key = e / per_row;
        const int d0 = (e % per_row) * 16;
        const int bo = (key >> 4) * T::kBlkBytes;
        const uint32_t src = (key >> 4) * T::kLoadBlk + swz8<D>(key & 15, d0 / 16);
        widen16(conv + bo + swz_offset(key & 15, d0), conv + bo + swz_offset(key & 15, d0 + 8),
                codes + src, false);
        widen16(conv + T::kKBytes + bo + swz_offset(key & 15, d0),
                conv + T::kKBytes + bo + swz_offset(key & 15, d0 + 8),
                codes + T::kLoadK + src, key < lead || key >= tail);
      }
      named_barrier(1, NWC * 32);
      if (!dead && lane == 0) mbar_arrive(empty0 + 8 * st);
      kst = smem_u32(conv);
    } else if (lead > 0 || tail < kTileKeys) {
      // Keys before the first loaded block or past pos_max have P = 0 for
      // every row here, but their V rows may hold stale NaN (slots >= L) or
      // whatever an earlier tile left (blocks not loaded): zero them so that
      // 0 * NaN cannot reach the MMA.
      uint8_t* vrows = smem + st * T::kStageBytes + T::kKBytes;
      const int per_row = (D / 64) * 8;  // 16-byte chunks per key row
      const int nlead = lead > 0 ? lead : 0;
      const int ntail = kTileKeys - tail;
      for (int e = threadIdx.x; !dead && e < (nlead + ntail) * per_row; e += NWC * 32) {
        const int r = e / per_row;
        const int key = r < nlead ? r : tail + (r - nlead);
        const int rem = e % per_row;
        *reinterpret_cast<uint4*>(vrows + (key >> 4) * T::kBlkBytes + (rem >> 3) * 2048 +
                                  (key & 15) * 128 + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async();
      named_barrier(1, NWC * 32);
    }
    if (dead) continue;
    const uint32_t vst = kst + T::kKBytes;

    // ---- S = Q K^T  (16 rows x 64 keys per warp)
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kk2 = 0; kk2 < D / 32; ++kk2) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int key = nt * 8 + kb_key;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kst + (key >> 4) * T::kBlkBytes + swz_offset(key & 15, kk2 * 32 + kb_d), b0, b1,
                b2, b3);
        mma_16816<FP8>(sc[nt], qa[2 * kk2][0], qa[2 * kk2][1], qa[2 * kk2][2], qa[2 * kk2][3], b0,
                       b1);
        mma_16816<FP8>(sc[nt], qa[2 * kk2 + 1][0], qa[2 * kk2 + 1][1], qa[2 * kk2 + 1][2],
                       qa[2 * kk2 + 1][3], b2, b3);
      }
    }
    // ---- scale, causal mask, online softmax
    const bool need_mask = tile0 + kTileKeys - 1 > wpos_min || (W > 0 && tile0 <= wpos_max - W);
    float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int key = tile0 + nt * 8 + 2 * (lane & 3);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float xa = sc[nt][c] * sclA;
        float xb = sc[nt][2 + c] * sclB;
        if (need_mask) {
          xa = (key + c <= posA && key + c >= loA) ? xa : -INFINITY;
          xb = (key + c <= posB && key + c >= loB) ? xb : -INFINITY;
        }
        sc[nt][c] = xa;
        sc[nt][2 + c] = xb;
        mxA = fmaxf(mxA, xa);
        mxB = fmaxf(mxB, xb);
      }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, off));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, off));
    }
    const float mnA = fmaxf(mA, mxA), mnB = fmaxf(mB, mxB);
    const float muA = mnA == -INFINITY ? 0.f : mnA;
    const float muB = mnB == -INFINITY ? 0.f : mnB;
    const float alA = exp2f(mA - muA), alB = exp2f(mB - muB);
    mA = mnA;
    mB = mnB;
    uint32_t pa[4][4];
    float sA = 0.f, sB = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int nt = 2 * ks + h;
        const uint32_t pA = pack2<FP8>(exp2f(sc[nt][0] - muA), exp2f(sc[nt][1] - muA));
        const uint32_t pB = pack2<FP8>(exp2f(sc[nt][2] - muB), exp2f(sc[nt][3] - muB));
        pa[ks][2 * h] = pA;
        pa[ks][2 * h + 1] = pB;
        sA += lo2<FP8>(pA) + hi2<FP8>(pA);
        sB += lo2<FP8>(pB) + hi2<FP8>(pB);
      }
    }
    lA = lA * alA + sA;
    lB = lB * alB + sB;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o[nd][0] *= alA;
      o[nd][1] *= alA;
      o[nd][2] *= alB;
      o[nd][3] *= alB;
    }
    // ---- O += P V
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int key = ks * 16 + vb_key;
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vst + (key >> 4) * T::kBlkBytes + swz_offset(key & 15, dp * 16 + vb_d), b0,
                      b1, b2, b3);
        mma_16816<FP8>(o[2 * dp], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
        mma_16816<FP8>(o[2 * dp + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
      }
    }
    __syncwarp();
    if (!FP8 && lane == 0) mbar_arrive(empty0 + 8 * st);
  }

#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }
  const float iA = lA > 0.f ? out_scale / lA : 0.f;
  const float iB = lB > 0.f ? out_scale / lB : 0.f;
  __nv_bfloat16* oA = out + (static_cast<int64_t>(q0 + jA) * Hq + kvh * G + rA % G) * D;
  __nv_bfloat16* oB = out + (static_cast<int64_t>(q0 + jB) * Hq + kvh * G + rB % G) * D;
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) {
    const int d = nd * 8 + 2 * (lane & 3);
    if (vA)
      *reinterpret_cast<__nv_bfloat162*>(oA + d) =
          __floats2bfloat162_rn(o[nd][0] * iA, o[nd][1] * iA);
    if (vB)
      *reinterpret_cast<__nv_bfloat162*>(oB + d) =
          __floats2bfloat162_rn(o[nd][2] * iB, o[nd][3] * iB);
  }
}

template <int D, int NS, bool FP8>
cudaError_t launch_prefill_t(const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const PrefillArgs& a, cudaStream_t stream) {
  constexpr int smem = prefill_smem_bytes<D, NS, FP8>();
  auto kfn = pkv_prefill_bf16_kernel<D, NS, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_mtiles, a.num_kv_heads, a.num_seqs);
  kfn<<<grid, (kConsumerWarps + 1) * 32, smem, stream>>>(kmap, vmap, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                const PrefillArgs& a, int head_size, bool fp8,
                                cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_mtiles == 0) return cudaSuccess;
  if (fp8) {  // code stages are released right after widening: a short ring suffices
    if (head_size == 128) return launch_prefill_t<128, 2, true>(kmap, vmap, a, stream);
    return launch_prefill_t<64, 4, true>(kmap, vmap, a, stream);
  }
  if (head_size == 128) return launch_prefill_t<128, 3, false>(kmap, vmap, a, stream);
  return launch_prefill_t<64, 4, false>(kmap, vmap, a, stream);
}

}  // namespace pkv
