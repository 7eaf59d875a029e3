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
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kTileKeys = 64;  // 4 cache blocks per stage

template <int D>
struct PrefillTile {
  static constexpr int kBlkBytes = D * 2 * kBlock;            // one block of K (or V)
  static constexpr int kKBytes = kBlkBytes * (kTileKeys / kBlock);
  static constexpr int kStageBytes = 2 * kKBytes;
};

template <int D, int NS>
constexpr int prefill_smem_bytes() {
  return 1024 + NS * PrefillTile<D>::kStageBytes + 2 * NS * 8;
}

template <int D, int NS>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32)
    pkv_prefill_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using T = PrefillTile<D>;
  constexpr int NWC = kConsumerWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * T::kStageBytes);
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
        bytes += ok[b] ? 2u * T::kBlkBytes : 0u;
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

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  const int kb_key = lane & 7;                          // K (B operand) ldmatrix rows
  const int kb_d = (lane >> 3) * 8;
  const int vb_key = (lane & 7) + ((lane >> 3) & 1) * 8;  // V (B operand, .trans)
  const int vb_d = (lane >> 4) * 8;

  for (int it = j0; it < ntiles; ++it) {
    const int st = (it - j0) % NS;
    if (!mbar_wait(full0 + 8 * st, ((it - j0) / NS) & 1)) {
      if (lane == 0) raise_error(a.err, PKV_ERR_TIMEOUT);
      break;
    }
    const uint32_t kst = smem_u32(smem + st * T::kStageBytes);
    const uint32_t vst = kst + T::kKBytes;
    const int tile0 = it * kTileKeys;
    const int lead = min(kTileKeys, b_lo * kBlock - tile0);      // keys not loaded (> 0 only at j0)
    const int tail = (it == ntiles - 1) ? pos_max + 1 - tile0 : kTileKeys;  // first unseen key
    if (lead > 0 || tail < kTileKeys) {
      // Keys before the first loaded block or past pos_max have P = 0 for
      // every row here, but their V rows may hold stale NaN (slots >= L) or
      // whatever an earlier tile left (blocks not loaded): zero them so that
      // 0 * NaN cannot reach the MMA.
      uint8_t* vrows = smem + st * T::kStageBytes + T::kKBytes;
      const int per_row = (D / 64) * 8;  // 16-byte chunks per key row
      const int nlead = lead > 0 ? lead : 0;
      const int ntail = kTileKeys - tail;
      for (int e = threadIdx.x; e < (nlead + ntail) * per_row; e += NWC * 32) {
        const int r = e / per_row;
        const int key = r < nlead ? r : tail + (r - nlead);
        const int rem = e % per_row;
        *reinterpret_cast<uint4*>(vrows + (key >> 4) * T::kBlkBytes + (rem >> 3) * 2048 +
                                  (key & 15) * 128 + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async();
      named_barrier(1, NWC * 32);
    }

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
        mma_bf16_16816(sc[nt], qa[2 * kk2][0], qa[2 * kk2][1], qa[2 * kk2][2], qa[2 * kk2][3], b0,
                       b1);
        mma_bf16_16816(sc[nt], qa[2 * kk2 + 1][0], qa[2 * kk2 + 1][1], qa[2 * kk2 + 1][2],
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
        float xa = sc[nt][c] * a.scale_log2;
        float xb = sc[nt][2 + c] * a.scale_log2;
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
        const uint32_t pA = pack_bf16(exp2f(sc[nt][0] - muA), exp2f(sc[nt][1] - muA));
        const uint32_t pB = pack_bf16(exp2f(sc[nt][2] - muB), exp2f(sc[nt][3] - muB));
        pa[ks][2 * h] = pA;
        pa[ks][2 * h + 1] = pB;
        sA += bf16_lo(pA) + bf16_hi(pA);
        sB += bf16_lo(pB) + bf16_hi(pB);
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
        mma_bf16_16816(o[2 * dp], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
  }

#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }
  const float iA = lA > 0.f ? 1.f / lA : 0.f;
  const float iB = lB > 0.f ? 1.f / lB : 0.f;
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

template <int D, int NS>
cudaError_t launch_prefill_t(const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const PrefillArgs& a, cudaStream_t stream) {
  constexpr int smem = prefill_smem_bytes<D, NS>();
  auto kfn = pkv_prefill_bf16_kernel<D, NS>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_mtiles, a.num_kv_heads, a.num_seqs);
  kfn<<<grid, (kConsumerWarps + 1) * 32, smem, stream>>>(kmap, vmap, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                const PrefillArgs& a, int head_size, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_mtiles == 0) return cudaSuccess;
  if (head_size == 128) return launch_prefill_t<128, 3>(kmap, vmap, a, stream);
  return launch_prefill_t<64, 4>(kmap, vmap, a, stream);
}

}  // namespace pkv
