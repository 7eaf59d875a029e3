// pkv_prefill_tc.cu -- paged varlen causal attention for chunked prefill on
// the 5th-generation tensor cores (tcgen05 + TMEM), bf16 in, fp32 accumulate.
//
// What it computes is the chunked-prefill definition of "Implémentation du
// cœur du moteur d'inférence haute performance vLLM", ch. 6 "Branche de
// masque": query j of a chunk of q_s new tokens of a sequence with L keys
// sits at absolute position L - q_s + j and attends keys 0 .. L - q_s + j,
// each read through the block table (ch. 6 "Flux des paramètres du chemin
// non-cascadé").  GQA: the G query heads of a kv head share every K/V tile.
//
// GB300 design (the dense contraction of the path):
//  * CTA = two 128-row query tiles x one kv head of one sequence (one CTA per
//    SM); a row is a (token, q head) pair with the head fastest, so each tile
//    holds 128/G tokens x G heads and is one TMA load per 64-column half
//    (box 64 x G heads x 128/G tokens, 128-byte swizzle), which lands exactly
//    in the K-major UMMA layout.
//  * warp 0 streams 64-key K/V tiles (4 cache blocks, one TMA box per block
//    and half) into a 4-stage ring shared by both query tiles; warp 1
//    allocates all 512 TMEM columns and one of its threads issues every MMA:
//        S_t  = Q_t K^T   (M=128, N=64, K=16 x D/16, operands from smem)
//        O_t += P_t V     (M=128, N=D,  K=16 x 4, P_t from TMEM, V MN-major)
//    for the two tiles t in turn, so the tensor core works on one tile while
//    the softmax of the other runs, and S_t of the next K/V tile is computed
//    as soon as the softmax has read the current one.
//  * warps 2-5 and 6-9 (one warpgroup per query tile) own one TMEM lane
//    (= one row) per thread: they load a row of S, apply the causal mask, keep
//    a lazily updated running max (O is rescaled in TMEM only when the max
//    grows by more than 2^8), write P (bf16) to TMEM for the second MMA, and at
//    the end read O, divide by the row sum and store bf16.  No shuffles: a
//    thread holds its whole row.
//  * every wait is an mbarrier with a bounded spin and a CTA-wide abort flag;
//    TMEM is freed on every path.
#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {

namespace {

constexpr int kTcRows = 128;      // UMMA M (rows of one query tile)
constexpr int kTcTiles = 2;       // query tiles per CTA
constexpr int kTcKeys = 64;       // keys per K/V tile
constexpr int kTcThreads = 320;   // load, MMA, 2 x 4 softmax warps
constexpr int kTcStages = 4;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S of tile t at 64t, P of tile t at 128 + 32t, O of tile t at 256 + 128t.
__host__ __device__ constexpr uint32_t col_s(int t) { return 64u * t; }
__host__ __device__ constexpr uint32_t col_p(int t) { return 128u + 32u * t; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
constexpr float kLazyRescale = 8.0f;  // log2 units: rescale O only past 2^8 growth

template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kTcRows * 128;       // 16 KB: 128 rows x 128 B
  static constexpr int kQTile = kHalves * kQHalf;
  static constexpr int kKvHalf = kTcKeys * 128;      // 8 KB: 64 keys x 128 B
  static constexpr int kKBytes = kHalves * kKvHalf;
  static constexpr int kStageBytes = 2 * kKBytes;    // K then V
};

struct TcShared {
  uint64_t q_full, drain;
  uint64_t s_full[kTcTiles], s_free[kTcTiles], p_full[kTcTiles], pv_done[kTcTiles];
  uint64_t kv_full[kTcStages], kv_empty[kTcStages];
  uint32_t tmem_base;
  int32_t abort;
};

template <int D>
constexpr int tc_smem_bytes() {
  // Whole-SM footprint: one CTA per SM (it owns all 512 TMEM columns).
  constexpr int need = 1024 + kTcTiles * TcLayout<D>::kQTile +
                       kTcStages * TcLayout<D>::kStageBytes + static_cast<int>(sizeof(TcShared));
  return need > 120 * 1024 ? need : 120 * 1024;
}

// Bounded wait that also gives up when another thread of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int32_t* abort, int32_t* err) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_test(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      raise_error(err, PKV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform version: lane 0 waits, the verdict is broadcast, and the other
// lanes then observe the (already completed) phase themselves.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                          int32_t* err) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  if (lane == 0) ok = wait_or_abort(bar, parity, abort, err);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok && lane != 0) ok = wait_or_abort(bar, parity, abort, err);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    pkv_prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using Lt = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                                   // [tile][half][128 rows x 128 B]
  uint8_t* sKV = smem + kTcTiles * Lt::kQTile;          // [stage][K halves | V halves]
  TcShared* sh = reinterpret_cast<TcShared*>(sKV + kTcStages * Lt::kStageBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int s = a.seq_begin + blockIdx.z;
  const int kvh = blockIdx.y;
  const int mtile = a.num_mtiles - 1 - blockIdx.x;  // heaviest first
  const int G = a.group;
  const int Hq = a.num_q_heads;
  const int tile_toks = kTcRows / G;                // tokens per query tile
  const int toks = kTcTiles * tile_toks;            // tokens per CTA

  const int L = __ldg(a.context_lens + s);
  const int q0 = __ldg(a.query_start_loc + s);
  const int qn = __ldg(a.query_start_loc + s + 1) - q0;
  const int tok0 = mtile * toks;
  const bool bad_rows = qn < 0 || q0 < 0 || static_cast<int64_t>(q0) + qn > a.num_tokens;
  if (bad_rows || qn == 0 || tok0 >= qn) {
    if (bad_rows && blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0)
      raise_error(a.err, PKV_ERR_QUERY_LEN);
    return;
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  const bool bad_len = (L < 1 || static_cast<int64_t>(L) > a.bt_stride * kBlock);
  if (bad_len || qn > L || qn > a.max_query_len) {
    if (threadIdx.x == 0 && mtile == 0 && kvh == 0)
      raise_error(a.err, bad_len ? PKV_ERR_CONTEXT_LEN : PKV_ERR_QUERY_LEN);
    const int nt = min(toks, qn - tok0);
    for (int i = threadIdx.x; i < nt * G * D; i += blockDim.x) {
      const int r = i / D;
      out[(static_cast<int64_t>(q0 + tok0 + r / G) * Hq + kvh * G + r % G) * D + i % D] =
          __float2bfloat16(0.f);
    }
    return;
  }
  const int tok_last = min(tok0 + toks, qn) - 1;
  const int ntq = (tok0 + tile_toks < qn) ? 2 : 1;  // query tiles holding a valid row
  const int pos_max = L - qn + tok_last;            // last key any row here can see
  const int ntiles = (pos_max + kTcKeys) / kTcKeys;
  const int nblk = (pos_max + kBlock) / kBlock;

  const uint32_t q_full = smem_u32(&sh->q_full), drain = smem_u32(&sh->drain);
  if (threadIdx.x == 0) {
    prefetch_tensor_map(&qmap);
    prefetch_tensor_map(&kmap);
    prefetch_tensor_map(&vmap);
    mbar_init(q_full, 1);
    mbar_init(drain, 1);
    for (int t = 0; t < kTcTiles; ++t) {
      mbar_init(smem_u32(&sh->s_full[t]), 1);
      mbar_init(smem_u32(&sh->s_free[t]), 4);
      mbar_init(smem_u32(&sh->p_full[t]), 4);
      mbar_init(smem_u32(&sh->pv_done[t]), 1);
    }
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(smem_u32(&sh->kv_full[i]), 1);
      mbar_init(smem_u32(&sh->kv_empty[i]), 1);
    }
    sh->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tc::alloc(smem_u32(&sh->tmem_base), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int32_t* abort = &sh->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t keep = policy_evict_normal();   // K/V tiles are re-read by the
    const int32_t* bt = a.block_tables + static_cast<int64_t>(s) * a.bt_stride;  // other row tiles
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, ntq * Lt::kQTile);
      for (int t = 0; t < ntq; ++t)
#pragma unroll
        for (int h = 0; h < Lt::kHalves; ++h)
          tma_load_3d(smem_u32(sQ + t * Lt::kQTile + h * Lt::kQHalf), &qmap, q_full, h * 64,
                      kvh * G, q0 + tok0 + t * tile_toks, keep);
    }
    int my_bid = -1;
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % kTcStages;
      if (it >= kTcStages &&
          !warp_wait(smem_u32(&sh->kv_empty[st]), ((it / kTcStages) - 1) & 1, abort, a.err))
        break;
      if ((it & 7) == 0) {  // block ids of the next 8 tiles, one per lane
        const int b = it * 4 + lane;
        my_bid = b < nblk ? __ldg(bt + b) : -1;
      }
      bool ok[4];
      int bid[4];
      uint32_t bytes = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        bid[b] = __shfl_sync(0xffffffffu, my_bid, (it & 7) * 4 + b);
        const bool in_range = it * 4 + b < nblk;
        ok[b] = in_range && bid[b] >= 0 && bid[b] < a.num_blocks;
        if (in_range && !ok[b] && lane == 0) raise_error(a.err, PKV_ERR_BLOCK_ID);
        bytes += ok[b] ? 2u * Lt::kHalves * 2048u : 0u;
      }
      if (lane == 0) {
        const uint32_t full = smem_u32(&sh->kv_full[st]);
        const uint32_t dst = smem_u32(sKV + st * Lt::kStageBytes);
        if (bytes == 0) {
          mbar_arrive(full);
        } else {
          mbar_arrive_expect_tx(full, bytes);
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            if (!ok[b]) continue;
#pragma unroll
            for (int h = 0; h < Lt::kHalves; ++h) {
              tma_load_3d(dst + h * Lt::kKvHalf + b * 2048, &kmap, full, h * 64, kvh,
                          bid[b] * kBlock, keep);
              tma_load_3d(dst + Lt::kKBytes + h * Lt::kKvHalf + b * 2048, &vmap, full, h * 64,
                          kvh, bid[b] * kBlock, keep);
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kTcRows, kTcKeys, 0, 0);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kTcRows, D, 0, 1);
      auto issue_s = [&](int t, int j) {
        const uint32_t q_addr = smem_u32(sQ + t * Lt::kQTile);
        const uint32_t k_addr = smem_u32(sKV + (j % kTcStages) * Lt::kStageBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;  // 16 bf16 = 32 B along the swizzled row
          const uint64_t da =
              tc::smem_desc_sw128(q_addr + (kk >> 2) * Lt::kQHalf + off, 16, 1024);
          const uint64_t db =
              tc::smem_desc_sw128(k_addr + (kk >> 2) * Lt::kKvHalf + off, 16, 1024);
          tc::mma_ss(tmem + col_s(t), da, db, idS, kk > 0 ? 1u : 0u);
        }
        tc::commit(smem_u32(&sh->s_full[t]));
      };
      auto issue_pv = [&](int t, int j) {
        const uint32_t v_addr =
            smem_u32(sKV + (j % kTcStages) * Lt::kStageBytes + Lt::kKBytes);
#pragma unroll
        for (int ks = 0; ks < kTcKeys / 16; ++ks) {
          const uint64_t dv = tc::smem_desc_sw128(v_addr + ks * 2048, Lt::kKvHalf, 1024);
          tc::mma_ts(tmem + col_o(t), tmem + col_p(t) + ks * 8, dv, idO,
                     (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::commit(smem_u32(&sh->pv_done[t]));
      };
      // Event loop: issue whichever MMA is ready, never blocking on one
      // tile while the other could use the tensor core.  Phases cannot run
      // more than one ahead of what this thread has seen, so parity probes
      // are unambiguous.
      int s_next[kTcTiles] = {0, 0};   // next tile index whose S is issued
      int pv_next[kTcTiles] = {0, 0};  // next tile index whose P V is issued
      int released = 0;                // K/V stages handed back to the producer
      bool ok = wait_or_abort(q_full, 0, abort, a.err);
      uint64_t idle_since = 0;
      while (ok) {
        bool progress = false;
        for (int t = 0; t < ntq; ++t) {
          const int js = s_next[t];
          if (js < ntiles &&
              mbar_test(smem_u32(&sh->kv_full[js % kTcStages]), (js / kTcStages) & 1) &&
              (js == 0 || mbar_test(smem_u32(&sh->s_free[t]), (js - 1) & 1))) {
            tc::fence_after_sync();
            issue_s(t, js);
            s_next[t] = js + 1;
            progress = true;
          }
          const int jp = pv_next[t];
          if (jp < s_next[t] && mbar_test(smem_u32(&sh->p_full[t]), jp & 1)) {
            tc::fence_after_sync();
            issue_pv(t, jp);
            pv_next[t] = jp + 1;
            progress = true;
          }
        }
        int done_pv = pv_next[0];
        if (ntq > 1) done_pv = min(done_pv, pv_next[1]);
        while (released < done_pv) {  // every P V of that stage is issued
          tc::commit(smem_u32(&sh->kv_empty[released % kTcStages]));
          ++released;
        }
        if (done_pv == ntiles) break;
        if (progress) {
          idle_since = 0;
        } else {
          const uint64_t now = global_timer_ns();
          if (idle_since == 0) {
            idle_since = now;
          } else if (*abort) {
            ok = false;
          } else if (now - idle_since > kWaitLimitNs) {
            *abort = 1;
            raise_error(a.err, PKV_ERR_TIMEOUT);
            ok = false;
          }
        }
      }
      // Every MMA issued here must finish before TMEM is released.
      tc::commit(drain);
      (void)mbar_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) >> 2;                // query tile of this warpgroup
    const int quarter = warp & 3;                 // TMEM lanes this warp may touch
    const int row = quarter * 32 + lane;          // tile row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int tok = tok0 + t * tile_toks + row / G;
    const int g = row % G;
    const bool valid = tok <= tok_last;
    const int pos = L - qn + (valid ? tok : tok_last);
    const int ts = ((warp - 2) & 3) * 32 + lane;  // 0..127 within the warpgroup
    const uint32_t b_sfull = smem_u32(&sh->s_full[t]), b_sfree = smem_u32(&sh->s_free[t]);
    const uint32_t b_pfull = smem_u32(&sh->p_full[t]), b_pvdone = smem_u32(&sh->pv_done[t]);
    const uint32_t tS = tmem + lane_off + col_s(t), tP = tmem + lane_off + col_p(t);
    const uint32_t tO = tmem + lane_off + col_o(t);
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool done = t < ntq;
    for (int j = 0; done && j < ntiles; ++j) {
      if (!warp_wait(b_sfull, j & 1, abort, a.err)) { done = false; break; }
      tc::fence_after_sync();
      uint32_t sr[2][32];
      tc::ld32(tS, sr[0]);
      tc::ld32(tS + 32, sr[1]);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sfree);
      // causal mask on raw scores (also hides keys >= L); scale > 0, so the
      // row max of the raw scores gives the max of the scaled ones
      const int key0 = j * kTcKeys;
      float x[kTcKeys];
#pragma unroll
      for (int c = 0; c < kTcKeys; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
      if (key0 + kTcKeys - 1 > pos) {
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) x[c] = (key0 + c > pos) ? -INFINITY : x[c];
      }
      // row max: four independent chains of three-input maxima
      float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int c = 4; c < kTcKeys; c += 8) {
        m4[0] = tc::max3(m4[0], x[c], x[c + 1]);
        m4[1] = tc::max3(m4[1], x[c + 2], x[c + 3]);
        m4[2] = tc::max3(m4[2], x[c + 4], x[c + 5]);
        m4[3] = tc::max3(m4[3], x[c + 6], x[c + 7]);
      }
      const float mt = tc::max3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;
      float alpha = 1.f;
      if (mt > m_used + kLazyRescale) {
        alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - mt);
        m_used = mt;
      }
      const float neg_mu = (m_used == -INFINITY) ? 0.f : -m_used;
      const uint64_t m2 = tc::pack_f32x2(sl2, sl2), b2 = tc::pack_f32x2(neg_mu, neg_mu);
      // P = 2^(s * scale*log2(e) - max): packed FMA, MUFU ex2, bf16 pairs; the
      // row sum adds the fp32 weights in four packed accumulators
      uint32_t pk[32];
      uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float y0, y1;
        tc::fma_f32x2(x[2 * c], x[2 * c + 1], m2, b2, y0, y1);
        y0 = ex2(y0);
        y1 = ex2(y1);
        pk[c] = pack_bf16(y0, y1);
        tc::add_f32x2(acc[c & 3], y0, y1);
      }
      const float ls = (tc::sum_f32x2(acc[0]) + tc::sum_f32x2(acc[1])) +
                       (tc::sum_f32x2(acc[2]) + tc::sum_f32x2(acc[3]));
      l = l * alpha + ls;
      if (j > 0) {
        if (!warp_wait(b_pvdone, (j - 1) & 1, abort, a.err)) { done = false; break; }
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {   // rescale O in TMEM
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc::ld32(tO + c0, o);
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tc::st32(tO + c0, o);
          }
          tc::wait_st();
        }
      }
      if (j == ntiles - 1 && key0 + kTcKeys > pos_max + 1) {
        // Keys past pos_max have P = 0 in every row, but their V rows may be
        // stale NaN or left over from an earlier tile: zero them before this
        // warpgroup's P V product may be issued.  Both warpgroups do it (the
        // MMAs of the two query tiles are issued in either order); the
        // second writes zeros over zeros.
        if (!warp_wait(smem_u32(&sh->kv_full[j % kTcStages]), (j / kTcStages) & 1, abort,
                       a.err)) { done = false; break; }
        uint8_t* vt = sKV + (j % kTcStages) * Lt::kStageBytes + Lt::kKBytes;
        const int first = pos_max + 1 - key0;
        const int per_row = Lt::kHalves * 8;
        for (int e = ts; e < (kTcKeys - first) * per_row; e += 128) {
          const int key = first + e / per_row;
          const int rem = e % per_row;
          *reinterpret_cast<uint4*>(vt + (rem >> 3) * Lt::kKvHalf + key * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async();
      }
      tc::st32(tP, pk);
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull);
    }
    if (done && warp_wait(b_pvdone, (ntiles - 1) & 1, abort, a.err)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = out + (static_cast<int64_t>(q0 + tok) * Hq + kvh * G + g) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tc::ld32(tO + c0, o);
        tc::wait_ld();
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            w[c] = pack_bf16(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_tc_t(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        const PrefillArgs& a, cudaStream_t stream) {
  constexpr int smem = tc_smem_bytes<D>();
  auto kfn = pkv_prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_mtiles, a.num_kv_heads, a.num_seqs);
  kfn<<<grid, kTcThreads, smem, stream>>>(qmap, kmap, vmap, a);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(int head_size, int group) {
  return (head_size == 64 || head_size == 128) && group >= 1 && group <= kTcRows &&
         kTcRows % group == 0;
}

int prefill_tc_tokens_per_tile(int group) { return kTcRows / group; }
int prefill_tc_tokens_per_cta(int group) { return kTcTiles * kTcRows / group; }

cudaError_t launch_prefill_tc(const CUtensorMap& qmap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const PrefillArgs& a, int head_size,
                              cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_mtiles == 0) return cudaSuccess;
  if (head_size == 128) return launch_tc_t<128>(qmap, kmap, vmap, a, stream);
  return launch_tc_t<64>(qmap, kmap, vmap, a, stream);
}

}  // namespace pkv
