// pkv_decode.cu -- paged decode attention (one query row per sequence), bf16,
// with split-K over the context and the log-sum-exp combine.
//
// What it computes: for each decode sequence s (context length L), kv head h
// and the G query heads of h (GQA, contiguous groups), the exact softmax
// attention of the query over keys 0..L-1, each fetched from block
// block_tables[s][p / 16] at offset p % 16 -- "Implémentation du cœur du
// moteur d'inférence haute performance vLLM", ch. 6 "Flux des paramètres du
// chemin non-cascadé" (seqused_k = seq_lens, block_table) and "Transformation
// de la disposition mémoire du KV cache" ([num_blocks, 16, Hkv, D] layout).
// Long contexts are split into chunks whose fp32 partial outputs and
// log-sum-exps go to a caller-provided buffer (ch. 6 "build() étape par
// étape", fourth step) and are merged by a second kernel (merge_attn_states in
// the ch. 6 sequence diagram).
//
// GB300 design (HBM-bound: every K/V byte is read once):
//  * grid = (split, kv head x 8-head group, sequence); 4 warps per CTA, each
//    warp owns every 4th cache block of the split and runs its own NS-deep
//    TMA ring: one 16-key block of K and of V (2 x 16 x D bf16) per stage,
//    loaded as 64-column boxes with the 128-byte swizzle (conflict-free
//    ldmatrix), completion on a per-stage mbarrier, evict-first L2 policy.
//  * keys sit on the MMA's M dimension and the query heads of the group on N:
//    S^T[16 keys x 8 heads] = K_blk . Q^T (m16n8k16, Q^T held in registers),
//    so one tile serves all G <= 8 heads and no head padding to 16 is needed.
//    The probabilities are rounded to bf16, transposed in registers
//    (movmatrix) into the B operand of O^T[D x 8] += V_blk^T . P^T
//    (ldmatrix.trans of the same swizzled V tile).  Online softmax in the
//    log2 domain; the denominator sums the same rounded weights the MMA uses.
//  * warps merge through shared memory; a CTA whose sequence needs one split
//    writes bf16 output, otherwise an fp32 partial + log-sum-exp.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kDecodeWarps = 4;

template <int D, bool FP8>
struct DecodeTile {
  static constexpr int kHalves = D / 64;             // 64-column TMA boxes per row
  static constexpr int kTileBytes = D * 2 * kBlock;  // one 16-key block of K (or V), bf16
  // what TMA lands per block: bf16 tiles, or e4m3 codes (D bytes per row)
  static constexpr int kLoadBytes = FP8 ? D * kBlock : kTileBytes;
  static constexpr int kStageBytes = 2 * kLoadBytes;
};

template <int D, int NS, bool FP8>
constexpr int decode_smem_bytes() {
  using T = DecodeTile<D, FP8>;
  return 1024 /* alignment slack */ + kDecodeWarps * NS * T::kStageBytes +
         kDecodeWarps * NS * 8 /* mbarriers */ + 2 * kDecodeWarps * 8 * 4 /* merge factors */;
}


// PREFIX: the cascade prefix launch.  The MMA's 8 columns are then (sequence,
// q head) pairs of every sequence of the batch (column gc of kv head kvh is
// sequence gc / G, q head kvh * G + gc % G), all reading the shared prefix
// keys [0, prefix_len) through sequence 0's block table; every column writes
// a partial.  Otherwise the columns are q heads of one sequence's query row.
template <int D, int NS, bool FP8, bool PREFIX>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    pkv_decode_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using T = DecodeTile<D, FP8>;
  constexpr int NW = kDecodeWarps;
  // Every CTA of this grid is resident once it runs this: the combine launch
  // that follows (programmatic, see launch_combine_bf16) may be scheduled
  // beside the grid's last CTAs; it waits for the grid's completion itself.
  asm volatile("griddepcontrol.launch_dependents;");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * NS * T::kStageBytes);
  float* merge_f = reinterpret_cast<float*>(bars + NW * NS);  // [NW][8] factors, [8] lse
  // Merge area of warp w ([8 heads][D] + m[8] + l[8] floats): the start of its
  // stage ring, free once its loads are consumed.
  static_assert(NS * T::kStageBytes >= (8 * D + 16) * 4, "merge area exceeds the ring");
  static_assert(T::kHalves >= 1, "head_size 64 or 128");
  auto merge_area = [&](int w) {
    return reinterpret_cast<float*>(smem + w * NS * T::kStageBytes);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int s = PREFIX ? 0 : blockIdx.z;  // block-table row (and sequence)
  const int ngsub = PREFIX ? a.prefix_col_groups : (a.group + 7) >> 3;
  const int kvh = blockIdx.y / ngsub;
  const int gsub = blockIdx.y - kvh * ngsub;
  const int G = a.group;
  const int Hq = a.num_q_heads;
  const bool reporter = (split == 0 && blockIdx.y == 0 && threadIdx.x == 0);

  int L, q0 = 0;
  if constexpr (PREFIX) {
    L = a.prefix_len;
  } else {
    L = __ldg(a.context_lens + s);
    q0 = __ldg(a.query_start_loc + s);
    const int qn = __ldg(a.query_start_loc + s + 1) - q0;
    // (cascade: the shared-prefix launch takes sequence t's query at row t)
    if (qn != 1 || q0 < 0 || q0 >= a.num_tokens || (a.key_begin_blocks > 0 && q0 != s)) {
      if (qn != 0 && reporter)
        raise_error(a.err, qn == 1 ? PKV_ERR_QUERY_LEN : PKV_ERR_DECODE_QLEN);
      return;
    }
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  // (cascade suffix: the query must sit after the shared prefix)
  if (L < 1 || static_cast<int64_t>(L) > a.bt_stride * kBlock || L > a.max_context_len ||
      (!PREFIX && L <= a.key_begin_blocks * kBlock)) {
    if (reporter) raise_error(a.err, PKV_ERR_CONTEXT_LEN);
    if (PREFIX) return;
    if (split == 0) {  // zero rows for a sequence with bad metadata
      for (int i = threadIdx.x; i < 8 * D; i += NW * 32) {
        const int g = gsub * 8 + i / D;
        if (g < G) out[(static_cast<int64_t>(q0) * Hq + kvh * G + g) * D + (i % D)] =
            __float2bfloat16(0.f);
      }
    }
    return;
  }
  // Keys the query sees: [kfirst, L) (the sliding window, if any; a cascade
  // suffix launch starts after the shared prefix); the splits cover the blocks
  // of that range only.
  const int kfirst = max((a.window > 0 && L > a.window) ? L - a.window : 0,
                         a.key_begin_blocks * kBlock);
  const int blk0 = kfirst / kBlock;
  const int nblk_seq = (L + kBlock - 1) / kBlock - blk0;
  const int nsplit = (nblk_seq + a.split_blocks - 1) / a.split_blocks;
  if (split >= nsplit) return;
  const int b_begin = blk0 + split * a.split_blocks;
  const int b_end = min(b_begin + a.split_blocks, blk0 + nblk_seq);
  const int nblk = b_end - b_begin;
  const int nb_w = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;  // <= 32 by construction

  if (threadIdx.x == 0) {
    prefetch_tensor_map(&kmap);
    prefetch_tensor_map(&vmap);
  }

  // Block ids of this warp's blocks: lane i holds its i-th block.
  int my_bid = -1;
  if (lane < nb_w)
    my_bid = __ldg(a.block_tables + static_cast<int64_t>(s) * a.bt_stride + b_begin + warp +
                   NW * lane);
  const bool my_ok = (my_bid >= 0 && my_bid < a.num_blocks);
  if (lane < nb_w && !my_ok) raise_error(a.err, PKV_ERR_BLOCK_ID);

  uint8_t* wbase = smem + warp * NS * T::kStageBytes;
  const uint32_t wbase_u = smem_u32(wbase);
  const uint32_t bar0 = smem_u32(bars + warp * NS);
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < NS; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
  }
  __syncwarp();

  const uint64_t policy = policy_evict_first();
  // Issues this warp's block i into stage i % NS (all lanes call; lane 0 acts).
  // Test hook: warp 0 withholds its first block (no copy, no arrival), so
  // that its wait for it runs out.
  const bool withheld = a.debug_stall != 0 && warp == 0;
  auto issue = [&](int i) {
    const int bid = __shfl_sync(0xffffffffu, my_bid, i);
    const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, i) != 0;
    if (lane == 0 && !(withheld && i == 0)) {
      const int st = i % NS;
      const uint32_t dst = wbase_u + st * T::kStageBytes;
      const uint32_t bar = bar0 + 8 * st;
      if (ok) {
        mbar_arrive_expect_tx(bar, T::kStageBytes);
        if constexpr (FP8) {  // one box of 16 rows x D codes per block
          tma_load_3d(dst, &kmap, bar, 0, kvh, bid * kBlock, policy);
          tma_load_3d(dst + T::kLoadBytes, &vmap, bar, 0, kvh, bid * kBlock, policy);
        } else {
#pragma unroll
          for (int h = 0; h < T::kHalves; ++h) {
            tma_load_3d(dst + h * 2048, &kmap, bar, h * 64, kvh, bid * kBlock, policy);
            tma_load_3d(dst + T::kTileBytes + h * 2048, &vmap, bar, h * 64, kvh, bid * kBlock,
                        policy);
          }
        }
      } else {
        mbar_arrive(bar);  // nothing to load: complete the phase empty
      }
    }
  };

  const int n_pro = nb_w < NS ? nb_w : NS;
  for (int i = 0; i < n_pro; ++i) issue(i);
  int issued = n_pro;  // blocks whose copies have been started

  // Q^T as the B operand: lane holds Q[g = lane/4][kk*16 + 2*(lane%4) + {0,1}]
  // (qb[kk][0]) and the same +8 (qb[kk][1]); heads past the group are zero.
  // FP8: the contraction runs over a permutation of d instead (any order
  // gives the same dot products), chosen so that a lane's K codes are
  // contiguous: step kk, k-slots {2t, 2t+1, 2t+8, 2t+9} (t = lane % 4) are
  // d = (D/4) t + 4 kk + {0, 1, 2, 3}.
  uint32_t qb[D / 16][2];
  {
    int g = gsub * 8 + (lane >> 2);
    bool gv = g < G;
    int qr = q0;
    if constexpr (PREFIX) {  // column -> (sequence, head in group); its query row
      const int sc = g / G;
      g -= sc * G;
      qr = sc < a.num_seqs ? __ldg(a.query_start_loc + sc) : -1;
      gv = qr >= 0 && qr < a.num_tokens;
    }
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const __nv_bfloat16*>(a.q) +
        (static_cast<int64_t>(gv ? qr : 0) * Hq + kvh * G + (gv ? g : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      if constexpr (FP8) {
        qb[kk][0] = gv ? __ldg(qrow + (D / 8) * (lane & 3) + 2 * kk) : 0u;
        qb[kk][1] = gv ? __ldg(qrow + (D / 8) * (lane & 3) + 2 * kk + 1) : 0u;
      } else {
        qb[kk][0] = gv ? __ldg(qrow + kk * 8 + (lane & 3)) : 0u;
        qb[kk][1] = gv ? __ldg(qrow + kk * 8 + 4 + (lane & 3)) : 0u;
      }
    }
  }

  // FP8: the MMAs run on fp16 operands.  K = code * k_descale folds into the
  // score scale, V = code * v_descale into the output; Q goes to fp16, a head
  // whose values exceed 2^14 scaled down by 2^e first and its scores up by 2^e.
  float scale_log2 = a.scale_log2, out_scale = 1.f;
  float col_scale[2] = {scale_log2, scale_log2};  // score scale of head columns c0, c0 + 1
  if constexpr (FP8) {
    scale_log2 *= __ldg(a.k_descale + static_cast<int64_t>(s) * a.num_kv_heads + kvh);
    out_scale = __ldg(a.v_descale + static_cast<int64_t>(s) * a.num_kv_heads + kvh);
    float amax = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int j = 0; j < 2; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(qb[kk][j])), fabsf(bf16_hi(qb[kk][j]))));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the 4 lanes of head lane/4
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int e = f16_row_exponent(amax);
    const float down = pow2f(-e);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
      for (int j = 0; j < 2; ++j) qb[kk][j] = bf16x2_to_f16x2(qb[kk][j], down);
    const int c0 = 2 * (lane & 3);
    col_scale[0] = scale_log2 * pow2f(__shfl_sync(0xffffffffu, e, 4 * c0));
    col_scale[1] = scale_log2 * pow2f(__shfl_sync(0xffffffffu, e, 4 * c0 + 4));
  }

  float o[D / 16][4];
#pragma unroll
  for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY};
  float l[2] = {0.f, 0.f};

  // Per-lane ldmatrix row/column pieces.
  const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8;   // QK: A = K (keys x d)
  const int k_dsub = (lane >> 4) * 8;
  const int v_row = (lane & 7) + ((lane >> 4) & 1) * 8;   // PV: A = V^T via .trans
  const int v_dsub = ((lane >> 3) & 1) * 8;
  const int r0 = lane >> 2;                                // score rows (keys) r0, r0 + 8
  bool timed_out = false;

  // One block's online-softmax step: scores sc (S^T: keys r0, r0 + 8 x head
  // columns c0, c0 + 1) of the block starting at key p0 -> probabilities as
  // the P^T operand (pb0: keys 0..7, pb1: keys 8..15); updates m, l and O.
  // The reference max m of a column moves only when a score exceeds it by more
  // than 8 (log2 units): the probabilities then stay below 2^8 (as exact in
  // 16 bits as any, summed in fp32), and the common case costs one warp vote
  // instead of a shuffle reduction and a rescale of O.  The exponent reference
  // cancels in O / l, so the result is the same softmax.
  auto softmax_step = [&](const float (&sc)[4], int p0, uint32_t& pb0, uint32_t& pb1) {
    // mask keys past the context (they may hold stale NaN) and before the window
    const bool v0 = p0 + r0 < L && p0 + r0 >= kfirst;
    const bool v1 = p0 + r0 + 8 < L && p0 + r0 + 8 >= kfirst;
    float x[4];
    x[0] = v0 ? sc[0] * col_scale[0] : -INFINITY;
    x[1] = v0 ? sc[1] * col_scale[1] : -INFINITY;
    x[2] = v1 ? sc[2] * col_scale[0] : -INFINITY;
    x[3] = v1 ? sc[3] * col_scale[1] : -INFINITY;
    const float lim0 = m[0] + 8.f, lim1 = m[1] + 8.f;
    const bool grow = x[0] > lim0 || x[1] > lim1 || x[2] > lim0 || x[3] > lim1;
    if (__any_sync(0xffffffffu, grow)) {
      // new reference: the column max over the block's keys (lanes of equal t)
      float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float alpha0 = mn0 == -INFINITY ? 1.f : exp2f(m[0] - mn0);
      const float alpha1 = mn1 == -INFINITY ? 1.f : exp2f(m[1] - mn1);
      m[0] = mn0;
      m[1] = mn1;
      l[0] *= alpha0;
      l[1] *= alpha1;
#pragma unroll
      for (int dt = 0; dt < D / 16; ++dt) {
        o[dt][0] *= alpha0;
        o[dt][1] *= alpha1;
        o[dt][2] *= alpha0;
        o[dt][3] *= alpha1;
      }
    }
    const float mu0 = m[0] == -INFINITY ? 0.f : m[0];  // all keys so far masked
    const float mu1 = m[1] == -INFINITY ? 0.f : m[1];
    const uint32_t pk0 = pack2<FP8>(exp2f(x[0] - mu0), exp2f(x[1] - mu1));  // key r0
    const uint32_t pk1 = pack2<FP8>(exp2f(x[2] - mu0), exp2f(x[3] - mu1));  // key r0 + 8
    l[0] += lo2<FP8>(pk0) + lo2<FP8>(pk1);
    l[1] += hi2<FP8>(pk0) + hi2<FP8>(pk1);
    pb0 = movmatrix_trans(pk0);  // P^T rows = heads
    pb1 = movmatrix_trans(pk1);
  };

  // FP8: this lane's fragment offsets inside a block's code tiles (the same
  // for every block): K rows r0, r0 + 8 at chunks (D/64) t + c; V rows 2t,
  // 2t+1, 2t+8, 2t+9 at the lane's D/8 bytes (see the loop below).
  constexpr int KC = D / 64;
  uint32_t koff[2][KC], voff[4];
  if constexpr (FP8) {
    const int t = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < KC; ++c) koff[h][c] = swz8<D>(r0 + 8 * h, KC * t + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int row = 2 * t + (q & 1) + 8 * (q >> 1);
      voff[q] = D == 128 ? swz8<D>(row, r0) : swz8<D>(row, r0 >> 1) + 8 * (r0 & 1);
    }
  }

  for (int i = 0; i < nb_w; ++i) {
    const int st = i % NS;
    const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, i) != 0;
    if (!mbar_wait(bar0 + 8 * st, (i / NS) & 1, wait_limit(a.wait_limit_ns))) {
      timed_out = true;
      break;
    }
    const int p0 = (b_begin + warp + NW * i) * kBlock;  // first key of the block
    if constexpr (FP8) {
      // The whole block goes to registers first, so that its stage is
      // refilled before the block is computed (all NS loads stay in flight).
      // K: rows r0 and r0 + 8, bytes [(D/4) t, (D/4) t + D/4) (the permuted d
      // above).  V: rows 2t, 2t+1, 2t+8, 2t+9, bytes [(D/8) r0, (D/8) r0 +
      // D/8): the PV output rows of step dt are d = (D/8) r0 + 2 dt + {0, 1},
      // a permutation of d undone in the merge.
      constexpr int VW = D / 32;  // 32-bit V words per lane and row
      const int t = lane & 3;
      uint4 kw[2][KC];
      uint32_t vw[4][VW];
      if (ok) {
        const uint8_t* kt = wbase + st * T::kStageBytes;
        const uint8_t* vt = kt + T::kLoadBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < KC; ++c) kw[h][c] = *reinterpret_cast<const uint4*>(kt + koff[h][c]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if constexpr (D == 128) {
            const uint4 u = *reinterpret_cast<const uint4*>(vt + voff[q]);
            vw[q][0] = u.x; vw[q][1] = u.y; vw[q][2] = u.z; vw[q][3] = u.w;
          } else {
            const uint2 u = *reinterpret_cast<const uint2*>(vt + voff[q]);
            vw[q][0] = u.x; vw[q][1] = u.y;
          }
        }
        if (p0 + kBlock > L) {  // the last block: rows past the context hold stale codes
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (p0 + 2 * t + (q & 1) + 8 * (q >> 1) >= L) {
#pragma unroll
              for (int w = 0; w < VW; ++w) vw[q][w] = 0u;
            }
        }
      }
      __syncwarp();
      if (i + NS < nb_w) {
        if (lane == 0) fence_proxy_async();
        issue(i + NS);
        ++issued;
      }
      if (ok) {
        // ---- S^T = K . Q^T  (16 keys x 8 heads), even/odd k steps in two
        //      accumulators to halve the dependent MMA chain
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t* w0 = reinterpret_cast<const uint32_t*>(&kw[0][kk / 4]);
          const uint32_t* w1 = reinterpret_cast<const uint32_t*>(&kw[1][kk / 4]);
          const uint2 x = e4m3x4_to_f16x4(w0[kk % 4]), y = e4m3x4_to_f16x4(w1[kk % 4]);
          mma_16816<true>((kk & 1) ? sd : sc, x.x, y.x, x.y, y.y, qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[j] += sd[j];
        uint32_t pb0, pb1;
        softmax_step(sc, p0, pb0, pb1);
        // ---- O^T += V^T . P^T
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
          // bytes 2dt, 2dt+1 of rows (2t, 2t+1) interleaved: (k0,d0) (k1,d0) (k0,d1) (k1,d1)
          const uint32_t sel = (dt & 1) ? 0x7362u : 0x5140u;
          const uint2 lo = e4m3x4_to_f16x4(prmt(vw[0][dt / 2], vw[1][dt / 2], sel));
          const uint2 hi = e4m3x4_to_f16x4(prmt(vw[2][dt / 2], vw[3][dt / 2], sel));
          mma_16816<true>(o[dt], lo.x, lo.y, hi.x, hi.y, pb0, pb1);
        }
      }
    } else {
      if (ok) {
        const uint32_t kbuf = wbase_u + st * T::kStageBytes;
        const uint32_t vbuf = kbuf + T::kTileBytes;
        // ---- S^T = K . Q^T  (16 keys x 8 heads), two accumulators as above
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kbuf + swz_offset(k_row, kk * 16 + k_dsub), a0, a1, a2, a3);
          mma_16816<false>((kk & 1) ? sd : sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[j] += sd[j];
        uint32_t pb0, pb1;
        softmax_step(sc, p0, pb0, pb1);
        // ---- the sequence's last, partial block: zero V rows past the context
        if (p0 + kBlock > L) {
          const int nvalid = L - p0;
          uint8_t* vrow = wbase + st * T::kStageBytes + T::kTileBytes;
          for (int e = lane; e < (kBlock - nvalid) * T::kHalves * 8; e += 32) {
            const int r = nvalid + e / (T::kHalves * 8);
            const int rem = e % (T::kHalves * 8);
            *reinterpret_cast<uint4*>(vrow + (rem >> 3) * 2048 + r * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async();  // before any later TMA write to this stage
          __syncwarp();
        }
        // ---- O^T += V^T . P^T
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(vbuf + swz_offset(v_row, dt * 16 + v_dsub), a0, a1, a2, a3);
          mma_16816<false>(o[dt], a0, a1, a2, a3, pb0, pb1);
        }
      }
      __syncwarp();
      if (i + NS < nb_w) {
        if (lane == 0) fence_proxy_async();
        issue(i + NS);
        ++issued;
      }
    }
  }

  if (timed_out) {
    if (lane == 0) raise_error(a.err, PKV_ERR_TIMEOUT);
    // Let every copy this warp issued land before the CTA's memory is released.
    for (int st = 0; st < NS && st < issued; ++st) {
      const int last = ((issued - 1 - st) / NS) * NS + st;  // last block issued into stage st
      if (withheld && last == 0) continue;                    // (never issued)
      (void)mbar_wait(bar0 + 8 * st, (last / NS) & 1);
    }
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  // Denominators: sum the per-lane parts over the 8 lanes sharing a column.
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
  }

  // ---- merge the warps through shared memory
  float* wo = merge_area(warp);  // [8 heads][D] then m[8], l[8]
#pragma unroll
  for (int dt = 0; dt < D / 16; ++dt) {
    // output rows r0 and r0 + 8 of step dt hold d and d + dd
    const int d = FP8 ? (D / 8) * r0 + 2 * dt : dt * 16 + r0;
    constexpr int dd = FP8 ? 1 : 8;
    const int c = 2 * (lane & 3);
    wo[c * D + d] = o[dt][0];
    wo[(c + 1) * D + d] = o[dt][1];
    wo[c * D + d + dd] = o[dt][2];
    wo[(c + 1) * D + d + dd] = o[dt][3];
  }
  if (lane < 4) {
    wo[8 * D + 2 * lane] = m[0];
    wo[8 * D + 2 * lane + 1] = m[1];
    wo[8 * D + 8 + 2 * lane] = l[0];
    wo[8 * D + 8 + 2 * lane + 1] = l[1];
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    const int c = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, merge_area(w)[8 * D + c]);
    float den = 0.f;
    float f[NW];
    for (int w = 0; w < NW; ++w) {
      const float* ww = merge_area(w);
      f[w] = (M == -INFINITY) ? 0.f : exp2f(ww[8 * D + c] - M);
      den += f[w] * ww[8 * D + 8 + c];
    }
    for (int w = 0; w < NW; ++w) merge_f[w * 8 + c] = den > 0.f ? f[w] * out_scale / den : 0.f;
    merge_f[NW * 8 + c] = den > 0.f ? M + log2f(den) : -INFINITY;
  }
  __syncthreads();

  const bool direct = !PREFIX && nsplit == 1 && !a.force_partial;
  for (int idx = threadIdx.x; idx < 8 * D; idx += NW * 32) {
    const int c = idx / D;
    const int d = idx - c * D;
    int g = gsub * 8 + c, seq = s;
    if constexpr (PREFIX) {
      seq = g / G;
      g -= seq * G;
      if (seq >= a.num_seqs) continue;
    } else if (g >= G) {
      continue;
    }
    float r = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) r += merge_f[w * 8 + c] * merge_area(w)[c * D + d];
    const int hq = kvh * G + g;
    if (direct) {
      out[(static_cast<int64_t>(q0) * Hq + hq) * D + d] = __float2bfloat16(r);
    } else {
      const int64_t row =
          (static_cast<int64_t>(seq) * Hq + hq) * a.max_splits + a.split_base + split;
      a.ws_o[row * D + d] = r;
      if (d == 0) a.ws_lse[row] = merge_f[NW * 8 + c];
    }
  }
}

// ---------------------------------------------------------------- combine
// One warp per (sequence, q head) whose context was split:
// out = sum_i 2^(lse_i - M) O_i / sum_i 2^(lse_i - M).  The step is
// latency-bound, so the split loop is unrolled eight deep: a lane issues the
// loads of eight partial rows (a float4 or float2 of the head each) and their
// log-sum-exps before it needs any of them.
constexpr int kCombineUnroll = 8;

template <int D>
__global__ void __launch_bounds__(128) pkv_combine_bf16_kernel(const DecodeArgs a) {
  constexpr int PER = D / 32;  // elements per lane
  static_assert(PER == 2 || PER % 4 == 0, "head_size 64 or a multiple of 128");
  // (a programmatic dependent launch: the decode grid's partials are visible
  // once this returns; a no-op after an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= a.num_seqs * a.num_q_heads) return;
  int q0, nsplit;
  int64_t row;   // (query row, q head) index of the split partials
  int hq;
  if (a.merge_rows_end > a.merge_rows_begin) {
    // Cascade merge of a chunked-prefill row: its prefix partials, then the
    // one partial over its own keys.  A row whose sequence's metadata is bad
    // (or that sits inside the shared prefix) is zeroed, as the attention
    // calls do.
    const int tok = a.merge_rows_begin + gw / a.num_q_heads;
    hq = gw - (tok - a.merge_rows_begin) * a.num_q_heads;
    q0 = tok;
    const int s = seq_of_row(a.query_start_loc, a.casc_seqs, tok);
    bool ok = s >= 0;
    if (ok) {
      const int L = __ldg(a.context_lens + s);
      const int qn = __ldg(a.query_start_loc + s + 1) - __ldg(a.query_start_loc + s);
      ok = qn >= 1 && L >= qn && static_cast<int64_t>(L) <= a.bt_stride * kBlock &&
           L <= a.max_context_len && L - qn >= a.key_begin_blocks * kBlock;
    }
    if (!ok) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) +
                         (static_cast<int64_t>(tok) * a.num_q_heads + hq) * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; e += 2)
        *reinterpret_cast<__nv_bfloat162*>(o + e) = __floats2bfloat162_rn(0.f, 0.f);
      return;
    }
    nsplit = a.prefix_splits + 1;
    row = (static_cast<int64_t>(tok) * a.num_q_heads + hq) * a.max_splits;
  } else {
    const int s = gw / a.num_q_heads;
    hq = gw - s * a.num_q_heads;
    const int L = __ldg(a.context_lens + s);
    q0 = __ldg(a.query_start_loc + s);
    const int qn = __ldg(a.query_start_loc + s + 1) - q0;
    if (qn != 1 || q0 < 0 || q0 >= a.num_tokens || L < 1 ||
        static_cast<int64_t>(L) > a.bt_stride * kBlock || L > a.max_context_len ||
        L <= a.key_begin_blocks * kBlock || (a.key_begin_blocks > 0 && q0 != s))
      return;
    const int kfirst = max((a.window > 0 && L > a.window) ? L - a.window : 0,
                           a.key_begin_blocks * kBlock);
    const int nblk_seq = (L + kBlock - 1) / kBlock - kfirst / kBlock;
    // prefix partials (cascade) first, then this row's own splits
    nsplit = a.prefix_splits + (nblk_seq + a.split_blocks - 1) / a.split_blocks;
    if (nsplit <= 1 && !a.force_partial) return;  // the decode kernel wrote this row directly
    row = (static_cast<int64_t>(s) * a.num_q_heads + hq) * a.max_splits;
  }
  const float* lse = a.ws_lse + row;
  float M = -INFINITY;
  for (int i = lane; i < nsplit; i += 32) M = fmaxf(M, lse[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float den = 0.f;
  if (M != -INFINITY) {
    const float* o = a.ws_o + row * D + lane * PER;
    for (int i0 = 0; i0 < nsplit; i0 += kCombineUnroll) {
      float v[kCombineUnroll][PER];
      float lv[kCombineUnroll];
#pragma unroll
      for (int u = 0; u < kCombineUnroll; ++u) {
        const int i = i0 + u;
        lv[u] = -INFINITY;
#pragma unroll
        for (int e = 0; e < PER; ++e) v[u][e] = 0.f;
        if (i < nsplit) {
          lv[u] = lse[i];
          const float* src = o + static_cast<int64_t>(i) * D;
          if constexpr (PER == 2) {
            *reinterpret_cast<float2*>(v[u]) = *reinterpret_cast<const float2*>(src);
          } else {
#pragma unroll
            for (int e = 0; e < PER; e += 4)
              *reinterpret_cast<float4*>(v[u] + e) = *reinterpret_cast<const float4*>(src + e);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kCombineUnroll; ++u) {
        const float w = (lv[u] == -INFINITY) ? 0.f : exp2f(lv[u] - M);
        den += w;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] += w * v[u][e];
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) +
                       (static_cast<int64_t>(q0) * a.num_q_heads + hq) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(out + e) =
        __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}

template <int D, int NS, bool FP8, bool PREFIX = false>
cudaError_t launch_decode_t(const CUtensorMap& kmap, const CUtensorMap& vmap,
                            const DecodeArgs& a, cudaStream_t stream) {
  constexpr int smem = decode_smem_bytes<D, NS, FP8>();
  auto kfn = pkv_decode_bf16_kernel<D, NS, FP8, PREFIX>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // prefix launch: (prefix split, kv head x column group); otherwise (split of
  // this launch, kv head x head group, sequence)
  const int ngsub = PREFIX ? a.prefix_col_groups : (a.group + 7) / 8;
  dim3 grid(PREFIX ? a.prefix_splits : a.max_splits - a.split_base, a.num_kv_heads * ngsub,
            PREFIX ? 1 : a.num_seqs);
  DecodeArgs b = a;
  debug_wait_settings(&b.wait_limit_ns, &b.debug_stall);
  kfn<<<grid, kDecodeWarps * 32, smem, stream>>>(kmap, vmap, b);
  return cudaGetLastError();
}

}  // namespace

// Stages per warp: 3 x 8 KB (head_size 128) keeps 2 CTAs (8 warps, up to 16
// blocks = 128 KB of K/V) in flight per SM.
// FP8 stages are half the size: 3-deep rings leave room for four CTAs per SM
// (16 warps), and a warp refills a stage as soon as its block is in registers.
// (Measured on GB300 decode batches: 3 stages beat 2 and 4.)
cudaError_t launch_decode_bf16(const CUtensorMap& kmap, const CUtensorMap& vmap,
                               const DecodeArgs& a, int head_size, bool fp8,
                               cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  if (fp8) {
    if (head_size == 128) return launch_decode_t<128, 3, true>(kmap, vmap, a, stream);
    return launch_decode_t<64, 6, true>(kmap, vmap, a, stream);
  }
  if (head_size == 128) return launch_decode_t<128, 3, false>(kmap, vmap, a, stream);
  return launch_decode_t<64, 4, false>(kmap, vmap, a, stream);
}

cudaError_t launch_cascade_prefix_bf16(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                       const DecodeArgs& a, int head_size, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.prefix_splits == 0) return cudaSuccess;
  if (head_size == 128) return launch_decode_t<128, 3, false, true>(kmap, vmap, a, stream);
  return launch_decode_t<64, 4, false, true>(kmap, vmap, a, stream);
}

cudaError_t launch_combine_bf16(const DecodeArgs& a, int head_size, cudaStream_t stream,
                                bool after_decode) {
  if (a.num_seqs == 0 || a.max_splits <= 1) return cudaSuccess;
  const int warps = a.num_seqs * a.num_q_heads;
  const int blocks = (warps + 3) / 4;
  // Right after the decode launch on the same stream, the combine is a
  // programmatic dependent launch: its CTAs are scheduled while the decode's
  // last CTAs still run and wait in griddepcontrol.wait for the decode
  // grid's completion (its partials visible), so the launch gap overlaps the
  // decode's tail instead of following it.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_decode ? 1 : 0;
  if (head_size == 128) return cudaLaunchKernelEx(&cfg, pkv_combine_bf16_kernel<128>, a);
  return cudaLaunchKernelEx(&cfg, pkv_combine_bf16_kernel<64>, a);
}

}  // namespace pkv
