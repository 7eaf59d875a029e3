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
//  * 12 warps.  Warp 8 streams 128-key K tiles and warp 10 V tiles (8 cache
//    blocks, one TMA box per block and half; block ids fetched four tiles
//    ahead) into one 5-slot ring shared by both query tiles, in the order the
//    products read them (K_0, V_0, K_1, V_1, ...); warp 9 allocates all 512
//    TMEM columns.  The products of query tile t,
//        S_t  = Q_t K^T   (M=128, N=128, K=16 x D/16, operands from smem)
//        O_t += P_t V     (M=128, N=D,   K=16 x 8, P_t from TMEM, V MN-major)
//    are issued by one thread of tile t's own softmax warpgroup right after
//    it has written P_t, each group of eight K-steps from one asm block: an
//    issuing thread whose SM sub-partition neighbours keep the FMA pipe busy
//    gets few issue slots (measured), and the warpgroup that has just
//    finished its softmax is the one whose instructions are ready.  The two
//    tiles take turns (S_0, S_1, then [P_0 V, S_0], [P_1 V, S_1], ...), so one
//    tile's softmax runs beside the other tile's products.  An M=128
//    tcgen05 MMA at N = 128 runs at the full rate (64 cycles per K-step),
//    S_t (128 columns) and O_t (D columns) per query tile fill the 512
//    columns, and P_t (bf16) is written over the first half of S_t's columns;
//    S_t of the next K/V tile follows P_t V in the same thread's order.
//  * warps 0-3 and 4-7 (one warpgroup per query tile) own one TMEM lane
//    (= one row) per thread: they load a row of S, apply the causal mask, keep
//    a lazily updated running max (O is rescaled in TMEM only when the max
//    grows by more than 2^8), write P (bf16) to TMEM for the second MMA, and at
//    the end read O, divide by the row sum and store bf16.  No shuffles: a
//    thread holds its whole row.  The V producer zeroes the rows of the first
//    and last V tiles that no row may see (stale data, NaN included, would
//    reach P V through 0 * NaN).
//  * the outputs of a full query tile go out through its Q slot in shared
//    memory and one TMA store per 64-column half.
//  * a launch that has the GPU to itself hands its CTAs out longest first
//    (each CTA ranks the (sequence, tile pair) units by the key tiles they
//    see and takes the one whose rank is its launch index), so the last wave
//    holds the short ones; beside a decode launch the plain order stays.
//  * every wait is an mbarrier with a bounded spin and a CTA-wide abort flag;
//    TMEM is freed on every path.
//  * FP8 (e4m3) cache: TMA lands each tile's codes (128 keys x D bytes, the
//    128- or 64-byte swizzle of the row width) in the first part of its ring
//    slot and warps 10 and 11 (D = 128: half the rows each; D = 64: warp 10)
//    widen them in place to fp16 in the bf16 tiles' layout (e4m3 is exact in fp16; codes are read before the fp16
//    rows written over them), then marks the slot full for the MMAs;
//    each softmax thread converts its own Q row to fp16 (a row beyond 2^14
//    scaled by 2^-e, its scores by 2^e) and the MMAs run on fp16 operands with
//    P in fp16.  The K descale folds into the score scale, the V descale into
//    the output.
#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {

namespace {

constexpr int kTcRows = 128;      // UMMA M (rows of one query tile)
constexpr int kTcTiles = 2;       // query tiles per CTA
constexpr int kTcKeys = 128;      // keys per K/V tile
// Warps: 0-3 softmax of query tile 0, 4-7 of query tile 1 (warpgroups 0 and
// 1: warp w reads TMEM lanes 32 (w % 4) ..), 8 the K producer (and the V
// producer with an FP8 cache), 9 TMEM allocation, 10 the V producer (bf16) or
// a widener (FP8), 11 a widener (FP8, D = 128; idle otherwise).  The launch
// gives each thread 168 registers; warpgroup 2 then hands registers back so
// that the softmax warpgroups run at 208 (2 x 128 x 208 + 128 x 80 =
// 384 x 168).
constexpr int kTcThreads = 384;
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 80;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kTcThreads * 168, "register split");
// One ring of K/V tile slots, filled in the order the products read them:
// K of key tile j is ring element 2j, V of key tile j element 2j + 1, element
// e in slot e % kRing.  (Separate K and V rings of 3 + 2 slots left V on the
// critical path: a V tile was issued only once the V two tiles back had been
// read, and its copy, ~1.5-2 us from L2, still in flight when P was ready.)
constexpr int kRing = 5;
__host__ __device__ constexpr int ring_slot(int e) { return e % kRing; }
__host__ __device__ constexpr uint32_t ring_phase(int e) {
  return static_cast<uint32_t>((e / kRing) & 1);
}
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S of tile t at 128t (P of tile t over its first 64 columns),
// O of tile t at 256 + 128t.
__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }
__host__ __device__ constexpr uint32_t col_p(int t) { return 128u * t; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
constexpr float kLazyRescale = 8.0f;  // log2 units: rescale O only past 2^8 growth

template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kTcRows * 128;       // 16 KB: 128 rows x 128 B
  static constexpr int kQTile = kHalves * kQHalf;
  static constexpr int kKvHalf = kTcKeys * 128;      // 16 KB: 128 keys x 128 B
  static constexpr int kTileBytes = kHalves * kKvHalf;  // one K (or V) tile
};

struct TcShared {
  uint64_t q_full, q_conv;
  uint64_t drain[kTcTiles];   // each tile's issuer: all its products complete
  uint64_t s_full[kTcTiles], p_full[kTcTiles], pv_done[kTcTiles];
  uint64_t kv_full[kRing], kv_empty[kRing];
  uint64_t kv_land[kRing];   // FP8 (and bf16 V edge tiles): landed, not yet ready
  uint64_t issued[kTcTiles];   // tile t's issuer has issued its next MMA group
  uint32_t tmem_base;
  int32_t abort;
  int32_t n_issued[2];   // bf16 producers: K / V tiles issued, for the drain
};

template <int D>
constexpr int tc_smem_bytes() {
  // Whole-SM footprint: one CTA per SM (it owns all 512 TMEM columns).
  constexpr int need = 1024 + kTcTiles * TcLayout<D>::kQTile +
                       kRing * TcLayout<D>::kTileBytes +
                       static_cast<int>(sizeof(TcShared));
  return need > 120 * 1024 ? need : 120 * 1024;
}

// Timeline of one CTA (profiling builds, -DPKV_TC_TIMELINE): %globaltimer
// stamps of the pipeline events of the CTA computing the last row-tile pair
// of the batch's second sequence, kv head 0.
#ifdef PKV_TC_TIMELINE
__device__ unsigned long long g_tc_timeline[4096];
#define TC_MARK(idx)                                         \
  do {                                                       \
    if (tl_on) g_tc_timeline[(idx)] = global_timer_ns();     \
  } while (0)
#else
#define TC_MARK(idx) \
  do {               \
  } while (0)
#endif

__device__ __forceinline__ void set_max_regs_inc_softmax() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
}
__device__ __forceinline__ void set_max_regs_dec_other() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
}

// Bounded wait that also gives up when another thread of the CTA has aborted.
// mbarrier.try_wait suspends the thread in hardware until the phase completes
// or a short time limit passes, so a waiting warp takes no issue slots from
// the softmax and MMA-issuing warps of its SM sub-partition.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int32_t* abort, int32_t* err,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      raise_error(err, PKV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform version: lane 0 waits, the verdict is broadcast, and the other
// lanes then observe the (already completed) phase themselves.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                          int32_t* err, uint64_t limit_ns) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  if (lane == 0) ok = wait_or_abort(bar, parity, abort, err, limit_ns);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok && lane != 0) ok = mbar_test(bar, parity);   // completed: observe it
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Widens one 128-key x 128 e4m3 tile (128-byte swizzled rows at `tile`) in
// place into the fp16 tile layout (two 64-column halves, 16 KB apart,
// 128-byte swizzled); all 32 lanes of the calling warp.  A batch covers 16
// rows: a lane reads its 16-code chunk of 4 rows (4 loads in flight), and
// only after the warp has read the whole batch does it write the batch's fp16
// chunks (those of half 0 overwrite the same rows' codes); batches touch
// disjoint rows, so two warps may widen batches [b0, b1) of the same tile.
__device__ __forceinline__ void widen_tile_fp8(uint8_t* tile, int lane, int b0, int b1) {
  const int c = lane & 7;           // chunk: columns 16c .. 16c + 15
  const int j = 2 * (c & 3);        // its first 8-column chunk within the half
  uint8_t* half = tile + (c >> 2) * (kTcKeys * 128);
#pragma unroll 1
  for (int b = b0; b < b1; ++b) {
    uint4 codes[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 16 * b + 4 * i + (lane >> 3);
      codes[i] = *reinterpret_cast<const uint4*>(tile + r * 128 + ((c ^ (r & 7)) << 4));
    }
    uint4 lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 x = e4m3x4_to_f16x4(codes[i].x), y = e4m3x4_to_f16x4(codes[i].y);
      const uint2 z = e4m3x4_to_f16x4(codes[i].z), w = e4m3x4_to_f16x4(codes[i].w);
      lo[i] = make_uint4(x.x, x.y, y.x, y.y);
      hi[i] = make_uint4(z.x, z.y, w.x, w.y);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 16 * b + 4 * i + (lane >> 3);
      *reinterpret_cast<uint4*>(half + r * 128 + ((j ^ (r & 7)) << 4)) = lo[i];
      *reinterpret_cast<uint4*>(half + r * 128 + (((j + 1) ^ (r & 7)) << 4)) = hi[i];
    }
  }
  __syncwarp();
}

// Zeroes the V rows [0, lead) and [tail, 128) that lie in rows [r0, r1) of
// one landed 128-key tile (bf16 or widened fp16 layout: D / 64 halves of 128
// rows x 128 B, 16 KB apart); the calling warp's 32 lanes share the stores.
// Those keys have P = 0 in every row, but their rows may hold stale data --
// NaN included -- which 0 * NaN would carry into P V.
template <int D>
__device__ __forceinline__ void zero_v_rows(uint8_t* vt, int lead, int tail, int r0, int r1,
                                            int lane) {
  constexpr int per_row = (D / 64) * 8;   // 16-byte chunks per row
  const int lead_end = min(max(lead, r0), r1);   // lead rows: [r0, lead_end)
  const int tail_beg = min(max(tail, r0), r1);   // tail rows: [tail_beg, r1)
  const int nlead = lead_end - r0;
  const int ntail = r1 - tail_beg;
  for (int e = lane; e < (nlead + ntail) * per_row; e += 32) {
    const int r = e / per_row;
    const int key = r < nlead ? r0 + r : tail_beg + (r - nlead);
    const int rem = e % per_row;
    *reinterpret_cast<uint4*>(vt + (rem >> 3) * (kTcKeys * 128) + key * 128 + (rem & 7) * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
}

// head_size 64: the tile's 128 code rows of 64 B (64-byte swizzle: chunk c of
// row r at r * 64 + ((c ^ (r / 2 % 4)) << 4)) land in its first 8 KB and
// widen into 128 fp16 rows of 128 B (128-byte swizzle).  Batch b (rows 16b ..
// 16b + 15) writes bytes [2048 b, 2048 b + 2048), the codes of batches 2b and
// 2b + 1; going from the last batch to the first, those were read earlier
// (or, for b = 0, by this batch before its writes).  A lane reads two 16-code
// chunks per batch.
__device__ __forceinline__ void widen_tile_fp8_d64(uint8_t* tile, int lane) {
  const int c = lane & 3;           // code chunk: columns 16c .. 16c + 15
#pragma unroll 1
  for (int b = kTcKeys / 16 - 1; b >= 0; --b) {
    uint4 codes[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 16 * b + 8 * i + (lane >> 2);
      codes[i] = *reinterpret_cast<const uint4*>(tile + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
    }
    uint4 lo[2], hi[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint2 x = e4m3x4_to_f16x4(codes[i].x), y = e4m3x4_to_f16x4(codes[i].y);
      const uint2 z = e4m3x4_to_f16x4(codes[i].z), w = e4m3x4_to_f16x4(codes[i].w);
      lo[i] = make_uint4(x.x, x.y, y.x, y.y);
      hi[i] = make_uint4(z.x, z.y, w.x, w.y);
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 16 * b + 8 * i + (lane >> 2);
      *reinterpret_cast<uint4*>(tile + r * 128 + (((2 * c) ^ (r & 7)) << 4)) = lo[i];
      *reinterpret_cast<uint4*>(tile + r * 128 + (((2 * c + 1) ^ (r & 7)) << 4)) = hi[i];
    }
    __syncwarp();
  }
}

// Which (sequence, row-tile pair, kv head) this CTA computes.  The block
// scheduler starts CTAs in launch order, so with `longest_first` the grid is
// handed out longest first (list scheduling): the units (sequence, pair) are
// ranked by the number of 128-key tiles their rows see (a chunk's last
// pairs, and longer contexts, see more), ties by index, and the kv heads of a
// unit are consecutive CTAs.  Every CTA ranks the units itself (at most
// kLptUnits costs, in shared memory scratch that the K/V ring later reuses).
// Otherwise, or with more than kLptUnits units (many waves, little tail), the
// grid keeps its plain order (heaviest pair of each sequence first).
// Measured on GB300, the 4 x 512-token chunks of the mixed 32 q / 8 kv head
// batch alone: 104 -> 88 us longest first; beside that batch's decode launch
// the plain order is better (140 vs 144 us for both): its short CTAs end
// early and the decode CTAs, HBM-bound, run beside the long tensor-bound ones.
constexpr int kLptUnits = 128;

struct TcWork {
  int s, kvh, mtile;
};

__device__ __forceinline__ int tc_unit_cost(const PrefillArgs& a, int u, int toks) {
  const int s = a.seq_begin + u / a.num_mtiles;
  const int tok0 = (u % a.num_mtiles) * toks;
  const int L = __ldg(a.context_lens + s);
  const int q0 = __ldg(a.query_start_loc + s);
  const int qn = __ldg(a.query_start_loc + s + 1) - q0;
  if (qn <= 0 || tok0 >= qn || L < qn) return 0;   // nothing (or an error) to do
  const int pos_max = L - qn + min(tok0 + toks, qn) - 1;
  const int pos_min = L - qn + tok0;
  const int lo_min = max(a.window > 0 ? pos_min - a.window + 1 : 0, a.key_begin);
  const int j0 = lo_min > 0 ? lo_min / kTcKeys : 0;
  return (pos_max + kTcKeys) / kTcKeys - j0 + 1;   // key tiles + the CTA's own overhead
}

// Called by every thread of the CTA (it synchronises the CTA twice).
__device__ __forceinline__ TcWork pick_work(const PrefillArgs& a, int toks, int32_t* scratch) {
  const int nu = a.num_seqs * a.num_mtiles;
  if (nu > kLptUnits) {   // (the launcher does not choose this kernel then)
    return TcWork{a.seq_begin + static_cast<int>(blockIdx.z), static_cast<int>(blockIdx.y),
                  a.num_mtiles - 1 - static_cast<int>(blockIdx.x)};
  }
  const int b = static_cast<int>(blockIdx.x) +
                static_cast<int>(gridDim.x) * (static_cast<int>(blockIdx.y) +
                                               static_cast<int>(gridDim.y) *
                                                   static_cast<int>(blockIdx.z));
  const int r = b / a.num_kv_heads;   // this CTA's unit rank
  int32_t* cost = scratch;            // [nu]
  int32_t* pick = scratch + kLptUnits;
  for (int u = threadIdx.x; u < nu; u += blockDim.x) cost[u] = tc_unit_cost(a, u, toks);
  if (threadIdx.x == 0) *pick = 0;
  __syncthreads();
  for (int u = threadIdx.x; u < nu; u += blockDim.x) {
    const int c = cost[u];
    int rank = 0;
    for (int v = 0; v < nu; ++v) {
      const int cv = cost[v];
      rank += (cv > c || (cv == c && v < u)) ? 1 : 0;
    }
    if (rank == r) *pick = u;
  }
  fence_proxy_async();   // the ring's TMA writes later land on this scratch
  __syncthreads();
  const int u = *pick;
  return TcWork{a.seq_begin + u / a.num_mtiles, b % a.num_kv_heads, u % a.num_mtiles};
}

// LPT: the longest-first instantiation (a separate kernel, so that the plain
// one keeps its work indices as launch coordinates and its register budget).
template <int D, bool FP8, bool LPT>
__global__ void __launch_bounds__(kTcThreads, 1)
    pkv_prefill_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ CUtensorMap omap, const PrefillArgs a) {
  using Lt = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                                   // [tile][half][128 rows x 128 B]
  uint8_t* sKV = smem + kTcTiles * Lt::kQTile;          // [slot][half][128 keys x 128 B]
  TcShared* sh = reinterpret_cast<TcShared*>(sKV + kRing * Lt::kTileBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Cascade prefix launch: one "sequence" whose rows are the batch's decode
  // rows (sequence t at row t), non-causal over the shared keys, one key split
  // per grid.z; otherwise grid.z is the sequence.
  const bool casc = a.cascade_prefix != 0;
  const int G = a.group;
  const int Hq = a.num_q_heads;
  const int tile_toks = kTcRows / G;                // tokens per query tile
  const int toks = kTcTiles * tile_toks;            // tokens per CTA
  int s, kvh, mtile;
  if constexpr (LPT) {
    const TcWork w = pick_work(a, toks, reinterpret_cast<int32_t*>(sKV));
    s = w.s;
    kvh = w.kvh;
    mtile = w.mtile;
  } else {
    s = casc ? 0 : a.seq_begin + blockIdx.z;
    kvh = blockIdx.y;
    mtile = a.num_mtiles - 1 - blockIdx.x;  // heaviest pair of each sequence first
  }

#ifdef PKV_TC_TIMELINE
  const bool tl_on = !casc && s == a.seq_begin + 1 && kvh == 0 && mtile == a.num_mtiles - 1;
#endif
  const int L = casc ? a.prefix_len : __ldg(a.context_lens + s);
  const int q0 = casc ? 0 : __ldg(a.query_start_loc + s);
  const int qn = casc ? a.num_seqs : __ldg(a.query_start_loc + s + 1) - q0;
  const int tok0 = mtile * toks;
  const bool bad_rows = qn < 0 || q0 < 0 || static_cast<int64_t>(q0) + qn > a.num_tokens;
  if (bad_rows || qn == 0 || tok0 >= qn) {
    if (bad_rows && mtile == 0 && kvh == 0 && threadIdx.x == 0)
      raise_error(a.err, PKV_ERR_QUERY_LEN);
    return;
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  const bool bad_len = (L < 1 || static_cast<int64_t>(L) > a.bt_stride * kBlock);
  if (casc && bad_len) {
    if (threadIdx.x == 0 && mtile == 0 && kvh == 0) raise_error(a.err, PKV_ERR_CONTEXT_LEN);
    return;
  }
  // (a cascade suffix row must sit after the shared prefix; its merge then
  // zeroes the rows of the sequence)
  const bool before_prefix = a.key_begin > 0 && L - qn < a.key_begin;
  if (!casc && (bad_len || qn > L || qn > a.max_query_len || before_prefix)) {
    if (threadIdx.x == 0 && mtile == 0 && kvh == 0)
      raise_error(a.err, (bad_len || before_prefix) ? PKV_ERR_CONTEXT_LEN : PKV_ERR_QUERY_LEN);
    if (a.key_begin > 0) return;   // (the merge writes the output rows)
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
  // last key any row here can see (cascade prefix: every shared key)
  const int pos_max = casc ? L - 1 : L - qn + tok_last;
  // With a sliding window, K/V tiles wholly before the lowest row's window
  // are never loaded (their block-table entries may hold the null block): the
  // CTA walks tiles j0 .. ntiles-1, ring positions 0 .. n_rel-1.  A cascade
  // prefix CTA walks its split's prefix_tiles tiles.
  const int pos_min = L - qn + tok0;
  // first key some row here sees: the lowest row's window start, or the end
  // of the shared prefix (cascade suffix launch)
  const int lo_min = max(a.window > 0 ? pos_min - a.window + 1 : 0, a.key_begin);
  const int j0 = casc ? static_cast<int>(blockIdx.z) * a.prefix_tiles
                      : (lo_min > 0 ? lo_min / kTcKeys : 0);
  const int ntiles =
      casc ? min(j0 + a.prefix_tiles, (L + kTcKeys - 1) / kTcKeys) : (pos_max + kTcKeys) / kTcKeys;
  const int n_rel = ntiles - j0;
  if (n_rel <= 0) return;
  // First cache block holding a key some row can see; blocks before it in
  // tile j0 are not loaded (their entries may be null) and their V rows are
  // zeroed instead.
  const int b_lo = casc ? j0 * (kTcKeys / kBlock) : (lo_min > 0 ? lo_min / kBlock : 0);
  const int nblk = (pos_max + kBlock) / kBlock;
  // V rows of the first tile before the first loaded block, and of the last
  // tile past pos_max, are zeroed once the tile has landed (zero_v_rows).
  const int v_lead = min(kTcKeys, b_lo * kBlock - j0 * kTcKeys);
  const int v_tail = pos_max + 1 - (ntiles - 1) * kTcKeys;
  auto v_edges = [&](int rel, int& lead, int& tail) {
    lead = rel == 0 ? v_lead : 0;
    tail = rel == n_rel - 1 ? v_tail : kTcKeys;
    return lead > 0 || tail < kTcKeys;
  };

  const uint32_t q_full = smem_u32(&sh->q_full);
  // the MMAs may read Q once it has landed (bf16) or been converted (FP8)
  const uint32_t q_ready = FP8 ? smem_u32(&sh->q_conv) : q_full;
  if (threadIdx.x == 0) {
    prefetch_tensor_map(&qmap);
    prefetch_tensor_map(&kmap);
    prefetch_tensor_map(&vmap);
    prefetch_tensor_map(&omap);
    mbar_init(q_full, 1);
    // one MMA-issuing thread per query tile, each committing its own products
    const uint32_t issuers = static_cast<uint32_t>(ntq);
    mbar_init(smem_u32(&sh->q_conv), 8);   // one arrival per softmax warp
    for (int t = 0; t < kTcTiles; ++t) {
      mbar_init(smem_u32(&sh->s_full[t]), 1);
      mbar_init(smem_u32(&sh->p_full[t]), 4);
      mbar_init(smem_u32(&sh->pv_done[t]), 1);
      mbar_init(smem_u32(&sh->issued[t]), 1);
      mbar_init(smem_u32(&sh->drain[t]), 1);
    }
    for (int i = 0; i < kRing; ++i) {
      // FP8 D = 128: both widening warps arrive (each widens half the rows)
      mbar_init(smem_u32(&sh->kv_full[i]), (FP8 && D == 128) ? 2 : 1);
      mbar_init(smem_u32(&sh->kv_empty[i]), issuers);
      mbar_init(smem_u32(&sh->kv_land[i]), 1);
    }
    sh->abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) tc::alloc(smem_u32(&sh->tmem_base), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  volatile int32_t* abort = &sh->abort;
  const uint64_t wlim = wait_limit(a.wait_limit_ns);
  TC_MARK(0);
#ifdef PKV_TC_TIMELINE
  const int cta_lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  if (threadIdx.x == 0 && cta_lin < 600) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_tc_timeline[2048 + 3 * cta_lin] = smid;
    g_tc_timeline[2048 + 3 * cta_lin + 1] = global_timer_ns();
  }
#endif

  // ---------------------------------------------------------- MMA issue
  constexpr uint32_t idS = FP8 ? tc::idesc_f16_f32(kTcRows, kTcKeys, 0, 0)
                               : tc::idesc_bf16_f32(kTcRows, kTcKeys, 0, 0);
  constexpr uint32_t idO = FP8 ? tc::idesc_f16_f32(kTcRows, D, 0, 1)
                               : tc::idesc_bf16_f32(kTcRows, D, 0, 1);
  // Shared-memory descriptors are built once: the address field is the
  // low 14 bits (address / 16) and never carries, so an operand at a
  // constant byte offset is the base descriptor plus offset / 16 -- one
  // add per MMA on the issuing thread, whose instructions compete with
  // the softmax warps for the same issue slots.
  const uint64_t dq0 = tc::smem_desc_sw128(smem_u32(sQ), 16, 1024);
  const uint64_t dk0 = tc::smem_desc_sw128(smem_u32(sKV), 16, 1024);
  const uint64_t dv0 = tc::smem_desc_sw128(smem_u32(sKV), Lt::kKvHalf, 1024);
  auto issue_s = [&](int t, int j) {
    const uint64_t da0 = dq0 + static_cast<uint64_t>((t * Lt::kQTile) >> 4);
    const uint64_t db0 =
        dk0 + static_cast<uint64_t>((ring_slot(2 * j) * Lt::kTileBytes) >> 4);
    const uint32_t d = tmem + col_s(t);
    // K-step k: 16 bf16 = 32 B along the swizzled 128-B row, 64 columns
    // per half (16 KB apart for both operands)
    static_assert(Lt::kQHalf == Lt::kKvHalf, "equal half strides");
    if constexpr (D == 128) {
      tc::mma_ss_x8<2, 4, 6, 1024, 1026, 1028, 1030, 2, 4, 6, 1024, 1026, 1028, 1030>(
          d, da0, db0, idS, 0u);
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc::mma_ss(d, da0 + (kk * 32 >> 4), db0 + (kk * 32 >> 4), idS, kk > 0 ? 1u : 0u);
    }
    tc::commit(smem_u32(&sh->s_full[t]));
  };
  auto issue_pv = [&](int t, int j) {
    const uint64_t db0 =
        dv0 + static_cast<uint64_t>((ring_slot(2 * j + 1) * Lt::kTileBytes) >> 4);
    tc::mma_ts_x8(tmem + col_o(t), tmem + col_p(t), db0, idO, j > 0 ? 1u : 0u);
    tc::commit(smem_u32(&sh->pv_done[t]));
  };


  if (warp >= 8) {
   set_max_regs_dec_other();
   if (warp == 8 || (!FP8 && warp == 10)) {
    // ------------------------------------------------------------ producers
    // bf16: warp 8 streams the K tiles and warp 10 the V tiles into their
    // ring slots, each waiting only for its own slots.  FP8: warp 8 streams
    // both (K of tile it before V of tile it - 1); warps 10 and 11 widen
    // them.
    const uint64_t keep = policy_evict_normal();   // K/V tiles are re-read by the
    const int32_t* bt = a.block_tables + static_cast<int64_t>(s) * a.bt_stride;  // other row tiles
    if (warp == 8 && lane == 0) {
      mbar_arrive_expect_tx(q_full, ntq * Lt::kQTile);
      for (int t = 0; t < ntq; ++t)
#pragma unroll
        for (int h = 0; h < Lt::kHalves; ++h)
          tma_load_3d(smem_u32(sQ + t * Lt::kQTile + h * Lt::kQHalf), &qmap, q_full, h * 64,
                      kvh * G, q0 + tok0 + t * tile_toks, keep);
    }
    constexpr int kBlocks = kTcKeys / kBlock;      // cache blocks per tile
    // Block ids of four consecutive tiles per warp-wide load: lane l holds
    // block l % 8 of ring position 4g + l / 8.  Group g + 1 is loaded while
    // group g is issued, so no tile waits on its ids.
    auto load_ids4 = [&](int g) {
      const int it = j0 + 4 * g + (lane >> 3);
      const int b = it * kBlocks + (lane & 7);
      return (it < ntiles && b < nblk) ? __ldg(bt + b) : -1;
    };
    // Issues the K (is_v = false) or V tile `it` into `dst`, completing on
    // `full`; its ids are lanes 8 sub .. 8 sub + 7 of `ids`.
    auto issue_tile = [&](int it, int ids, int sub, bool is_v, uint32_t dst, uint32_t full) {
      bool ok[kBlocks];
      int bid[kBlocks];
      uint32_t bytes = 0;
#pragma unroll
      for (int b = 0; b < kBlocks; ++b) {
        bid[b] = __shfl_sync(0xffffffffu, ids, 8 * sub + b);
        const int blk = it * kBlocks + b;
        const bool in_range = blk < nblk && blk >= b_lo;
        ok[b] = in_range && bid[b] >= 0 && bid[b] < a.num_blocks;
        if (!is_v && in_range && !ok[b] && lane == 0) raise_error(a.err, PKV_ERR_BLOCK_ID);
        bytes += ok[b] ? (FP8 ? 16u * D : Lt::kHalves * 2048u) : 0u;
      }
      if (lane == 0) {
        if (bytes == 0) {
          mbar_arrive(full);
        } else {
          mbar_arrive_expect_tx(full, bytes);
#pragma unroll
          for (int b = 0; b < kBlocks; ++b) {
            if (!ok[b]) continue;
            if constexpr (FP8) {  // 16 rows x D codes: rows b*16 .. b*16+15 of the tile
              tma_load_3d(dst + b * 16 * D, is_v ? &vmap : &kmap, full, 0, kvh, bid[b] * kBlock,
                          keep);
            } else {
#pragma unroll
              for (int h = 0; h < Lt::kHalves; ++h)
                tma_load_3d(dst + h * Lt::kKvHalf + b * 2048, is_v ? &vmap : &kmap, full,
                            h * 64, kvh, bid[b] * kBlock, keep);
            }
          }
        }
      }
    };
    int g_cur = load_ids4(0), g_nxt = load_ids4(1);
    // Test hook: the K producer withholds the first K tile (no copy, no
    // arrival), so that the waits for it run out.
    const bool withhold_k0 = a.debug_stall != 0;
    // Before the CTA's shared memory is released every copy a producer
    // started must have landed.  Only the last use of a slot can still be in
    // flight: element e's slot is refilled by element e + kRing only after e
    // has been read (so has landed).  Waits on a slot's barrier with e's
    // parity are then exact (no later phase of that barrier exists).
    // n_k / n_v: K / V tiles this warp issued (ring positions 0 .. n - 1),
    // n_k_all / n_v_all: by either producer; `skip`: a ring element whose
    // copy was already waited for (or never started).
    auto drain = [&](int n_k, int n_v, int n_k_all, int n_v_all, bool land, int skip) {
      for (int e = 0; e < 2 * max(n_k, n_v); ++e) {
        const bool mine_k = !(e & 1) && (e >> 1) < n_k, mine_v = (e & 1) && (e >> 1) < n_v;
        if (!(mine_k || mine_v) || e == skip) continue;
        const int nx = e + kRing;   // the slot's next element: issued?
        if ((nx & 1) ? (nx >> 1) < n_v_all : (nx >> 1) < n_k_all) continue;
        const int st = ring_slot(e);
        const uint32_t bar = smem_u32(land ? &sh->kv_land[st] : &sh->kv_full[st]);
        if (lane == 0) (void)mbar_wait(bar, ring_phase(e));
      }
      __syncwarp();
    };
    if constexpr (!FP8) {
      const bool is_v = warp == 10;
      uint32_t land_phase = 0;   // parity of each slot's next kv_land phase (V edges)
      int n_issued = 0, pending_land = -1, pending_e = -1;
      for (int rel = 0; rel < n_rel; ++rel) {
        if (rel > 0 && (rel & 3) == 0) {
          g_cur = g_nxt;
          g_nxt = load_ids4((rel >> 2) + 1);
        }
        const int e = 2 * rel + (is_v ? 1 : 0);
        const int st = ring_slot(e);
        if (e >= kRing && !warp_wait(smem_u32(&sh->kv_empty[st]), ring_phase(e - kRing), abort,
                                     a.err, wlim))
          break;
        int lead, tail;
        const bool edge = is_v && v_edges(rel, lead, tail);
        if (!(!is_v && rel == 0 && withhold_k0))
          issue_tile(j0 + rel, g_cur, rel & 3, is_v, smem_u32(sKV + st * Lt::kTileBytes),
                     smem_u32(edge ? &sh->kv_land[st] : &sh->kv_full[st]));
        n_issued = rel + 1;
        if (lane == 0) TC_MARK((is_v ? 200 : 100) + (rel & 63));
        if (edge) {   // landed, edge rows zeroed, then full
          pending_land = st;
          pending_e = e;
          if (!warp_wait(smem_u32(&sh->kv_land[st]), (land_phase >> st) & 1u, abort, a.err, wlim))
            break;
          pending_land = -1;
          land_phase ^= 1u << st;
          zero_v_rows<D>(sKV + st * Lt::kTileBytes, lead, tail, 0, kTcKeys, lane);
          fence_proxy_async();   // generic writes, then the tensor core reads
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sh->kv_full[st]));
        }
      }
      // An edge tile whose landing wait gave up is still in flight on
      // kv_land; the other tiles' copies complete on kv_full.
      if (pending_land >= 0 && lane == 0)
        (void)mbar_wait(smem_u32(&sh->kv_land[pending_land]), (land_phase >> pending_land) & 1u);
      if (lane == 0) sh->n_issued[is_v ? 1 : 0] = n_issued;
      named_barrier(3, 64);   // warps 8 and 10: both counts final
      drain(is_v ? 0 : n_issued, is_v ? n_issued : 0, sh->n_issued[0], sh->n_issued[1], false,
            pending_land >= 0 ? pending_e : (withhold_k0 && !is_v ? 0 : -1));
    } else {
      // one warp, ring elements in order: K(0), V(0), K(1), ...
      int k_issued = 0, v_issued = 0;
      for (int e = 0; e < 2 * n_rel; ++e) {
        const int rel = e >> 1;
        const bool is_v = (e & 1) != 0;
        if (!is_v && rel > 0 && (rel & 3) == 0) {
          g_cur = g_nxt;
          g_nxt = load_ids4((rel >> 2) + 1);
        }
        const int st = ring_slot(e);
        if (e >= kRing && !warp_wait(smem_u32(&sh->kv_empty[st]), ring_phase(e - kRing), abort,
                                     a.err, wlim))
          break;
        // (the codes land on kv_land; warps 10 and 11 widen them, then kv_full)
        if (!(e == 0 && withhold_k0))
          issue_tile(j0 + rel, g_cur, rel & 3, is_v, smem_u32(sKV + st * Lt::kTileBytes),
                     smem_u32(&sh->kv_land[st]));
        (is_v ? v_issued : k_issued) = rel + 1;
        if (lane == 0) TC_MARK((is_v ? 200 : 100) + (rel & 63));
      }
      drain(k_issued, v_issued, k_issued, v_issued, true, withhold_k0 ? 0 : -1);
    }
    if (warp == 8 && lane == 0) (void)mbar_wait(q_full, 0);   // the query tiles too
    __syncwarp();
   } else if (FP8 && (warp == 10 || (D == 128 && warp == 11))) {
    // ------------------------------------------------- widen e4m3 tiles (FP8)
    // Ring elements in order, so that each wait on a slot's kv_land is for
    // the phase after the last one this warp saw there.  D = 128: warp 10
    // widens rows 0-63 and warp 11 rows 64-127 of every tile.  D = 64: the
    // in-place widening overwrites later rows' codes with earlier rows' fp16
    // (it runs from the last rows to the first), so warp 10 takes whole tiles.
    const int r0 = D == 128 ? 64 * (warp - 10) : 0;
    const int r1 = D == 128 ? r0 + 64 : kTcKeys;
    for (int e = 0; e < 2 * n_rel; ++e) {
      const int st = ring_slot(e);
      if (!warp_wait(smem_u32(&sh->kv_land[st]), ring_phase(e), abort, a.err, wlim)) break;
      uint8_t* tile = sKV + st * Lt::kTileBytes;
      if constexpr (D == 128)
        widen_tile_fp8(tile, lane, r0 / 16, r1 / 16);
      else
        widen_tile_fp8_d64(tile, lane);
      int lead, tail;
      if ((e & 1) && v_edges(e >> 1, lead, tail)) {
        __syncwarp();
        zero_v_rows<D>(tile, lead, tail, r0, r1, lane);
      }
      fence_proxy_async();   // generic writes, then the tensor core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->kv_full[st]));
    }
   }
  } else {
    // ------------------------------------------------------------ softmax
    set_max_regs_inc_softmax();
    const int t = warp >> 2;                      // query tile of this warpgroup
    const int quarter = warp & 3;                 // TMEM lanes this warp may touch
    const int row = quarter * 32 + lane;          // tile row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int tok = tok0 + t * tile_toks + row / G;
    const int g = row % G;
    const bool valid = tok <= tok_last;
    const int pos = casc ? L - 1 : L - qn + (valid ? tok : tok_last);
    const uint32_t b_sfull = smem_u32(&sh->s_full[t]);
    const uint32_t b_pfull = smem_u32(&sh->p_full[t]), b_pvdone = smem_u32(&sh->pv_done[t]);
    const uint32_t tS = tmem + lane_off + col_s(t), tP = tmem + lane_off + col_p(t);
    const uint32_t tO = tmem + lane_off + col_o(t);
    float sl2 = a.scale_log2;
    float out_scale = 1.f;
    if constexpr (FP8) {
      // descales of this (sequence, kv head) -- a cascade prefix row's own
      // sequence (rows are the batch's query tokens); this thread's Q row to
      // fp16
      const int ds =
          casc ? max(seq_of_row(a.query_start_loc, a.casc_seqs, valid ? tok : tok_last), 0) : s;
      sl2 *= __ldg(a.k_descale + static_cast<int64_t>(ds) * a.num_kv_heads + kvh);
      out_scale = __ldg(a.v_descale + static_cast<int64_t>(ds) * a.num_kv_heads + kvh);
      bool qok = warp_wait(q_full, 0, abort, a.err, wlim);
      if (qok) {
        uint8_t* qrow = sQ + t * Lt::kQTile + row * 128;
        uint4 v[2 * 8];
        float amax = 0.f;
#pragma unroll
        for (int h = 0; h < Lt::kHalves; ++h)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            v[h * 8 + j] = *reinterpret_cast<const uint4*>(qrow + h * Lt::kQHalf + ((j ^ (row & 7)) << 4));
            const uint32_t w[4] = {v[h * 8 + j].x, v[h * 8 + j].y, v[h * 8 + j].z, v[h * 8 + j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
          }
        const int ex = f16_row_exponent(amax);
        const float down = pow2f(-ex);
        sl2 *= pow2f(ex);
#pragma unroll
        for (int h = 0; h < Lt::kHalves; ++h)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 u = v[h * 8 + j];
            *reinterpret_cast<uint4*>(qrow + h * Lt::kQHalf + ((j ^ (row & 7)) << 4)) =
                make_uint4(bf16x2_to_f16x2(u.x, down), bf16x2_to_f16x2(u.y, down),
                           bf16x2_to_f16x2(u.z, down), bf16x2_to_f16x2(u.w, down));
          }
        fence_proxy_async();   // generic writes, then the tensor core reads
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->q_conv));
    }
    float m_used = -INFINITY, l = 0.f;
    bool done = t < ntq;
    // first key this row sees (its window; after the shared prefix in a
    // cascade suffix launch)
    const int lo = max(a.window > 0 ? pos - a.window + 1 : 0, a.key_begin);
    // Thread 0 of the warpgroup issues its tile's MMAs.  Handing them to
    // a separate MMA warp costs a wake-up per product, and that warp, sharing
    // its SM sub-partition with two softmax warps that have instructions ready
    // most of the time, gets few issue slots (measured on GB300: an issuing
    // thread beside one FMA-bound warp gets an MMA out every ~240 cycles
    // instead of 64).  Per tile the order is S(0), P(0) V, S(1), P(1) V, ...:
    // S(j + 1) overwrites the columns P(j) lives in, and one thread's MMAs
    // execute in issue order.
    // The two tiles' issuers take turns -- S0(0), S1(0), then groups
    // [P0(j) V, S0(j + 1)], [P1(j) V, S1(j + 1)], ... -- so that each tile's
    // softmax runs while the tensor core works on the other tile's products
    // (left to themselves the two tiles fall into step and their softmaxes
    // contend).  issued[t] completes one phase per group tile t has issued,
    // its S(0) being phase 0; a turn waits for the other tile's previous
    // group, which cannot run two phases ahead of the waiter.
    // (tile t's issuer sits on SM sub-partition t, apart from the other tile's)
    const bool issuer = done && quarter == t && lane == 0;
    const bool paired = ntq > 1;
    const uint32_t my_issued = smem_u32(&sh->issued[t]);
    const uint32_t other_issued = smem_u32(&sh->issued[t ^ 1]);
    if (issuer) {
      if (wait_or_abort(q_ready, 0, abort, a.err, wlim) &&
          wait_or_abort(smem_u32(&sh->kv_full[ring_slot(0)]), ring_phase(0), abort, a.err, wlim) &&
          (t == 0 || wait_or_abort(other_issued, 0, abort, a.err, wlim))) {
        tc::fence_after_sync();
        TC_MARK(300 + 64 * t);
        issue_s(t, 0);
        tc::commit(smem_u32(&sh->kv_empty[ring_slot(0)]));
        mbar_arrive(my_issued);
      }
    }
    __syncwarp();
    for (int j = 0; done && j < n_rel; ++j) {
      // S_t(j) complete (its commit also covers P_t(j - 1) V, so O_t is stable)
      if (!warp_wait(b_sfull, j & 1, abort, a.err, wlim)) { done = false; break; }
      tc::fence_after_sync();
      if (quarter == 0 && lane == 0) TC_MARK(700 + 64 * t + (j & 63));
      if (t == 0 && quarter > 0 && lane == 0 && j < 32) TC_MARK(1030 + 32 * (quarter - 1) + j);
      float x[kTcKeys];
#pragma unroll
      for (int c0 = 0; c0 < kTcKeys; c0 += 32) {
        uint32_t r[32];
        tc::ld32(tS + c0, r);
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c0 + c] = __uint_as_float(r[c]);
      }
      tc::wait_ld();
      // causal mask on raw scores (also hides keys >= L); scale > 0, so the
      // row max of the raw scores gives the max of the scaled ones
      const int key0 = (j0 + j) * kTcKeys;
      // (warp-uniform branches: the votes below need every lane)
      if (__any_sync(0xffffffffu, key0 + kTcKeys - 1 > pos || key0 < lo)) {
        // visible columns [nlo, nvis) of this row (rows that see the whole
        // tile keep every column); one compare per element where no row of
        // the warp has a lower bound in this tile
        const int nvis = pos - key0 + 1;
        const int nlo = lo - key0;
        if (__any_sync(0xffffffffu, nlo > 0)) {
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c)
            x[c] = (c < nvis && c >= nlo) ? x[c] : -INFINITY;
        } else {
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c) x[c] = c < nvis ? x[c] : -INFINITY;
        }
      }
      // row max: four independent chains of three-input maxima
      float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int c = 4; c < kTcKeys - 4; c += 8) {
        m4[0] = tc::max3(m4[0], x[c], x[c + 1]);
        m4[1] = tc::max3(m4[1], x[c + 2], x[c + 3]);
        m4[2] = tc::max3(m4[2], x[c + 4], x[c + 5]);
        m4[3] = tc::max3(m4[3], x[c + 6], x[c + 7]);
      }
      m4[0] = tc::max3(m4[0], x[kTcKeys - 4], x[kTcKeys - 3]);
      m4[1] = tc::max3(m4[1], x[kTcKeys - 2], x[kTcKeys - 1]);
      const float mt = tc::max3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;
      float alpha = 1.f;
      if (mt > m_used + kLazyRescale) {
        alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - mt);
        m_used = mt;
      }
      const float neg_mu = (m_used == -INFINITY) ? 0.f : -m_used;
      const uint64_t m2 = tc::pack_f32x2(sl2, sl2), b2 = tc::pack_f32x2(neg_mu, neg_mu);
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {   // rescale O in TMEM
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tc::ld32(tO + c0, o);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tc::st32(tO + c0, o);
        }
      }
      // P = 2^(s * scale*log2(e) - max): packed FMA, MUFU ex2, bf16 pairs
      // written over S's first 64 columns; the row sum adds the fp32 weights
      uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
      for (int c0 = 0; c0 < kTcKeys / 2; c0 += 32) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int k = 2 * (c0 + c);
          float y0, y1;
          tc::fma_f32x2(x[k], x[k + 1], m2, b2, y0, y1);
          y0 = ex2(y0);
          y1 = ex2(y1);
          pk[c] = pack2<FP8>(y0, y1);
          tc::add_f32x2(acc[c & 3], y0, y1);
        }
        tc::st32(tP + c0, pk);
      }
      const float ls = (tc::sum_f32x2(acc[0]) + tc::sum_f32x2(acc[1])) +
                       (tc::sum_f32x2(acc[2]) + tc::sum_f32x2(acc[3]));
      l = l * alpha + ls;
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull);
      if (quarter == 0 && lane == 0) TC_MARK(900 + 64 * t + (j & 63));
      if (t == 0 && lane == 0) TC_MARK(1700 + 64 * quarter + (j & 63));
      if (issuer) {
        // (a failed wait leaves the other warps to give up on s_full)
        // this tile's group j: after the other tile's group j - 1 (tile 0)
        // or group j (tile 1), i.e. the other barrier's phase j or j + 1
        bool go = wait_or_abort(b_pfull, j & 1, abort, a.err, wlim);
        if (go) TC_MARK(1528 + 64 * t + (j & 63));
        go = go && wait_or_abort(smem_u32(&sh->kv_full[ring_slot(2 * j + 1)]),
                                 ring_phase(2 * j + 1), abort, a.err, wlim);
        if (go) TC_MARK(1400 + 64 * t + (j & 63));
        if (go && (!paired || wait_or_abort(other_issued, (j + t) & 1, abort, a.err, wlim))) {
          tc::fence_after_sync();
          TC_MARK(500 + 64 * t + (j & 63));
          issue_pv(t, j);
          tc::commit(smem_u32(&sh->kv_empty[ring_slot(2 * j + 1)]));
          const int jn = j + 1;
          if (jn < n_rel && wait_or_abort(smem_u32(&sh->kv_full[ring_slot(2 * jn)]),
                                          ring_phase(2 * jn), abort, a.err, wlim)) {
            tc::fence_after_sync();
            TC_MARK(300 + 64 * t + (jn & 63));
            issue_s(t, jn);
            tc::commit(smem_u32(&sh->kv_empty[ring_slot(2 * jn)]));
          }
          mbar_arrive(my_issued);
        }
      }
      __syncwarp();
    }
    if (issuer) {   // every MMA this thread issued completes before TMEM is freed
      tc::commit(smem_u32(&sh->drain[t]));
      (void)mbar_wait(smem_u32(&sh->drain[t]), 0);
    }
    __syncwarp();
    if (casc || a.key_begin > 0) {
      if (done && warp_wait(b_pvdone, (n_rel - 1) & 1, abort, a.err, wlim)) {
        // cascade prefix (split blockIdx.z) or suffix (split split_base): the
        // row's normalised partial and log2-sum-exp (in the scaled log2 domain
        // of m_used) for the merge
        tc::fence_after_sync();
        const float inv = l > 0.f ? out_scale / l : 0.f;
        const int64_t wrow = (static_cast<int64_t>(q0 + tok) * Hq + kvh * G + g) * a.max_splits +
                             (casc ? static_cast<int>(blockIdx.z) : a.split_base);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tc::ld32(tO + c0, o);
          tc::wait_ld();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(a.ws_o + wrow * D + c0);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                   __uint_as_float(o[4 * v + 2]) * inv,
                                   __uint_as_float(o[4 * v + 3]) * inv);
          }
        }
        if (valid) a.ws_lse[wrow] = l > 0.f ? m_used + log2f(l) : -INFINITY;
      }
    } else if (t < ntq) {
      const bool ok = done && warp_wait(b_pvdone, (n_rel - 1) & 1, abort, a.err, wlim);
      // every row of the tile is a query row of this sequence
      const bool full_tile = tok0 + (t + 1) * tile_toks - 1 <= tok_last;
      float inv = 0.f;
      uint32_t o[D];   // the whole O row: every load in flight before one wait
      if (ok) {
        tc::fence_after_sync();
        if (quarter == 0 && lane == 0) TC_MARK(1300 + t);
        inv = l > 0.f ? out_scale / l : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32)
          tc::ld32(tO + c0, *reinterpret_cast<uint32_t(*)[32]>(o + c0));
        tc::wait_ld();
      }
      if (full_tile) {
        // The rows go out through the tile's Q slot (its products have all
        // completed: pv_done's last phase covers every MMA of the tile), in
        // the swizzled layout Q arrived in, then one TMA store per 64-column
        // half -- a row per thread written straight to memory would make
        // every store instruction touch 32 rows.
        uint8_t* srow = sQ + t * Lt::kQTile + row * 128;
        if (ok) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 8) {
            uint32_t w[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
              w[c] = pack_bf16(__uint_as_float(o[c0 + 2 * c]) * inv,
                               __uint_as_float(o[c0 + 2 * c + 1]) * inv);
            const int h = c0 / 64, j = (c0 % 64) / 8;
            *reinterpret_cast<uint4*>(srow + h * Lt::kQHalf + ((j ^ (row & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async();   // generic writes, then the TMA engine reads
        }
        // the tile's four warps (named barrier 1 + t); no store unless all wrote
        const bool all = named_barrier_and(1 + t, 128, ok);
        if (all && quarter == 0 && lane == 0) {
#pragma unroll
          for (int h = 0; h < Lt::kHalves; ++h)
            tma_store_3d(&omap, smem_u32(sQ + t * Lt::kQTile + h * Lt::kQHalf), h * 64, kvh * G,
                         q0 + tok0 + t * tile_toks);
          bulk_commit_group();
          bulk_wait_group_read0();   // shared memory stays until the reads are done
        }
      } else if (ok && valid) {
        __nv_bfloat16* orow = out + (static_cast<int64_t>(q0 + tok) * Hq + kvh * G + g) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 8) {
          uint32_t w[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            w[c] = pack_bf16(__uint_as_float(o[c0 + 2 * c]) * inv,
                             __uint_as_float(o[c0 + 2 * c + 1]) * inv);
          *reinterpret_cast<uint4*>(orow + c0) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  TC_MARK(1);
#ifdef PKV_TC_TIMELINE
  if (threadIdx.x == 0 && cta_lin < 600) g_tc_timeline[2048 + 3 * cta_lin + 2] = global_timer_ns();
#endif
  if (warp == 9) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}

#ifdef PKV_TC_TIMELINE
}  // namespace
extern "C" int pkv_tc_timeline(unsigned long long* host, int n) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_tc_timeline,
                                               sizeof(unsigned long long) * (n < 4096 ? n : 4096)));
}
extern "C" int pkv_tc_timeline_clear() {
  static unsigned long long zeros[4096];
  return static_cast<int>(cudaMemcpyToSymbol(g_tc_timeline, zeros, sizeof(zeros)));
}
namespace {
#endif

template <int D, bool FP8>
cudaError_t launch_tc_t(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        const CUtensorMap& omap, const PrefillArgs& a, cudaStream_t stream) {
  constexpr int smem = tc_smem_bytes<D>();
  const bool lpt = a.longest_first && !a.cascade_prefix &&
                   static_cast<int64_t>(a.num_seqs) * a.num_mtiles <= kLptUnits;
  auto kfn = lpt ? pkv_prefill_tc_kernel<D, FP8, true> : pkv_prefill_tc_kernel<D, FP8, false>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // cascade prefix: grid.z = prefix key splits
  const int gz = a.cascade_prefix ? (a.prefix_len + a.prefix_tiles * kTcKeys - 1) /
                                        (a.prefix_tiles * kTcKeys)
                                  : a.num_seqs;
  dim3 grid(a.num_mtiles, a.num_kv_heads, gz);
  PrefillArgs b = a;
  debug_wait_settings(&b.wait_limit_ns, &b.debug_stall);
  kfn<<<grid, kTcThreads, smem, stream>>>(qmap, kmap, vmap, omap, b);
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
                              const CUtensorMap& vmap, const CUtensorMap& omap,
                              const PrefillArgs& a, int head_size, bool fp8, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_mtiles == 0) return cudaSuccess;
  if (fp8)
    return head_size == 128 ? launch_tc_t<128, true>(qmap, kmap, vmap, omap, a, stream)
                            : launch_tc_t<64, true>(qmap, kmap, vmap, omap, a, stream);
  if (head_size == 128) return launch_tc_t<128, false>(qmap, kmap, vmap, omap, a, stream);
  return launch_tc_t<64, false>(qmap, kmap, vmap, omap, a, stream);
}

}  // namespace pkv
