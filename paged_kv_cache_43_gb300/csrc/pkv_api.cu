// pkv_api.cu -- the C ABI of include/pkv.h: host-side argument checks, the
// split-K plan, TMA descriptor encoding and kernel dispatch.
//
// Nothing here allocates device memory or synchronises, except
// pkv_get_error(), which is documented as synchronising.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Per-device error word (PKV_ERR_* bits), OR-ed by the kernels.
__device__ int32_t g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per device: the stream that a mixed batch's prefill launch (and a cascade
// call's shared-prefix launch) runs on while the decode launches run on the
// caller's stream, created once at the device's greatest priority (so that
// the block scheduler hands freed SMs to the tensor-core tiles first and the
// short decode CTAs fill their tail), and the events that fork it from the
// caller's stream and join it back.  `mu`
// keeps the record-wait-launch-record-wait sequence of one call from
// interleaving with another thread's.  side == nullptr: not available (the
// launches then stay on the caller's stream).
struct SideStream {
  std::mutex mu;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream g_side[kMaxDevices];

// The CUDA error behind the most recent PKV_E_CUDA (process-wide).
std::atomic<int> g_last_cuda_error{0};

int cuda_fail(cudaError_t e) {
  g_last_cuda_error.store(static_cast<int>(e));
  return PKV_E_CUDA;
}

// Returns PKV_E_CUDA from the enclosing function when a CUDA call fails.
#define PKV_TRY(expr)                                   \
  do {                                                  \
    const cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_);        \
  } while (0)

void make_side_stream(SideStream* s) {
  int least = 0, greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return;
  cudaStream_t st = nullptr;
  cudaEvent_t f = nullptr, j = nullptr;
  if (cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, greatest) == cudaSuccess &&
      cudaEventCreateWithFlags(&f, cudaEventDisableTiming) == cudaSuccess &&
      cudaEventCreateWithFlags(&j, cudaEventDisableTiming) == cudaSuccess) {
    s->side = st;
    s->fork = f;
    s->join = j;
    return;
  }
  if (j) cudaEventDestroy(j);
  if (f) cudaEventDestroy(f);
  if (st) cudaStreamDestroy(st);
  cudaGetLastError();
}

// Device-side address of the error word and the SM count, once per device
// (with the device's side stream).
int device_state(int32_t** err, int* num_sms, int* device = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_E_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    PKV_TRY(cudaGetSymbolAddress(&p, g_error_word));
    int sms = 0;
    PKV_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    make_side_stream(&g_side[dev]);
    g_err_ptr[dev] = static_cast<int32_t*>(p);
    g_num_sms[dev] = sms;
  }
  *err = g_err_ptr[dev];
  *num_sms = g_num_sms[dev];
  if (device) *device = dev;
  return PKV_OK;
}

// Whether work may be forked from `st` onto the side stream: the side stream
// is idle (not part of any capture), or it already belongs to the capture
// that `st` is in.  A side stream held by another thread's capture is left
// alone.
bool side_usable(cudaStream_t side, cudaStream_t st) {
  cudaStreamCaptureStatus ss = cudaStreamCaptureStatusNone, cs = cudaStreamCaptureStatusNone;
  unsigned long long sid = 0, cid = 0;
  if (cudaStreamGetCaptureInfo(side, &ss, &sid) != cudaSuccess ||
      cudaStreamGetCaptureInfo(st, &cs, &cid) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (ss == cudaStreamCaptureStatusNone) return cs != cudaStreamCaptureStatusInvalidated;
  return ss == cudaStreamCaptureStatusActive && cs == cudaStreamCaptureStatusActive && sid == cid;
}

// Fork-join around the device's side stream.  begin() makes the side stream
// wait for the work already on `st` and holds the side stream's lock;
// stream() is then where the forked launches go (the side stream, or `st`
// itself when the side stream is missing or held by another capture); join()
// makes `st` wait for them.  The destructor joins too (error paths), so a
// capture on `st` never ends with unjoined work.
class SideFork {
 public:
  SideFork(int dev, cudaStream_t st) : ss_(g_side[dev]), st_(st), pst_(st) {}
  SideFork(const SideFork&) = delete;
  SideFork& operator=(const SideFork&) = delete;
  ~SideFork() { (void)join(); }
  int begin() {
    if (ss_.side == nullptr) return PKV_OK;
    lock_ = std::unique_lock<std::mutex>(ss_.mu);
    if (!side_usable(ss_.side, st_)) return PKV_OK;
    PKV_TRY(cudaEventRecord(ss_.fork, st_));
    PKV_TRY(cudaStreamWaitEvent(ss_.side, ss_.fork, 0));
    pst_ = ss_.side;
    return PKV_OK;
  }
  cudaStream_t stream() const { return pst_; }
  int join() {
    if (pst_ == st_) return PKV_OK;
    pst_ = st_;
    cudaError_t e = cudaEventRecord(ss_.join, ss_.side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st_, ss_.join, 0);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
  }

 private:
  SideStream& ss_;
  cudaStream_t st_, pst_;
  std::unique_lock<std::mutex> lock_;
};

int encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr)
      return PKV_E_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  *fn = g_encode;
  return PKV_OK;
}

// TMA descriptor of one cache viewed as a 3-D tensor
// (head_size, num_kv_heads, num_blocks * 16).  bf16: a box of 64 columns x 1
// head x 16 rows (one cache block of one head, 128 bytes wide) with the
// 128-byte swizzle.  FP8 (e4m3 codes as bytes): a box of the whole head row x
// 1 head x 16 rows with the swizzle of the row's width (128 or 64 bytes), which
// keeps the kernels' per-lane fragment reads free of bank conflicts.
// The L2 fill size is capped at one head row (64, 128 or 256 bytes): a wider
// fill would pull the neighbouring kv head's row, which another CTA reads at
// some other time, and double the DRAM traffic of narrow rows.
int encode_cache_map(CUtensorMap* map, const void* base, const pkv_cache_desc& c) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  if (int st = encode_fn(&fn)) return st;
  const bool fp8 = c.dtype == PKV_FP8_E4M3;
  const cuuint64_t eb = fp8 ? 1 : 2;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(c.head_size) * eb;
  const CUtensorMapL2promotion promo =
      row_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                       : (row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                           : CU_TENSOR_MAP_L2_PROMOTION_L2_64B);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(c.head_size),
                              static_cast<cuuint64_t>(c.num_kv_heads),
                              static_cast<cuuint64_t>(c.num_blocks) * c.block_size};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(c.head_size) * eb,
                                 static_cast<cuuint64_t>(c.num_kv_heads) * c.head_size * eb};
  const cuuint32_t box[3] = {fp8 ? static_cast<cuuint32_t>(c.head_size) : 64u, 1,
                             static_cast<cuuint32_t>(c.block_size)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  (fp8 && row_bytes == 64) ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_128B,
                  promo,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_E_CUDA;
}

// TMA descriptor of the bf16 query tensor [num_tokens, num_q_heads, D] viewed
// as (D, Hq, T) with a box of 64 columns x `group` heads x 128/group tokens:
// one box is the 128-row (token, head) tile of one kv head, 128 bytes wide.
int encode_query_map(CUtensorMap* map, const void* q, int num_tokens, int num_q_heads,
                     int head_size, int group) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  if (int st = encode_fn(&fn)) return st;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_size),
                              static_cast<cuuint64_t>(num_q_heads),
                              static_cast<cuuint64_t>(num_tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_size) * 2,
                                 static_cast<cuuint64_t>(num_q_heads) * head_size * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group),
                             static_cast<cuuint32_t>(prefill_tc_tokens_per_tile(group))};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_E_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cache(const pkv_cache_desc* c) {
  if (c == nullptr) return PKV_E_NULL;
  if (c->dtype != PKV_F32 && c->dtype != PKV_BF16 && c->dtype != PKV_FP8_E4M3) return PKV_E_DTYPE;
  if (c->block_size != kBlock) return PKV_E_SHAPE;
  if (c->head_size != 64 && c->head_size != 128) return PKV_E_SHAPE;
  if (c->num_kv_heads < 1 || c->num_blocks < 0) return PKV_E_SHAPE;
  // TMA coordinates of cache rows are int32.
  if (static_cast<int64_t>(c->num_blocks) * c->block_size > INT32_MAX) return PKV_E_SHAPE;
  return PKV_OK;
}

// How the batch is cut: decode run, prefill rest, split-K chunk.
struct Plan {
  int num_decode = 0;     // sequences [0, num_decode) go to the decode kernel
  int split_blocks = 0;   // cache blocks per decode split
  int max_splits = 0;
  size_t ws_o_bytes = 0;  // fp32 partial outputs
  size_t ws_bytes = 0;    // total workspace
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_meta(const pkv_cache_desc* c, const pkv_attn_meta* m) {
  if (m == nullptr) return PKV_E_NULL;
  if (m->num_seqs < 0 || m->num_tokens < 0 || m->max_query_len < 0 || m->max_context_len < 0 ||
      m->block_table_stride < 1)
    return PKV_E_META;
  if (m->num_q_heads < 1 || m->num_q_heads % c->num_kv_heads != 0) return PKV_E_GQA;
  if (m->num_q_heads > 65535) return PKV_E_SHAPE;
  if (m->num_decode_seqs < -1 || m->num_decode_seqs > m->num_seqs) return PKV_E_META;
  if (m->sliding_window < 0) return PKV_E_META;
  if (m->kv_split_tokens != 0 &&
      (m->kv_split_tokens < 64 || m->kv_split_tokens > 2048 || m->kv_split_tokens % 64 != 0))
    return PKV_E_META;
  return PKV_OK;
}

// Cache blocks per decode split (CTA).  Measured on GB300 decode batches: 1024
// keys (512 KB of K+V per kv head at D=128) by default; 2048 for long contexts
// (>= 16K keys), which halves the split partials and the CTAs that find
// nothing to do; shorter chunks only while the batch would have fewer CTAs
// than SMs.  A CTA's fixed costs (barriers, Q, the first TMA round trip, its
// partial and the merge's read of it) outweigh more parallelism well before
// the GPU is full twice over: 2 sequences x 8 kv heads x 32K keys run in 51 us
// with 2048-key splits against 65 us with 512-key ones, 4 x 32 heads x 4K keys
// in 46 against 49 us, 8 x 8 kv heads x 2K keys in 23 against 25 us.
// `max_blocks`: blocks the longest row reads; `units`: (sequence, kv head,
// 8-head group) triples.
// Then the longest row's splits are evened out: their number is its blocks
// over that size rounded to nearest rather than up, each ceil(blocks / n)
// long and at most 128 (the kernel's 32 blocks per warp).  A 1024-key window
// spans 65 blocks: one split of 65, not 64 + 1, which would also cost a
// merge pass (measured with 1024-key windows: 146 -> 141 us on the
// 64 x 32-head batch, 112 -> 104 us on 256 x 8 kv heads, 27 -> 20 us on
// 16 x 8 kv heads).
int choose_split_blocks(int max_blocks, int64_t units, int num_sms, int kv_split_tokens) {
  if (kv_split_tokens > 0) return kv_split_tokens / kBlock;
  auto ctas = [&](int sb) { return units * ((max_blocks + sb - 1) / sb); };
  int split_blocks = 64;
  if (max_blocks * kBlock >= 16384 && ctas(128) >= num_sms) split_blocks = 128;
  while (split_blocks > 4 && ctas(split_blocks) < num_sms) split_blocks /= 2;
  if (max_blocks > 0) {
    constexpr int kMaxSplitBlocks = 128;
    int n = (max_blocks + split_blocks / 2) / split_blocks;
    n = std::max(n, (max_blocks + kMaxSplitBlocks - 1) / kMaxSplitBlocks);
    n = std::max(n, 1);
    split_blocks = (max_blocks + n - 1) / n;
  }
  return split_blocks;
}

int make_plan(const pkv_cache_desc* c, const pkv_attn_meta* m, int num_sms, Plan* p) {
  if (int st = check_cache(c)) return st;
  if (int st = check_meta(c, m)) return st;
  *p = Plan{};
  if (c->dtype == PKV_F32) return PKV_OK;  // one kernel, no workspace
  int nd = 0;
  if (m->max_query_len <= 1) nd = m->num_seqs;
  else if (m->num_decode_seqs >= 0) nd = m->num_decode_seqs;
  p->num_decode = nd;
  if (nd == 0) return PKV_OK;
  // Blocks a decode query may read: the whole context, or the window's span
  // (which can straddle one block boundary more than W / 16 blocks do).
  int max_blocks = (m->max_context_len + kBlock - 1) / kBlock;
  if (m->sliding_window > 0) {
    const int wb = (m->sliding_window + kBlock - 1) / kBlock + 1;
    if (wb < max_blocks) max_blocks = wb;
  }
  const int g_sub = (m->num_q_heads / c->num_kv_heads + 7) / 8;
  const int split_blocks = choose_split_blocks(
      max_blocks, static_cast<int64_t>(nd) * c->num_kv_heads * g_sub, num_sms, m->kv_split_tokens);
  p->split_blocks = split_blocks;
  p->max_splits = max_blocks > 0 ? (max_blocks + split_blocks - 1) / split_blocks : 1;
  if (p->max_splits > 1) {
    const size_t rows = static_cast<size_t>(nd) * m->num_q_heads * p->max_splits;
    p->ws_o_bytes = round_up(rows * c->head_size * sizeof(float), 256);
    p->ws_bytes = p->ws_o_bytes + round_up(rows * sizeof(float), 256);
  }
  return PKV_OK;
}

// Cascade attention over a decode batch whose sequences share their first
// P = common_prefix_blocks blocks: a prefix launch (every row against the
// shared keys, P blocks cut into prefix_splits chunks), a suffix launch (each
// row against its own keys after the prefix, the usual splits) and the
// combine, which merges prefix and suffix partials.  Workspace rows hold
// prefix_splits + suffix_max_splits partials.
struct CascadePlan {
  bool tc_prefix = false;    // shared keys on the tcgen05 kernel (G divides 128)
  int prefix_tiles = 0;      // tcgen05 prefix: 128-key tiles per CTA
  int prefix_mtiles = 0;     // tcgen05 prefix: query-row tiles
  int prefix_blocks = 0;
  int prefix_split_blocks = 0;
  int prefix_splits = 0;
  int num_decode = 0;        // leading decode sequences (one query row each)
  int rows = 0;              // query rows of the prefix launch (tokens)
  int col_groups = 0;        // 8-column groups of (sequence, q head in group) per kv head
  int split_blocks = 0;      // suffix split size
  int max_splits = 0;        // prefix_splits + the longest suffix's splits
  size_t ws_o_bytes = 0;
  size_t ws_bytes = 0;
};

int make_cascade_plan(const pkv_cache_desc* c, const pkv_attn_meta* m, int32_t prefix_blocks,
                      int num_sms, CascadePlan* p) {
  if (int st = check_cache(c)) return st;
  if (c->dtype != PKV_BF16 && c->dtype != PKV_FP8_E4M3) return PKV_E_DTYPE;
  if (int st = check_meta(c, m)) return st;
  // no window, and a prefix that every query follows; chunked-prefill rows
  // after num_decode_seqs decode sequences
  const bool chunks = m->max_query_len > 1;
  if (m->sliding_window != 0 || prefix_blocks < 1 || prefix_blocks > m->block_table_stride ||
      static_cast<int64_t>(prefix_blocks) * kBlock >= m->max_context_len ||
      (chunks && (m->num_decode_seqs < 0 || m->num_decode_seqs > m->num_seqs)))
    return PKV_E_META;
  *p = CascadePlan{};
  p->prefix_blocks = prefix_blocks;
  const int G = m->num_q_heads / c->num_kv_heads;
  // chunk rows: the shared keys and each chunk's own keys both on the tcgen05
  // kernel (group sizes dividing 128)
  if (chunks && !prefill_tc_supported(c->head_size, G)) return PKV_E_SHAPE;
  p->num_decode = chunks ? m->num_decode_seqs : m->num_seqs;
  p->rows = chunks ? m->num_tokens : m->num_seqs;
  p->col_groups = static_cast<int>((static_cast<int64_t>(m->num_seqs) * G + 7) / 8);
  // e4m3 caches: the shared keys only on the widening tcgen05 kernel
  if (c->dtype == PKV_FP8_E4M3 && !prefill_tc_supported(c->head_size, G)) return PKV_E_SHAPE;
  if (prefill_tc_supported(c->head_size, G)) {
    // tcgen05: all decode rows of a kv head in 128-row tiles, at least two
    // 128-key tiles per CTA, about half the SMs (their partials are merged)
    p->tc_prefix = true;
    const int per_cta = prefill_tc_tokens_per_cta(G);
    p->prefix_mtiles = (p->rows + per_cta - 1) / per_cta;
    const int ktiles = (prefix_blocks * kBlock + 127) / 128;
    const int64_t units = static_cast<int64_t>(p->prefix_mtiles) * c->num_kv_heads;
    int tiles = static_cast<int>((ktiles * units + num_sms / 2 - 1) / (num_sms / 2));
    tiles = tiles < 2 ? 2 : (tiles > ktiles ? ktiles : tiles);
    p->prefix_tiles = tiles;
    p->prefix_splits = (ktiles + tiles - 1) / tiles;
  } else {
    // mma.sync decode kernel over 8 (sequence, head) columns per CTA: 1024-key
    // chunks, shorter while the launch would not fill the GPU twice
    const int64_t prefix_units = static_cast<int64_t>(c->num_kv_heads) * p->col_groups;
    int psb = 64;
    while (psb > 4 && prefix_units * ((prefix_blocks + psb - 1) / psb) < 4LL * num_sms) psb /= 2;
    p->prefix_split_blocks = psb;
    p->prefix_splits = (prefix_blocks + psb - 1) / psb;
  }
  const int suffix_blocks = (m->max_context_len + kBlock - 1) / kBlock - prefix_blocks;
  const int g_sub = (G + 7) / 8;
  p->split_blocks = choose_split_blocks(
      suffix_blocks, static_cast<int64_t>(std::max(p->num_decode, 1)) * c->num_kv_heads * g_sub,
      num_sms, m->kv_split_tokens);
  // decode rows: the longest suffix's splits; chunk rows: one suffix partial
  p->max_splits = p->prefix_splits + (suffix_blocks + p->split_blocks - 1) / p->split_blocks;
  const size_t rows = static_cast<size_t>(p->rows) * m->num_q_heads * p->max_splits;
  p->ws_o_bytes = round_up(rows * c->head_size * sizeof(float), 256);
  p->ws_bytes = p->ws_o_bytes + round_up(rows * sizeof(float), 256);
  return PKV_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int attention_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens,
                   const int32_t* query_start_loc, float scale, const float* k_descale,
                   const float* v_descale, const pkv_cache_desc* cache,
                   const pkv_attn_meta* meta, void* workspace, size_t workspace_bytes,
                   void* stream);

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_write(const void* k, const void* v, const int64_t* slot_mapping,
                         int32_t num_tokens, void* k_cache, void* v_cache,
                         const pkv_cache_desc* cache, void* stream) {
  if (int st = check_cache(cache)) return st;
  if (cache->dtype == PKV_FP8_E4M3) return PKV_E_DTYPE;  // pkv_write_fp8
  if (num_tokens < 0) return PKV_E_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_E_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_E_ALIGN;
  int32_t* err;
  int sms;
  if (int st = device_state(&err, &sms)) return st;
  const int ebytes = cache->dtype == PKV_BF16 ? 2 : 4;
  WriteArgs a{};
  a.k = k;
  a.v = v;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.err = err;
  a.num_slots = static_cast<int64_t>(cache->num_blocks) * cache->block_size;
  a.num_tokens = num_tokens;
  a.row_vecs = cache->num_kv_heads * cache->head_size * ebytes / 16;
  a.k_scale = a.v_scale = nullptr;
  a.head_size = cache->head_size;
  return launch_write(a, as_stream(stream), sms) == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

extern "C" int pkv_write_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                             int32_t num_tokens, void* k_cache, void* v_cache,
                             const float* k_scale, const float* v_scale,
                             const pkv_cache_desc* cache, void* stream) {
  if (int st = check_cache(cache)) return st;
  if (cache->dtype != PKV_FP8_E4M3) return PKV_E_DTYPE;
  if (num_tokens < 0) return PKV_E_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PKV_E_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return PKV_E_ALIGN;
  int32_t* err;
  int sms;
  if (int st = device_state(&err, &sms)) return st;
  WriteArgs a{};
  a.k = k;
  a.v = v;
  a.slot_mapping = slot_mapping;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.err = err;
  a.num_slots = static_cast<int64_t>(cache->num_blocks) * cache->block_size;
  a.num_tokens = num_tokens;
  a.row_vecs = cache->num_kv_heads * cache->head_size / 16;  // 16 codes per vector
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.head_size = cache->head_size;
  return launch_write_fp8(a, as_stream(stream), sms) == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

extern "C" size_t pkv_attention_workspace_size(const pkv_cache_desc* cache,
                                               const pkv_attn_meta* meta) {
  int32_t* err;
  int sms;
  if (device_state(&err, &sms) != PKV_OK) return static_cast<size_t>(-1);
  Plan p;
  if (make_plan(cache, meta, sms, &p) != PKV_OK) return static_cast<size_t>(-1);
  return p.ws_bytes;
}

extern "C" int pkv_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             const int32_t* query_start_loc, float scale,
                             const pkv_cache_desc* cache, const pkv_attn_meta* meta,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (cache != nullptr && cache->dtype == PKV_FP8_E4M3) return PKV_E_DTYPE;  // pkv_attention_fp8
  return attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                        scale, nullptr, nullptr, cache, meta, workspace, workspace_bytes, stream);
}

extern "C" int pkv_attention_fp8(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, const int32_t* query_start_loc,
                                 float scale, const float* k_descale, const float* v_descale,
                                 const pkv_cache_desc* cache, const pkv_attn_meta* meta,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (cache == nullptr) return PKV_E_NULL;
  if (cache->dtype != PKV_FP8_E4M3) return PKV_E_DTYPE;
  if (meta != nullptr && meta->num_seqs > 0 && meta->num_tokens > 0) {
    if (!k_descale || !v_descale) return PKV_E_NULL;
    if ((reinterpret_cast<uintptr_t>(k_descale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_descale) & 3u))
      return PKV_E_ALIGN;
  }
  return attention_impl(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                        scale, k_descale, v_descale, cache, meta, workspace, workspace_bytes,
                        stream);
}

namespace pkv {
namespace {

int attention_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens,
                   const int32_t* query_start_loc, float scale, const float* k_descale,
                   const float* v_descale, const pkv_cache_desc* cache,
                   const pkv_attn_meta* meta, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int32_t* err;
  int sms, dev;
  if (int st = device_state(&err, &sms, &dev)) return st;
  Plan p;
  if (int st = make_plan(cache, meta, sms, &p)) return st;
  if (meta->num_seqs == 0 || meta->num_tokens == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start_loc)
    return PKV_E_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_start_loc) & 3u))
    return PKV_E_ALIGN;
  if (p.ws_bytes > 0) {
    if (workspace == nullptr || workspace_bytes < p.ws_bytes) return PKV_E_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_E_ALIGN;
  }
  const cudaStream_t st = as_stream(stream);
  const float LOG2E = 1.4426950408889634f;

  if (cache->dtype == PKV_F32) {
    F32Args a{};
    a.out = static_cast<float*>(out);
    a.q = static_cast<const float*>(q);
    a.k_cache = static_cast<const float*>(k_cache);
    a.v_cache = static_cast<const float*>(v_cache);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start_loc = query_start_loc;
    a.err = err;
    a.bt_stride = meta->block_table_stride;
    a.num_seqs = meta->num_seqs;
    a.num_tokens = meta->num_tokens;
    a.num_q_heads = meta->num_q_heads;
    a.num_kv_heads = cache->num_kv_heads;
    a.head_size = cache->head_size;
    a.num_blocks = cache->num_blocks;
    a.window = meta->sliding_window;
    a.scale = scale;
    return launch_attention_f32(a, st) == cudaSuccess ? PKV_OK : PKV_E_CUDA;
  }

  if (cache->num_blocks == 0) return PKV_E_SHAPE;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  CUtensorMap kmap, vmap;
  if (int e = encode_cache_map(&kmap, k_cache, *cache)) return e;
  if (int e = encode_cache_map(&vmap, v_cache, *cache)) return e;
  const int G = meta->num_q_heads / cache->num_kv_heads;

  const int npf = meta->num_seqs - p.num_decode;
  auto decode_part = [&](cudaStream_t st) -> int {
    DecodeArgs d{};
    d.out = out;
    d.q = q;
    d.block_tables = block_tables;
    d.context_lens = context_lens;
    d.query_start_loc = query_start_loc;
    d.ws_o = p.ws_bytes ? static_cast<float*>(workspace) : nullptr;
    d.ws_lse = p.ws_bytes ? reinterpret_cast<float*>(static_cast<char*>(workspace) + p.ws_o_bytes)
                          : nullptr;
    d.err = err;
    d.bt_stride = meta->block_table_stride;
    d.num_seqs = p.num_decode;
    d.num_q_heads = meta->num_q_heads;
    d.num_kv_heads = cache->num_kv_heads;
    d.group = G;
    d.num_blocks = cache->num_blocks;
    d.split_blocks = p.split_blocks;
    d.max_splits = p.max_splits;
    d.num_tokens = meta->num_tokens;
    d.max_context_len = meta->max_context_len;
    d.window = meta->sliding_window;
    d.k_descale = k_descale;
    d.v_descale = v_descale;
    d.scale_log2 = scale * LOG2E;
    PKV_TRY(launch_decode_bf16(kmap, vmap, d, cache->head_size, fp8, st));
    PKV_TRY(launch_combine_bf16(d, cache->head_size, st, /*after_decode=*/true));
    return PKV_OK;
  };
  auto prefill_part = [&](cudaStream_t st) -> int {
    PrefillArgs f{};
    f.out = out;
    f.q = q;
    f.block_tables = block_tables;
    f.context_lens = context_lens;
    f.query_start_loc = query_start_loc;
    f.err = err;
    f.bt_stride = meta->block_table_stride;
    f.seq_begin = p.num_decode;
    f.num_seqs = npf;
    f.num_q_heads = meta->num_q_heads;
    f.num_kv_heads = cache->num_kv_heads;
    f.group = G;
    f.num_blocks = cache->num_blocks;
    f.num_tokens = meta->num_tokens;
    f.max_query_len = meta->max_query_len;
    f.window = meta->sliding_window;
    f.k_descale = k_descale;
    f.v_descale = v_descale;
    f.scale_log2 = scale * LOG2E;
    f.longest_first = p.num_decode == 0 ? 1 : 0;   // alone on the GPU, or beside decode
    if (prefill_tc_supported(cache->head_size, G)) {
      // tcgen05/TMEM kernel: two tiles of 128/G tokens x G heads per CTA.
      const int toks = prefill_tc_tokens_per_cta(G);
      f.num_mtiles = (meta->max_query_len + toks - 1) / toks;
      CUtensorMap qmap, omap;
      if (int e = encode_query_map(&qmap, q, meta->num_tokens, meta->num_q_heads,
                                   cache->head_size, G))
        return e;
      if (int e = encode_query_map(&omap, out, meta->num_tokens, meta->num_q_heads,
                                   cache->head_size, G))
        return e;
      PKV_TRY(launch_prefill_tc(qmap, kmap, vmap, omap, f, cache->head_size, fp8, st));
    } else {
      // group sizes that do not divide 128 rows: mma.sync kernel, 64 rows per
      // CTA.
      const int64_t rows = static_cast<int64_t>(meta->max_query_len) * G;
      f.num_mtiles = static_cast<int32_t>((rows + kPrefillRows - 1) / kPrefillRows);
      PKV_TRY(launch_prefill_bf16(kmap, vmap, f, cache->head_size, fp8, st));
    }
    return PKV_OK;
  };
  if (p.num_decode == 0) return prefill_part(st);
  if (npf == 0) return decode_part(st);
  // Decode and prefill rows in one batch: the prefill launch goes first, on
  // the device's high-priority side stream forked from the caller's stream,
  // and the decode launches follow on the caller's stream, so that the short
  // decode CTAs fill the SMs that the prefill's last wave leaves idle; the
  // side stream is joined back before the call returns.  (Measured on GB300,
  // the mixed 48-decode + 4 x 512-token-chunk batch of 32 q / 8 kv heads:
  // attention 170 us in one stream, 143 us forked.)
  SideFork fork(dev, st);
  if (int e = fork.begin()) return e;
  int rc = prefill_part(fork.stream());
  if (rc == PKV_OK) rc = decode_part(st);
  const int jr = fork.join();
  return rc != PKV_OK ? rc : jr;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_use_cascade(const pkv_attn_meta* meta, int32_t common_prefix_blocks) {
  // The gate the [book] gives for cascade attention: a common prefix of at
  // least 256 tokens, at least 8 requests, no sliding window.  Then, in place
  // of the pages' rough CTA/wave model, rules measured on GB300 (32 q / 8 kv
  // heads, head_size 128; the prefix launch on the side stream beside the
  // suffix launches):
  //  * decode rows (own keys U[128, 1024]): the plain call already meets
  //    repeated prefix reads in L2, so the cascade wins once the prefix is
  //    >= 512 tokens and the repeated prefix keys (sequences - 1) x prefix
  //    reach 16K (1.09x at 64 x 512, 1.17x at 16 x 2048, 1.19x at 8 x 8192,
  //    3.6x at 64 x 8192, 6.0x at 256 x 8192; 0.83-0.96x below, and at every
  //    256-token prefix);
  //  * with chunked-prefill rows: their prefix work is a dense contraction
  //    either way (the cascade saves K/V reads, not flops) and costs a second
  //    pass and a merge, so the cascade wins only for at most 512 chunk rows
  //    beside a prefix of >= 4096 tokens (1.14-1.22x with 0, 16 or 48 decode
  //    rows; 4 x 512 chunk rows: 0.58-0.93x at every prefix up to 4096).
  if (meta == nullptr) return 0;
  const int64_t p = static_cast<int64_t>(common_prefix_blocks) * kBlock;
  const bool pages_gate = p >= 256 && meta->num_seqs >= 8 && meta->sliding_window == 0;
  const bool chunks = meta->max_query_len > 1;
  if (!pages_gate || p >= meta->max_context_len) return 0;
  if (!chunks)
    return p >= 512 && (static_cast<int64_t>(meta->num_seqs) - 1) * p >= 16384 ? 1 : 0;
  if (meta->num_decode_seqs < 0 || meta->num_decode_seqs > meta->num_seqs) return 0;
  const int64_t chunk_rows = static_cast<int64_t>(meta->num_tokens) - meta->num_decode_seqs;
  return chunk_rows <= 512 && p >= 4096 ? 1 : 0;
}

extern "C" size_t pkv_attention_cascade_workspace_size(const pkv_cache_desc* cache,
                                                       const pkv_attn_meta* meta,
                                                       int32_t common_prefix_blocks) {
  int32_t* err;
  int sms;
  if (device_state(&err, &sms) != PKV_OK) return static_cast<size_t>(-1);
  CascadePlan p;
  if (make_cascade_plan(cache, meta, common_prefix_blocks, sms, &p) != PKV_OK)
    return static_cast<size_t>(-1);
  return p.ws_bytes;
}

namespace pkv {
namespace {

int cascade_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens,
                 const int32_t* query_start_loc, float scale, int32_t common_prefix_blocks,
                 const float* k_descale, const float* v_descale, const pkv_cache_desc* cache,
                 const pkv_attn_meta* meta, void* workspace, size_t workspace_bytes,
                 void* stream);

}  // namespace
}  // namespace pkv

extern "C" int pkv_attention_cascade(void* out, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables,
                                     const int32_t* context_lens, const int32_t* query_start_loc,
                                     float scale, int32_t common_prefix_blocks,
                                     const pkv_cache_desc* cache, const pkv_attn_meta* meta,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (cache != nullptr && cache->dtype == PKV_FP8_E4M3) return PKV_E_DTYPE;  // _fp8 variant
  return cascade_impl(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                      scale, common_prefix_blocks, nullptr, nullptr, cache, meta, workspace,
                      workspace_bytes, stream);
}

extern "C" int pkv_attention_cascade_fp8(void* out, const void* q, const void* k_cache,
                                         const void* v_cache, const int32_t* block_tables,
                                         const int32_t* context_lens,
                                         const int32_t* query_start_loc, float scale,
                                         int32_t common_prefix_blocks, const float* k_descale,
                                         const float* v_descale, const pkv_cache_desc* cache,
                                         const pkv_attn_meta* meta, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (cache == nullptr) return PKV_E_NULL;
  if (cache->dtype != PKV_FP8_E4M3) return PKV_E_DTYPE;
  if (meta != nullptr && meta->num_seqs > 0 && meta->num_tokens > 0) {
    if (!k_descale || !v_descale) return PKV_E_NULL;
    if ((reinterpret_cast<uintptr_t>(k_descale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_descale) & 3u))
      return PKV_E_ALIGN;
  }
  return cascade_impl(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                      scale, common_prefix_blocks, k_descale, v_descale, cache, meta, workspace,
                      workspace_bytes, stream);
}

namespace pkv {
namespace {

int cascade_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens,
                 const int32_t* query_start_loc, float scale, int32_t common_prefix_blocks,
                 const float* k_descale, const float* v_descale, const pkv_cache_desc* cache,
                 const pkv_attn_meta* meta, void* workspace, size_t workspace_bytes,
                 void* stream) {
  const bool fp8 = cache != nullptr && cache->dtype == PKV_FP8_E4M3;
  int32_t* err;
  int sms, dev;
  if (int st = device_state(&err, &sms, &dev)) return st;
  CascadePlan p;
  if (int st = make_cascade_plan(cache, meta, common_prefix_blocks, sms, &p)) return st;
  if (meta->num_seqs == 0 || meta->num_tokens == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start_loc)
    return PKV_E_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_start_loc) & 3u))
    return PKV_E_ALIGN;
  if (workspace == nullptr || workspace_bytes < p.ws_bytes) return PKV_E_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_E_ALIGN;
  if (cache->num_blocks == 0) return PKV_E_SHAPE;
  CUtensorMap kmap, vmap;
  if (int e = encode_cache_map(&kmap, k_cache, *cache)) return e;
  if (int e = encode_cache_map(&vmap, v_cache, *cache)) return e;
  const cudaStream_t st = as_stream(stream);
  DecodeArgs d{};
  d.out = out;
  d.q = q;
  d.block_tables = block_tables;
  d.context_lens = context_lens;
  d.query_start_loc = query_start_loc;
  d.ws_o = static_cast<float*>(workspace);
  d.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.ws_o_bytes);
  d.err = err;
  d.bt_stride = meta->block_table_stride;
  d.num_seqs = meta->num_seqs;
  d.num_q_heads = meta->num_q_heads;
  d.num_kv_heads = cache->num_kv_heads;
  d.group = meta->num_q_heads / cache->num_kv_heads;
  d.num_blocks = cache->num_blocks;
  d.max_splits = p.max_splits;
  d.num_tokens = meta->num_tokens;
  d.max_context_len = meta->max_context_len;
  d.scale_log2 = scale * 1.4426950408889634f;
  d.k_descale = k_descale;
  d.v_descale = v_descale;
  d.force_partial = 1;
  d.prefix_splits = p.prefix_splits;
  // The prefix and suffix launches write disjoint split slots and meet only
  // in the merge: the prefix goes on the side stream (high priority; the
  // tcgen05 prefix grid is sized to about half the SMs) and the suffix on
  // the caller's stream beside it, joined before the merge.
  SideFork fork(dev, st);
  if (int e = fork.begin()) return e;
  const cudaStream_t pst = fork.stream();
  // prefix: every row against the shared keys, through sequence 0's table
  if (p.tc_prefix) {
    PrefillArgs f{};
    f.out = out;
    f.q = q;
    f.block_tables = block_tables;
    f.context_lens = context_lens;
    f.query_start_loc = query_start_loc;
    f.err = err;
    f.bt_stride = meta->block_table_stride;
    f.num_seqs = p.rows;              // the prefix launch's rows: query tokens
    f.casc_seqs = meta->num_seqs;
    f.num_q_heads = meta->num_q_heads;
    f.num_kv_heads = cache->num_kv_heads;
    f.group = d.group;
    f.num_blocks = cache->num_blocks;
    f.num_mtiles = p.prefix_mtiles;
    f.num_tokens = meta->num_tokens;
    f.max_query_len = 1;
    f.scale_log2 = d.scale_log2;
    f.cascade_prefix = 1;
    f.prefix_len = p.prefix_blocks * kBlock;
    f.prefix_tiles = p.prefix_tiles;
    f.max_splits = p.max_splits;
    f.ws_o = d.ws_o;
    f.ws_lse = d.ws_lse;
    f.k_descale = k_descale;
    f.v_descale = v_descale;
    CUtensorMap qmap;
    if (int e = encode_query_map(&qmap, q, meta->num_tokens, meta->num_q_heads,
                                 cache->head_size, d.group))
      return e;
    PKV_TRY(launch_prefill_tc(qmap, kmap, vmap, qmap, f, cache->head_size, fp8, pst));  // (no output map: workspace rows)
  } else {
    DecodeArgs pa = d;
    pa.split_blocks = p.prefix_split_blocks;
    pa.prefix_len = p.prefix_blocks * kBlock;
    pa.prefix_col_groups = p.col_groups;
    PKV_TRY(launch_cascade_prefix_bf16(kmap, vmap, pa, cache->head_size, pst));
  }
  // suffix: each row against its own keys after the prefix (decode rows on
  // the split-K decode kernel, chunk rows causally on the tcgen05 kernel);
  // then the merges
  DecodeArgs sa = d;
  sa.num_seqs = p.num_decode;
  sa.split_blocks = p.split_blocks;
  sa.key_begin_blocks = p.prefix_blocks;
  sa.split_base = p.prefix_splits;
  PKV_TRY(launch_decode_bf16(kmap, vmap, sa, cache->head_size, fp8, st));
  const int npf = meta->num_seqs - p.num_decode;
  if (npf > 0) {
    PrefillArgs f{};
    f.out = out;
    f.q = q;
    f.block_tables = block_tables;
    f.context_lens = context_lens;
    f.query_start_loc = query_start_loc;
    f.err = err;
    f.bt_stride = meta->block_table_stride;
    f.seq_begin = p.num_decode;
    f.num_seqs = npf;
    f.num_q_heads = meta->num_q_heads;
    f.num_kv_heads = cache->num_kv_heads;
    f.group = d.group;
    f.num_blocks = cache->num_blocks;
    f.num_tokens = meta->num_tokens;
    f.max_query_len = meta->max_query_len;
    f.k_descale = k_descale;
    f.v_descale = v_descale;
    f.scale_log2 = d.scale_log2;
    const int toks = prefill_tc_tokens_per_cta(d.group);
    f.num_mtiles = (meta->max_query_len + toks - 1) / toks;
    f.key_begin = p.prefix_blocks * kBlock;
    f.split_base = p.prefix_splits;
    f.max_splits = p.max_splits;
    f.ws_o = d.ws_o;
    f.ws_lse = d.ws_lse;
    CUtensorMap qmap;
    if (int e = encode_query_map(&qmap, q, meta->num_tokens, meta->num_q_heads,
                                 cache->head_size, d.group))
      return e;
    PKV_TRY(launch_prefill_tc(qmap, kmap, vmap, qmap, f, cache->head_size, fp8, st));  // (workspace rows)
  }
  if (int e = fork.join()) return e;
  PKV_TRY(launch_combine_bf16(sa, cache->head_size, st));
  if (npf > 0) {
    // chunk rows are the query tokens after the decode rows
    DecodeArgs mr = sa;
    mr.merge_rows_begin = p.num_decode;
    mr.merge_rows_end = meta->num_tokens;
    mr.num_seqs = meta->num_tokens - p.num_decode;
    mr.casc_seqs = meta->num_seqs;
    PKV_TRY(launch_combine_bf16(mr, cache->head_size, st));
  }
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

namespace pkv {
namespace {
// Test hook (pkv_debug_wait_test): 0 = off.
std::atomic<uint64_t> g_debug_wait_limit_ns{0};
std::atomic<int32_t> g_debug_stall{0};
constexpr uint64_t kDebugWaitLimitNs = 20000;   // 20 us
}  // namespace

void debug_wait_settings(uint64_t* limit_ns, int32_t* stall) {
  *limit_ns = g_debug_wait_limit_ns.load(std::memory_order_relaxed);
  *stall = g_debug_stall.load(std::memory_order_relaxed);
}
}  // namespace pkv

extern "C" int pkv_debug_wait_test(int enable) {
  pkv::g_debug_wait_limit_ns.store(enable ? pkv::kDebugWaitLimitNs : 0);
  pkv::g_debug_stall.store(enable ? 1 : 0);
  return PKV_OK;
}

extern "C" int pkv_get_error(int32_t* error_bits, int clear) {
  if (error_bits == nullptr) return PKV_E_NULL;
  int32_t* err;
  int sms;
  if (int st = device_state(&err, &sms)) return st;
  PKV_TRY(cudaDeviceSynchronize());
  PKV_TRY(cudaMemcpy(error_bits, err, sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (clear) {
    PKV_TRY(cudaMemset(err, 0, sizeof(int32_t)));
    PKV_TRY(cudaDeviceSynchronize());
  }
  return PKV_OK;
}

extern "C" int pkv_last_cuda_error(void) { return g_last_cuda_error.load(); }

extern "C" const char* pkv_last_cuda_error_string(void) {
  return cudaGetErrorString(static_cast<cudaError_t>(g_last_cuda_error.load()));
}

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_E_NULL: return "a required pointer is NULL";
    case PKV_E_DTYPE:
      return "dtype not supported by this call (PKV_F32/PKV_BF16: pkv_write, pkv_attention; "
             "PKV_FP8_E4M3: pkv_write_fp8, pkv_attention_fp8)";
    case PKV_E_SHAPE: return "unsupported or out-of-range shape (block_size 16, head_size 64/128)";
    case PKV_E_GQA: return "num_q_heads is not a multiple of num_kv_heads";
    case PKV_E_WORKSPACE: return "workspace missing or smaller than pkv_attention_workspace_size";
    case PKV_E_ALIGN: return "pointer not aligned (16 B tensors, 4 B int32 metadata, 256 B workspace)";
    case PKV_E_CUDA: return "CUDA launch or driver call failed";
    case PKV_E_META: return "inconsistent pkv_attn_meta";
    default: return "unknown status";
  }
}
