// pkv_internal.h -- argument blocks and launchers shared between the C-ABI
// front end (pkv_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Keys per cache block; the only block size the kernels take.
constexpr int kBlock = 16;

struct WriteArgs {
  const void* k;
  const void* v;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  int32_t* err;
  int64_t num_slots;    // num_blocks * block_size
  int32_t num_tokens;
  int32_t row_vecs;     // 16-byte vectors per token row (num_kv_heads*head_size*bytes/16)
  // FP8 cache: per-kv-head quantisation scales (null otherwise)
  const float* k_scale;
  const float* v_scale;
  int32_t head_size;
};

// Split-K decode over sequences [0, num_seqs) (each with one query row).
struct DecodeArgs {
  void* out;                     // bf16 [T, Hq, D]
  const void* q;                 // bf16 [T, Hq, D]
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  float* ws_o;                   // [num_seqs, Hq, max_splits, D] fp32 (split > 1 only)
  float* ws_lse;                 // [num_seqs, Hq, max_splits]   log2-domain
  int32_t* err;
  int64_t bt_stride;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;                 // num_q_heads / num_kv_heads
  int32_t num_blocks;
  int32_t split_blocks;          // cache blocks per split
  int32_t max_splits;
  int32_t num_tokens;            // rows of q/out: query_start_loc must stay inside
  int32_t max_context_len;       // bound the split buffer was sized for
  int32_t window;                // sliding window (keys per query), 0 = none
  const float* k_descale;        // FP8 cache: [num_seqs_total, Hkv] (null otherwise)
  const float* v_descale;
  float scale_log2;              // scale * log2(e)
  // Cascade attention (all zero otherwise).
  int32_t key_begin_blocks;      // suffix launch: a sequence's keys start at this block
  int32_t split_base;            // first workspace split slot this launch writes
  int32_t force_partial;         // write partials even when a row has one split
  int32_t prefix_splits;         // combine: leading split slots that hold prefix partials
  int32_t prefix_len;            // prefix launch: the shared keys [0, prefix_len)
  int32_t prefix_col_groups;     // prefix launch: 8-column groups per kv head
  // Combine over token rows [merge_rows_begin, merge_rows_end) (> begin: the
  // cascade merge of chunked-prefill rows, each with prefix_splits prefix
  // partials and one suffix partial); 0, 0 otherwise.
  int32_t merge_rows_begin;
  int32_t merge_rows_end;
  int32_t casc_seqs;             // sequences of the batch (rows mode: row -> sequence)
  // Test hook (pkv_debug_wait_test): main-loop wait limit (0 = the default)
  // and, when set, warp 0 of every CTA withholds its first block load so
  // that its wait runs out.
  uint64_t wait_limit_ns;
  int32_t debug_stall;
};

// Varlen causal attention over sequences [seq_begin, seq_begin + num_seqs).
struct PrefillArgs {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int32_t* err;
  int64_t bt_stride;
  int32_t seq_begin;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t num_blocks;
  int32_t num_mtiles;            // grid.x: row tiles of the longest sequence
  int32_t num_tokens;
  int32_t max_query_len;
  int32_t window;                // sliding window (keys per query), 0 = none
  const float* k_descale;        // FP8 cache: [num_seqs_total, Hkv] (null otherwise)
  const float* v_descale;
  float scale_log2;
  // tcgen05 kernel: hand the CTAs out longest first (a launch that has the
  // GPU to itself); 0 keeps the plain order, whose short CTAs finish early
  // and leave SMs to a decode launch running beside it.
  int32_t longest_first;
  // Cascade prefix launch of the tcgen05 kernel (cascade_prefix = 1): the
  // decode rows 0 .. num_seqs - 1 (row t = sequence t) against the shared keys
  // [0, prefix_len) of block-table row 0, prefix_tiles 128-key tiles per CTA
  // (grid.z = prefix split); normalised fp32 partials and log2-sum-exps go to
  // ws_o / ws_lse at split slot blockIdx.z of rows [seq, q head, max_splits].
  int32_t cascade_prefix;
  int32_t prefix_len;
  int32_t prefix_tiles;
  int32_t max_splits;
  float* ws_o;
  float* ws_lse;
  // Cascade prefix launch: the batch's sequences (query_start_loc has
  // casc_seqs + 1 entries), to find each row's sequence for its descales.
  int32_t casc_seqs;
  // Cascade suffix launch of the tcgen05 kernel (key_begin > 0): every row
  // sees only keys >= key_begin (the shared prefix is the prefix launch's),
  // and writes its normalised fp32 partial and log2-sum-exp to ws_o / ws_lse
  // at split slot split_base of rows [token, q head, max_splits].
  int32_t key_begin;
  int32_t split_base;
  // Test hook (pkv_debug_wait_test), tcgen05 kernel: main-loop wait limit (0
  // = the default) and, when set, the K producer withholds the CTA's first K
  // tile so that the waits for it run out.
  uint64_t wait_limit_ns;
  int32_t debug_stall;
};

// Settings of the test hook, applied to the decode and tcgen05 prefill
// launches made after pkv_debug_wait_test (pkv_api.cu).
void debug_wait_settings(uint64_t* limit_ns, int32_t* stall);

// fp32 I/O: one CTA per (query row, q head), every sequence.
struct F32Args {
  float* out;
  const float* q;
  const float* k_cache;
  const float* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start_loc;
  int32_t* err;
  int64_t bt_stride;
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_size;
  int32_t num_blocks;
  int32_t window;                // sliding window (keys per query), 0 = none
  float scale;
};

cudaError_t launch_write(const WriteArgs& a, cudaStream_t stream, int num_sms);
cudaError_t launch_write_fp8(const WriteArgs& a, cudaStream_t stream, int num_sms);
// fp8 = true: the caches hold e4m3 codes (the maps are uint8, unswizzled).
cudaError_t launch_decode_bf16(const CUtensorMap& kmap, const CUtensorMap& vmap,
                               const DecodeArgs& a, int head_size, bool fp8,
                               cudaStream_t stream);
// after_decode: launched right after launch_decode_bf16 on the same stream
// (a programmatic dependent launch; false when other work sits between them).
cudaError_t launch_combine_bf16(const DecodeArgs& a, int head_size, cudaStream_t stream,
                                bool after_decode = false);
// Cascade prefix launch: every decode row of the batch (all sequences, all q
// heads) against the shared prefix keys, read once per 8 columns; partials to
// split slots [0, prefix_splits).
cudaError_t launch_cascade_prefix_bf16(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                       const DecodeArgs& a, int head_size, cudaStream_t stream);
cudaError_t launch_prefill_bf16(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                const PrefillArgs& a, int head_size, bool fp8,
                                cudaStream_t stream);
cudaError_t launch_attention_f32(const F32Args& a, cudaStream_t stream);

// tcgen05 prefill: query tiles of 128 rows = (128 / group) tokens x group heads,
// two tiles per CTA.
bool prefill_tc_supported(int head_size, int group);
int prefill_tc_tokens_per_tile(int group);
int prefill_tc_tokens_per_cta(int group);
// fp8 = true: e4m3 caches, widened to fp16 in shared memory.
// omap: the output tensor viewed like qmap (full query tiles of a plain
// launch leave through it; cascade launches write the workspace instead).
cudaError_t launch_prefill_tc(const CUtensorMap& qmap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const CUtensorMap& omap,
                              const PrefillArgs& a, int head_size, bool fp8,
                              cudaStream_t stream);

// Rows of the prefill kernel's query tile (grid.x covers ceil(q_len*G / this)).
constexpr int kPrefillRows = 64;

}  // namespace pkv
