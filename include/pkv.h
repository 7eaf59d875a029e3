/*
 * pkv.h -- C ABI of libpkv: paged KV-cache write and PagedAttention on one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [book]   "Implémentation du cœur du moteur d'inférence haute performance
 *            vLLM" (AiReadCodeBooks); ch. 5 "slot_mapping et la block table",
 *            ch. 6 "Transformation de la disposition mémoire du KV cache",
 *            "Structure des métadonnées", "Flux des paramètres du chemin
 *            non-cascadé", "Branche de masque", "Écriture du KV cache",
 *            "build() étape par étape".
 *   [gpuhub] "Khám phá vLLM: Giải phẫu hệ thống suy luận LLM thông lượng cao";
 *            note under "KV cache manager" (block bytes), "allocate_slots"
 *            step 1 (ceil(n/16) blocks), "Chạy forward pass" (flattened batch).
 *
 * Conventions shared by every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, on the
 *     current CUDA device, 16-byte aligned, densely packed (row-major, no
 *     padding) in the layout stated at the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work: they never allocate device memory,
 *     never synchronise and never copy device data to the host, so they may be
 *     captured into a CUDA graph.
 *   - The first call on a device (with it current) also creates the
 *     library's side stream there (non-blocking, the device's greatest
 *     priority) and two events; make that first call before any stream
 *     capture.  pkv_attention(_fp8/_static_scratch) on a batch with both
 *     decode and prefill rows enqueues its prefill launch, and the cascade
 *     calls their shared-prefix launch, on the side stream, forked from
 *     `stream` by an event after the work already on `stream` and joined
 *     back to `stream` before the call's last launch, so that work enqueued on
 *     `stream` afterwards sees the whole result, inside a graph capture too.
 *     A side stream that another thread's capture holds is not used (the
 *     call then runs on `stream` alone).
 *   - A call returns PKV_OK or a negative PKV_E_* for a host-side argument
 *     error, in which case nothing was enqueued.  PKV_E_CUDA means a launch
 *     failed; cudaGetLastError() holds the reason.
 *   - Errors that depend on device data (a slot past the pool, a block id
 *     outside [0, num_blocks), a context length outside
 *     [1, block_table_stride * block_size], more queries than keys, a
 *     "decode" sequence with a query length other than 1) never trap: the
 *     offending item is skipped and a bit is OR-ed into a per-device error
 *     word that pkv_get_error() returns.  Output rows of a sequence with a
 *     metadata error are zero; with a bad block id they are unspecified.
 *     Every other sequence is unaffected.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) -------------------------------------- */
#define PKV_OK 0
#define PKV_E_NULL (-1)        /* a required pointer is NULL                     */
#define PKV_E_DTYPE (-2)       /* dtype not supported by this call               */
#define PKV_E_SHAPE (-3)       /* unsupported head_size / block_size, or a size  */
                               /* is negative or too large                       */
#define PKV_E_GQA (-4)         /* num_q_heads not a multiple of num_kv_heads     */
#define PKV_E_WORKSPACE (-5)   /* workspace smaller than pkv_attention_workspace_size */
#define PKV_E_ALIGN (-6)       /* a pointer is not 16-byte aligned               */
#define PKV_E_CUDA (-7)        /* a kernel launch or driver call failed          */
#define PKV_E_META (-8)        /* inconsistent pkv_attn_meta fields              */

/* ---- device error-word bits (see pkv_get_error) ------------------------- */
#define PKV_ERR_SLOT (1 << 0)        /* pkv_write: slot >= num_blocks*block_size  */
#define PKV_ERR_BLOCK_ID (1 << 1)    /* block id outside [0, num_blocks)         */
#define PKV_ERR_CONTEXT_LEN (1 << 2) /* context_lens[s] < 1 with queries, or     */
                                     /* > block_table_stride * block_size        */
#define PKV_ERR_QUERY_LEN (1 << 3)   /* query length < 0 or > context_lens[s]    */
#define PKV_ERR_DECODE_QLEN (1 << 4) /* a sequence below num_decode_seqs whose   */
                                     /* query length is not 1                    */
#define PKV_ERR_TIMEOUT (1 << 5)     /* an on-chip wait gave up (bounded spin)   */

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Shape of the paged KV cache ([book] ch. 6 "Transformation de la disposition
 * mémoire du KV cache": separate K and V caches, each
 * [num_blocks, block_size, num_kv_heads, head_size]).  One block of both
 * caches takes 2 * block_size * num_kv_heads * head_size * dtype_bytes bytes
 * ([gpuhub] note under "KV cache manager").
 * Supported: block_size 16, head_size 64 or 128, dtype PKV_BF16, PKV_F32 or
 * PKV_FP8_E4M3 (e4m3 codes; [book] ch. 6 "Matrice de capacités": fp8 cache
 * dtypes), the last through pkv_write_fp8 / pkv_attention_fp8 only. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_size;
  int32_t dtype; /* pkv_dtype */
} pkv_cache_desc;

/* Host-side description of one attention batch ([book] ch. 6 "Structure des
 * métadonnées"): the batch is flattened into num_tokens query rows
 * ([gpuhub] "Chạy forward pass"), sequence s owning rows
 * query_start_loc[s] .. query_start_loc[s+1]-1. */
typedef struct {
  int32_t num_seqs;           /* S                                              */
  int32_t num_tokens;         /* T = query_start_loc[S] (rows of q and out)     */
  int32_t num_q_heads;        /* Hq, a multiple of num_kv_heads (GQA)           */
  int32_t block_table_stride; /* int32 entries per block_tables row (>= 1)      */
  int32_t max_query_len;      /* >= every query length; 1 means pure decode.    */
                              /* A longer sequence sets PKV_ERR_QUERY_LEN and   */
                              /* its rows are unspecified                       */
  int32_t max_context_len;    /* >= every context_lens[s]; sizes split-K.  A    */
                              /* decode sequence past it sets                   */
                              /* PKV_ERR_CONTEXT_LEN (rows zero)                */
  int32_t num_decode_seqs;    /* sequences 0..n-1 have query length 1 (the      */
                              /* decode run of a mixed batch); -1 = unknown     */
  int32_t sliding_window;     /* W > 0: query at position pos sees only keys    */
                              /* pos - W < p <= pos ([book] ch. 6 causal window */
                              /* (w, 0), ch. 2 sliding_window); block-table     */
                              /* entries before that range are never read, so   */
                              /* they may hold the null block.  0 = no window   */
  int32_t kv_split_tokens;    /* split-K chunk in keys for decode: 0 = choose   */
                              /* automatically, else a multiple of 64 in        */
                              /* [64, 2048]                                     */
} pkv_attn_meta;

/* KV-cache write ([book] ch. 6 "Écriture du KV cache"; ch. 5 on the -1 padding
 * of slot_mapping): for every token t < num_tokens with slot =
 * slot_mapping[t] >= 0, copies k[t] and v[t] (num_kv_heads * head_size
 * elements each, bit for bit) into row `slot` of the caches, i.e. block
 * slot / block_size, offset slot % block_size.  Slots < 0 are padding and are
 * skipped.  A slot >= num_blocks * block_size is skipped and sets
 * PKV_ERR_SLOT.  Two tokens with the same slot: the row written is one of
 * the two (unspecified which).
 *   k, v          [num_tokens, num_kv_heads, head_size], cache dtype
 *   slot_mapping  int64 [num_tokens]
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_size]
 * num_tokens == 0 is a no-op. */
int pkv_write(const void *k, const void *v, const int64_t *slot_mapping,
              int32_t num_tokens, void *k_cache, void *v_cache,
              const pkv_cache_desc *cache, void *stream);

/* FP8 KV-cache write: as pkv_write, but k and v are bf16 and each element is
 * stored as the e4m3 code of k / k_scale[h] (v / v_scale[h]), h its kv head:
 * the quotient is an fp32 division rounded to nearest, then rounded to the
 * nearest e4m3 value (ties to the even code), magnitudes above 448 clamped to
 * 448; a NaN input gives a NaN code.
 *   k, v              bf16 [num_tokens, num_kv_heads, head_size]
 *   k_cache, v_cache  uint8 e4m3 [num_blocks, block_size, num_kv_heads, head_size]
 *   k_scale, v_scale  fp32 [num_kv_heads] (device)
 * cache->dtype must be PKV_FP8_E4M3. */
int pkv_write_fp8(const void *k, const void *v, const int64_t *slot_mapping,
                  int32_t num_tokens, void *k_cache, void *v_cache, const float *k_scale,
                  const float *v_scale, const pkv_cache_desc *cache, void *stream);

/* Bytes of scratch workspace pkv_attention needs for this batch shape (the
 * split buffer of [book] ch. 6 "build() étape par étape", fourth step: one
 * fp32 partial output and one log-sum-exp per split, head and decode
 * sequence).  0 when no split is needed.  Returns (size_t)-1 for an invalid
 * description. */
size_t pkv_attention_workspace_size(const pkv_cache_desc *cache,
                                    const pkv_attn_meta *meta);

/* PagedAttention ([book] ch. 6 "Flux des paramètres du chemin non-cascadé":
 * cu_seqlens_q = query_start_loc, seqused_k = seq_lens; "Branche de masque").
 * For each sequence s with L = context_lens[s] keys (history plus this step's
 * new tokens, which pkv_write must already have stored) and q_s query rows,
 * query row j sits at absolute position L - q_s + j and attends the keys
 * p <= L - q_s + j; key p is read from block block_tables[s][p / block_size],
 * offset p % block_size.  Query head hq uses kv head hq / (num_q_heads /
 * num_kv_heads).  out[t][hq] = softmax(scale * q[t][hq] . K^T) V, accumulated
 * in fp32 and rounded to the cache dtype (round to nearest even).
 *   out, q            [num_tokens, num_q_heads, head_size], cache dtype
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_size]
 *   block_tables      int32 [num_seqs, block_table_stride]; entries past
 *                     ceil(L / block_size) are never read
 *   context_lens      int32 [num_seqs]
 *   query_start_loc   int32 [num_seqs + 1], non-decreasing, [0] = 0,
 *                     [num_seqs] <= num_tokens (a sequence whose rows fall
 *                     outside [0, num_tokens) sets PKV_ERR_QUERY_LEN and is
 *                     skipped)
 *   workspace         device scratch of at least
 *                     pkv_attention_workspace_size() bytes (may be NULL when
 *                     that is 0); its contents need no initialisation.
 * A sequence with q_s = 0 produces nothing.  Rows of out that belong to no
 * sequence are not written. */
int pkv_attention(void *out, const void *q, const void *k_cache,
                  const void *v_cache, const int32_t *block_tables,
                  const int32_t *context_lens, const int32_t *query_start_loc,
                  float scale, const pkv_cache_desc *cache,
                  const pkv_attn_meta *meta, void *workspace,
                  size_t workspace_bytes, void *stream);

/* Bytes of the fixed scratch array behind pkv_attention_static_scratch. */
#define PKV_STATIC_SCRATCH_BYTES (64u << 20) /* 64 MiB per GPU */

/* pkv_attention for callers that cannot allocate device memory.  The pages
 * have no counterpart to this call; it exists for users of this library.
 *
 * Who needs it: a caller that has no way to hand pkv_attention a workspace,
 * such as a plugin inside a host framework that owns every device
 * allocation through its own pool (a stray cudaMalloc there can synchronise
 * the device and escapes the pool's accounting), or a decode loop that must
 * never enter the allocator.
 *
 * What it does: exactly pkv_attention (same arguments, same results), with
 * the split-K workspace taken from a fixed array of PKV_STATIC_SCRATCH_BYTES
 * inside the library instead of from the caller.  Every GPU on which the
 * library's device code is loaded holds that array until the process exits.
 * The call itself allocates nothing and frees nothing.
 *
 * Limits and sharing:
 *   - A batch whose workspace (pkv_attention_workspace_size) exceeds
 *     PKV_STATIC_SCRATCH_BYTES is rejected with PKV_E_WORKSPACE before
 *     anything is enqueued; a larger kv_split_tokens shrinks the need.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; nothing in it has to start at zero (each call writes every
 *     partial it reads).  Calls whose GPU work overlaps (e.g. on two streams
 *     without ordering) race on the array: order them.
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture. */
int pkv_attention_static_scratch(void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *context_lens,
                                 const int32_t *query_start_loc, float scale,
                                 const pkv_cache_desc *cache,
                                 const pkv_attn_meta *meta, void *stream);

/* PagedAttention over an FP8 (e4m3) cache: as pkv_attention with q and out in
 * bf16, and K = code value * k_descale[s][h], V = code value * v_descale[s][h]
 * for sequence s, kv head h ([book] ch. 6 "Flux des paramètres du chemin
 * non-cascadé": descales shaped (num_sequences, num_kv_heads)).  For the
 * result to be the attention of the written K/V, k_descale[s][h] must equal
 * the k_scale the blocks were written with (likewise for V).
 *   k_descale, v_descale  fp32 [num_seqs, num_kv_heads] (device)
 * Workspace as for pkv_attention (same size function). */
int pkv_attention_fp8(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *context_lens,
                      const int32_t *query_start_loc, float scale, const float *k_descale,
                      const float *v_descale, const pkv_cache_desc *cache,
                      const pkv_attn_meta *meta, void *workspace, size_t workspace_bytes,
                      void *stream);

/* Cascade attention ([book] ch. 6: "Structure des métadonnées", the cascade
 * fields use_cascade / common_prefix_len / cu_prefix_query_lens; the sequence
 * diagram, where the cascade branch runs a prefix call over every query token
 * and a suffix call and merges them with merge_attn_states; "Réflexion de
 * conception", the use_cascade_attention gate).  For a batch -- decode rows,
 * or meta->num_decode_seqs decode sequences followed by chunked-prefill
 * sequences -- whose sequences' first common_prefix_blocks block-table entries
 * name the same physical blocks (the caller guarantees it; sequence 0's
 * entries are read): the shared prefix keys are attended once for all query
 * rows (K/V read once per 128-row tile of rows instead of once per sequence),
 * each row's own keys after the prefix separately (causally inside a chunk),
 * and the partial results merged.  Same result as pkv_attention (arguments as
 * there).  Every query row must sit after the prefix: L - q_len >=
 * 16 * common_prefix_blocks for a chunk, L > 16 * common_prefix_blocks for a
 * decode row (else the sequence's rows are zeroed and PKV_ERR_CONTEXT_LEN
 * set).  With chunk rows the group size must divide 128 (PKV_E_SHAPE) and
 * num_decode_seqs be given (>= 0, PKV_E_META otherwise).  bf16 caches only
 * (PKV_E_DTYPE otherwise); PKV_E_META for a window, or a prefix outside
 * [1, min(block_table_stride, (max_context_len - 1) / 16)].  The workspace
 * is required (size from the function below).  e4m3 caches:
 * pkv_attention_cascade_fp8 (PKV_E_DTYPE here). */
size_t pkv_attention_cascade_workspace_size(const pkv_cache_desc *cache,
                                            const pkv_attn_meta *meta,
                                            int32_t common_prefix_blocks);
int pkv_attention_cascade(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *context_lens,
                          const int32_t *query_start_loc, float scale,
                          int32_t common_prefix_blocks, const pkv_cache_desc *cache,
                          const pkv_attn_meta *meta, void *workspace, size_t workspace_bytes,
                          void *stream);
/* Cascade attention over e4m3 caches: as pkv_attention_cascade with the
 * descales of pkv_attention_fp8 (fp32 [num_seqs, num_kv_heads], device; each
 * row uses its own sequence's descales, the shared keys included).  The shared
 * keys run on the tcgen05 kernel, so the group size must divide 128
 * (PKV_E_SHAPE otherwise); workspace size from
 * pkv_attention_cascade_workspace_size with the e4m3 cache descriptor. */
int pkv_attention_cascade_fp8(void *out, const void *q, const void *k_cache,
                              const void *v_cache, const int32_t *block_tables,
                              const int32_t *context_lens, const int32_t *query_start_loc,
                              float scale, int32_t common_prefix_blocks, const float *k_descale,
                              const float *v_descale, const pkv_cache_desc *cache,
                              const pkv_attn_meta *meta, void *workspace, size_t workspace_bytes,
                              void *stream);
/* Whether to use cascade attention, host only.  1 when the [book]'s gate
 * passes (common prefix >= 256 tokens, >= 8 sequences, no sliding window, a
 * prefix shorter than the longest context) and a cost rule measured on GB300
 * says it pays (the [book]'s own rule is a rough CTA/wave model): decode
 * batches, prefix >= 512 tokens and (num_seqs - 1) * prefix tokens >= 16384;
 * batches with chunked-prefill rows (num_decode_seqs given), at most 512
 * chunk rows and a prefix >= 4096 tokens; else 0. */
int pkv_use_cascade(const pkv_attn_meta *meta, int32_t common_prefix_blocks);

/* Reads (and, if clear != 0, resets) the current device's error word: the OR
 * of PKV_ERR_* bits raised by kernels since the last clear.  SYNCHRONISES the
 * device first.  Returns PKV_OK or PKV_E_CUDA. */
int pkv_get_error(int32_t *error_bits, int clear);

/* TEST HOOK for the timeout path; no counterpart in the pages.  Every on-chip
 * wait of the kernels gives up after a bounded time (1 s), sets
 * PKV_ERR_TIMEOUT, lets the CTA's own copies in flight land, frees its tensor
 * memory and returns.  With enable != 0, the decode and tcgen05 prefill
 * launches this process makes afterwards (on any device, from any thread)
 * wait at most 20 us and withhold their first key block or tile, so that
 * those waits run out and the attention calls return with PKV_ERR_TIMEOUT
 * set and meaningless output; enable = 0 restores normal launches.  Host
 * only; never synchronises.  Returns PKV_OK. */
int pkv_debug_wait_test(int enable);

/* Static, human-readable text for a status code. */
const char *pkv_status_string(int status);

/* The CUDA runtime error (cudaError_t as int, 0 = none yet) behind the most
 * recent PKV_E_CUDA any call of this library returned in this process, and
 * its text.  Host only; never synchronises. */
int pkv_last_cuda_error(void);
const char *pkv_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
