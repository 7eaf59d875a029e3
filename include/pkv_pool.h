/* pkv_pool.h -- host-side KV-cache block pool: the free queue, the null
 * block, reference counts and the prefix cache, with the per-request
 * allocation that yields block-table rows and slot mappings for pkv_write /
 * pkv_attention.
 *
 * Follows "Implémentation du cœur du moteur d'inférence haute performance
 * vLLM" ch. 4 §4.1 (pool of blocks, doubly linked free queue kept in eviction
 * order, null block = first block taken from the head, never counted, a
 * placeholder for positions that need no block, e.g. those a sliding window
 * skips), §4.3 (allocation in three phases, failing without side effects when
 * blocks are short) and §4.4 (longest leading run of cached full-block hashes,
 * capped at num_tokens - 1 tokens; a new block pops the queue head, drops its
 * cached hash and is counted; released blocks without a hash go to the head
 * (LIFO), with a hash to the tail (FIFO = LRU eviction); newly full blocks
 * enter the hash map; a hit block leaves the queue if unreferenced and is
 * counted), and "Khám phá vLLM: Giải phẫu hệ thống suy luận LLM thông lượng
 * cao", "KV cache manager" / "allocate_slots" (ceil(n / block_size) blocks
 * for n tokens, taken from the front of the free queue).
 *
 * Choices the pages leave open: a block's hash chains on its parent's,
 * h_i = FNV-1a-64(h_{i-1} as 8 little-endian bytes, then the block's token ids
 * as 4 little-endian bytes each), h_{-1} = 0; a lookup takes the oldest block
 * filed under a hash; a request releases its blocks last to first.
 *
 * Host memory only; no call touches the GPU.  Not thread-safe: one pool is
 * driven by one host thread (the scheduler's).  Block ids are int32 in
 * [0, num_blocks); slots are block * block_size + offset (int64), the
 * slot_mapping pkv_write takes.  Status: PKV_OK, or a negative PKV_E_* code
 * (pkv.h) / PKV_E_REQUEST below; pkv_pool_allocate_slots returns
 * PKV_POOL_NO_SPACE (positive) when the pool is short, changing nothing. */
#ifndef PKV_POOL_H_
#define PKV_POOL_H_

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_POOL_NO_SPACE 1    /* not enough free blocks; nothing changed        */
#define PKV_E_REQUEST (-10)    /* unknown request id, duplicate id, or a call out */
                               /* of order (admit after allocation)               */

typedef struct pkv_pool pkv_pool; /* opaque; owned by the caller of create/destroy */

/* A pool of num_blocks blocks of block_size tokens (>= 1 each).  The null
 * block (id 0) is reserved at once.  enable_caching = 0 turns the prefix
 * cache off (no hashing, no hits).  Returns NULL on bad sizes or no memory. */
pkv_pool *pkv_pool_create(int32_t num_blocks, int32_t block_size, int32_t enable_caching);
void pkv_pool_destroy(pkv_pool *pool);

/* Blocks in the free queue (unreferenced, cached ones included). */
int32_t pkv_pool_num_free(const pkv_pool *pool);
/* Id of the null block (0). */
int32_t pkv_pool_null_block(const pkv_pool *pool);
/* Blocks currently filed in the prefix-cache map. */
int32_t pkv_pool_num_cached(const pkv_pool *pool);

/* Registers request req_id with its known token ids (copied). */
int pkv_pool_add_request(pkv_pool *pool, int64_t req_id, const int32_t *tokens,
                         int32_t num_tokens);
/* Appends generated token ids to a request (copied). */
int pkv_pool_append_tokens(pkv_pool *pool, int64_t req_id, const int32_t *tokens,
                           int32_t num_tokens);
/* One sampled token for each of num_reqs requests (req_ids[i] gets
 * tokens[i]), in one call.  Stops at the first unknown id (PKV_E_REQUEST). */
int pkv_pool_append_token_batch(pkv_pool *pool, const int64_t *req_ids, const int32_t *tokens,
                                int32_t num_reqs);
/* Prefix-cache lookup for a request that holds no blocks yet: the hit blocks
 * become its first blocks (shared, counted) and *num_cached_tokens (a multiple
 * of block_size) tokens count as computed. */
int pkv_pool_admit(pkv_pool *pool, int64_t req_id, int32_t *num_cached_tokens);
/* Makes room for the request's next num_new_tokens positions.  With
 * sliding_window W > 0, blocks wholly before key (first new position - W + 1)
 * are released and replaced by the null block first.  Writes the new
 * positions' slots to slot_mapping[0 .. num_new_tokens) (may be NULL), files
 * newly full blocks whose tokens are known in the prefix cache, and advances
 * the request's computed count.  PKV_POOL_NO_SPACE: nothing changed. */
int pkv_pool_allocate_slots(pkv_pool *pool, int64_t req_id, int32_t num_new_tokens,
                            int32_t sliding_window, int64_t *slot_mapping);
/* One scheduler step's allocations in one call: pkv_pool_allocate_slots for
 * req_ids[i] with num_new_tokens[i], i = 0, 1, ... in order, the slots packed
 * back to back into slot_mapping (sum of num_new_tokens entries; may be NULL).
 * Stops at the first request the pool cannot serve; *num_done = requests
 * served (the rest untouched).  Returns PKV_OK when all were served, else
 * PKV_POOL_NO_SPACE or the first error. */
int pkv_pool_allocate_slots_batch(pkv_pool *pool, const int64_t *req_ids,
                                  const int32_t *num_new_tokens, int32_t num_reqs,
                                  int32_t sliding_window, int64_t *slot_mapping,
                                  int32_t *num_done);
/* Releases every block of the request (last to first) and forgets it. */
int pkv_pool_free_request(pkv_pool *pool, int64_t req_id);

/* The request's block ids (position order, null block where released): up to
 * capacity ids to row; *num_blocks = the full count. */
int pkv_pool_block_table(const pkv_pool *pool, int64_t req_id, int32_t *row, int32_t capacity,
                         int32_t *num_blocks);
/* Rows of a block_tables array [num_reqs, stride] for pkv_attention: request
 * req_ids[i]'s ids, the rest of the row -1.  PKV_E_SHAPE if a row is longer
 * than stride. */
int pkv_pool_build_block_tables(const pkv_pool *pool, const int64_t *req_ids, int32_t num_reqs,
                                int32_t *block_tables, int32_t stride);
/* Tokens of the request counted as computed. */
int pkv_pool_num_computed(const pkv_pool *pool, int64_t req_id, int32_t *num_computed);

/* Introspection (tests, debugging): a block's reference count and cached hash
 * (*has_hash = 0: none), and the free queue in eviction order (head first; up
 * to capacity ids, *n = its length). */
int pkv_pool_block_state(const pkv_pool *pool, int32_t block, int32_t *ref_cnt, uint64_t *hash,
                         int32_t *has_hash);
int pkv_pool_free_queue(const pkv_pool *pool, int32_t *out, int32_t capacity, int32_t *n);

#ifdef __cplusplus
}
#endif

#endif /* PKV_POOL_H_ */
