"""Oracle of the host block pool: free queue, null block, reference counts and
the prefix-cache hash map, with the request-level allocation that turns them
into block-table rows and slot mappings.

TEST INFRASTRUCTURE ONLY (see the package docstring): plain Python lists and
dicts, no attempt at speed, sharing nothing with the library's C++ pool.

Sources (page title, then section):

* "Implémentation du cœur du moteur d'inférence haute performance vLLM",
  ch. 4 §4.1 (the pool holds every block and a doubly linked free queue kept
  in eviction order; the null block is the first block taken from the head of
  that queue, is never reference-counted and stands in for positions that need
  no real block, e.g. those a sliding window skips), §4.3 (allocation in three
  phases: drop what is no longer needed and check that enough blocks are free,
  take the prefix-cache hits, allocate blocks for the new tokens; fail without
  side effects when blocks are short) and §4.4 (a cache hit is the longest run
  of leading full-block hashes found in the map, capped at num_tokens - 1
  tokens; taking a new block pops the head of the free queue, drops the block's
  cached hash and raises its count; releasing puts blocks without a hash at the
  head (LIFO reuse) and blocks with a hash at the tail (FIFO, i.e. LRU
  eviction); newly full blocks get their hash inserted in the map, an older
  hash of the same block being removed first; touching a hit block takes it out
  of the free queue if its count is 0, then raises the count).
* "Khám phá vLLM: Giải phẫu hệ thống suy luận LLM thông lượng cao", "KV cache
  manager" and "allocate_slots" (ceil(n / 16) blocks for n tokens, e.g. 2 for a
  17-token prefill; blocks come from the front of the free queue; requests keep
  their block lists; finished requests return their blocks to the queue).

Readings where the pages are silent (stated once here, relied on by the tests):

* Block hash: a chain, hash_i = FNV-1a-64(hash_{i-1} as 8 little-endian bytes
  followed by the block's 16 token ids as 4 little-endian bytes each), with
  hash_{-1} = 0.  (The pages fix no hash function; FNV-1a is a published
  64-bit hash whose definition both sides implement.)
* A map entry can hold several blocks with the same hash; a lookup takes the
  entry's oldest block.
* A request releases its blocks last to first, so that under LRU the deepest
  blocks of a cached prefix leave before its root.
* A hit, like any block the request holds, is released with the request.
"""
from __future__ import annotations

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit: for each byte, xor it in, then multiply by the prime."""
    h = FNV_OFFSET
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent: int, tokens) -> int:
    """hash of one full block chained on its parent's hash (reading above)."""
    data = parent.to_bytes(8, "little") + b"".join(
        (t & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


class Request:
    def __init__(self, tokens):
        self.tokens = list(tokens)      # every token id known so far
        self.blocks = []                # block ids, position order (null = 0)
        self.num_computed = 0           # tokens whose KV has been (or is being) written


class Pool:
    """The block pool plus the per-request bookkeeping of the KV-cache manager."""

    def __init__(self, num_blocks: int, block_size: int = 16, caching: bool = True):
        assert num_blocks >= 1
        self.bs = block_size
        self.caching = caching
        self.ref = [0] * num_blocks
        self.hash = [None] * num_blocks
        # free queue in eviction order: index 0 is the head
        self.free = list(range(num_blocks))
        # the null block is the first block taken from the head (§4.1)
        self.null_block = self.free.pop(0)
        self.map = {}                   # hash -> [block ids], oldest first
        self.reqs = {}

    # ---------------------------------------------------------------- blocks
    def num_free(self) -> int:
        return len(self.free)

    def _evict_hash(self, b):
        h = self.hash[b]
        if h is None:
            return
        self.map[h].remove(b)
        if not self.map[h]:
            del self.map[h]
        self.hash[b] = None

    def _get_new_blocks(self, n):
        """pop n blocks from the head; drop their cached hash; count them (§4.4)."""
        out = []
        for _ in range(n):
            b = self.free.pop(0)
            self._evict_hash(b)
            self.ref[b] += 1
            out.append(b)
        return out

    def _touch(self, blocks):
        """a hit block leaves the free queue if unreferenced, then is counted (§4.4)."""
        for b in blocks:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1

    def _free_blocks(self, blocks):
        """release in the given order; unhashed to the head, hashed to the tail (§4.4)."""
        for b in blocks:
            if b == self.null_block:
                continue
            self.ref[b] -= 1
            assert self.ref[b] >= 0
            if self.ref[b] == 0:
                if self.hash[b] is None:
                    self.free.insert(0, b)
                else:
                    self.free.append(b)

    def _cache_block(self, b, h):
        """enter a newly full block in the map, replacing an older hash (§4.4)."""
        if self.hash[b] == h:
            return
        self._evict_hash(b)
        self.hash[b] = h
        self.map.setdefault(h, []).append(b)

    # -------------------------------------------------------------- requests
    def _full_hashes(self, tokens, n_blocks):
        hs, parent = [], 0
        for i in range(n_blocks):
            parent = block_hash(parent, tokens[i * self.bs:(i + 1) * self.bs])
            hs.append(parent)
        return hs

    def add_request(self, req_id, tokens):
        assert req_id not in self.reqs
        self.reqs[req_id] = Request(tokens)

    def computed_blocks(self, req_id):
        """longest run of leading full-block hashes present in the map, capped so
        that at least the last token is computed (§4.4).  No side effects."""
        r = self.reqs[req_id]
        if not self.caching or r.blocks:
            return []
        cap = (len(r.tokens) - 1) // self.bs if r.tokens else 0
        hits = []
        for h in self._full_hashes(r.tokens, cap):
            if h not in self.map:
                break
            hits.append(self.map[h][0])
        return hits

    def admit(self, req_id) -> int:
        """take the prefix-cache hits of a new request; returns the cached tokens."""
        r = self.reqs[req_id]
        assert not r.blocks and r.num_computed == 0, "admit once, before any allocation"
        hits = self.computed_blocks(req_id)
        self._touch(hits)
        r.blocks = list(hits)
        r.num_computed = len(hits) * self.bs
        return r.num_computed

    def allocate_slots(self, req_id, num_new_tokens, window: int = 0):
        """blocks for the next num_new_tokens positions of the request and their
        slots (block * bs + offset); None (and no change) when blocks are short."""
        r = self.reqs[req_id]
        bs = self.bs
        first = r.num_computed
        end = first + num_new_tokens
        # phase 1: blocks wholly before every new token's window become the null
        # block and go back to the pool; check that enough blocks are free
        drop = []
        if window > 0:
            keep_from = max(0, first - window + 1)   # first key any new token sees
            for i in range(min(keep_from // bs, len(r.blocks))):
                if r.blocks[i] != self.null_block:
                    drop.append(i)
        need = -(-end // bs) - len(r.blocks)
        if need > len(self.free) + sum(1 for i in drop if self.ref[r.blocks[i]] == 1):
            return None
        if drop:
            freed = [r.blocks[i] for i in drop]
            for i in drop:
                r.blocks[i] = self.null_block
            self._free_blocks(list(reversed(freed)))
        # phase 3: new blocks for the new tokens
        if need > 0:
            r.blocks.extend(self._get_new_blocks(need))
        slots = [r.blocks[p // bs] * bs + p % bs for p in range(first, end)]
        r.num_computed = end
        # newly full blocks whose tokens are known enter the prefix cache
        if self.caching:
            n_full = min(end, len(r.tokens)) // bs
            for i, h in enumerate(self._full_hashes(r.tokens, n_full)):
                if r.blocks[i] != self.null_block:
                    self._cache_block(r.blocks[i], h)
        return slots

    def append_token(self, req_id, token):
        self.reqs[req_id].tokens.append(int(token))

    def free_request(self, req_id):
        r = self.reqs.pop(req_id)
        self._free_blocks(list(reversed(r.blocks)))

    def block_table(self, req_id):
        return list(self.reqs[req_id].blocks)

    def num_computed(self, req_id) -> int:
        return self.reqs[req_id].num_computed

    def cached_blocks(self) -> int:
        return sum(len(v) for v in self.map.values())
