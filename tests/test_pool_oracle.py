"""Pins of the block-pool oracle (oracle/pool.py) against what the pages state
about the block pool and allocate_slots, and against published FNV-1a test
vectors.  Each test names the behaviour it pins; a plausible slip in the
oracle (wrong queue end, missing hash eviction, uncapped hit, wrong slot
formula, leaked reference) fails at least one of them."""
import pytest

from oracle import pool as P


def test_fnv1a64_published_vectors():
    # FNV-1a 64-bit test vectors from the algorithm's reference list
    assert P.fnv1a64(b"") == 0xCBF29CE484222325
    assert P.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert P.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_chains_on_parent_and_tokens():
    t = list(range(16))
    h0 = P.block_hash(0, t)
    assert h0 == P.fnv1a64(bytes(8) + b"".join(x.to_bytes(4, "little") for x in t))
    assert P.block_hash(h0, t) != h0                 # the parent enters the hash
    assert P.block_hash(0, t[::-1]) != h0            # so does the token order


def test_null_block_is_first_from_the_head_and_never_handed_out():
    p = P.Pool(8)
    assert p.null_block == 0 and p.num_free() == 7
    p.add_request("a", list(range(7 * 16)))
    assert p.allocate_slots("a", 7 * 16) is not None
    assert 0 not in p.block_table("a") and p.num_free() == 0


def test_seventeen_tokens_take_two_blocks_from_the_front():
    """[gpuhub] "allocate_slots": ceil(17/16) = 2 blocks, from the queue front."""
    p = P.Pool(10)
    p.add_request("a", list(range(17)))
    slots = p.allocate_slots("a", 17)
    assert p.block_table("a") == [1, 2]
    assert slots == [1 * 16 + i for i in range(16)] + [2 * 16]   # slot = block*16 + offset
    assert p.num_free() == 9 - 2


def test_allocation_failure_changes_nothing():
    p = P.Pool(4)
    p.add_request("a", list(range(40)))
    assert p.allocate_slots("a", 40) is not None            # 3 blocks: all free ones
    p.add_request("b", list(range(100, 120)))
    before = (list(p.free), list(p.ref))
    assert p.allocate_slots("b", 20) is None
    assert (list(p.free), list(p.ref)) == before and p.block_table("b") == []


def test_unhashed_blocks_are_reused_lifo():
    p = P.Pool(10, caching=False)
    p.add_request("a", list(range(32)))
    p.allocate_slots("a", 32)                               # blocks 1, 2
    p.free_request("a")                                     # released 2 then 1: head = 1, 2
    p.add_request("b", list(range(16)))
    p.allocate_slots("b", 16)
    assert p.block_table("b") == [1]                        # first freed-last, back at the head


def test_hashed_blocks_go_to_the_tail_and_are_evicted_last():
    p = P.Pool(6)
    p.add_request("a", list(range(32)))
    p.allocate_slots("a", 32)                               # blocks 1, 2 become full: hashed
    p.free_request("a")
    assert p.free == [3, 4, 5, 2, 1]                        # tail, deepest block first
    p.add_request("b", list(range(1000, 1048)))
    p.allocate_slots("b", 48)                               # takes 3, 4, 5: cache survives
    assert p.block_table("b") == [3, 4, 5] and p.cached_blocks() >= 2


def test_reusing_a_cached_block_evicts_its_hash():
    p = P.Pool(3)                                           # two usable blocks
    p.add_request("a", list(range(32)))
    p.allocate_slots("a", 32)                               # blocks 1, 2, both cached
    p.free_request("a")
    assert p.cached_blocks() == 2 and p.free == [2, 1]
    p.add_request("b", list(range(500, 516)))
    p.allocate_slots("b", 16)                               # pops block 2: its hash goes
    assert p.block_table("b") == [2]
    assert p.hash[2] == P.block_hash(0, list(range(500, 516)))   # now b's own full block
    assert p.cached_blocks() == 2
    p.add_request("c", list(range(32)) + [5])
    assert p.admit("c") == 16                               # root still cached, child evicted


def test_prefix_hit_touches_and_shares_blocks():
    p = P.Pool(10)
    prompt = list(range(48))
    p.add_request("a", prompt)
    p.allocate_slots("a", 48)                               # 3 full blocks cached
    p.add_request("b", prompt + [7, 8])
    assert p.admit("b") == 48                               # hit all three
    assert p.block_table("b") == p.block_table("a")
    assert all(p.ref[b] == 2 for b in p.block_table("a"))
    slots = p.allocate_slots("b", 2)
    assert len(p.block_table("b")) == 4 and slots[0] == p.block_table("b")[3] * 16
    p.free_request("a")
    assert all(p.ref[b] == 1 for b in p.block_table("b")[:3])
    assert p.num_free() == 9 - 4                            # shared blocks stay out of the queue


def test_hit_of_a_free_cached_block_leaves_the_queue():
    p = P.Pool(10)
    p.add_request("a", list(range(32)))
    p.allocate_slots("a", 32)
    p.free_request("a")
    n = p.num_free()
    p.add_request("b", list(range(32)) + [1])
    assert p.admit("b") == 32
    assert p.num_free() == n - 2 and all(b not in p.free for b in p.block_table("b"))


def test_hit_is_capped_so_the_last_token_is_computed():
    """[book] §4.4: at most num_tokens - 1 tokens come from the cache."""
    p = P.Pool(10)
    p.add_request("a", list(range(32)))
    p.allocate_slots("a", 32)
    p.add_request("b", list(range(32)))                     # same 32 tokens
    assert p.admit("b") == 16                               # (32 - 1) // 16 = 1 block


def test_sliding_window_swaps_dead_blocks_for_the_null_block():
    p = P.Pool(10, caching=False)
    p.add_request("a", list(range(64)))
    p.allocate_slots("a", 64)                               # blocks 1..4
    free0 = p.num_free()
    p.append_token("a", 99)
    # the next token sits at position 64 and with W = 20 sees keys 45..64:
    # blocks 0 and 1 (keys 0..31) are dead
    slots = p.allocate_slots("a", 1, window=20)
    bt = p.block_table("a")
    assert bt[:2] == [p.null_block, p.null_block] and bt[2:4] == [3, 4]
    assert slots == [bt[4] * 16]
    assert p.num_free() == free0 + 2 - 1


def test_decode_appends_a_block_every_sixteen_tokens():
    p = P.Pool(10)
    p.add_request("a", list(range(16)))
    p.allocate_slots("a", 16)
    for i in range(17):
        p.append_token("a", 1000 + i)
        p.allocate_slots("a", 1)
    assert len(p.block_table("a")) == 3 and p.num_computed("a") == 33
    assert p.cached_blocks() == 2                           # blocks 0 and 1 full and known


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_reference_counts_match_holders(seed):
    """Invariant: a block's count equals the number of live requests holding it,
    and a block is in the free queue iff its count is 0."""
    import random
    rng = random.Random(seed)
    p = P.Pool(40)
    live = []
    sys_prompt = list(range(40))
    for step in range(300):
        op = rng.random()
        if op < 0.3 or not live:
            rid = step
            toks = (sys_prompt if rng.random() < 0.5 else []) + [rng.randrange(1000) for _ in range(rng.randrange(1, 40))]
            p.add_request(rid, toks)
            cached = p.admit(rid)
            if p.allocate_slots(rid, len(toks) - cached) is None:
                p.free_request(rid)
            else:
                live.append(rid)
        elif op < 0.8:
            rid = rng.choice(live)
            p.append_token(rid, rng.randrange(1000))
            if p.allocate_slots(rid, 1) is None:
                p.free_request(rid)
                live.remove(rid)
        else:
            rid = live.pop(rng.randrange(len(live)))
            p.free_request(rid)
        holders = {}
        for rid in live:
            for b in p.block_table(rid):
                if b != p.null_block:
                    holders[b] = holders.get(b, 0) + 1
        for b in range(1, 40):
            assert p.ref[b] == holders.get(b, 0)
            assert (b in p.free) == (p.ref[b] == 0)
        assert len(set(p.free)) == len(p.free)


def test_popping_a_cached_block_drops_it_from_the_map():
    p = P.Pool(3)
    p.add_request("a", list(range(32)))
    p.allocate_slots("a", 32)
    p.free_request("a")                                     # queue [2, 1], both cached
    p.add_request("b", [7] * 10)                            # partial block: never cached
    p.allocate_slots("b", 10)                               # pops block 2
    assert p.cached_blocks() == 1
    p.add_request("c", list(range(32)) + [5])
    assert p.admit("c") == 16                               # the child hash left with block 2


def test_hash_chains_so_equal_blocks_at_other_positions_miss():
    x, y = list(range(16)), list(range(100, 116))
    p = P.Pool(10)
    p.add_request("a", x + y)
    p.allocate_slots("a", 32)
    p.add_request("b", y + [1])                             # y, but as a first block
    assert p.admit("b") == 0


@pytest.mark.parametrize("window,dead", [(17, 3), (18, 2), (33, 2), (34, 1)])
def test_window_boundary_blocks(window, dead):
    """position 64 with window W sees keys 65 - W .. 64: blocks wholly before
    key 65 - W are dead (W = 17: key 48 starts block 3, so 3 dead)."""
    p = P.Pool(10, caching=False)
    p.add_request("a", list(range(64)))
    p.allocate_slots("a", 64)
    p.append_token("a", 1)
    p.allocate_slots("a", 1, window=window)
    bt = p.block_table("a")
    assert bt[:dead] == [p.null_block] * dead and p.null_block not in bt[dead:]
