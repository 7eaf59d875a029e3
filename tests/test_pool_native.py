"""The C++ block pool (libpkv.so, include/pkv_pool.h) against the oracle
(oracle/pool.py) on seeded random request traces: every slot, block table,
reference count, cached hash and the free queue's order must be identical
after every operation (integer work: bit-exact).  Host only, no GPU."""
import random

import pytest

from oracle import pool as O
from paged_kv_cache_43_gb300 import build
from paged_kv_cache_43_gb300 import pool as N


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _same_state(o, n, live, nb):
    assert n.num_free() == o.num_free()
    assert n.free_queue() == o.free
    assert n.cached_blocks() == o.cached_blocks()
    for b in range(nb):
        assert n.block_state(b) == (o.ref[b], o.hash[b]), b
    for rid in live:
        assert n.block_table(rid) == o.block_table(rid)
        assert n.num_computed(rid) == o.num_computed(rid)


def _trace(seed, nb, caching, window, steps=400, vocab=50, max_prompt=80, max_own=40,
           check_every=1):
    rng = random.Random(seed)
    o, n = O.Pool(nb, caching=caching), N.BlockPool(nb, caching=caching)
    assert n.null_block == o.null_block
    prompts = [[rng.randrange(vocab) for _ in range(rng.randrange(16, max_prompt))]
               for _ in range(3)]
    live, next_id = [], 0
    for step in range(steps):
        op = rng.random()
        if op < 0.25 or not live:
            rid = next_id
            next_id += 1
            base = rng.choice(prompts) if rng.random() < 0.7 else []
            toks = base + [rng.randrange(vocab) for _ in range(rng.randrange(1, max_own))]
            o.add_request(rid, toks)
            n.add_request(rid, toks)
            assert n.admit(rid) == o.admit(rid)
            # prefill in one or two chunks
            todo = len(toks) - o.num_computed(rid)
            chunk = todo if rng.random() < 0.5 else max(1, todo // 2)
            so = o.allocate_slots(rid, chunk, window)
            sn = n.allocate_slots(rid, chunk, window)
            assert (sn is None) == (so is None)
            if so is None:
                o.free_request(rid)
                n.free_request(rid)
            else:
                assert list(sn) == so
                live.append(rid)
        elif op < 0.8:
            rid = rng.choice(live)
            todo = len(o.reqs[rid].tokens) - o.num_computed(rid)
            if todo <= 0:
                t = rng.randrange(vocab)
                o.append_token(rid, t)
                n.append_token(rid, t)
                todo = 1
            so = o.allocate_slots(rid, todo, window)
            sn = n.allocate_slots(rid, todo, window)
            assert (sn is None) == (so is None)
            if so is None:
                live.remove(rid)
                o.free_request(rid)
                n.free_request(rid)
            else:
                assert list(sn) == so
        else:
            rid = live.pop(rng.randrange(len(live)))
            o.free_request(rid)
            n.free_request(rid)
        if step % check_every == check_every - 1:
            _same_state(o, n, live, nb)
    _same_state(o, n, live, nb)
    n.close()


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("nb,caching,window", [(24, True, 0), (64, True, 0), (24, False, 0),
                                                (40, True, 40), (40, True, 17), (16, False, 9)])
def test_native_pool_matches_oracle_on_random_traces(seed, nb, caching, window):
    _trace(seed * 131 + nb, nb, caching, window)


@pytest.mark.parametrize("seed", range(2))
def test_native_pool_matches_oracle_with_thousands_of_cached_blocks(seed):
    """A pool of 3000 blocks with a large vocabulary: the prefix table grows
    several times and most evictions remove an entry (backward-shift
    deletion under collisions); the full state is compared every 50
    operations and at the end."""
    _trace(seed + 77, 3000, True, 0, steps=1500, vocab=32000, max_prompt=400, max_own=300,
           check_every=50)


def test_block_tables_rows_and_errors():
    n = N.BlockPool(20)
    n.add_request(7, list(range(40)))
    n.admit(7)
    n.allocate_slots(7, 40)
    n.add_request(9, list(range(100, 110)))
    n.admit(9)
    n.allocate_slots(9, 10)
    bt = n.block_tables([7, 9], 4)
    assert bt.tolist() == [[1, 2, 3, -1], [4, -1, -1, -1]]
    with pytest.raises(Exception):
        n.block_tables([7], 2)                 # row longer than the stride
    with pytest.raises(Exception):
        n.add_request(7, [1])                  # duplicate id
    with pytest.raises(Exception):
        n.admit(7)                             # admit after allocation
    with pytest.raises(Exception):
        n.free_request(12345)                  # unknown id
    n.close()


def test_batch_allocation_equals_one_by_one():
    rng = random.Random(9)
    a, b = N.BlockPool(30), N.BlockPool(30)
    for rid in range(6):
        toks = [rng.randrange(50) for _ in range(rng.randrange(5, 40))]
        for p in (a, b):
            p.add_request(rid, toks)
            p.admit(rid)
    want = [rng.randrange(1, 30) for _ in range(6)]
    slots, done = a.allocate_slots_batch(list(range(6)), want)
    one, served = [], 0
    for rid in range(6):
        s = b.allocate_slots(rid, want[rid])
        if s is None:
            break
        one += list(s)
        served += 1
    assert list(slots) == one and done == served
    assert a.free_queue() == b.free_queue()
    a.close()
    b.close()


def test_batch_append_equals_one_by_one():
    a, b = N.BlockPool(30), N.BlockPool(30)
    for p in (a, b):
        for rid in range(3):
            p.add_request(rid, [1, 2, 3])
            p.admit(rid)
            p.allocate_slots(rid, 3)
    a.append_token_batch([0, 1, 2], [7, 8, 9])
    for rid, t in zip(range(3), [7, 8, 9]):
        b.append_token(rid, t)
    for p in (a, b):
        for rid in range(3):
            p.allocate_slots(rid, 1)
    assert [a.block_table(r) for r in range(3)] == [b.block_table(r) for r in range(3)]
    a.close()
    b.close()
