"""The decode loop's host logic on CPU (scheduling, prefix hits, recompute
preemption, block tables and slots from the C++ pool), with the two kernel
calls replaced by stand-ins that record what they were given.  Checks the
invariants the kernels rely on: slots of one step are distinct and inside
the blocks the tables list, context_lens = last position + 1, decode rows
lead the batch, and every request finishes with its full token count."""
import numpy as np
import pytest
import torch

from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import decode_loop as DL


@pytest.fixture(autouse=True)
def _stub_kernels(monkeypatch):
    build.build()
    calls = []

    def write(k, v, slots, kc, vc, stream=None):
        calls.append(("write", slots.clone()))

    def attention(out, q, kc, vc, bt, cl, qsl, scale, **kw):
        out.zero_()
        calls.append(("attn", bt.clone(), cl.clone(), qsl.clone(), kw))

    monkeypatch.setattr(DL.pkv, "write", write)
    monkeypatch.setattr(DL.pkv, "attention", attention)
    return calls


@pytest.mark.parametrize("num_blocks,caching,window", [(96, True, 0), (14, True, 0),
                                                        (14, False, 0), (40, True, 33)])
def test_host_loop_invariants(_stub_kernels, num_blocks, caching, window):
    rng = np.random.default_rng(5)
    loop = DL.DecodeLoop(num_blocks=num_blocks, num_q_heads=4, num_kv_heads=2, head_size=64,
                         caching=caching, window=window, max_batch_tokens=160, device="cpu")
    system = [int(x) for x in rng.integers(0, 512, 40)]
    want = {}
    for i in range(8):
        p = system + [int(x) for x in rng.integers(0, 512, int(rng.integers(3, 30)))]
        n = int(rng.integers(5, 25))
        want[loop.add_request(p, n)] = len(p) + n
    finished, preempted, steps = {}, 0, 0
    reqs = {}
    while not loop.done():
        st = loop.step()
        assert st is not None
        steps += 1
        preempted += len(st.preempted)
        slots = st.slot_mapping.numpy()
        assert len(set(slots.tolist())) == len(slots)          # distinct slots in a step
        bt = st.block_tables.numpy()
        for i, rid in enumerate(st.req_ids):
            pos = st.positions[i]
            assert int(st.context_lens[i]) == pos[-1] + 1
            q0 = int(st.query_start_loc[i])
            for j, p in enumerate(pos):
                assert slots[q0 + j] == bt[i, p // 16] * 16 + p % 16
                assert bt[i, p // 16] != loop.pool.null_block
        ql = st.q_lens
        nd = next((i for i, x in enumerate(ql) if x != 1), len(ql))
        assert all(x > 1 for x in ql[nd:])                      # decode rows lead
        for rid in st.finished:
            finished[rid] = True
        assert steps < 1000
    assert set(finished) == set(want)
    if num_blocks == 14:
        assert preempted > 0
    assert loop.pool.num_free() == num_blocks - 1             # everything returned


@pytest.mark.parametrize("caching", [True, False])
def test_host_loop_prefills_long_prompts_in_chunks(_stub_kernels, caching):
    """Prompts longer than the token budget are prefilled over several steps:
    every chunk fits the budget left after that step's decode rows, a
    request's chunks cover its prompt positions once and in order, it samples
    nothing before its prompt is done, and everything finishes."""
    rng = np.random.default_rng(11)
    budget = 48
    loop = DL.DecodeLoop(num_blocks=200, num_q_heads=4, num_kv_heads=2, head_size=64,
                         caching=caching, max_batch_tokens=budget, device="cpu")
    system = [int(x) for x in rng.integers(0, 512, 70)]
    want, prompt_len = {}, {}
    for i in range(6):
        p = system + [int(x) for x in rng.integers(0, 512, int(rng.integers(10, 90)))]
        n = int(rng.integers(3, 12))
        rid = loop.add_request(p, n)
        want[rid], prompt_len[rid] = len(p) + n, len(p)
    covered = {rid: [] for rid in want}
    chunked = set()
    done, steps = set(), 0
    while not loop.done():
        st = loop.step()
        assert st is not None
        steps += 1
        assert sum(st.q_lens) <= budget              # the token budget holds every step
        for i, rid in enumerate(st.req_ids):
            pos = st.positions[i]
            assert pos == list(range(pos[0], pos[0] + len(pos)))
            if pos[-1] + 1 < prompt_len[rid]:
                chunked.add(rid)
                assert rid not in st.finished
            covered[rid].extend(pos)
        done |= set(st.finished)
        assert steps < 2000
    assert done == set(want)
    assert chunked                               # some prompt did take several steps
    for rid, pos in covered.items():
        assert max(pos) == want[rid] - 2         # the last sampled token is never computed
    assert loop.pool.num_free() == 200 - 1


def test_more_decodes_than_the_budget_wait_their_turn():
    """With more running decodes than the token budget, a step takes only as
    many rows as the budget allows (oldest first); the rest wait, and all
    finish."""
    loop = DL.DecodeLoop(num_blocks=200, num_q_heads=4, num_kv_heads=2, head_size=64,
                         caching=False, max_batch_tokens=4, device="cpu")
    rng = np.random.default_rng(5)
    rids = [loop.add_request([int(x) for x in rng.integers(0, 512, 3)], 6) for _ in range(7)]
    done, steps = set(), 0
    while not loop.done():
        st = loop.step()
        assert st is not None and 0 < sum(st.q_lens) <= 4
        done |= set(st.finished)
        steps += 1
        assert steps < 500
    assert done == set(rids)
