"""The block pool driving the kernels in a decode loop (prefix caching,
sliding window, recompute preemption): every step's write and attention are
checked against the oracle replaying the same writes into its own cache, and
each (request, position) output must not depend on caching or preemption."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import workloads as W
from paged_kv_cache_43_gb300.decode_loop import DecodeLoop

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    pkv.load()
    pkv.get_error(clear=True)
    yield
    assert pkv.get_error(clear=True) == 0


def _run(num_blocks, caching, window=0, check=True, hq=8, hkv=2, d=128, seed=3):
    rng = np.random.default_rng(seed)
    loop = DecodeLoop(num_blocks=num_blocks, num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                      caching=caching, window=window, max_batch_tokens=160, seed=seed)
    system = [int(x) for x in rng.integers(0, 512, 40)]
    for i in range(8):
        tail = [int(x) for x in rng.integers(0, 512, int(rng.integers(3, 30)))]
        loop.add_request(system + tail, max_new_tokens=int(rng.integers(5, 25)))
    A = W.as_oracle_array
    kc = A(loop.k_cache).copy()     # all NaN: nothing of the CUDA path's state
    vc = A(loop.v_cache).copy()
    rows = {}
    preempted = 0
    steps = 0
    while not loop.done():
        st = loop.step()
        assert st is not None, "pool too small to make progress"
        steps += 1
        preempted += len(st.preempted)
        torch.cuda.synchronize()
        assert pkv.get_error() == 0
        if check:
            assert oracle.write(A(st.k_new), A(st.v_new), A(st.slot_mapping), kc, vc) == 0
            exp, status = oracle.attention(A(st.q), kc, vc, A(st.block_tables), A(st.context_lens),
                                           A(st.query_start_loc), loop.scale, window=window)
            assert not status.any()
            got = st.out.float().cpu().numpy().astype(np.float64)
            assert np.isfinite(got).all()
            assert np.abs(got - exp).max() <= 2e-2
        q0 = st.query_start_loc.cpu().numpy()
        for i, rid in enumerate(st.req_ids):
            for j, p in enumerate(st.positions[i]):
                rows[(rid, p)] = st.out[q0[i] + j].float().cpu()
        assert steps < 500
    return rows, preempted, loop


def test_decode_loop_with_prefix_cache_matches_oracle_every_step():
    rows_c, _, loop = _run(num_blocks=96, caching=True)
    assert loop.pool.cached_blocks() > 0
    rows_n, _, _ = _run(num_blocks=96, caching=False, check=False)
    # a hit reuses another request's blocks: the rows a request computes are
    # the same as without the cache (cached positions are not recomputed)
    common = set(rows_c) & set(rows_n)
    assert len(common) > 100
    assert max(float((rows_c[k] - rows_n[k]).abs().max()) for k in common) <= 2e-2


def test_decode_loop_preempts_and_recomputes():
    rows_small, preempted, _ = _run(num_blocks=14, caching=True)
    assert preempted > 0
    rows_big, _, _ = _run(num_blocks=96, caching=True, check=False)
    common = set(rows_small) & set(rows_big)
    assert len(common) > 100
    assert max(float((rows_small[k] - rows_big[k]).abs().max()) for k in common) <= 2e-2


@pytest.mark.parametrize("window", [16, 33])
def test_decode_loop_with_sliding_window(window):
    rows, _, loop = _run(num_blocks=64, caching=False, window=window)
    assert len(rows) > 100


def test_decode_loop_takes_cascade_on_a_long_shared_prompt():
    """70 requests behind a 1104-token system prompt: after the first prefill
    the others hit the prefix cache, and their decode steps share 69 blocks,
    which passes pkv_use_cascade; every step still matches the oracle."""
    rng = np.random.default_rng(8)
    loop = DecodeLoop(num_blocks=70 * 72 + 200, num_q_heads=32, num_kv_heads=8, head_size=128,
                      caching=True, max_batch_tokens=20000, seed=8, max_pos=2048,
                      use_cascade=True)
    system = [int(x) for x in rng.integers(0, 512, 69 * 16)]
    for _ in range(70):
        loop.add_request(system + [int(x) for x in rng.integers(0, 512, int(rng.integers(3, 12)))],
                         max_new_tokens=4)
    A = W.as_oracle_array
    kc, vc = A(loop.k_cache).copy(), A(loop.v_cache).copy()
    used = 0
    while not loop.done():
        st = loop.step()
        assert st is not None
        torch.cuda.synchronize()
        assert pkv.get_error() == 0
        used += st.cascade_blocks > 0
        assert oracle.write(A(st.k_new), A(st.v_new), A(st.slot_mapping), kc, vc) == 0
        exp, status = oracle.attention(A(st.q), kc, vc, A(st.block_tables), A(st.context_lens),
                                       A(st.query_start_loc), loop.scale)
        assert not status.any()
        got = st.out.float().cpu().numpy().astype(np.float64)
        assert np.abs(got - exp).max() <= 2e-2
    assert used >= 2
