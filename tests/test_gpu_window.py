"""Sliding-window attention on the GPU against the oracle: a query at position
pos sees keys pos - W < p <= pos.  Block-table entries wholly before every
window may hold the null block and must not be read."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import workloads as W
from tests.support import as_f64, compact_subproblem, max_err, nan_like, oracle_step

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


def _run(wl, window, **kw):
    g = wl.to("cuda")
    out = nan_like(g.q)
    pkv.run_step(g, out, sliding_window=window, **kw)
    torch.cuda.synchronize()
    return g, out


EDGE_CTX = [1, 2, 15, 16, 17, 33, 64, 65, 129, 300, 1000]


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 1000])
@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (32, 8, 128), (8, 1, 64)])
def test_decode_window(window, hq, hkv, d):
    wl = W.make_workload([1] * len(EDGE_CTX), EDGE_CTX, num_q_heads=hq, num_kv_heads=hkv,
                         head_size=d, dtype=torch.bfloat16, seed=window + hq + d)
    exp, _, _, _ = oracle_step(wl, window=window)
    for split in (0, 64):
        _, out = _run(wl, window, kv_split_tokens=split)
        assert max_err(out, exp) <= 2e-2


@pytest.mark.parametrize("window", [1, 7, 64, 130, 500])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (3, 1), (8, 8)])
def test_prefill_window(window, hq, hkv):
    """128 % G == 0 runs the tcgen05 kernel, G = 3 the mma.sync one."""
    q_lens = [1, 5, 64, 130, 1, 200, 33]
    ctx = [40, 5, 300, 130, 700, 900, 1000]
    wl = W.make_workload(q_lens, ctx, num_q_heads=hq, num_kv_heads=hkv, head_size=128,
                         dtype=torch.bfloat16, seed=window * 7 + hq)
    exp, _, _, _ = oracle_step(wl, window=window)
    _, out = _run(wl, window)
    assert max_err(out, exp) <= 2e-2


@pytest.mark.parametrize("window", [1, 10, 40])
def test_f32_window(window):
    wl = W.make_workload([1, 3, 17, 1], [17, 40, 70, 100], num_q_heads=4, num_kv_heads=2,
                         head_size=64, dtype=torch.float32, seed=window)
    exp, _, _, _ = oracle_step(wl, window=window)
    _, out = _run(wl, window)
    assert max_err(out, exp) <= 1e-5


def test_null_blocks_before_the_window_are_never_read():
    window = 48
    q_lens = [1, 1, 40, 100]
    ctx = [500, 333, 400, 900]
    wl = W.make_workload(q_lens, ctx, num_q_heads=32, num_kv_heads=8, head_size=128,
                         dtype=torch.bfloat16, seed=5)
    exp, _, _, _ = oracle_step(wl, window=window)
    g = wl.to("cuda")
    pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    for s, (n, L) in enumerate(zip(q_lens, ctx)):
        first_visible = max(0, L - n - window + 1)   # lowest key any row of s sees
        g.block_tables[s, : first_visible // 16] = -1
    out = nan_like(g.q)
    pkv.attention(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                  g.query_start_loc, g.scale, max_query_len=100, max_context_len=900,
                  num_decode_seqs=2, sliding_window=window)
    torch.cuda.synchronize()
    assert pkv.get_error() == 0
    assert max_err(out, exp) <= 2e-2


def test_full_size_long_context_window_sampled():
    window = 4096
    g = W.workload(5, device="cuda")
    pre_k, pre_v = g.k_cache.clone(), g.v_cache.clone()
    out = nan_like(g.q)
    pkv.run_step(g, out, sliding_window=window)
    torch.cuda.synchronize()
    assert pkv.get_error() == 0
    seqs = [0, 7, 15]
    P, rows = compact_subproblem(g, seqs, pre_k, pre_v, window=window)
    exp, st = oracle.attention(P.q, P.k_cache, P.v_cache, P.block_tables, P.context_lens,
                               P.query_start_loc, g.scale, window=window)
    assert not st.any()
    assert max_err(out[torch.as_tensor(rows, device="cuda")], exp) <= 2e-2
