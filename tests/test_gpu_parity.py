"""CUDA path vs the CPU oracle, element by element, through the C ABI.

KV write: bit-exact.  Attention: max |error| <= 1e-5 (fp32 I/O) or 2e-2 (bf16
I/O) against the fp64 oracle.  Output buffers start as NaN so that a row the
kernels fail to write shows up.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import workloads as W
from tests.support import (TOL, as_f64, compact_subproblem, max_err, nan_like, oracle_step,
                           raw_bytes)

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


def _run(wl_cpu, **kw):
    g = wl_cpu.to("cuda")
    out = nan_like(g.q)
    pkv.run_step(g, out, **kw)
    torch.cuda.synchronize()
    return g, out


# ------------------------------------------------------------ five workloads

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_step_matches_oracle_small(n):
    wl = W.workload(n, small=(n != 1))
    exp, st, kc, vc = oracle_step(wl)
    assert not st.any()
    g, out = _run(wl)
    assert raw_bytes(g.k_cache) == kc.tobytes() and raw_bytes(g.v_cache) == vc.tobytes()
    err = max_err(out, exp)
    assert err <= TOL[wl.dtype], err
    assert pkv.get_error() == 0


@pytest.mark.parametrize("split", [64, 128, 192, 512, 2048])
@pytest.mark.parametrize("n", [2, 5])
def test_split_k_chunk_sizes(n, split):
    wl = W.workload(n, small=True)
    exp, _, _, _ = oracle_step(wl)
    _, out = _run(wl, kv_split_tokens=split)
    assert max_err(out, exp) <= TOL[wl.dtype]
    assert pkv.get_error() == 0


def test_decode_rows_through_prefill_kernel():
    """Decode sequences handed to the varlen kernel (num_decode_seqs = 0)."""
    wl = W.workload(3, small=True)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    out = nan_like(g.q)
    pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    pkv.attention(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                  g.query_start_loc, g.scale, max_query_len=2,
                  max_context_len=g.max_context_len, num_decode_seqs=0)
    assert max_err(out, exp) <= TOL[wl.dtype]


def test_mixed_batch_with_unknown_decode_run():
    wl = W.workload(4, small=True)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    out = nan_like(g.q)
    pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    pkv.attention(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                  g.query_start_loc, g.scale, max_query_len=g.max_query_len,
                  max_context_len=g.max_context_len, num_decode_seqs=-1)
    assert max_err(out, exp) <= TOL[wl.dtype]


# ------------------------------------------------------------ edge shapes

EDGE_CTX = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (8, 1), (16, 2), (12, 4), (32, 2)])
def test_decode_edge_lengths_and_groups(hq, hkv, d):
    wl = W.make_workload([1] * len(EDGE_CTX), EDGE_CTX, num_q_heads=hq, num_kv_heads=hkv,
                         head_size=d, dtype=torch.bfloat16, seed=hq * 100 + hkv + d)
    exp, _, _, _ = oracle_step(wl)
    for split in (0, 64):
        _, out = _run(wl, kv_split_tokens=split)
        assert max_err(out, exp) <= 2e-2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 8), (3, 1), (16, 1), (64, 8), (6, 2),
                                    (128, 1)])
def test_prefill_edge_chunks(hq, hkv, d):
    """Group sizes dividing 128 run the tcgen05 kernel, others (3) the mma.sync one."""
    q_lens = [1, 5, 16, 63, 64, 65, 97, 1, 40]
    ctx = [1, 5, 40, 63, 130, 65, 97, 2, 200]   # includes whole-prompt chunks
    wl = W.make_workload(q_lens, ctx, num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                         dtype=torch.bfloat16, seed=7 * hq + d)
    exp, _, _, _ = oracle_step(wl)
    _, out = _run(wl)
    assert max_err(out, exp) <= 2e-2


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_full_tiles_one_head_per_group(d):
    """G = 1: a query tile is 128 tokens, so only chunks of 128 tokens or more
    have full tiles, whose rows leave through shared memory and a TMA store
    (a box of one head x 128 tokens).  The 129- and 300-token chunks end in a
    partial tile written row by row; the 128-token chunk has no second tile."""
    q_lens = [128, 129, 256, 300, 1]
    ctx = [128, 500, 256, 700, 50]
    wl = W.make_workload(q_lens, ctx, num_q_heads=8, num_kv_heads=8, head_size=d,
                         dtype=torch.bfloat16, seed=5 + d)
    exp, _, _, _ = oracle_step(wl)
    _, out = _run(wl)
    assert max_err(out, exp) <= 2e-2


@pytest.mark.parametrize("d", [64, 128])
def test_f32_decode_and_prefill(d):
    wl = W.make_workload([1, 3, 17, 1], [17, 40, 70, 100], num_q_heads=4, num_kv_heads=2,
                         head_size=d, dtype=torch.float32, seed=d)
    exp, _, _, _ = oracle_step(wl)
    _, out = _run(wl)
    assert max_err(out, exp) <= 1e-5


def test_empty_queries_and_empty_batch():
    wl = W.make_workload([1, 0, 3, 0], [20, 30, 40, 50], num_q_heads=8, num_kv_heads=2,
                         head_size=128, dtype=torch.bfloat16, seed=3)
    exp, _, _, _ = oracle_step(wl)
    _, out = _run(wl)
    assert max_err(out, exp) <= 2e-2
    # zero tokens: both calls are no-ops
    g = wl.to("cuda")
    e = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    pkv.write(e[:, :2], e[:, :2], torch.empty(0, dtype=torch.int64, device="cuda"),
              g.k_cache, g.v_cache)
    assert pkv.get_error() == 0


# ------------------------------------------------------------ KV write

def test_write_skips_padding_and_flags_out_of_range():
    wl = W.workload(3, small=True)
    g = wl.to("cuda")
    A = W.as_oracle_array
    slots = A(wl.slot_mapping).copy()
    slots[2] = -1
    slots[5] = wl.num_blocks * 16 + 3          # past the pool
    kc, vc = A(wl.k_cache).copy(), A(wl.v_cache).copy()
    assert oracle.write(A(wl.k_new), A(wl.v_new), slots, kc, vc) == 1
    pkv.write(g.k_new, g.v_new, torch.from_numpy(slots).cuda(), g.k_cache, g.v_cache)
    assert pkv.get_error() == pkv.ERR_SLOT
    assert raw_bytes(g.k_cache) == kc.tobytes() and raw_bytes(g.v_cache) == vc.tobytes()


# ------------------------------------------------------------ bad device data

def test_bad_block_id_flags_and_spares_other_sequences():
    wl = W.workload(2, small=True)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    g.block_tables[1, 0] = wl.num_blocks + 5
    out = nan_like(g.q)
    pkv.run_step(g, out)
    assert pkv.get_error() & pkv.ERR_BLOCK_ID
    others = [t for t in range(g.q.shape[0]) if t != 1]
    assert max_err(out, exp, rows=others) <= 2e-2


def test_bad_lengths_zero_rows_and_flag():
    wl = W.make_workload([1, 1, 4, 3], [20, 30, 40, 50], num_q_heads=8, num_kv_heads=2,
                         head_size=128, dtype=torch.bfloat16, seed=11)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    g.context_lens[0] = 0                  # decode row with no keys
    g.context_lens[2] = 3                  # 4 queries but 3 keys
    out = nan_like(g.q)
    pkv.attention(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                  g.query_start_loc, g.scale, max_query_len=4, max_context_len=50,
                  num_decode_seqs=2)
    bits = pkv.get_error()
    assert bits & pkv.ERR_CONTEXT_LEN and bits & pkv.ERR_QUERY_LEN
    o = as_f64(out)
    assert (o[0] == 0).all() and (o[2:6] == 0).all()
    assert max_err(out, exp, rows=[1, 6, 7, 8]) <= 2e-2


def test_decode_run_with_long_query_is_flagged():
    wl = W.make_workload([1, 2, 1], [20, 30, 40], num_q_heads=4, num_kv_heads=4,
                         head_size=64, dtype=torch.bfloat16, seed=12)
    g = wl.to("cuda")
    out = torch.zeros_like(g.q)
    pkv.attention(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                  g.query_start_loc, g.scale, max_query_len=2, max_context_len=40,
                  num_decode_seqs=3)
    assert pkv.get_error() & pkv.ERR_DECODE_QLEN


# ------------------------------------------------------------ host-side errors

def test_host_argument_errors():
    import ctypes
    lib = pkv.load()
    wl = W.workload(2, small=True).to("cuda")
    desc = pkv.cache_desc(wl.k_cache)
    meta = pkv.attn_meta(wl.q, wl.block_tables, wl.context_lens, max_query_len=1,
                         max_context_len=wl.max_context_len, kv_split_tokens=64)
    out = torch.empty_like(wl.q)
    need = pkv.workspace_size(wl.k_cache, meta)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(**over):
        args = dict(out=out.data_ptr(), q=wl.q.data_ptr(), kc=wl.k_cache.data_ptr(),
                    vc=wl.v_cache.data_ptr(), bt=wl.block_tables.data_ptr(),
                    cl=wl.context_lens.data_ptr(), qsl=wl.query_start_loc.data_ptr(),
                    desc=desc, meta=meta, ws=ws.data_ptr(), wsb=need)
        args.update(over)
        return lib.pkv_attention(args["out"], args["q"], args["kc"], args["vc"], args["bt"],
                                 args["cl"], args["qsl"], ctypes.c_float(wl.scale),
                                 ctypes.byref(args["desc"]), ctypes.byref(args["meta"]),
                                 args["ws"], args["wsb"], s)

    assert call() == 0
    assert call(q=0) == -1
    assert call(wsb=need - 1) == -5
    assert call(ws=0) == -5
    assert call(out=out.data_ptr() + 2) == -6
    bad = pkv.CacheDesc(desc.num_blocks, 16, desc.num_kv_heads, 96, desc.dtype)
    assert call(desc=bad) == -3
    bad = pkv.CacheDesc(desc.num_blocks, 32, desc.num_kv_heads, 128, desc.dtype)
    assert call(desc=bad) == -3
    bad = pkv.CacheDesc(desc.num_blocks, 16, desc.num_kv_heads, 128, 7)
    assert call(desc=bad) == -2
    m2 = pkv.AttnMeta(*[getattr(meta, f) for f, _ in pkv.AttnMeta._fields_])
    m2.num_q_heads = 33
    assert call(meta=m2) == -4
    m2.num_q_heads = meta.num_q_heads
    m2.kv_split_tokens = 100
    assert call(meta=m2) == -8
    torch.cuda.synchronize()
    assert pkv.get_error() == 0


# ------------------------------------------------------------ full sizes

def _sample_seqs(ctx, k):
    order = np.argsort(ctx)
    pick = {int(order[0]), int(order[-1])}
    pick.update(int(x) for x in order[np.linspace(0, len(order) - 1, k).astype(int)])
    return sorted(pick)


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_full_size_step_sampled_against_oracle(n):
    """Full-size workload, the launch configuration the bench times: the write
    is compared over the whole pool, attention on sampled sequences."""
    g = W.workload(n, device="cuda")
    pre_k, pre_v = g.k_cache.clone(), g.v_cache.clone()
    out = nan_like(g.q)
    pkv.run_step(g, out)
    torch.cuda.synchronize()
    assert pkv.get_error() == 0
    assert torch.isfinite(out.float()).all()
    # write: every new row landed, nothing else moved (oracle write on CPU)
    A = W.as_oracle_array
    kc, vc = A(pre_k).copy(), A(pre_v).copy()
    assert oracle.write(A(g.k_new), A(g.v_new), A(g.slot_mapping), kc, vc) == 0
    assert np.array_equal(A(g.k_cache), kc) and np.array_equal(A(g.v_cache), vc)
    del kc, vc
    # attention: every row of sampled decode sequences, a few rows of each
    # prefill chunk
    nd = g.num_decode_seqs
    dec = _sample_seqs(g.ctx_lens[:nd], 6) if nd else []
    P, rows = compact_subproblem(g, dec, pre_k, pre_v) if dec else (None, [])
    if dec:
        exp, st = oracle.attention(P.q, P.k_cache, P.v_cache, P.block_tables,
                                   P.context_lens, P.query_start_loc, g.scale)
        assert not st.any()
        err = max_err(out[torch.as_tensor(rows, device="cuda")], exp)
        assert err <= 2e-2, err
    # every row and head of every prefill chunk (the tcgen05 kernel's tile
    # pairs, row tails and key tails all live in these 512-row chunks)
    pf = list(range(nd, g.num_seqs))
    if pf:
        P, rows = compact_subproblem(g, pf, pre_k, pre_v)
        exp, st = oracle.attention(P.q, P.k_cache, P.v_cache, P.block_tables,
                                   P.context_lens, P.query_start_loc, g.scale)
        assert not st.any()
        err = max_err(out[torch.as_tensor(rows, device="cuda")], exp)
        assert err <= 2e-2, err


# ------------------------------------------------------------ CUDA graphs

def test_step_captured_in_a_cuda_graph_replays_correctly():
    """The calls only enqueue work (no allocation, no synchronisation), so a
    whole step -- write, split-K attention, combine -- can be captured once and
    replayed; replays pick up new inputs written into the same buffers."""
    wl = W.workload(5, small=True)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=1,
                         max_context_len=g.max_context_len, kv_split_tokens=128)
    ws = torch.empty(pkv.workspace_size(g.k_cache, meta), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    out = torch.empty_like(g.q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # first call on the device: set-up outside the capture
        pkv.run_step(g, out, workspace=ws, kv_split_tokens=128)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkv.run_step(g, out, workspace=ws, kv_split_tokens=128)
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert max_err(out, exp) <= 2e-2
    # new queries in the same buffer, replay again
    q2 = torch.randn(wl.q.shape, generator=torch.Generator().manual_seed(99)).to(wl.q.dtype)
    wl2 = W.Workload(**{k: getattr(wl, k) for k in wl.__dataclass_fields__})
    wl2.q = q2
    exp2, _, _, _ = oracle_step(wl2)
    g.q.copy_(q2)
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert max_err(out, exp2) <= 2e-2
    assert pkv.get_error() == 0
