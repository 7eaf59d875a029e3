"""Cascade attention on the GPU against the oracle: a batch whose sequences
share their first P blocks, the prefix attended once for all rows (tcgen05
kernel when the group size divides 128 -- G = 1, 4, 8 here -- else, for decode
rows, the mma.sync decode kernel over (sequence, head) columns -- G = 3), each
row's own keys after it (decode rows on the split-K decode kernel, chunked
prefill rows causally on the tcgen05 kernel), the partials merged.  The
result must be the plain attention (oracle) within the bf16 tolerance, and
equal pkv_attention's within it."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import workloads as W
from tests.support import TOL, max_err, nan_like, oracle_step

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


def _shared(S, pblocks, hq, hkv, d, lo, hi, seed, dtype=torch.bfloat16):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(max(lo, pblocks * 16 + 1), hi, S, endpoint=True)
    return W.make_workload([1] * S, ctx, num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                           dtype=dtype, seed=seed, shared_prefix_blocks=pblocks,
                           shared_seqs=tuple(range(S)))


def _cascade(wl, pblocks, **kw):
    g = wl.to("cuda")
    out = nan_like(g.q)
    pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    pkv.attention_cascade(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                          g.query_start_loc, g.scale, pblocks,
                          max_context_len=g.max_context_len, **kw)
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S,hq,hkv", [(8, 8, 8), (16, 32, 8), (3, 64, 8), (40, 8, 2), (1, 4, 4),
                                     (9, 12, 4), (200, 32, 8)])
@pytest.mark.parametrize("pblocks", [1, 5, 64])
def test_cascade_matches_oracle(S, hq, hkv, d, pblocks):
    wl = _shared(S, pblocks, hq, hkv, d, 2, pblocks * 16 + 700, seed=S * 7 + pblocks + d)
    exp, st, _, _ = oracle_step(wl)
    assert not st.any()
    g, out = _cascade(wl, pblocks)
    assert max_err(out, exp) <= TOL[torch.bfloat16]
    assert pkv.get_error() == 0


@pytest.mark.parametrize("split", [0, 64, 256, 2048])
def test_cascade_split_sizes_and_long_suffixes(split):
    wl = _shared(12, 20, 32, 8, 128, 1000, 9000, seed=split + 1)
    exp, _, _, _ = oracle_step(wl)
    _, out = _cascade(wl, 20, kv_split_tokens=split)
    assert max_err(out, exp) <= TOL[torch.bfloat16]


def test_cascade_equals_plain_attention():
    wl = _shared(24, 16, 32, 8, 128, 300, 3000, seed=5)
    g, out_c = _cascade(wl, 16)
    out_p = nan_like(g.q)
    pkv.attention(out_p, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                  g.query_start_loc, g.scale, max_query_len=1, max_context_len=g.max_context_len)
    torch.cuda.synchronize()
    assert float((out_c.float() - out_p.float()).abs().max()) <= 2e-2


def test_cascade_of_workload4_sharing_sequences():
    """The mixed workload's 16 decode sequences that share 64 blocks, as one
    cascade call (the rest of the batch goes through pkv_attention)."""
    wl = W.workload(4, small=False)
    nsh = len(wl.shared_seqs)
    sub = W.make_workload(wl.q_lens[:nsh], wl.ctx_lens[:nsh], num_q_heads=32, num_kv_heads=8,
                          head_size=128, seed=44, shared_prefix_blocks=wl.shared_prefix_blocks,
                          shared_seqs=tuple(range(nsh)))
    exp, _, _, _ = oracle_step(sub)
    _, out = _cascade(sub, wl.shared_prefix_blocks)
    assert max_err(out, exp) <= TOL[torch.bfloat16]


def test_cascade_row_inside_the_prefix_is_flagged_and_zeroed():
    wl = _shared(8, 4, 8, 2, 128, 100, 400, seed=3)
    g = wl.to("cuda")
    pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    cl = g.context_lens.clone()
    cl[2] = 4 * 16                           # its query would sit inside the prefix
    out = nan_like(g.q)
    pkv.attention_cascade(out, g.q, g.k_cache, g.v_cache, g.block_tables, cl,
                          g.query_start_loc, g.scale, 4, max_context_len=g.max_context_len)
    assert pkv.get_error() == pkv.ERR_CONTEXT_LEN
    assert float(out[2].float().abs().max()) == 0.0
    A = W.as_oracle_array
    exp, _, _, _ = oracle_step(wl)
    rows = [r for r in range(8) if r != 2]
    assert max_err(out, exp, rows=rows) <= TOL[torch.bfloat16]


def test_cascade_host_errors():
    lib = pkv.load()
    wl = _shared(8, 16, 8, 2, 128, 300, 600, seed=1)
    g = wl.to("cuda")
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=1,
                         max_context_len=g.max_context_len)
    mw = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=1,
                       max_context_len=g.max_context_len, sliding_window=64)
    desc = pkv.cache_desc(g.k_cache)
    E_META = -8
    for bad in (pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=2,
                              max_context_len=g.max_context_len), mw):
        assert lib.pkv_attention_cascade_workspace_size(ctypes.byref(desc), ctypes.byref(bad),
                                                        16) == ctypes.c_size_t(-1).value
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(g.q)
    args = (out.data_ptr(), g.q.data_ptr(), g.k_cache.data_ptr(), g.v_cache.data_ptr(),
            g.block_tables.data_ptr(), g.context_lens.data_ptr(), g.query_start_loc.data_ptr(),
            ctypes.c_float(g.scale))
    mq = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=2,
                       max_context_len=g.max_context_len)
    assert lib.pkv_attention_cascade(*args, 16, ctypes.byref(desc), ctypes.byref(mq),
                                     ws.data_ptr(), ws.numel(), None) == E_META
    assert lib.pkv_attention_cascade(*args, 0, ctypes.byref(desc), ctypes.byref(meta),
                                     ws.data_ptr(), ws.numel(), None) == E_META
    assert lib.pkv_attention_cascade(*args, 16, ctypes.byref(desc), ctypes.byref(meta),
                                     None, 0, None) == -5           # PKV_E_WORKSPACE
    torch.cuda.synchronize()
    assert pkv.get_error() == 0


def test_cascade_captured_in_a_cuda_graph_replays_correctly():
    wl = _shared(24, 16, 32, 8, 128, 300, 3000, seed=6)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=1,
                         max_context_len=g.max_context_len)
    ws = torch.empty(pkv.cascade_workspace_size(g.k_cache, meta, 16), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(g.q)
    s = torch.cuda.Stream()

    def step():
        pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, stream=s)
        pkv.attention_cascade(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                              g.query_start_loc, g.scale, 16, max_context_len=g.max_context_len,
                              workspace=ws, stream=s)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert max_err(out, exp) <= TOL[torch.bfloat16]
    assert pkv.get_error() == 0


# ------------------------------------------------------------ e4m3 caches

@pytest.mark.parametrize("S,hq,hkv,pblocks,d", [(8, 8, 8, 1, 128), (16, 32, 8, 5, 128),
                                                (40, 8, 2, 64, 128), (200, 32, 8, 5, 128),
                                                (3, 64, 8, 16, 128), (8, 8, 8, 1, 64),
                                                (16, 32, 8, 5, 64), (40, 8, 2, 64, 64)])
def test_cascade_fp8_matches_oracle(S, hq, hkv, pblocks, d):
    """Descales drawn per (sequence, kv head): every row, the shared keys
    included, must use its own sequence's.  head_size 64 and 128."""
    from tests.support import fp8_scale_tensors, gpu_fp8_caches, oracle_step_fp8
    wl = _shared(S, pblocks, hq, hkv, d, 2, pblocks * 16 + 700, seed=S + pblocks + d)
    g = wl.to("cuda")
    ks, vs, _, _ = fp8_scale_tensors(hkv, S, 13)
    rng = np.random.default_rng(S * 3 + pblocks)
    kd = torch.from_numpy(rng.uniform(0.002, 0.03, (S, hkv)).astype(np.float32)).cuda()
    vd = torch.from_numpy(rng.uniform(0.005, 0.04, (S, hkv)).astype(np.float32)).cuda()
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    pkv.write_fp8(g.k_new, g.v_new, g.slot_mapping, kc8, vc8, ks, vs)
    out = nan_like(g.q)
    pkv.attention_cascade_fp8(out, g.q, kc8, vc8, g.block_tables, g.context_lens,
                              g.query_start_loc, g.scale, pblocks, kd, vd,
                              max_context_len=g.max_context_len)
    torch.cuda.synchronize()
    exp, st, _, _ = oracle_step_fp8(wl, ks, vs, kd, vd)
    assert not st.any()
    assert max_err(out, exp) <= TOL[torch.bfloat16]
    assert pkv.get_error() == 0


def test_cascade_fp8_shapes_without_the_tcgen05_prefix_are_refused():
    lib = pkv.load()
    for hq, hkv, d in ((12, 4, 128), (12, 4, 64)):          # group 3
        wl = _shared(8, 4, hq, hkv, d, 100, 300, seed=2)
        g = wl.to("cuda")
        kc8 = torch.zeros(g.k_cache.shape, dtype=torch.uint8, device="cuda")
        meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=1,
                             max_context_len=g.max_context_len)
        desc = pkv.cache_desc(kc8)
        assert lib.pkv_attention_cascade_workspace_size(ctypes.byref(desc), ctypes.byref(meta),
                                                        4) == ctypes.c_size_t(-1).value
        with pytest.raises(pkv.PkvError):
            kd = torch.ones((8, hkv), dtype=torch.float32, device="cuda")
            pkv.attention_cascade_fp8(torch.zeros_like(g.q), g.q, kc8, kc8, g.block_tables,
                                      g.context_lens, g.query_start_loc, g.scale, 4, kd, kd,
                                      max_context_len=g.max_context_len,
                                      workspace=torch.empty(1 << 20, dtype=torch.uint8,
                                                            device="cuda"))
    torch.cuda.synchronize()
    assert pkv.get_error() == 0


# ------------------------------------------------- chunked-prefill rows

def _shared_mixed(nd, chunks, pblocks, hq, hkv, d, seed, extra_hi=600):
    """nd decode sequences then one chunk of each length in `chunks`, every
    sequence sharing its first pblocks blocks; every query row after them."""
    rng = np.random.default_rng(seed)
    P = pblocks * 16
    q_lens = [1] * nd + list(chunks)
    ctx = [P + int(q) + int(rng.integers(0, extra_hi)) for q in q_lens]
    return W.make_workload(q_lens, ctx, num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                           seed=seed, shared_prefix_blocks=pblocks,
                           shared_seqs=tuple(range(len(q_lens))))


MIXED = [(0, (1, 5, 97), 1, 8, 8, 128), (3, (17, 128, 200), 5, 32, 8, 128),
         (6, (64, 511), 64, 32, 8, 128), (2, (40, 300), 17, 16, 1, 128),
         (4, (33, 129), 5, 32, 8, 64), (1, (256,), 8, 128, 1, 128)]


@pytest.mark.parametrize("nd,chunks,pblocks,hq,hkv,d", MIXED)
def test_cascade_with_chunked_prefill_rows(nd, chunks, pblocks, hq, hkv, d):
    """Decode rows and prefill chunks in one cascade call: every row of every
    chunk equals the plain attention, and the oracle's own cascade split
    (prefix state merged with the causal suffix state) agrees with both."""
    wl = _shared_mixed(nd, chunks, pblocks, hq, hkv, d, seed=nd * 31 + pblocks + d)
    exp, st, kc, vc = oracle_step(wl)
    assert not st.any()
    A = W.as_oracle_array
    P = oracle.Problem(A(wl.q), kc, vc, A(wl.block_tables), A(wl.context_lens),
                       A(wl.query_start_loc), wl.scale)
    assert np.abs(oracle.cascade(P, pblocks * 16) - exp).max() < 1e-9
    g, out = _cascade(wl, pblocks, max_query_len=wl.max_query_len, num_decode_seqs=nd)
    assert max_err(out, exp) <= TOL[torch.bfloat16]
    assert pkv.get_error() == 0


@pytest.mark.parametrize("nd,chunks,pblocks,hq,hkv,d", MIXED[:3] + MIXED[4:5])
def test_cascade_fp8_with_chunked_prefill_rows(nd, chunks, pblocks, hq, hkv, d):
    from tests.support import fp8_scale_tensors, gpu_fp8_caches, oracle_step_fp8
    wl = _shared_mixed(nd, chunks, pblocks, hq, hkv, d, seed=nd * 17 + pblocks + d)
    g = wl.to("cuda")
    S = g.num_seqs
    ks, vs, _, _ = fp8_scale_tensors(hkv, S, 5)
    rng = np.random.default_rng(nd + pblocks)
    kd = torch.from_numpy(rng.uniform(0.002, 0.03, (S, hkv)).astype(np.float32)).cuda()
    vd = torch.from_numpy(rng.uniform(0.005, 0.04, (S, hkv)).astype(np.float32)).cuda()
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    pkv.write_fp8(g.k_new, g.v_new, g.slot_mapping, kc8, vc8, ks, vs)
    out = nan_like(g.q)
    pkv.attention_cascade_fp8(out, g.q, kc8, vc8, g.block_tables, g.context_lens,
                              g.query_start_loc, g.scale, pblocks, kd, vd,
                              max_context_len=g.max_context_len, max_query_len=g.max_query_len,
                              num_decode_seqs=nd)
    torch.cuda.synchronize()
    exp, st, _, _ = oracle_step_fp8(wl, ks, vs, kd, vd)
    assert not st.any()
    assert max_err(out, exp) <= TOL[torch.bfloat16]
    assert pkv.get_error() == 0


def test_cascade_chunk_inside_the_prefix_is_zeroed_and_flagged():
    """A chunk whose first row sits inside the shared prefix breaks the
    cascade's contract: its rows come out zero with PKV_ERR_CONTEXT_LEN; the
    other sequences are unaffected."""
    wl = _shared_mixed(2, (40, 50), 4, 8, 2, 128, seed=3)
    bad = 3                                          # the chunk of 50 rows
    L = int(wl.ctx_lens[bad])
    wl.ctx_lens[bad] = 4 * 16 + 10                   # L - q_len < 64 shared keys
    wl.context_lens[bad] = int(wl.ctx_lens[bad])
    good = [0, 1, 2]
    exp, st, _, _ = oracle_step(wl)
    g, out = _cascade(wl, 4, max_query_len=wl.max_query_len, num_decode_seqs=2)
    qsl = wl.query_start_loc.numpy()
    rows_good = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in good])
    rows_bad = np.arange(qsl[bad], qsl[bad + 1])
    assert max_err(out, exp, rows_good) <= TOL[torch.bfloat16]
    assert not out[torch.from_numpy(rows_bad).cuda()].float().any()
    assert pkv.get_error(clear=True) & (1 << 2)
    assert L > 0


def test_cascade_chunk_rows_refused_without_their_kernels():
    g = _shared_mixed(1, (20,), 4, 12, 4, 128, seed=4).to("cuda")     # group 3
    with pytest.raises(pkv.PkvError):
        pkv.attention_cascade(torch.zeros_like(g.q), g.q, g.k_cache, g.v_cache, g.block_tables,
                              g.context_lens, g.query_start_loc, g.scale, 4,
                              max_context_len=g.max_context_len, max_query_len=20,
                              num_decode_seqs=1,
                              workspace=torch.empty(1 << 24, dtype=torch.uint8, device="cuda"))
    g = _shared_mixed(1, (20,), 4, 8, 2, 128, seed=5).to("cuda")
    with pytest.raises(pkv.PkvError):                                  # decode count unknown
        pkv.attention_cascade(torch.zeros_like(g.q), g.q, g.k_cache, g.v_cache, g.block_tables,
                              g.context_lens, g.query_start_loc, g.scale, 4,
                              max_context_len=g.max_context_len, max_query_len=20,
                              num_decode_seqs=-1,
                              workspace=torch.empty(1 << 24, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert pkv.get_error() == 0
