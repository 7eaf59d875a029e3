"""FP8 (e4m3) KV cache on the GPU against the oracle: pkv_write_fp8 must give
the oracle's codes bit for bit (fp32 division by the kv head's scale, round to
nearest even, clamp to 448); pkv_attention_fp8 must match the oracle's
attention over decode(code) * descale within the bf16 tolerance."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import workloads as W
from tests.support import (TOL, as_f64, compact_subproblem_fp8, fp8_scale_tensors,
                           gpu_fp8_caches, max_err, nan_like, oracle_fp8_caches,
                           oracle_step_fp8, raw_bytes)

pytestmark = pytest.mark.gpu
TOL_FP8 = TOL[torch.bfloat16]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    pkv.load()
    pkv.get_error(clear=True)
    yield
    assert pkv.get_error(clear=True) == 0


def _step(g, kc8, vc8, ks, vs, kd, vd, **kw):
    """This step's write into the e4m3 caches, then attention."""
    out = nan_like(g.q)
    pkv.write_fp8(g.k_new, g.v_new, g.slot_mapping, kc8, vc8, ks, vs)
    kw.setdefault("max_query_len", g.max_query_len)
    kw.setdefault("max_context_len", g.max_context_len)
    kw.setdefault("num_decode_seqs", g.num_decode_seqs)
    pkv.attention_fp8(out, g.q, kc8, vc8, g.block_tables, g.context_lens, g.query_start_loc,
                      g.scale, kd, vd, **kw)
    torch.cuda.synchronize()
    return out


def _run(wl, seed=11, window=0, **kw):
    g = wl.to("cuda")
    ks, vs, kd, vd = fp8_scale_tensors(g.num_kv_heads, g.num_seqs, seed)
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    out = _step(g, kc8, vc8, ks, vs, kd, vd, sliding_window=window, **kw)
    exp, st, kc, vc = oracle_step_fp8(wl, ks, vs, kd, vd, window=window)
    assert not st.any()
    return out, exp, (kc8, vc8), (kc, vc)


# ------------------------------------------------------------ write

@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_write_fp8_codes_bit_exact(n):
    wl = W.workload(n, small=True)
    out, exp, (kc8, vc8), (kc, vc) = _run(wl)
    assert raw_bytes(kc8) == kc.tobytes() and raw_bytes(vc8) == vc.tobytes()
    assert max_err(out, exp) <= TOL_FP8
    assert pkv.get_error() == 0


def test_write_fp8_clamps_and_keeps_signs():
    """Scales small enough that a large share of N(0, 1) values saturate at
    +-448, and values that underflow to (signed) zero and subnormals."""
    wl = W.make_workload([3, 1, 20], [40, 17, 60], num_q_heads=8, num_kv_heads=4,
                         head_size=128, seed=91)
    g = wl.to("cuda")
    ks = torch.tensor([0.002, 0.05, 1e-3, 300.0], dtype=torch.float32, device="cuda")
    vs = torch.tensor([40.0, 0.004, 0.02, 1.0], dtype=torch.float32, device="cuda")
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    pkv.write_fp8(g.k_new, g.v_new, g.slot_mapping, kc8, vc8, ks, vs)
    torch.cuda.synchronize()
    kc, vc = oracle_fp8_caches(wl, ks, vs)
    A = W.as_oracle_array
    assert oracle.write_fp8(A(wl.k_new), A(wl.v_new), A(wl.slot_mapping), kc, vc, A(ks),
                            A(vs)) == 0
    assert raw_bytes(kc8) == kc.tobytes() and raw_bytes(vc8) == vc.tobytes()
    codes = kc8.cpu().numpy()
    assert ((codes & 0x7F) == 0x7E).any()          # saturated at 448
    assert ((codes & 0x7F) == 0).any()             # flushed to (signed) zero


def test_write_fp8_padding_and_out_of_range_slot():
    wl = W.make_workload([1, 1], [20, 40], num_q_heads=4, num_kv_heads=2, head_size=64,
                         seed=5)
    g = wl.to("cuda")
    ks, vs, _, _ = fp8_scale_tensors(2, 2, 3)
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    before_k, before_v = kc8.clone(), vc8.clone()
    nslots = g.num_blocks * 16
    slots = torch.tensor([-1, nslots], dtype=torch.int64, device="cuda")
    pkv.write_fp8(g.k_new, g.v_new, slots, kc8, vc8, ks, vs)
    assert pkv.get_error() == pkv.ERR_SLOT
    assert torch.equal(kc8, before_k) and torch.equal(vc8, before_v)


def test_float8_dtype_tensors_are_accepted():
    wl = W.workload(2, small=True)
    g = wl.to("cuda")
    ks, vs, kd, vd = fp8_scale_tensors(g.num_kv_heads, g.num_seqs, 11)
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    kf, vf = kc8.view(torch.float8_e4m3fn), vc8.view(torch.float8_e4m3fn)
    out = _step(g, kf, vf, ks, vs, kd, vd)
    exp, _, kc, vc = oracle_step_fp8(wl, ks, vs, kd, vd)
    assert raw_bytes(kc8) == kc.tobytes()
    assert max_err(out, exp) <= TOL_FP8


# ------------------------------------------------------------ attention

@pytest.mark.parametrize("split", [0, 64, 192, 2048])
@pytest.mark.parametrize("n", [2, 5])
def test_fp8_decode_split_sizes(n, split):
    out, exp, _, _ = _run(W.workload(n, small=True), kv_split_tokens=split)
    assert max_err(out, exp) <= TOL_FP8
    assert pkv.get_error() == 0


EDGE_CTX = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (8, 1), (12, 4), (32, 2)])
def test_fp8_decode_edge_lengths_and_groups(hq, hkv, d):
    wl = W.make_workload([1] * len(EDGE_CTX), EDGE_CTX, num_q_heads=hq, num_kv_heads=hkv,
                         head_size=d, seed=hq * 100 + hkv + d)
    for split in (0, 64):
        out, exp, _, _ = _run(wl, kv_split_tokens=split)
        assert max_err(out, exp) <= TOL_FP8


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (32, 8), (3, 1), (16, 1), (128, 1)])
def test_fp8_prefill_edge_chunks(hq, hkv, d):
    q_lens = [1, 5, 16, 63, 64, 65, 97, 1, 40]
    ctx = [1, 5, 40, 63, 130, 65, 97, 2, 200]
    wl = W.make_workload(q_lens, ctx, num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                         seed=7 * hq + d)
    out, exp, _, _ = _run(wl)
    assert max_err(out, exp) <= TOL_FP8


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_prefill_full_tiles_one_head_per_group(d):
    """G = 1 with chunks of 128 tokens or more: full query tiles (TMA-stored
    rows) and partial ones, over widened e4m3 tiles."""
    wl = W.make_workload([128, 129, 256, 300, 1], [128, 500, 256, 700, 50], num_q_heads=8,
                         num_kv_heads=8, head_size=d, seed=9 + d)
    out, exp, _, _ = _run(wl)
    assert max_err(out, exp) <= TOL_FP8


def test_fp8_mixed_batch_with_prefix_sharing():
    out, exp, _, _ = _run(W.workload(4, small=True))
    assert max_err(out, exp) <= TOL_FP8


@pytest.mark.parametrize("window", [1, 17, 100, 1000])
def test_fp8_sliding_window(window):
    wl = W.make_workload([1, 1, 1, 40, 1, 64], [1, 300, 1000, 400, 2000, 1500],
                         num_q_heads=16, num_kv_heads=4, head_size=128, seed=window)
    out, exp, _, _ = _run(wl, window=window)
    assert max_err(out, exp) <= TOL_FP8


def test_fp8_descales_are_per_sequence_and_head():
    """Descales unrelated to the write scales, different for every (sequence,
    kv head): a swapped or shared index shows up as a wrong output."""
    wl = W.make_workload([1, 1, 1, 30, 1], [50, 700, 129, 200, 1000], num_q_heads=16,
                         num_kv_heads=4, head_size=128, seed=23)
    g = wl.to("cuda")
    ks, vs, _, _ = fp8_scale_tensors(4, 5, 29)
    rng = np.random.default_rng(31)
    # the size of real descales (so that K/V stay O(1)), but drawn per entry
    kd = torch.from_numpy(rng.uniform(0.002, 0.03, (5, 4)).astype(np.float32)).cuda()
    vd = torch.from_numpy(rng.uniform(0.005, 0.04, (5, 4)).astype(np.float32)).cuda()
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    for split in (0, 64):
        kc8b, vc8b = kc8.clone(), vc8.clone()
        out = _step(g, kc8b, vc8b, ks, vs, kd, vd, kv_split_tokens=split)
        exp, st, _, _ = oracle_step_fp8(wl, ks, vs, kd, vd)
        assert not st.any()
        assert max_err(out, exp) <= TOL_FP8


def _sample_seqs(ctx, k):
    order = np.argsort(ctx)
    pick = {int(order[0]), int(order[-1])}
    pick.update(int(x) for x in order[np.linspace(0, len(order) - 1, k).astype(int)])
    return sorted(pick)


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_fp8_full_size_step_sampled_against_oracle(n):
    """Full-size workload with an e4m3 cache, the launch configuration the
    bench's FP8 line times: the write is compared on the new tokens' slots, the
    attention on sampled sequences."""
    g = W.workload(n, device="cuda")
    ks, vs, kd, vd = fp8_scale_tensors(g.num_kv_heads, g.num_seqs, 11)
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    out = _step(g, kc8, vc8, ks, vs, kd, vd)
    assert pkv.get_error() == 0
    assert torch.isfinite(out.float()).all()
    # the new tokens' rows against the oracle's quantisation of the same rows
    A = W.as_oracle_array
    T, hkv, d = g.k_new.shape
    kq = np.full((T, 1, hkv, d), 0, np.uint8)
    vq = kq.copy()
    assert oracle.write_fp8(A(g.k_new), A(g.v_new), np.arange(T, dtype=np.int64), kq, vq,
                            A(ks), A(vs)) == 0
    nb = g.num_blocks
    got_k = kc8.view(nb * 16, hkv, d).index_select(0, g.slot_mapping).cpu().numpy()
    got_v = vc8.view(nb * 16, hkv, d).index_select(0, g.slot_mapping).cpu().numpy()
    assert np.array_equal(got_k, kq[:, 0]) and np.array_equal(got_v, vq[:, 0])
    nd = g.num_decode_seqs
    dec = _sample_seqs(g.ctx_lens[:nd], 6) if nd else []
    if dec:
        P, rows = compact_subproblem_fp8(g, dec, ks, vs, kd, vd)
        exp, st = oracle.attention(P.q, P.k_cache, P.v_cache, P.block_tables, P.context_lens,
                                   P.query_start_loc, g.scale, k_descale=P.k_descale,
                                   v_descale=P.v_descale)
        assert not st.any()
        err = max_err(out[torch.as_tensor(rows, device="cuda")], exp)
        assert err <= TOL_FP8, err
    # every row and head of every prefill chunk
    pf = list(range(nd, g.num_seqs))
    if pf:
        P, rows = compact_subproblem_fp8(g, pf, ks, vs, kd, vd)
        exp, st = oracle.attention(P.q, P.k_cache, P.v_cache, P.block_tables,
                                   P.context_lens, P.query_start_loc, g.scale,
                                   k_descale=P.k_descale, v_descale=P.v_descale)
        assert not st.any()
        err = max_err(out[torch.as_tensor(rows, device="cuda")], exp)
        assert err <= TOL_FP8, err


# ------------------------------------------------------------ host errors

def test_fp8_host_argument_errors():
    lib = pkv.load()
    wl = W.make_workload([1], [20], num_q_heads=4, num_kv_heads=2, head_size=64, seed=1)
    g = wl.to("cuda")
    ks, vs, kd, vd = fp8_scale_tensors(2, 1, 3)
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    d8 = pkv.cache_desc(kc8)
    dbf = pkv.cache_desc(g.k_cache)
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=1,
                         max_context_len=20)
    out = torch.zeros_like(g.q)
    args = lambda c, dsc: (out.data_ptr(), g.q.data_ptr(), c.data_ptr(), c.data_ptr(),
                           g.block_tables.data_ptr(), g.context_lens.data_ptr(),
                           g.query_start_loc.data_ptr(), ctypes.c_float(0.125))
    E_NULL, E_DTYPE = -1, -2
    # the bf16 entry points refuse an e4m3 cache, the fp8 ones a bf16 cache
    assert lib.pkv_attention(*args(kc8, d8), ctypes.byref(d8), ctypes.byref(meta), None, 0,
                             None) == E_DTYPE
    assert lib.pkv_write(g.k_new.data_ptr(), g.v_new.data_ptr(), g.slot_mapping.data_ptr(), 1,
                         kc8.data_ptr(), vc8.data_ptr(), ctypes.byref(d8), None) == E_DTYPE
    assert lib.pkv_attention_fp8(*args(g.k_cache, dbf), kd.data_ptr(), vd.data_ptr(),
                                 ctypes.byref(dbf), ctypes.byref(meta), None, 0,
                                 None) == E_DTYPE
    assert lib.pkv_write_fp8(g.k_new.data_ptr(), g.v_new.data_ptr(), g.slot_mapping.data_ptr(),
                             1, g.k_cache.data_ptr(), g.v_cache.data_ptr(), ks.data_ptr(),
                             vs.data_ptr(), ctypes.byref(dbf), None) == E_DTYPE
    # descales and scales are required
    assert lib.pkv_attention_fp8(*args(kc8, d8), None, vd.data_ptr(), ctypes.byref(d8),
                                 ctypes.byref(meta), None, 0, None) == E_NULL
    assert lib.pkv_write_fp8(g.k_new.data_ptr(), g.v_new.data_ptr(), g.slot_mapping.data_ptr(),
                             1, kc8.data_ptr(), vc8.data_ptr(), None, vs.data_ptr(),
                             ctypes.byref(d8), None) == E_NULL
    torch.cuda.synchronize()
    assert pkv.get_error() == 0


def test_fp8_step_captured_in_a_cuda_graph_replays_correctly():
    """Quantising write + e4m3 attention (decode split-K, combine and the
    tcgen05 prefill with its widening warps) captured once and replayed."""
    wl = W.workload(4, small=True)
    g = wl.to("cuda")
    ks, vs, kd, vd = fp8_scale_tensors(g.num_kv_heads, g.num_seqs, 11)
    kc8, vc8 = gpu_fp8_caches(g, ks, vs)
    exp, _, _, _ = oracle_step_fp8(wl, ks, vs, kd, vd)
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=g.max_query_len,
                         max_context_len=g.max_context_len, num_decode_seqs=g.num_decode_seqs,
                         kv_split_tokens=128)
    ws = torch.empty(max(pkv.workspace_size(kc8, meta), 1), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(g.q)
    s = torch.cuda.Stream()

    def step():
        pkv.write_fp8(g.k_new, g.v_new, g.slot_mapping, kc8, vc8, ks, vs, stream=s)
        pkv.attention_fp8(out, g.q, kc8, vc8, g.block_tables, g.context_lens,
                          g.query_start_loc, g.scale, kd, vd, max_query_len=g.max_query_len,
                          max_context_len=g.max_context_len, num_decode_seqs=g.num_decode_seqs,
                          kv_split_tokens=128, workspace=ws, stream=s)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert max_err(out, exp) <= TOL_FP8
    assert pkv.get_error() == 0
