"""Batches with both decode and prefill rows: pkv_attention enqueues the
prefill launch on the library's high-priority side stream, forked from the
caller's stream and joined back to it, and the decode launches on the
caller's stream.  These tests check that the fork and join keep the call's
stream semantics: the prefill sees the KV write enqueued just before it, work
enqueued after the call sees the whole output, the pair can be captured into
a CUDA graph, calls from several host threads on their own streams do not
mix, and a side stream held by another thread's capture is left alone."""
import threading

import numpy as np
import pytest
import torch

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


def _mixed(seed, small=True):
    wl = W.workload(4, small=small, seed=seed)
    assert 0 < wl.num_decode_seqs < wl.num_seqs          # both kinds of rows
    return wl


def _ws(g):
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=g.max_query_len,
                         max_context_len=g.max_context_len, num_decode_seqs=g.num_decode_seqs)
    return torch.empty(max(pkv.workspace_size(g.k_cache, meta), 256), dtype=torch.uint8,
                       device="cuda")


def test_forked_step_on_a_fresh_stream_sees_its_write_and_is_seen_after():
    """write + attention enqueued back to back on a new stream, then a copy of
    the output on the same stream: no host synchronisation in between."""
    wl = _mixed(17)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    ws = _ws(g)
    out = nan_like(g.q)
    host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            out.fill_(float("nan"))
            pkv.run_step(g, out, workspace=ws, stream=s)
            host.copy_(out, non_blocking=True)
    s.synchronize()
    assert max_err(host, exp) <= TOL[torch.bfloat16]


def test_forked_step_captured_in_a_cuda_graph_replays_correctly():
    wl = _mixed(18)
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    ws = _ws(g)
    out = torch.empty_like(g.q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.run_step(g, out, workspace=ws, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkv.run_step(g, out, workspace=ws, stream=s)
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert max_err(out, exp) <= TOL[torch.bfloat16]


def test_calls_from_several_threads_on_their_own_streams():
    """Four host threads, each with its own batch, stream and buffers, call
    the step 20 times; every result equals the single-threaded one bit for
    bit (the kernels are deterministic)."""
    gs = [_mixed(30 + i).to("cuda") for i in range(4)]
    wss = [_ws(g) for g in gs]
    ref = []
    for g, ws in zip(gs, wss):
        o = nan_like(g.q)
        pkv.run_step(g, o, workspace=ws)
        ref.append(o)
    torch.cuda.synchronize()
    outs = [nan_like(g.q) for g in gs]
    bad = []

    def work(i):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(20):
                outs[i].fill_(float("nan"))
                pkv.run_step(gs[i], outs[i], workspace=wss[i], stream=s)
                if not torch.equal(outs[i].view(torch.int16), ref[i].view(torch.int16)):
                    bad.append(i)
                    return

    th = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    torch.cuda.synchronize()
    assert not bad


def test_side_stream_held_by_another_threads_capture_is_left_alone():
    """Thread A captures a forked step (the side stream joins A's capture);
    while A's capture is open, thread B runs a forked step eagerly on its own
    stream, which must not touch the side stream.  Both results are right."""
    wla, wlb = _mixed(41), _mixed(42)
    expa, _, _, _ = oracle_step(wla)
    expb, _, _, _ = oracle_step(wlb)
    ga, gb = wla.to("cuda"), wlb.to("cuda")
    wsa, wsb = _ws(ga), _ws(gb)
    outa, outb = torch.empty_like(ga.q), nan_like(gb.q)
    sa = torch.cuda.Stream()
    with torch.cuda.stream(sa):
        pkv.run_step(ga, outa, workspace=wsa, stream=sa)
    torch.cuda.synchronize()
    captured, b_done = threading.Event(), threading.Event()
    errs = []

    def thread_a():
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=sa, capture_error_mode="thread_local"):
                pkv.run_step(ga, outa, workspace=wsa, stream=sa)
                captured.set()
                if not b_done.wait(60):
                    raise RuntimeError("thread B did not finish")
            outa.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            errs.append(("A", repr(e)))
            captured.set()

    def thread_b():
        try:
            if not captured.wait(60):
                raise RuntimeError("thread A did not capture")
            sb = torch.cuda.Stream()
            with torch.cuda.stream(sb):
                pkv.run_step(gb, outb, workspace=wsb, stream=sb)
            sb.synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            errs.append(("B", repr(e)))
        finally:
            b_done.set()

    ta, tb = threading.Thread(target=thread_a), threading.Thread(target=thread_b)
    ta.start()
    tb.start()
    ta.join()
    tb.join()
    assert not errs, errs
    assert max_err(outa, expa) <= TOL[torch.bfloat16]
    assert max_err(outb, expb) <= TOL[torch.bfloat16]


def test_forked_full_size_mixed_batch_matches_the_single_stream_order():
    """Workload 4 at full size: the forked call equals the decode and prefill
    halves run one after the other on one stream, bit for bit."""
    wl = W.workload(4, device="cuda")
    pkv.write(wl.k_new, wl.v_new, wl.slot_mapping, wl.k_cache, wl.v_cache)
    nd = wl.num_decode_seqs
    ws = _ws(wl)
    out = nan_like(wl.q)
    pkv.attention(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
                  wl.query_start_loc, wl.scale, max_query_len=wl.max_query_len,
                  max_context_len=wl.max_context_len, num_decode_seqs=nd, workspace=ws)
    ref = nan_like(wl.q)
    pkv.attention(ref[:nd], wl.q[:nd], wl.k_cache, wl.v_cache, wl.block_tables[:nd],
                  wl.context_lens[:nd], wl.query_start_loc[:nd + 1], wl.scale, max_query_len=1,
                  max_context_len=wl.max_context_len, workspace=ws)
    pkv.attention(ref[nd:], wl.q[nd:], wl.k_cache, wl.v_cache, wl.block_tables[nd:],
                  wl.context_lens[nd:], (wl.query_start_loc[nd:] - nd).contiguous(), wl.scale,
                  max_query_len=wl.max_query_len, max_context_len=wl.max_context_len,
                  num_decode_seqs=0)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert np.isfinite(out.float().cpu().numpy()).all()


def test_cascade_forked_prefix_on_a_fresh_stream_is_ordered():
    """Cascade: the shared-prefix launch goes on the side stream beside the
    suffix launch; write + cascade + a copy of the output, back to back on a
    new stream, three times, with no host synchronisation in between."""
    rng = np.random.default_rng(7)
    S, P = 24, 16
    ctx = rng.integers(P * 16 + 1, P * 16 + 900, S, endpoint=True)
    wl = W.make_workload([1] * S, ctx, num_q_heads=32, num_kv_heads=8, head_size=128, seed=7,
                         shared_prefix_blocks=P, shared_seqs=tuple(range(S)))
    exp, _, _, _ = oracle_step(wl)
    g = wl.to("cuda")
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, max_query_len=1,
                         max_context_len=g.max_context_len)
    ws = torch.empty(pkv.cascade_workspace_size(g.k_cache, meta, P), dtype=torch.uint8,
                     device="cuda")
    out = nan_like(g.q)
    host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            out.fill_(float("nan"))
            pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, stream=s)
            pkv.attention_cascade(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                  g.query_start_loc, g.scale, P,
                                  max_context_len=g.max_context_len, workspace=ws, stream=s)
            host.copy_(out, non_blocking=True)
    s.synchronize()
    assert max_err(host, exp) <= TOL[torch.bfloat16]
