"""pkv_attention_static_scratch: the attention call for callers that cannot
allocate device memory (for example a plugin whose host framework owns every
device allocation, or a decode loop that must not enter the allocator).  It
takes its split-K workspace from a fixed array inside the library instead of
from the caller.

Checked through the C ABI against pkv_attention with a caller workspace, bit
for bit, on two calls in a row after a different batch has filled the array
with other partial results (the array keeps the previous call's contents,
which must not leak into the next result), and against the fp64 oracle; plus
the rejection of a batch that needs more scratch than the array holds.  This
file is collected last so that a run that stops at the first failure has
already run every other test.
"""
import pytest
import torch

from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import workloads as W
from tests.support import max_err, oracle_step

pytestmark = pytest.mark.gpu

PKV_E_WORKSPACE = -5
TOL = 2e-2   # the bf16 tolerance of the parity tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    pkv.load()
    pkv.get_error(clear=True)


def _kw(g, split):
    return dict(max_query_len=g.max_query_len, max_context_len=g.max_context_len,
                num_decode_seqs=g.num_decode_seqs, kv_split_tokens=split)


def _attend(fn, g, split):
    out = torch.full_like(g.q, float("nan"))
    st = fn(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
            g.query_start_loc, g.scale, **_kw(g, split))
    return st, out


@pytest.mark.parametrize("n,split", [(2, 128), (5, 0), (4, 64)])
def test_static_scratch_matches_workspace_call_twice(n, split):
    # A different, larger batch first (long contexts cut into many 64-key
    # splits), so that the scratch array holds other partial results when the
    # tested batch runs: none of them may leak into its output.
    big = W.workload(5, small=True).to("cuda")
    pkv.write(big.k_new, big.v_new, big.slot_mapping, big.k_cache, big.v_cache)
    st, _ = _attend(pkv.attention_static_scratch, big, 64)
    assert st == 0, pkv.status_string(st)

    wl = W.workload(n, small=True)
    exp, ost, _, _ = oracle_step(wl)
    assert not ost.any()
    g = wl.to("cuda")
    pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, **_kw(g, split))
    need = pkv.workspace_size(g.k_cache, meta)
    assert 0 < need <= pkv.STATIC_SCRATCH_BYTES      # the scratch really is used
    _, ref = _attend(pkv.attention, g, split)      # (raises on a bad status)
    for _ in range(2):
        st, out = _attend(pkv.attention_static_scratch, g, split)
        assert st == 0, pkv.status_string(st)
        torch.cuda.synchronize()
        # the same kernels and split plan as the workspace call: bit for bit
        assert torch.equal(out, ref)
        assert max_err(out, exp) <= TOL
    assert pkv.get_error() == 0


def test_static_scratch_rejects_batches_beyond_its_size():
    g = W.workload(2, small=True).to("cuda")
    # valid (1024 splits of 64 keys) but ~101 MB of split-K workspace
    big = dict(max_query_len=1, max_context_len=1 << 16, num_decode_seqs=-1,
               kv_split_tokens=64)
    meta = pkv.attn_meta(g.q, g.block_tables, g.context_lens, **big)
    assert pkv.workspace_size(g.k_cache, meta) > pkv.STATIC_SCRATCH_BYTES
    out = torch.zeros_like(g.q)
    st = pkv.attention_static_scratch(out, g.q, g.k_cache, g.v_cache, g.block_tables,
                                      g.context_lens, g.query_start_loc, g.scale, **big)
    assert st == PKV_E_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any()                                   # nothing was enqueued
    assert pkv.get_error() == 0
