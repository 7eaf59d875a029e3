"""The timeout path of the kernels' bounded waits, run out on purpose through
the test hook pkv_debug_wait_test (each CTA withholds its first key block or
tile and waits at most 20 us for it): the attention call returns, the device
error word carries PKV_ERR_TIMEOUT, and the context stays usable -- the next
normal calls on the same device (which need the tensor memory the aborted
CTAs held, and the shared memory their copies were landing in) match the
oracle with a clean error word.  No fault, trap or hang is involved: the waits
are bounded and the withheld copy is simply never started."""
import pytest
import torch

from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import workloads as W
from tests.support import (TOL, fp8_scale_tensors, gpu_fp8_caches, max_err, oracle_step,
                           oracle_step_fp8)

pytestmark = pytest.mark.gpu

PKV_ERR_TIMEOUT = 1 << 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    pkv.load()
    pkv.get_error(clear=True)
    yield
    pkv.debug_wait_test(False)


# decode rows split over several CTAs (32 q / 8 kv heads, 128-key splits), and
# a mixed batch whose prefill chunks run on the tcgen05 kernel beside its
# decode rows
BATCHES = {"decode": (3, 128), "mixed": (4, 0)}


@pytest.mark.parametrize("name", sorted(BATCHES))
@pytest.mark.parametrize("fp8", [False, True])
def test_waits_run_out_then_the_device_recovers(name, fp8):
    n, split = BATCHES[name]
    wl = W.workload(n, small=True)
    g = wl.to("cuda")
    kw = dict(max_query_len=g.max_query_len, max_context_len=g.max_context_len,
              num_decode_seqs=g.num_decode_seqs, kv_split_tokens=split)
    if fp8:
        ks, vs, kd, vd = fp8_scale_tensors(g.num_kv_heads, g.num_seqs, 21)
        kc, vc = gpu_fp8_caches(g, ks, vs)
        pkv.write_fp8(g.k_new, g.v_new, g.slot_mapping, kc, vc, ks, vs)
        exp, st, _, _ = oracle_step_fp8(wl, ks.cpu(), vs.cpu(), kd.cpu(), vd.cpu())

        def call(out):
            pkv.attention_fp8(out, g.q, kc, vc, g.block_tables, g.context_lens,
                              g.query_start_loc, g.scale, kd, vd, **kw)
        tol = 2e-2
    else:
        pkv.write(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
        exp, st, _, _ = oracle_step(wl)

        def call(out):
            pkv.attention(out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                          g.query_start_loc, g.scale, **kw)
        tol = TOL[torch.bfloat16]
    assert not st.any()
    torch.cuda.synchronize()
    assert pkv.get_error(clear=True) == 0

    pkv.debug_wait_test(True)
    try:
        for _ in range(2):
            out = torch.zeros_like(g.q)
            call(out)                                   # returns: nothing hangs
            torch.cuda.synchronize()
            assert pkv.get_error(clear=True) & PKV_ERR_TIMEOUT
    finally:
        pkv.debug_wait_test(False)

    for _ in range(2):                                  # the device is usable again
        out = torch.full_like(g.q, float("nan"))
        call(out)
        torch.cuda.synchronize()
        assert pkv.get_error(clear=True) == 0
        assert max_err(out, exp) <= tol
