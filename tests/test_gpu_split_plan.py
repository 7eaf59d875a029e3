"""The decode split plan, read back through pkv_attention_workspace_size (a
host call that needs the device only for its SM count): 1024-key chunks by
default, 2048 for contexts of 16K keys or more, halved only while the batch
would have fewer CTAs than SMs, then the longest row's splits evened out
(count rounded to nearest, at most 128 blocks each).  Expectations are for a
152-SM GB300."""
import ctypes

import pytest
import torch

from paged_kv_cache_43_gb300 import build, pkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("expectations are for 152 SMs")
    build.build()
    pkv.load()


def ws_bytes(S, hq, hkv, max_ctx, window=0, split=0, d=128):
    desc = pkv.CacheDesc(1 << 20, 16, hkv, d, 1)          # bf16
    meta = pkv.AttnMeta(S, S, hq, (max_ctx + 15) // 16, 1, max_ctx, S, window, split)
    n = pkv.load().pkv_attention_workspace_size(ctypes.byref(desc), ctypes.byref(meta))
    assert n != ctypes.c_size_t(-1).value
    return int(n)


def expect(S, hq, splits, d=128):
    if splits == 1:
        return 0
    up = lambda x: (x + 255) // 256 * 256
    rows = S * hq * splits
    return up(rows * d * 4) + up(rows * 4)


@pytest.mark.parametrize("S,hq,hkv,ctx,window,split,splits", [
    (64, 32, 32, 4096, 0, 0, 4),        # 256 blocks / 64
    (64, 32, 32, 4096, 1024, 0, 1),     # a 1024-key window spans 65 blocks: one split
    (16, 64, 8, 32768, 4096, 0, 4),     # 257 blocks: 4 splits of 65, not 5 of 64 (+1)
    (16, 64, 8, 32768, 4096, 1024, 5),  # an explicit size is taken as given
    (16, 64, 8, 32768, 0, 0, 16),       # >= 16K keys: 128-block splits
    (2, 64, 8, 32768, 0, 0, 16),        # 16 units x 16 splits >= 152 CTAs: still 128
    (8, 32, 8, 2048, 0, 0, 4),          # 32 units: 64 -> 32 blocks (128 -> 256 CTAs)
    (1, 1, 1, 4096, 0, 0, 64),          # one unit: down to 4-block splits
    (16, 32, 32, 1100, 0, 0, 1),        # 69 blocks, 512 units: one split of 69
])
def test_split_plan(S, hq, hkv, ctx, window, split, splits):
    assert ws_bytes(S, hq, hkv, ctx, window, split) == expect(S, hq, splits)
