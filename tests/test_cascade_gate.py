"""The cascade gate (pkv_use_cascade) on the host: the pages' conditions
(>= 256 shared tokens, >= 8 sequences, no sliding window) plus this build's
(a key after the prefix) and the cost rules measured on GB300 (decode rows;
chunked-prefill rows)."""
import pytest

from paged_kv_cache_43_gb300 import build, pkv


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    pkv.load()


def M(S, mcl, mq=1, w=0):
    # AttnMeta(num_seqs, num_tokens, q heads, stride, max_query_len,
    #          max_context_len, num_decode_seqs, window, split)
    return pkv.AttnMeta(S, S, 8, 600, mq, mcl, -1, w, 0)


@pytest.mark.parametrize("S,mcl,pblocks,want", [
    (64, 3000, 128, True),      # 64 x 2048 shared keys (measured 1.83x)
    (16, 9000, 512, True),      # 16 x 8192 (1.62x)
    (256, 3000, 128, True),     # (2.3x)
    (16, 3000, 128, True),      # 15 x 2048 = 30K >= 16K (1.17x)
    (8, 9000, 512, True),       # 7 x 8192 = 57K (1.19x)
    (64, 1000, 32, True),       # 64 x 512: 63 x 512 = 32K (1.09x)
    (16, 2000, 64, False),      # 15 x 1024 < 16K: plain wins (0.89x)
    (8, 3000, 128, False),      # 7 x 2048 < 16K (0.89x)
    (256, 1000, 16, False),     # prefix < 512 tokens (0.96x)
    (7, 90000, 4096, False),    # < 8 sequences: the pages' gate
    (64, 3000, 15, False),      # < 256 tokens: the pages' gate
    (64, 2048, 128, False),     # no key after the prefix
])
def test_gate(S, mcl, pblocks, want):
    assert pkv.use_cascade(M(S, mcl), pblocks) == want


def test_gate_rejects_windows():
    assert not pkv.use_cascade(M(64, 3000, w=64), 128)


def Mx(nd, chunk_rows, mcl, mq):
    # nd decode sequences then chunked-prefill sequences holding chunk_rows rows
    S = nd + max(1, chunk_rows // mq)
    return pkv.AttnMeta(S, nd + chunk_rows, 8, 600, mq, mcl, nd, 0, 0)


@pytest.mark.parametrize("nd,rows,mq,mcl,pblocks,want", [
    (48, 512, 512, 7000, 256, True),    # one 512-token chunk, 4096 shared (measured 1.14x)
    (16, 512, 512, 7000, 256, True),    # (1.14x)
    (47, 512, 512, 7000, 256, True),    # >= 8 sequences either way
    (48, 512, 512, 5000, 128, False),   # 2048 shared: 0.90x
    (48, 2048, 512, 7000, 256, False),  # 4 x 512 chunk rows: 0.93x
    (16, 2048, 256, 7000, 256, False),  # 8 x 256: 0.81x
    (48, 512, 512, 7000, -1, False),    # (no prefix)
])
def test_gate_with_chunk_rows(nd, rows, mq, mcl, pblocks, want):
    assert pkv.use_cascade(Mx(nd, rows, mcl, mq), max(pblocks, 0)) == want


def test_gate_with_chunk_rows_needs_the_decode_count():
    m = Mx(48, 512, 7000, 512)
    m.num_decode_seqs = -1
    assert not pkv.use_cascade(m, 256)
