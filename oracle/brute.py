"""Second, independent oracle: numpy brute force for tiny inputs.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Unlike ``pkv_oracle.c`` it never walks a block table key by key and keeps no
running state: for each sequence it first gathers all of its keys into a dense
[L, Hkv, D] array through the block table (the PagedAttention mapping of the
vLLM core book, ch. 5 "slot_mapping et la block table"), then applies a plain
masked softmax over a full score matrix.  Query j of a chunk of q_s queries sits
at absolute position L - q_s + j (ch. 6 "Branche de masque").
"""
from __future__ import annotations

import numpy as np


def widen(a: np.ndarray) -> np.ndarray:
    """float32 -> float64; uint16 bf16 bit patterns -> float64 (exact)."""
    if a.dtype == np.float32:
        return a.astype(np.float64)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise TypeError(a.dtype)


def dense_kv(k_cache, v_cache, block_row, L):
    """Keys/values 0..L-1 of one sequence as dense [L, Hkv, D] float64."""
    nb, bs, hkv, d = k_cache.shape
    blocks = np.asarray(block_row[: -(-L // bs)], dtype=np.int64)
    flat_k = widen(k_cache).reshape(nb * bs, hkv, d)
    flat_v = widen(v_cache).reshape(nb * bs, hkv, d)
    slots = (blocks[:, None] * bs + np.arange(bs)[None, :]).reshape(-1)[:L]
    return flat_k[slots], flat_v[slots]


def attention(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale,
              window=0):
    """float64 [T, Hq, D]; valid inputs only.  ``window`` W > 0 restricts the
    query at position pos to keys pos - W < p <= pos."""
    qf = widen(q)
    T, hq, d = qf.shape
    hkv = k_cache.shape[2]
    g = hq // hkv
    out = np.zeros((T, hq, d), dtype=np.float64)
    for s in range(len(context_lens)):
        q0, q1 = int(query_start_loc[s]), int(query_start_loc[s + 1])
        n, L = q1 - q0, int(context_lens[s])
        if n == 0:
            continue
        K, V = dense_kv(k_cache, v_cache, block_tables[s], L)
        pos = L - n + np.arange(n)                       # absolute positions
        visible = np.arange(L)[None, :] <= pos[:, None]  # [n, L]
        if window > 0:
            visible &= np.arange(L)[None, :] > (pos[:, None] - window)
        for h in range(hq):
            kv = h // g
            x = scale * (qf[q0:q1, h, :] @ K[:, kv, :].T)  # [n, L]
            x = np.where(visible, x, -np.inf)
            w = np.exp(x - x.max(axis=1, keepdims=True))
            out[q0:q1, h, :] = (w @ V[:, kv, :]) / w.sum(axis=1, keepdims=True)
    return out
