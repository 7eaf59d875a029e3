"""Seeded synthetic inputs for the paged KV-cache write and PagedAttention.

This module only draws inputs: context lengths, block placements, slot
mappings and N(0, 1) tensors.  It computes no attention and is shared by the
CUDA path's tests/bench and the CPU oracle's tests, which is why it sits on its
own and imports neither.

The five workloads follow the serving scenarios the vLLM pages describe
(decode batches, GQA, chunked prefill mixed with decode, prefix-shared blocks,
long contexts).  The pages name no public dataset; every input here is
synthetic.  Layout (vLLM core book, ch. 6 "Transformation de la disposition
mémoire du KV cache"): caches are [num_blocks, block_size=16, num_kv_heads,
head_size], K and V separate.  Block ids are drawn without replacement from a
pool ~10% larger than needed; ``block_tables`` rows past a sequence's last
block hold -1 (never to be read).  Slots that hold no live key -- unused pool
blocks, the tail of each last block, and the slots this step's new tokens will
be written to -- are filled with NaN so that any read outside the context, or
before the write, shows up.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16
SEED_BASE = 4300          # seed of workload n is SEED_BASE + n

WORKLOAD_NAMES = {
    1: "tiny-decode-f32",
    2: "llama7b-decode-bf16",
    3: "gqa8b-decode-bf16",
    4: "mixed-prefill-prefix-bf16",
    5: "longctx70b-decode-bf16",
}


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    num_blocks: int
    q: torch.Tensor                 # [T, Hq, D]
    k_new: torch.Tensor             # [T, Hkv, D]  this step's new keys
    v_new: torch.Tensor             # [T, Hkv, D]
    slot_mapping: torch.Tensor      # int64 [T]
    k_cache: torch.Tensor           # [NB, 16, Hkv, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor      # int32 [S, max_blocks]
    context_lens: torch.Tensor      # int32 [S]   keys per seq incl. new tokens
    query_start_loc: torch.Tensor   # int32 [S+1]
    scale: float
    num_decode_seqs: int            # leading run of sequences with one query
    q_lens: np.ndarray = field(repr=False, default=None)
    ctx_lens: np.ndarray = field(repr=False, default=None)
    shared_prefix_blocks: int = 0
    shared_seqs: tuple = ()

    @property
    def block_size(self) -> int:
        return BLOCK_SIZE

    @property
    def num_seqs(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_query_len(self) -> int:
        return int(self.q_lens.max()) if self.q_lens.size else 0

    @property
    def max_context_len(self) -> int:
        return int(self.ctx_lens.max()) if self.ctx_lens.size else 0

    def to(self, device) -> "Workload":
        out = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("q", "k_new", "v_new", "slot_mapping", "k_cache", "v_cache",
                  "block_tables", "context_lens", "query_start_loc"):
            setattr(out, k, getattr(self, k).to(device))
        return out


def _blocks_for(n_tokens: int) -> int:
    """Blocks that hold n tokens at 16 tokens per block (ceil)."""
    return -(-int(n_tokens) // BLOCK_SIZE)


def make_workload(q_lens, ctx_lens, *, num_q_heads, num_kv_heads, head_size,
                  dtype=torch.bfloat16, seed=0, device="cpu", num_blocks=None,
                  pool_slack=1.1, shared_prefix_blocks=0, shared_seqs=(),
                  poison=True, bt_pad=0, scale=None, name="custom",
                  contiguous_blocks=False) -> Workload:
    """Draw one batch.

    q_lens[s] new tokens end sequence s, which then holds ctx_lens[s] keys
    (the new ones included).  ``shared_seqs`` list sequences whose first
    ``shared_prefix_blocks`` block-table entries are the same physical blocks.
    ``contiguous_blocks`` lays sequences out in pool order (block ids 0, 1, ...)
    instead of a seeded random placement.
    """
    q_lens = np.asarray(q_lens, dtype=np.int64)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    S = int(ctx_lens.shape[0])
    assert q_lens.shape == (S,)
    rng = np.random.default_rng(seed)
    nblk = np.array([_blocks_for(L) for L in ctx_lens], dtype=np.int64)
    shared_seqs = tuple(int(s) for s in shared_seqs)
    if shared_seqs:
        assert all(nblk[s] > shared_prefix_blocks for s in shared_seqs)
        assert all(ctx_lens[s] - q_lens[s] >= shared_prefix_blocks * BLOCK_SIZE
                   for s in shared_seqs), "new tokens must not land in shared blocks"
    unique_needed = int(nblk.sum()) - max(len(shared_seqs) - 1, 0) * shared_prefix_blocks
    if num_blocks is None:
        num_blocks = max(int(math.ceil(pool_slack * unique_needed)), 1)
    assert num_blocks >= unique_needed
    order = np.arange(num_blocks) if contiguous_blocks else rng.permutation(num_blocks)
    stride = int(nblk.max()) + bt_pad if S else 1
    bt = np.full((S, max(stride, 1)), -1, dtype=np.int32)
    cursor = 0
    shared_ids = None
    if shared_seqs:
        shared_ids = order[cursor:cursor + shared_prefix_blocks]
        cursor += shared_prefix_blocks
    for s in range(S):
        start = 0
        if s in shared_seqs:
            bt[s, :shared_prefix_blocks] = shared_ids
            start = shared_prefix_blocks
        take = int(nblk[s]) - start
        bt[s, start:start + take] = order[cursor:cursor + take]
        cursor += take

    # Slots of this step's new tokens (positions L - q .. L - 1) and of the
    # history they attend to.
    slot_list = []
    live = np.zeros(num_blocks * BLOCK_SIZE, dtype=bool)
    for s in range(S):
        L, n = int(ctx_lens[s]), int(q_lens[s])
        pos = np.arange(L)
        slots = bt[s, pos // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + pos % BLOCK_SIZE
        live[slots[: L - n]] = True
        slot_list.append(slots[L - n:])
    slot_mapping = np.concatenate(slot_list) if slot_list else np.zeros(0, np.int64)
    qsl = np.zeros(S + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    T = int(qsl[-1])

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    shape_c = (num_blocks, BLOCK_SIZE, num_kv_heads, head_size)
    k_cache = torch.randn(shape_c, generator=gen, device=device, dtype=torch.float32).to(dtype)
    v_cache = torch.randn(shape_c, generator=gen, device=device, dtype=torch.float32).to(dtype)
    q = torch.randn((T, num_q_heads, head_size), generator=gen, device=device,
                    dtype=torch.float32).to(dtype)
    k_new = torch.randn((T, num_kv_heads, head_size), generator=gen, device=device,
                        dtype=torch.float32).to(dtype)
    v_new = torch.randn((T, num_kv_heads, head_size), generator=gen, device=device,
                        dtype=torch.float32).to(dtype)
    if poison:
        dead = torch.from_numpy(~live).to(device)
        k_cache.view(num_blocks * BLOCK_SIZE, -1)[dead] = float("nan")
        v_cache.view(num_blocks * BLOCK_SIZE, -1)[dead] = float("nan")

    # Decode sequences (one query) form the leading run, as a mixed batch orders
    # them; count that run.
    nd = 0
    while nd < S and q_lens[nd] == 1:
        nd += 1
    return Workload(
        name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_size=head_size, num_blocks=num_blocks, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.from_numpy(slot_mapping).to(device),
        k_cache=k_cache, v_cache=v_cache,
        block_tables=torch.from_numpy(bt).to(device),
        context_lens=torch.from_numpy(ctx_lens.astype(np.int32)).to(device),
        query_start_loc=torch.from_numpy(qsl).to(device),
        scale=float(scale if scale is not None else 1.0 / math.sqrt(head_size)),
        num_decode_seqs=nd, q_lens=q_lens, ctx_lens=ctx_lens,
        shared_prefix_blocks=shared_prefix_blocks if shared_seqs else 0,
        shared_seqs=shared_seqs)


def _uniform_int(rng, lo, hi, n):
    return rng.integers(lo, hi, size=n, endpoint=True)


def _log_uniform_int(rng, lo, hi, n):
    return np.floor(np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))).astype(np.int64)


def lengths(n: int, small: bool = False, seed: int | None = None, num_seqs: int | None = None):
    """(q_lens, ctx_lens, extra kwargs) of workload n.  ``small`` keeps the head
    layout but shrinks batch and context so that the oracle finishes in seconds
    while the kernels still see several tiles, splits and ragged tails.
    ``num_seqs`` overrides the batch size of the decode workloads 2, 3 and 5
    (same length distribution)."""
    rng = np.random.default_rng(SEED_BASE + n if seed is None else seed)
    if n == 1:
        return np.ones(4, np.int64), np.array([17, 33, 64, 100]), {}
    if n == 2:
        S, hi = (6, 1200) if small else (64, 4096)
        S = num_seqs or S
        return np.ones(S, np.int64), _uniform_int(rng, 128, hi, S), {}
    if n == 3:
        S, hi = (24, 2048) if small else (256, 8192)
        S = num_seqs or S
        return np.ones(S, np.int64), _log_uniform_int(rng, 64, hi, S), {}
    if n == 4:
        if small:
            nd, npf, chunk, nsh, shb, hi = 6, 2, 96, 3, 8, 700
        else:
            nd, npf, chunk, nsh, shb, hi = 48, 4, 512, 16, 64, 4096
        ctx_sh = _uniform_int(rng, shb * 16 + 1, hi, nsh)
        ctx_dec = _uniform_int(rng, 256, hi, nd - nsh)
        ctx_pf = _uniform_int(rng, max(256, chunk), hi, npf)
        ctx = np.concatenate([ctx_sh, ctx_dec, ctx_pf])
        q = np.concatenate([np.ones(nd, np.int64), np.full(npf, chunk, np.int64)])
        return q, ctx, dict(shared_prefix_blocks=shb, shared_seqs=tuple(range(nsh)))
    if n == 5:
        S, lo, hi = (2, 3000, 6000) if small else (16, 16384, 32768)
        S = num_seqs or S
        return np.ones(S, np.int64), _uniform_int(rng, lo, hi, S), {}
    raise ValueError(n)


HEADS = {1: (4, 4, 64), 2: (32, 32, 128), 3: (32, 8, 128), 4: (32, 8, 128), 5: (64, 8, 128)}


def workload(n: int, *, small: bool = False, device="cpu", poison=True,
             seed: int | None = None, num_seqs: int | None = None) -> Workload:
    """Workload n (1..5) at full size, or its small parity variant."""
    seed = SEED_BASE + n if seed is None else seed
    q_lens, ctx, extra = lengths(n, small=small, seed=seed, num_seqs=num_seqs)
    hq, hkv, d = HEADS[n]
    kw = dict(num_q_heads=hq, num_kv_heads=hkv, head_size=d, seed=seed, device=device,
              poison=poison, name=WORKLOAD_NAMES[n] + ("-small" if small else ""), **extra)
    if n == 1:
        return make_workload(q_lens, ctx, dtype=torch.float32, num_blocks=64,
                             scale=1.0 / 8.0, **kw)
    return make_workload(q_lens, ctx, dtype=torch.bfloat16, **kw)


def history_slots(wl: Workload) -> np.ndarray:
    """Sorted unique cache slots of the keys written before this step
    (positions 0 .. L - q_s - 1 of every sequence), for filling a cache of
    another dtype from the same history."""
    bt = wl.block_tables.cpu().numpy()
    parts = []
    for s in range(wl.num_seqs):
        pos = np.arange(int(wl.ctx_lens[s]) - int(wl.q_lens[s]))
        parts.append(bt[s, pos // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + pos % BLOCK_SIZE)
    return np.unique(np.concatenate(parts)) if parts else np.zeros(0, np.int64)


def fp8_scales(num_kv_heads: int, seed: int, lo: float = 0.008, hi: float = 0.03) -> np.ndarray:
    """Per-kv-head fp32 quantisation scales for an e4m3 cache, drawn uniformly
    in [lo, hi] (N(0, 1) data then spans roughly 1/8 .. 1/2 of the e4m3 range)."""
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=num_kv_heads).astype(np.float32)


E4M3_NAN_CODE = 0x7F   # filler for slots with no live key (an e4m3 NaN)


def cache_bytes_per_block(num_kv_heads: int, head_size: int, dtype: torch.dtype) -> int:
    """Bytes the two caches allocate per block, measured from real tensors."""
    k = torch.empty((1, BLOCK_SIZE, num_kv_heads, head_size), dtype=dtype)
    v = torch.empty_like(k)
    return k.numel() * k.element_size() + v.numel() * v.element_size()


def as_oracle_array(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view for the oracle: float32 stays float32; bf16 becomes its
    uint16 bit patterns."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    return t.numpy()
