"""A serving-style decode loop over the host block pool and the kernels.

The loop is the consumer the pages describe for the pool ("Khám phá vLLM: Giải
phẫu hệ thống suy luận LLM thông lượng cao", "allocate_slots" and "Chạy
forward pass"; "Implémentation du cœur du moteur d'inférence haute
performance vLLM" ch. 4 §4.3 on allocation and recompute preemption): each
step gives every decoding request one token, every request still in its
prompt its next chunk, and admits waiting requests (prefix-cache hits first,
then the first chunk of their remaining prompt) while the token budget and
the pool allow -- a prompt longer than the budget is prefilled in chunks over
several steps -- preempts the most recently admitted request
when a decode finds no block (its blocks go back; it is re-admitted later and
recomputes what the cache no longer holds), writes the step's K/V rows with
pkv_write at the pool's slots and runs pkv_attention over the pool's block
tables — or, for a decode-only step whose requests share leading blocks and
when pkv_use_cascade says it pays ("Implémentation du cœur ... vLLM", ch. 6:
the scheduler's common_prefix_len feeding use_cascade), cascade attention.

There is no model: a token's q, k and v rows are a fixed function of (token
id, position) — rows of seeded N(0, 1) tables summed in fp32 and rounded to
the cache dtype — which is the one property of real K/V that prefix caching
relies on (equal prefixes give equal K/V).  "Sampling" draws a request's n-th
generated token from a generator seeded by (seed, request id, n), so a
request's tokens do not depend on how it was batched, cached or preempted.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch

from . import pkv
from .pool import BlockPool


@dataclass
class Req:
    rid: int
    tokens: list                 # prompt + generated ids
    max_new: int
    generated: int = 0
    admitted_order: int = 0


@dataclass
class Step:
    """What one step ran (host copies of the metadata; device tensors)."""
    req_ids: list
    q_lens: list
    slot_mapping: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    query_start_loc: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    out: torch.Tensor
    positions: list = field(default_factory=list)   # per request: new positions
    preempted: list = field(default_factory=list)
    finished: list = field(default_factory=list)
    cascade_blocks: int = 0                         # > 0: cascade over this prefix


class DecodeLoop:
    def __init__(self, *, num_blocks: int, num_q_heads: int, num_kv_heads: int, head_size: int,
                 dtype=torch.bfloat16, device="cuda", caching: bool = True, window: int = 0,
                 vocab: int = 512, max_pos: int = 8192, max_batch_tokens: int = 4096,
                 seed: int = 0, scale: float | None = None, use_cascade: bool = False):
        self.pool = BlockPool(num_blocks, 16, caching)
        self.hq, self.hkv, self.d = num_q_heads, num_kv_heads, head_size
        self.dtype, self.device, self.window = dtype, torch.device(device), window
        self.max_batch_tokens = max_batch_tokens
        self.scale = scale if scale is not None else 1.0 / float(np.sqrt(head_size))
        g = torch.Generator().manual_seed(seed)
        tab = lambda n, h: torch.randn((n, h, head_size), generator=g) * 0.7
        self.tq, self.tk, self.tv = tab(vocab, num_q_heads), tab(vocab, num_kv_heads), tab(vocab, num_kv_heads)
        self.pq, self.pk, self.pv = tab(max_pos, num_q_heads), tab(max_pos, num_kv_heads), tab(max_pos, num_kv_heads)
        self.vocab, self.seed = vocab, seed
        self.use_cascade = use_cascade
        shape = (num_blocks, 16, num_kv_heads, head_size)
        self.k_cache = torch.full(shape, float("nan"), dtype=dtype, device=self.device)
        self.v_cache = torch.full(shape, float("nan"), dtype=dtype, device=self.device)
        self.waiting: deque = deque()
        self.running: list = []
        self._next_id = 0
        self._order = 0

    # ------------------------------------------------------------------ rows
    def rows(self, token_ids, positions):
        """q, k, v rows of (token, position) pairs, in the cache dtype (host)."""
        t = torch.as_tensor(token_ids, dtype=torch.long)
        p = torch.as_tensor(positions, dtype=torch.long)
        q = (self.tq[t] + self.pq[p]).to(self.dtype)
        k = (self.tk[t] + self.pk[p]).to(self.dtype)
        v = (self.tv[t] + self.pv[p]).to(self.dtype)
        return q, k, v

    # -------------------------------------------------------------- requests
    def add_request(self, prompt, max_new_tokens: int) -> int:
        rid = self._next_id
        self._next_id += 1
        self.waiting.append(Req(rid, [int(x) for x in prompt], int(max_new_tokens)))
        return rid

    def _preempt(self, r: Req):
        """recompute preemption: blocks back to the pool, request back in front."""
        self.pool.free_request(r.rid)
        self.running.remove(r)
        self.waiting.appendleft(r)

    def done(self) -> bool:
        return not self.waiting and not self.running

    # ------------------------------------------------------------------ step
    def step(self) -> Step | None:
        sched = []        # (req, positions, slots)
        preempted = []
        budget = self.max_batch_tokens
        # running requests, oldest first: a decoding request computes its last
        # sampled token; one still in its prompt computes its next chunk, as
        # much of the rest as the token budget leaves (decodes go first)
        order = sorted(self.running, key=lambda x: (self.pool.num_computed(x.rid) + 1 <
                                                    len(x.tokens), x.admitted_order))
        for r in order:
            if r not in self.running:
                continue
            while True:
                pos = self.pool.num_computed(r.rid)
                rest = len(r.tokens) - pos
                n = min(1 if rest <= 1 else rest, budget)
                if n <= 0:
                    break                        # no budget left for its next row(s)
                slots = self.pool.allocate_slots(r.rid, n, self.window)
                if slots is not None:
                    sched.append((r, list(range(pos, pos + n)), slots))
                    budget -= n
                    break
                victim = max(self.running, key=lambda x: x.admitted_order)
                self._preempt(victim)
                preempted.append(victim.rid)
                budget += sum(len(s[1]) for s in sched if s[0] is victim)   # its rows go back
                sched = [s for s in sched if s[0] is not victim]
                if victim is r:
                    break
        # waiting requests: prefix hits, then the first chunk of the rest of
        # their known tokens (chunked prefill: at most the budget left)
        while self.waiting and budget > 0:
            r = self.waiting[0]
            self.pool.add_request(r.rid, r.tokens)
            cached = self.pool.admit(r.rid)
            n = min(len(r.tokens) - cached, budget)
            first = cached
            slots = self.pool.allocate_slots(r.rid, n, self.window)
            if slots is None:
                self.pool.free_request(r.rid)
                break
            self.waiting.popleft()
            self._order += 1
            r.admitted_order = self._order
            self.running.append(r)
            sched.append((r, list(range(first, first + n)), slots))
            budget -= n
        if not sched:
            return None
        # decode rows first (the kernels' decode run), then prefill chunks
        sched.sort(key=lambda s: len(s[1]) > 1)
        return self._run(sched, preempted)

    def _run(self, sched, preempted) -> Step:
        dev = self.device
        toks, poss, slots, q_lens, ids, ctx = [], [], [], [], [], []
        for r, positions, sl in sched:
            toks += [r.tokens[p] for p in positions]
            poss += positions
            slots += [int(x) for x in sl]
            q_lens.append(len(positions))
            ids.append(r.rid)
            ctx.append(positions[-1] + 1)
        q, k, v = self.rows(toks, poss)
        q, k, v = q.to(dev), k.to(dev), v.to(dev)
        stride = max(-(-c // 16) for c in ctx)
        bt = torch.from_numpy(self.pool.block_tables(ids, stride)).to(dev)
        cl = torch.tensor(ctx, dtype=torch.int32, device=dev)
        qsl = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32, device=dev)
        sm = torch.tensor(slots, dtype=torch.int64, device=dev)
        out = torch.empty_like(q)
        nd = 0
        while nd < len(q_lens) and q_lens[nd] == 1:
            nd += 1
        pkv.write(k, v, sm, self.k_cache, self.v_cache)
        casc = 0
        if self.use_cascade and nd == len(q_lens) and self.window == 0:
            # leading blocks every row of the step shares (the common prefix)
            rows = self.pool.block_tables(ids, stride)
            same = np.all(rows == rows[:1], axis=0) & (rows[0] != self.pool.null_block)
            casc = int(np.argmin(same)) if not same.all() else stride
            casc = min(casc, (min(ctx) - 1) // 16)   # every query after the prefix
            meta = pkv.attn_meta(q, bt, cl, max_query_len=1, max_context_len=max(ctx))
            if casc == 0 or not pkv.use_cascade(meta, casc):
                casc = 0
        if casc:
            pkv.attention_cascade(out, q, self.k_cache, self.v_cache, bt, cl, qsl, self.scale,
                                  casc, max_context_len=max(ctx))
        else:
            pkv.attention(out, q, self.k_cache, self.v_cache, bt, cl, qsl, self.scale,
                          max_query_len=max(q_lens), max_context_len=max(ctx),
                          num_decode_seqs=nd, sliding_window=self.window)
        # sample: every scheduled request gets its next token; finished ones leave
        finished = []
        for r, positions, _ in sched:
            if positions[-1] + 1 < len(r.tokens):
                continue                  # a prompt chunk short of the end: nothing to sample
            rng = np.random.default_rng((self.seed, r.rid, r.generated))
            r.tokens.append(int(rng.integers(self.vocab)))
            self.pool.append_token(r.rid, r.tokens[-1])
            r.generated += 1
            if r.generated >= r.max_new:
                finished.append(r.rid)
                self.pool.free_request(r.rid)
                self.running.remove(r)
        return Step(ids, q_lens, sm, bt, cl, qsl, q, k, v, out, [s[1] for s in sched],
                    preempted, finished, casc)
