"""Shared helpers for the GPU parity tests: run the oracle on CPU copies of a
workload (its own KV write, then attention) and compare with the CUDA path."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_43_gb300 import workloads as W

# Tolerances on max |out - oracle| (fp32 accumulate in both kernels).
TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


def oracle_step(wl, window=0):
    """Oracle result of one step on a CPU workload: (out fp64, status, k_cache,
    v_cache) after the oracle's own write of this step's tokens."""
    A = W.as_oracle_array
    kc, vc = A(wl.k_cache).copy(), A(wl.v_cache).copy()
    bad = oracle.write(A(wl.k_new), A(wl.v_new), A(wl.slot_mapping), kc, vc)
    assert bad == 0
    out, st = oracle.attention(A(wl.q), kc, vc, A(wl.block_tables), A(wl.context_lens),
                               A(wl.query_start_loc), wl.scale, window=window)
    return out, st, kc, vc


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def raw_bytes(t: torch.Tensor) -> bytes:
    return W.as_oracle_array(t).tobytes()


def max_err(got: torch.Tensor, exp: np.ndarray, rows=None) -> float:
    g = as_f64(got)
    if rows is not None:
        g, exp = g[rows], exp[rows]
    assert np.isfinite(g).all(), "non-finite output"
    return float(np.abs(g - exp).max()) if g.size else 0.0


def nan_like(t: torch.Tensor) -> torch.Tensor:
    return torch.full_like(t, float("nan"))


def compact_subproblem(wl_gpu, seqs, pre_k, pre_v, window=0):
    """CPU oracle inputs for the sequences `seqs` of a GPU workload: their
    blocks gathered (from the pre-write pools pre_k/pre_v) into a compact pool,
    block tables renumbered, the oracle's own write of their new tokens
    applied.  Returns (oracle.Problem, token index map)."""
    bt = wl_gpu.block_tables.cpu().numpy()
    cl = wl_gpu.context_lens.cpu().numpy()
    qsl = wl_gpu.query_start_loc.cpu().numpy()
    ids = []
    for s in seqs:
        nb = -(-int(cl[s]) // W.BLOCK_SIZE)
        ids.extend(int(b) for b in bt[s, :nb])
    uniq = sorted(set(ids))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.int64, device=pre_k.device)
    kc = W.as_oracle_array(pre_k.index_select(0, idx)).copy()
    vc = W.as_oracle_array(pre_v.index_select(0, idx)).copy()
    stride = bt.shape[1]
    sub_bt = np.full((len(seqs), stride), -1, np.int32)
    sub_cl = np.zeros(len(seqs), np.int32)
    sub_qsl = np.zeros(len(seqs) + 1, np.int32)
    rows = []
    for i, s in enumerate(seqs):
        nb = -(-int(cl[s]) // W.BLOCK_SIZE)
        sub_bt[i, :nb] = [remap[int(b)] for b in bt[s, :nb]]
        sub_cl[i] = cl[s]
        rows.extend(range(int(qsl[s]), int(qsl[s + 1])))
        sub_qsl[i + 1] = sub_qsl[i] + (qsl[s + 1] - qsl[s])
    rows = np.array(rows, dtype=np.int64)
    rows_t = torch.from_numpy(rows).to(pre_k.device)
    q = W.as_oracle_array(wl_gpu.q.index_select(0, rows_t))
    kn = W.as_oracle_array(wl_gpu.k_new.index_select(0, rows_t))
    vn = W.as_oracle_array(wl_gpu.v_new.index_select(0, rows_t))
    # slots of the new tokens, renumbered into the compact pool
    slots = wl_gpu.slot_mapping.cpu().numpy()[rows]
    blk, off = slots // W.BLOCK_SIZE, slots % W.BLOCK_SIZE
    sub_slots = np.array([remap[int(b)] * W.BLOCK_SIZE + int(o) for b, o in zip(blk, off)],
                         np.int64)
    assert oracle.write(kn, vn, sub_slots, kc, vc) == 0
    P = oracle.Problem(q, kc, vc, sub_bt, sub_cl, sub_qsl, wl_gpu.scale, window)
    return P, rows


# ------------------------------------------------------------ FP8 (e4m3) cache

def fp8_scale_tensors(hkv, num_seqs, seed, device="cuda"):
    """(k_scale, v_scale) fp32 [Hkv] and the matching descales [S, Hkv] (each
    sequence reads the cache with the scales it was written with)."""
    ks = W.fp8_scales(hkv, seed)
    vs = W.fp8_scales(hkv, seed + 1)
    kd = np.tile(ks, (num_seqs, 1))
    vd = np.tile(vs, (num_seqs, 1))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return t(ks), t(vs), t(kd), t(vd)


def gpu_fp8_caches(g, k_scale, v_scale):
    """e4m3 caches on the GPU holding the workload's history, quantised by
    pkv_write_fp8 from the bf16 pool; every other slot holds the NaN code."""
    from paged_kv_cache_43_gb300 import pkv
    nb, bs, hkv, d = g.k_cache.shape
    kc8 = torch.full(g.k_cache.shape, W.E4M3_NAN_CODE, dtype=torch.uint8, device=g.q.device)
    vc8 = torch.full_like(kc8, W.E4M3_NAN_CODE)
    slots = torch.from_numpy(W.history_slots(g)).to(g.q.device)
    kh = g.k_cache.view(nb * bs, hkv, d).index_select(0, slots).contiguous()
    vh = g.v_cache.view(nb * bs, hkv, d).index_select(0, slots).contiguous()
    pkv.write_fp8(kh, vh, slots, kc8, vc8, k_scale, v_scale)
    return kc8, vc8


def oracle_fp8_caches(wl, k_scale, v_scale):
    """The oracle's e4m3 caches of the workload's history (same recipe)."""
    A = W.as_oracle_array
    nb, bs, hkv, d = wl.k_cache.shape
    ks, vs = A(k_scale), A(v_scale)
    kc = np.full((nb, bs, hkv, d), W.E4M3_NAN_CODE, np.uint8)
    vc = kc.copy()
    slots = W.history_slots(wl)
    kb = A(wl.k_cache).reshape(nb * bs, hkv, d)[slots]
    vb = A(wl.v_cache).reshape(nb * bs, hkv, d)[slots]
    assert oracle.write_fp8(kb, vb, slots, kc, vc, ks, vs) == 0
    return kc, vc


def oracle_step_fp8(wl, k_scale, v_scale, k_descale, v_descale, window=0):
    """Oracle result of one FP8 step: history quantised, this step's tokens
    quantised into it, attention with the descales.  (out, status, kc, vc)."""
    A = W.as_oracle_array
    ks, vs = A(k_scale), A(v_scale)
    kc, vc = oracle_fp8_caches(wl, k_scale, v_scale)
    assert oracle.write_fp8(A(wl.k_new), A(wl.v_new), A(wl.slot_mapping), kc, vc, ks, vs) == 0
    out, st = oracle.attention(A(wl.q), kc, vc, A(wl.block_tables), A(wl.context_lens),
                               A(wl.query_start_loc), wl.scale, window=window,
                               k_descale=A(k_descale), v_descale=A(v_descale))
    return out, st, kc, vc


def compact_subproblem_fp8(g, seqs, k_scale, v_scale, k_descale, v_descale, window=0):
    """compact_subproblem for an FP8 step: the sequences' bf16 blocks (g's bf16
    pool is the pre-step history) gathered into a compact pool, quantised by the
    oracle (history, then this step's tokens).  Returns (oracle.Problem, rows)."""
    A = W.as_oracle_array
    bt = g.block_tables.cpu().numpy()
    cl = g.context_lens.cpu().numpy()
    qsl = g.query_start_loc.cpu().numpy()
    ids = []
    for s in seqs:
        ids.extend(int(b) for b in bt[s, :-(-int(cl[s]) // W.BLOCK_SIZE)])
    uniq = sorted(set(ids))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.int64, device=g.q.device)
    kb = A(g.k_cache.index_select(0, idx))
    vb = A(g.v_cache.index_select(0, idx))
    nbc, bs, hkv, d = kb.shape
    kc = np.full(kb.shape, W.E4M3_NAN_CODE, np.uint8)
    vc = kc.copy()
    stride = bt.shape[1]
    sub_bt = np.full((len(seqs), stride), -1, np.int32)
    sub_cl = np.zeros(len(seqs), np.int32)
    sub_qsl = np.zeros(len(seqs) + 1, np.int32)
    rows, hist = [], []
    for i, s in enumerate(seqs):
        nb = -(-int(cl[s]) // W.BLOCK_SIZE)
        sub_bt[i, :nb] = [remap[int(b)] for b in bt[s, :nb]]
        sub_cl[i] = cl[s]
        n = int(qsl[s + 1] - qsl[s])
        pos = np.arange(int(cl[s]) - n)
        hist.append(sub_bt[i, pos // bs].astype(np.int64) * bs + pos % bs)
        rows.extend(range(int(qsl[s]), int(qsl[s + 1])))
        sub_qsl[i + 1] = sub_qsl[i] + n
    hist = np.unique(np.concatenate(hist))
    ks, vs = A(k_scale), A(v_scale)
    assert oracle.write_fp8(kb.reshape(-1, hkv, d)[hist], vb.reshape(-1, hkv, d)[hist], hist,
                            kc, vc, ks, vs) == 0
    rows = np.array(rows, dtype=np.int64)
    rows_t = torch.from_numpy(rows).to(g.q.device)
    slots = g.slot_mapping.cpu().numpy()[rows]
    sub_slots = np.array([remap[int(b)] * bs + int(o)
                          for b, o in zip(slots // bs, slots % bs)], np.int64)
    assert oracle.write_fp8(A(g.k_new.index_select(0, rows_t)),
                            A(g.v_new.index_select(0, rows_t)), sub_slots, kc, vc, ks, vs) == 0
    sel = np.asarray(seqs, dtype=np.int64)
    P = oracle.Problem(A(g.q.index_select(0, rows_t)), kc, vc, sub_bt, sub_cl, sub_qsl, g.scale,
                       window, A(k_descale)[sel], A(v_descale)[sel])
    return P, rows
