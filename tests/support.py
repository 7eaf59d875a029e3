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
