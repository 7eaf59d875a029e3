"""Pins of the CPU oracle to facts outside itself.

Each test ties the oracle to something other than its own formula: values the
pages print (tests/golden/block_bytes.json), hand-worked examples
(tests/golden/hand_examples.json), a library routine (torch's float64
scaled_dot_product_attention, with its own GQA and causal handling), the
second brute-force oracle, invariances that a wrong index breaks, and closed
forms.  Runs on CPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from paged_kv_cache_43_gb300 import workloads as W
from tests.support import oracle_step

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _oracle_args(wl):
    A = W.as_oracle_array
    return (A(wl.q), A(wl.k_cache), A(wl.v_cache), A(wl.block_tables),
            A(wl.context_lens), A(wl.query_start_loc), wl.scale)


def _written(wl):
    """Workload with this step's new K/V already written (by the oracle)."""
    kc, vc = W.as_oracle_array(wl.k_cache).copy(), W.as_oracle_array(wl.v_cache).copy()
    bad = oracle.write(W.as_oracle_array(wl.k_new), W.as_oracle_array(wl.v_new),
                       W.as_oracle_array(wl.slot_mapping), kc, vc)
    assert bad == 0
    A = W.as_oracle_array
    return (A(wl.q), kc, vc, A(wl.block_tables), A(wl.context_lens),
            A(wl.query_start_loc), wl.scale)


# ---------------------------------------------------------------- page facts

def test_block_bytes_formula_matches_pages():
    g = _load("block_bytes.json")
    for c in g["cases"]:
        dt = {"float32": torch.float32, "bfloat16": torch.bfloat16}[c["dtype"]]
        got = W.cache_bytes_per_block(c["num_kv_heads"], c["head_size"], dt)
        assert got == c["bytes_per_block"], c
        # and the generator's pools hold exactly that many bytes per block
        wl = W.make_workload([1], [3], num_q_heads=c["num_kv_heads"],
                             num_kv_heads=c["num_kv_heads"], head_size=c["head_size"],
                             dtype=dt, num_blocks=2)
        per_block = (wl.k_cache.numel() * wl.k_cache.element_size()
                     + wl.v_cache.numel() * wl.v_cache.element_size()) // wl.num_blocks
        assert per_block == c["bytes_per_block"]


def test_blocks_per_sequence_ceil16():
    g = _load("block_bytes.json")
    for n_tok, n_blk in g["blocks_for_tokens"]:
        wl = W.make_workload([1], [n_tok], num_q_heads=1, num_kv_heads=1, head_size=64,
                             dtype=torch.float32)
        assert int((wl.block_tables[0] >= 0).sum()) == n_blk
    wl = W.workload(1)
    per_seq = (wl.block_tables >= 0).sum(dim=1).tolist()
    assert per_seq == g["workload1_blocks"]["blocks"]
    ids = wl.block_tables[wl.block_tables >= 0]
    assert ids.numel() == g["workload1_blocks"]["total"] == len(set(ids.tolist()))
    assert int(ids.max()) < 64 and wl.num_blocks == 64


# ---------------------------------------------------------- hand-worked cases

def _hand_problem(case, g):
    D, bs, nb = g["head_size"], g["block_size"], g["num_blocks"]
    hkv, hq = case["kv_heads"], case["q_heads"]
    kc = np.full((nb, bs, hkv, D), np.nan, dtype=np.float32)
    vc = np.full((nb, bs, hkv, D), np.nan, dtype=np.float32)
    blk = g["block_table"][0]
    L = case["context_len"]
    for p in range(L):
        kc[blk, p, :, :] = g["keys"][p]
        vc[blk, p, :, :] = g["values"][p]
    q = np.array(case["queries"], dtype=np.float32).reshape(case["query_len"], hq, D)
    bt = np.array([g["block_table"]], dtype=np.int32)
    return q, kc, vc, bt, np.array([L], np.int32), np.array([0, case["query_len"]], np.int32)


@pytest.mark.parametrize("idx", range(4))
def test_hand_examples(idx):
    g = _load("hand_examples.json")
    case = g["cases"][idx]
    q, kc, vc, bt, cl, qsl = _hand_problem(case, g)
    exp = np.array(case["expected"], dtype=np.float64)
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, 1.0)
    assert st.tolist() == [0]
    np.testing.assert_allclose(out, exp, atol=g["tolerance"], rtol=0)
    out_b = brute.attention(q, kc, vc, bt, cl, qsl, 1.0)
    np.testing.assert_allclose(out_b, exp, atol=g["tolerance"], rtol=0)


# ------------------------------------------------- library routine: torch SDPA

def _sdpa(q, k, v, scale, causal):
    """torch float64 SDPA, [n, Hq, D] x [L, Hkv, D] -> [n, Hq, D]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, is_causal=causal, scale=scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (8, 1)])
def test_decode_matches_library_dense_attention(hq, hkv):
    ctx = [1, 15, 16, 17, 40, 100]
    wl = W.make_workload([1] * len(ctx), ctx, num_q_heads=hq, num_kv_heads=hkv,
                         head_size=64, dtype=torch.float32, seed=7, contiguous_blocks=True)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    assert not st.any()
    # Identity placement: sequence s's keys are pool rows in order.
    flat_k = kc.reshape(-1, hkv, 64).astype(np.float64)
    flat_v = vc.reshape(-1, hkv, 64).astype(np.float64)
    for s, L in enumerate(ctx):
        first = int(bt[s, 0]) * 16
        ref = _sdpa(q[s:s + 1].astype(np.float64), flat_k[first:first + L],
                    flat_v[first:first + L], sc, causal=False)
        np.testing.assert_allclose(out[s:s + 1], ref, atol=1e-12, rtol=1e-12)


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 1)])
def test_full_prompt_matches_library_causal_attention(hq, hkv):
    L = 37
    wl = W.make_workload([L], [L], num_q_heads=hq, num_kv_heads=hkv, head_size=64,
                         dtype=torch.float32, seed=11, contiguous_blocks=True)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    assert not st.any()
    flat_k = kc.reshape(-1, hkv, 64)[:L].astype(np.float64)
    flat_v = vc.reshape(-1, hkv, 64)[:L].astype(np.float64)
    ref = _sdpa(q.astype(np.float64), flat_k, flat_v, sc, causal=True)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=1e-12)


def test_chunk_equals_tail_of_full_prompt():
    """A prefill chunk of the last n queries must give the last n rows of the
    full-prompt result (the causal offset q_abs = q_idx + L - n)."""
    L, n = 70, 23
    wl = W.make_workload([L], [L], num_q_heads=4, num_kv_heads=2, head_size=64,
                         dtype=torch.float32, seed=3)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    full, _ = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    chunk, st = oracle.attention(q[L - n:], kc, vc, bt, cl, np.array([0, n], np.int32), sc)
    assert not st.any()
    np.testing.assert_array_equal(chunk, full[L - n:])


# ------------------------------------------------------------- invariances

def test_block_relabelling_is_bit_identical():
    q_lens, ctx, _ = W.lengths(3, small=True)
    ctx = ctx[:6]
    wl = W.make_workload(q_lens[:6], ctx, num_q_heads=8, num_kv_heads=2, head_size=64,
                         dtype=torch.bfloat16, seed=5)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    assert not st.any()
    rng = np.random.default_rng(0)
    perm = rng.permutation(kc.shape[0])          # new id of old block b = perm[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, st2 = oracle.attention(q, kc2, vc2, bt2, cl, qsl, sc)
    assert not st2.any()
    np.testing.assert_array_equal(out, out2)


def test_prefix_shared_blocks_read_through_every_table():
    """Two sequences whose tables share their first blocks see the same
    history: with equal queries, equal lengths and new tokens equal too,
    outputs must be identical although the tails live in other blocks."""
    wl = W.make_workload([1, 1], [50, 50], num_q_heads=2, num_kv_heads=2, head_size=64,
                         dtype=torch.float32, seed=9, shared_prefix_blocks=3,
                         shared_seqs=(0, 1))
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    assert (bt[0, :3] == bt[1, :3]).all() and bt[0, 3] != bt[1, 3]
    # make the private tail block of seq 1 a copy of seq 0's, and equal queries
    kc[bt[1, 3]] = kc[bt[0, 3]]
    vc[bt[1, 3]] = vc[bt[0, 3]]
    q[1] = q[0]
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    assert not st.any()
    np.testing.assert_array_equal(out[0], out[1])


# ------------------------------------------------------------- closed forms

def test_equal_keys_give_mean_of_visible_values():
    wl = W.make_workload([1, 5], [29, 40], num_q_heads=2, num_kv_heads=1, head_size=64,
                         dtype=torch.float32, seed=2)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    kc[:] = 0.5                       # every key identical -> uniform scores
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    assert not st.any()
    for s, (n, L) in enumerate([(1, 29), (5, 40)]):
        for j in range(n):
            pos = L - n + j
            rows = [int(bt[s, p // 16]) * 16 + p % 16 for p in range(pos + 1)]
            mean = vc.reshape(-1, 1, 64)[rows, 0, :].astype(np.float64).mean(axis=0)
            t = int(qsl[s]) + j
            for h in range(2):
                np.testing.assert_allclose(out[t, h], mean, atol=1e-13, rtol=0)


def test_single_key_and_dominant_key():
    wl = W.make_workload([1, 1], [1, 33], num_q_heads=1, num_kv_heads=1, head_size=64,
                         dtype=torch.float32, seed=4)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    # context length 1 -> exactly V[0]
    out, _ = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    v0 = vc[bt[0, 0], 0, 0].astype(np.float64)
    np.testing.assert_array_equal(out[0, 0], v0)
    # one key aligned with q and much larger than the rest -> its V
    p_dom = 20
    slot = int(bt[1, p_dom // 16]) * 16 + p_dom % 16
    kf = kc.reshape(-1, 1, 64)
    kf[slot, 0] = q[1, 0] * 40.0
    out, _ = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    np.testing.assert_allclose(out[1, 0], vc.reshape(-1, 1, 64)[slot, 0], atol=1e-9)


# ----------------------------------------------- second oracle (brute force)

@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_c_oracle_agrees_with_brute_force(n):
    if n == 1:
        wl = W.workload(1)
    else:
        q_lens, ctx, extra = W.lengths(n, small=True)
        keep = slice(0, 4) if n != 4 else slice(None)
        if n == 4:
            q_lens = np.minimum(q_lens, 20)
        wl = W.make_workload(q_lens[keep], np.minimum(ctx[keep], 400), num_q_heads=W.HEADS[n][0],
                             num_kv_heads=W.HEADS[n][1], head_size=64,
                             dtype=torch.bfloat16, seed=n,
                             **({} if n != 4 else dict(shared_prefix_blocks=2, shared_seqs=(0, 1, 2))))
    args = _written(wl)
    out, st = oracle.attention(*args)
    assert not st.any()
    ref = brute.attention(*args)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=1e-10)


# ------------------------------------------------------- split and merge

def test_partial_states_merge_to_full_result():
    wl = W.make_workload([1, 30], [300, 200], num_q_heads=4, num_kv_heads=2, head_size=64,
                         dtype=torch.bfloat16, seed=12)
    args = _written(wl)
    full, _ = oracle.attention(*args)
    P = oracle.Problem(*args)
    rng = np.random.default_rng(1)
    for s, j in [(0, 0), (1, 0), (1, 17), (1, 29)]:
        L, n = int(args[4][s]), int(args[5][s + 1] - args[5][s])
        cuts = np.sort(rng.choice(np.arange(1, L), size=5, replace=False))
        edges = [0, *cuts.tolist(), L]
        for hq in range(4):
            ms, ls, accs = [], [], []
            for lo, hi in zip(edges[:-1], edges[1:]):
                st, m, l, acc = oracle.row_state(P, s, hq, j, lo, hi)
                assert st == 0
                ms.append(m); ls.append(l); accs.append(acc)
            merged = oracle.merge(ms, ls, accs)
            t = int(args[5][s]) + j
            np.testing.assert_allclose(merged, full[t, hq], atol=1e-12, rtol=0)
    # a range past the causal limit is empty: m = -inf, l = 0
    st, m, l, acc = oracle.row_state(P, 1, 0, 0, 190, 200)
    assert st == 0 and m == -math.inf and l == 0.0 and not acc.any()


# --------------------------------------------------------------- KV write

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_write_matches_numpy_scatter_and_skips_padding(dtype):
    wl = W.make_workload([1, 3, 2], [20, 35, 16], num_q_heads=2, num_kv_heads=2,
                         head_size=64, dtype=dtype, seed=6)
    A = W.as_oracle_array
    kc, vc = A(wl.k_cache).copy(), A(wl.v_cache).copy()
    kn, vn = A(wl.k_new), A(wl.v_new)
    slots = A(wl.slot_mapping).copy()
    slots[1] = -1                                  # padding entry
    exp_k, exp_v = kc.copy(), vc.copy()
    nb, bs = kc.shape[:2]
    fk = exp_k.reshape(nb * bs, *kc.shape[2:])
    fv = exp_v.reshape(nb * bs, *vc.shape[2:])
    keep = slots >= 0
    fk[slots[keep]] = kn[keep]
    fv[slots[keep]] = vn[keep]
    assert oracle.write(kn, vn, slots, kc, vc) == 0
    assert kc.tobytes() == exp_k.tobytes() and vc.tobytes() == exp_v.tobytes()
    # the skipped slot still holds its poison
    skipped = A(wl.slot_mapping)[1]
    raw = kc.reshape(nb * bs, -1)[skipped]
    assert np.isnan(raw.astype(np.float32) if dtype == torch.float32 else
                    brute.widen(raw)).all()


def test_write_counts_out_of_range_slots():
    kc = np.zeros((2, 16, 1, 64), np.float32)
    vc = np.zeros_like(kc)
    k = np.ones((2, 1, 64), np.float32)
    n_bad = oracle.write(k, k, np.array([5, 32], np.int64), kc, vc)
    assert n_bad == 1 and kc.reshape(32, 64)[5].tolist() == [1.0] * 64


def test_metadata_errors_zero_rows():
    wl = W.make_workload([1, 1], [20, 30], num_q_heads=2, num_kv_heads=2, head_size=64,
                         dtype=torch.float32, seed=8)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    cl = cl.copy()
    cl[0] = 0                                      # queries but no keys
    bt = bt.copy()
    bt[1, 1] = 999                                 # block id past the pool
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, sc)
    assert st.tolist() == [1, 2]
    assert (out[0] == 0).all() and np.isnan(out[1]).all()


# ------------------------------------------------------------ sliding window

def test_window_wider_than_context_is_full_attention():
    wl = W.make_workload([1, 7, 1], [40, 55, 90], num_q_heads=4, num_kv_heads=2, head_size=64,
                         dtype=torch.bfloat16, seed=21)
    args = _written(wl)
    full, _ = oracle.attention(*args)
    wide, st = oracle.attention(*args, window=90)
    assert not st.any()
    np.testing.assert_array_equal(full, wide)


def test_window_of_one_gives_the_query_own_value():
    wl = W.make_workload([1, 5], [37, 50], num_q_heads=2, num_kv_heads=1, head_size=64,
                         dtype=torch.float32, seed=22)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    out, st = oracle.attention(q, kc, vc, bt, cl, qsl, sc, window=1)
    assert not st.any()
    vf = vc.reshape(-1, 1, 64).astype(np.float64)
    for s, (n, L) in enumerate([(1, 37), (5, 50)]):
        for j in range(n):
            pos = L - n + j
            slot = int(bt[s, pos // 16]) * 16 + pos % 16
            t = int(qsl[s]) + j
            for h in range(2):
                np.testing.assert_array_equal(out[t, h], vf[slot, 0])


@pytest.mark.parametrize("window", [2, 16, 17, 40])
def test_window_matches_brute_force(window):
    wl = W.make_workload([1, 20, 1, 33], [70, 64, 17, 100], num_q_heads=8, num_kv_heads=2,
                         head_size=64, dtype=torch.bfloat16, seed=23)
    args = _written(wl)
    out, st = oracle.attention(*args, window=window)
    assert not st.any()
    np.testing.assert_allclose(out, brute.attention(*args, window=window), atol=1e-12,
                               rtol=1e-10)


def test_window_never_reads_blocks_before_the_window():
    """Entries for blocks wholly before every query's window may hold the null
    block (here: an invalid id); results must not change."""
    wl = W.make_workload([1, 4], [100, 90], num_q_heads=2, num_kv_heads=2, head_size=64,
                         dtype=torch.bfloat16, seed=24)
    q, kc, vc, bt, cl, qsl, sc = _written(wl)
    out, _ = oracle.attention(q, kc, vc, bt, cl, qsl, sc, window=20)
    bt2 = bt.copy()
    bt2[0, : (100 - 20) // 16] = -1              # keys < 80 are outside every window
    bt2[1, : (90 - 4 - 20 + 1) // 16] = -1       # first query at 86 sees keys > 66
    out2, st = oracle.attention(q, kc, vc, bt2, cl, qsl, sc, window=20)
    assert not st.any()
    np.testing.assert_array_equal(out, out2)


# ------------------------------------------------------------ FP8 (e4m3) cache

def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2          # 0x7F, 0xFF
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rounding_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 100, 2000),
                        rng.uniform(-2 ** -6, 2 ** -6, 2000),             # subnormal range
                        [1.0625, 1.1875, 2 ** -10, 3 * 2 ** -10, -0.0, 440.0, 447.9]])
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_clamps_beyond_the_largest_finite():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-500.0) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_fp8_write_quantises_per_head_and_skips_padding():
    wl = W.make_workload([1, 3], [20, 35], num_q_heads=4, num_kv_heads=2, head_size=64,
                         dtype=torch.bfloat16, seed=31)
    A = W.as_oracle_array
    nb = wl.num_blocks
    kc = np.full((nb, 16, 2, 64), 0x7F, np.uint8)
    vc = kc.copy()
    slots = A(wl.slot_mapping).copy()
    slots[0] = -1
    ks = np.array([0.5, 2.0], np.float32)
    vs = np.array([1.25, 0.125], np.float32)
    assert oracle.write_fp8(A(wl.k_new), A(wl.v_new), slots, kc, vc, ks, vs) == 0
    # expectation built with torch: fp32 division by the head's scale, then
    # torch's e4m3 cast (values here stay inside +-448)
    for t in range(len(slots)):
        if slots[t] < 0:
            continue
        for cache, src, sc in ((kc, wl.k_new, ks), (vc, wl.v_new, vs)):
            x = src[t].float() / torch.from_numpy(sc)[:, None]
            assert float(x.abs().max()) <= 448
            ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(cache.reshape(-1, 2, 64)[slots[t]], ref)
    assert (kc.reshape(-1, 2, 64)[A(wl.slot_mapping)[0]] == 0x7F).all()   # padding skipped


def test_fp8_attention_equals_bf16_attention_on_representable_values():
    """Codes times power-of-two descales are exact in bf16: the fp8 path must
    give the bf16 path's result."""
    wl = W.make_workload([1, 6, 1], [45, 70, 33], num_q_heads=8, num_kv_heads=2,
                         head_size=64, dtype=torch.bfloat16, seed=32)
    A = W.as_oracle_array
    rng = np.random.default_rng(1)
    nb = wl.num_blocks
    codes_k = rng.integers(0, 0x7E, size=(nb, 16, 2, 64), dtype=np.uint8) | \
        (rng.integers(0, 2, size=(nb, 16, 2, 64), dtype=np.uint8) << 7)
    codes_v = rng.integers(0, 0x7E, size=(nb, 16, 2, 64), dtype=np.uint8)
    kd = np.array([[2.0 ** -6, 2.0 ** -5], [2.0 ** -7, 2.0 ** -6], [2.0 ** -5, 2.0 ** -8]],
                  np.float32)
    vd = np.array([[0.5, 0.25], [1.0, 0.5], [0.125, 1.0]], np.float32)
    dec = np.vectorize(oracle.e4m3_decode)
    kval, vval = dec(codes_k), dec(codes_v)
    out8, st = oracle.attention(A(wl.q), codes_k, codes_v, A(wl.block_tables),
                                A(wl.context_lens), A(wl.query_start_loc), wl.scale,
                                k_descale=kd, v_descale=vd)
    assert not st.any()
    # same values as bf16 caches, sequence by sequence (descales differ per sequence)
    for s in range(3):
        k16 = torch.from_numpy(kval * kd[s][None, None, :, None]).to(torch.bfloat16)
        v16 = torch.from_numpy(vval * vd[s][None, None, :, None]).to(torch.bfloat16)
        assert torch.equal(k16.double(), torch.from_numpy(kval * kd[s][None, None, :, None]))
        ref, _ = oracle.attention(A(wl.q), A(k16), A(v16), A(wl.block_tables),
                                  A(wl.context_lens), A(wl.query_start_loc), wl.scale)
        q0, q1 = int(wl.query_start_loc[s]), int(wl.query_start_loc[s + 1])
        np.testing.assert_allclose(out8[q0:q1], ref[q0:q1], atol=1e-12, rtol=0)


# ------------------------------------------------------- cascade

@pytest.mark.parametrize("hq,hkv,pblocks", [(4, 4, 3), (8, 2, 8), (8, 1, 1)])
def test_cascade_decomposition_equals_attention(hq, hkv, pblocks):
    """Prefix state (shared keys) merged with the suffix state = the plain
    attention of each decode row (ch. 6 cascade branch + merge_attn_states)."""
    S = 6
    rng = np.random.default_rng(hq + pblocks)
    ctx = rng.integers(pblocks * 16 + 1, pblocks * 16 + 90, S)
    wl = W.make_workload([1] * S, ctx, num_q_heads=hq, num_kv_heads=hkv, head_size=64,
                         dtype=torch.float32, seed=17 + pblocks, shared_prefix_blocks=pblocks,
                         shared_seqs=tuple(range(S)))
    exp, _, kc, vc = oracle_step(wl)
    A = W.as_oracle_array
    P = oracle.Problem(A(wl.q), kc, vc, A(wl.block_tables), A(wl.context_lens),
                       A(wl.query_start_loc), wl.scale)
    got = oracle.cascade(P, pblocks * 16)
    np.testing.assert_allclose(got, exp, atol=1e-12, rtol=0)


@pytest.mark.parametrize("q_lens,pblocks", [([5, 1, 17, 3], 2), ([33, 16, 1], 4), ([1, 1, 40], 1)])
def test_cascade_decomposition_equals_attention_for_chunks(q_lens, pblocks):
    """The same with chunked-prefill rows (ch. 6: the prefix call covers every
    query token of the batch): each chunk row's state over the shared keys
    merged with its causal state over its own keys = its plain attention."""
    S = len(q_lens)
    rng = np.random.default_rng(sum(q_lens) + pblocks)
    ctx = [pblocks * 16 + q + int(rng.integers(0, 60)) for q in q_lens]
    wl = W.make_workload(q_lens, ctx, num_q_heads=8, num_kv_heads=2, head_size=64,
                         dtype=torch.float32, seed=23 + pblocks, shared_prefix_blocks=pblocks,
                         shared_seqs=tuple(range(S)))
    exp, _, kc, vc = oracle_step(wl)
    A = W.as_oracle_array
    P = oracle.Problem(A(wl.q), kc, vc, A(wl.block_tables), A(wl.context_lens),
                       A(wl.query_start_loc), wl.scale)
    got = oracle.cascade(P, pblocks * 16)
    np.testing.assert_allclose(got, exp, atol=1e-12, rtol=0)


def test_cascade_refuses_a_row_inside_the_prefix():
    wl = W.make_workload([4], [40], num_q_heads=2, num_kv_heads=2, head_size=64,
                         dtype=torch.float32, seed=3)
    exp, _, kc, vc = oracle_step(wl)
    A = W.as_oracle_array
    P = oracle.Problem(A(wl.q), kc, vc, A(wl.block_tables), A(wl.context_lens),
                       A(wl.query_start_loc), wl.scale)
    with pytest.raises(AssertionError):
        oracle.cascade(P, 48)     # rows at positions 36..39 < 48
