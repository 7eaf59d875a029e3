"""Benchmark of the paged KV-cache hot path on GB300.

One step = one pass of the whole path over one synthetic decode batch: the KV
write of this step's new tokens (pkv_write), then paged attention over the
updated cache (pkv_attention: split-K decode kernel + combine).  The default
workload is the LLaMA-7B-shaped decode batch (32 q = 32 kv heads, head_size
128, bf16, 64 sequences, context lengths uniform in [128, 4096]).

Metric: KV bytes moved per second (algorithmic bytes / device time), with the
fraction of the measured HBM copy bandwidth and decode tokens/s.  Inputs are
resident in HBM before timing; the KV pool (~2.4 GB) is far larger than L2, so
no flush is needed between steps.  `--impl reference` times the CPU oracle on
a bounded sample of the same workload instead.

Launch: `python bench.py [--gpus N --steps K --warmup W]`; for N > 1 under
torchrun each rank runs its own seeded batch of the same shape (sequences are
independent: weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged-attn KV GB/s and % of GB300 HBM peak; decode tokens/s at batch"
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "paged_kv_cache_43_gb300", "csrc")


# ----------------------------------------------------------------- helpers

def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def rank_seed(workload: int, rank: int) -> int:
    """Each rank draws its own batch of the same shape (independent replicas)."""
    from paged_kv_cache_43_gb300 import workloads as W
    return W.SEED_BASE + workload + 1000 * rank


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time: the whole job is done when it is."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moves its own bytes in the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak(sustained: bool = False):
    """Measured dense bf16 tensor throughput (TFLOP/s): the burst figure for a
    launch timed alone, the sustained one for a launch inside a long step."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as f:
            return float(json.load(f)[key]), "measured " + key
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback " + key


def attention_flops(wl, seqs, window=0):
    """4 * head_size flops per (query row, q head, visible key): the two
    products of the attention definition (scores and weighted sum)."""
    f = 0
    for s in seqs:
        L, n = int(wl.ctx_lens[s]), int(wl.q_lens[s])
        vis = L - n + np.arange(n, dtype=np.int64) + 1       # keys 0 .. pos
        if window > 0:
            vis = np.minimum(vis, window)
        f += int(vis.sum())
    return f * wl.num_q_heads * 4 * wl.head_size


def sub_batch(wl, s0, s1):
    """Sequences [s0, s1) of a workload as a batch of their own over the same
    caches (views of its tensors; query_start_loc rebased)."""
    from paged_kv_cache_43_gb300 import workloads as W
    qsl = wl.query_start_loc.cpu().numpy()
    t0, t1 = int(qsl[s0]), int(qsl[s1])
    out = W.Workload(**{k: getattr(wl, k) for k in wl.__dataclass_fields__})
    for name in ("q", "k_new", "v_new", "slot_mapping"):
        setattr(out, name, getattr(wl, name)[t0:t1])
    out.block_tables = wl.block_tables[s0:s1]
    out.context_lens = wl.context_lens[s0:s1]
    out.query_start_loc = (wl.query_start_loc[s0:s1 + 1] - t0).contiguous()
    out.q_lens, out.ctx_lens = wl.q_lens[s0:s1], wl.ctx_lens[s0:s1]
    out.num_decode_seqs = max(0, min(wl.num_decode_seqs, s1) - s0)
    out.shared_seqs = ()
    return out


def decode_source_hash() -> str:
    """sha256 over what the decode kernel is compiled from: its source, the
    common device header and its argument struct (DecodeArgs, the text of its
    definition in pkv_internal.h; the other structs there do not reach it)."""
    h = hashlib.sha256()
    for name in ("pkv_decode.cu", "pkv_common.cuh"):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(CSRC, "pkv_internal.h"), "rb") as f:
        text = f.read()
    a = text.index(b"struct DecodeArgs {")
    h.update(text[a:text.index(b"};", a) + 2])
    return h.hexdigest()


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha256") != decode_source_hash():
        return None
    return rec.get("per_workload", {}).get(workload_name)


def algorithmic_bytes(wl, window=0, fp8=False):
    """Bytes the step must move at minimum.
    attention: each K and V row some query of its sequence can see, once (one
    byte per element for an e4m3 cache); q read, out written, the block-table
    entries of those rows and per-sequence metadata (and descales) read;
    write: new K/V rows read and written (as codes for e4m3), slots read."""
    e = wl.q.element_size()
    ekv = 1 if fp8 else e
    hkv, d, hq = wl.num_kv_heads, wl.head_size, wl.num_q_heads
    ctx = wl.ctx_lens.astype(np.int64)
    if window > 0:   # keys [L - q_s - W + 1, L) are visible to some row
        ctx = ctx - np.maximum(0, ctx - wl.q_lens.astype(np.int64) - window + 1)
    kv = int(ctx.sum()) * hkv * d * ekv * 2
    qo = 2 * wl.num_tokens * hq * d * e
    meta = int(np.ceil(ctx / 16).sum()) * 4 + wl.num_seqs * 4 + (wl.num_seqs + 1) * 4
    if fp8:
        meta += 2 * wl.num_seqs * hkv * 4
    attn = kv + qo + meta
    write = 2 * wl.num_tokens * hkv * d * (e + ekv) + wl.num_tokens * 8
    if fp8:
        write += 2 * hkv * 4
    return attn, write, kv


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"pkv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9 or p[0] != self.gpu:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx = max(mx, float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- oracle leg

def oracle_sample(wl_gpu, seqs, kv_heads=None, fp8=None):
    """CPU inputs (compact pool) for the sequences `seqs`, with this step's new
    tokens, for the oracle.  Must be taken before any step has run, so that
    no oracle input passes through the CUDA path.  `kv_heads` keeps only the
    first kv heads (and their query-head groups).  `fp8` = (k_scale, v_scale,
    k_descale, v_descale) as numpy: the sample's history is quantised to e4m3
    by the oracle (every other slot holds the NaN code)."""
    from paged_kv_cache_43_gb300 import workloads as W
    bt = wl_gpu.block_tables.cpu().numpy()
    cl = wl_gpu.context_lens.cpu().numpy()
    qsl = wl_gpu.query_start_loc.cpu().numpy()
    g = wl_gpu.num_q_heads // wl_gpu.num_kv_heads
    hkv = wl_gpu.num_kv_heads if kv_heads is None else kv_heads
    uniq = sorted({int(b) for s in seqs for b in bt[s, :-(-int(cl[s]) // 16)]})
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.int64, device=wl_gpu.k_cache.device)
    kc = W.as_oracle_array(wl_gpu.k_cache.index_select(0, idx)[:, :, :hkv]).copy()
    vc = W.as_oracle_array(wl_gpu.v_cache.index_select(0, idx)[:, :, :hkv]).copy()
    sub_bt = np.full((len(seqs), bt.shape[1]), -1, np.int32)
    rows, sub_qsl = [], [0]
    for i, s in enumerate(seqs):
        nb = -(-int(cl[s]) // 16)
        sub_bt[i, :nb] = [remap[int(b)] for b in bt[s, :nb]]
        rows.extend(range(int(qsl[s]), int(qsl[s + 1])))
        sub_qsl.append(len(rows))
    rows_t = torch.tensor(rows, dtype=torch.int64, device=wl_gpu.q.device)
    slots = wl_gpu.slot_mapping.cpu().numpy()[rows]
    sub_slots = np.array([remap[int(x) // 16] * 16 + int(x) % 16 for x in slots], np.int64)
    A = W.as_oracle_array
    smp = dict(q=A(wl_gpu.q.index_select(0, rows_t)[:, : hkv * g]),
               k_new=A(wl_gpu.k_new.index_select(0, rows_t)[:, :hkv]),
               v_new=A(wl_gpu.v_new.index_select(0, rows_t)[:, :hkv]),
               slots=sub_slots, k_cache=kc, v_cache=vc, bt=sub_bt,
               cl=cl[seqs].astype(np.int32), qsl=np.array(sub_qsl, np.int32),
               scale=wl_gpu.scale, rows=rows)
    if fp8 is not None:
        import oracle
        ks, vs, kd, vd = (np.ascontiguousarray(a) for a in fp8)
        ks, vs = ks[:hkv].copy(), vs[:hkv].copy()
        kd, vd = kd[seqs][:, :hkv].copy(), vd[seqs][:, :hkv].copy()
        hist = []
        for i, s in enumerate(seqs):
            pos = np.arange(int(cl[s]) - int(qsl[s + 1] - qsl[s]))
            hist.append(sub_bt[i, pos // 16].astype(np.int64) * 16 + pos % 16)
        hist = np.unique(np.concatenate(hist))
        d = kc.shape[3]
        k8 = np.full(kc.shape, W.E4M3_NAN_CODE, np.uint8)
        v8 = k8.copy()
        assert oracle.write_fp8(kc.reshape(-1, hkv, d)[hist], vc.reshape(-1, hkv, d)[hist],
                                hist, k8, v8, ks, vs) == 0
        smp.update(k_cache=k8, v_cache=v8, fp8=(ks, vs, kd, vd))
    return smp


def oracle_pass(sample, window=0):
    """One oracle step on a sample: its own KV write, then attention."""
    import oracle
    kc, vc = sample["k_cache"].copy(), sample["v_cache"].copy()
    if "fp8" in sample:
        ks, vs, kd, vd = sample["fp8"]
        oracle.write_fp8(sample["k_new"], sample["v_new"], sample["slots"], kc, vc, ks, vs)
        out, _ = oracle.attention(sample["q"], kc, vc, sample["bt"], sample["cl"],
                                  sample["qsl"], sample["scale"], window=window,
                                  k_descale=kd, v_descale=vd)
        return out
    oracle.write(sample["k_new"], sample["v_new"], sample["slots"], kc, vc)
    out, _ = oracle.attention(sample["q"], kc, vc, sample["bt"], sample["cl"], sample["qsl"],
                              sample["scale"], window=window)
    return out


def sample_bytes(sample, window=0):
    """Algorithmic bytes of one oracle pass over a sample (same accounting as
    algorithmic_bytes)."""
    ekv = sample["k_cache"].dtype.itemsize
    e = sample["q"].dtype.itemsize
    hkv, d = sample["k_cache"].shape[2], sample["k_cache"].shape[3]
    hq = sample["q"].shape[1]
    cl = sample["cl"].astype(np.int64)
    if window > 0:
        qn = np.diff(sample["qsl"]).astype(np.int64)
        cl = cl - np.maximum(0, cl - qn - window + 1)
    keys = int(cl.sum())
    t = int(sample["qsl"][-1])
    return keys * hkv * d * ekv * 2 + 2 * t * hq * d * e + 2 * t * hkv * d * (e + ekv)


def cpu_baseline(samples, name, num_seqs, window=0, budget_s=12.0):
    """The oracle, as it stands, over pre-step samples of the workload (one
    sequence each, all heads) until about budget_s of CPU time is spent."""
    import oracle
    spent, nbytes, passes = 0.0, 0, 0
    while spent < budget_s:
        for smp in samples:
            t0 = time.perf_counter()
            oracle_pass(smp, window)
            spent += time.perf_counter() - t0
            nbytes += sample_bytes(smp, window)
        passes += 1
    return {"value": round(nbytes / spent / 1e9, 4), "unit": "GB/s",
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{len(samples)} of {num_seqs} sequences (all heads) of {name}, "
                      f"{passes} passes: fp64 KV write + attention per sequence, "
                      f"{spent:.1f} s wall on the host cores"}


# ----------------------------------------------------------------- arms

class KVCache:
    """The caches a step runs on and the two calls of the step.  bf16: the
    workload's own pool.  fp8: e4m3 pools whose history is quantised from the
    workload's bf16 pool by pkv_write_fp8 (setup, not timed), per-kv-head
    scales drawn from the workload's seed; every sequence reads with the
    scales its blocks were written with."""

    def __init__(self, wl, fp8, seed, kv_split, window):
        from paged_kv_cache_43_gb300 import pkv
        from paged_kv_cache_43_gb300 import workloads as W
        self.pkv, self.wl, self.fp8 = pkv, wl, fp8
        self.meta_kw = dict(max_query_len=wl.max_query_len, max_context_len=wl.max_context_len,
                            num_decode_seqs=wl.num_decode_seqs, kv_split_tokens=kv_split,
                            sliding_window=window)
        dev = wl.q.device
        if not fp8:
            self.k, self.v = wl.k_cache, wl.v_cache
            self.np_scales = None
            return
        ks = W.fp8_scales(wl.num_kv_heads, seed)
        vs = W.fp8_scales(wl.num_kv_heads, seed + 1)
        kd, vd = np.tile(ks, (wl.num_seqs, 1)), np.tile(vs, (wl.num_seqs, 1))
        self.np_scales = (ks, vs, kd, vd)
        self.ks, self.vs, self.kd, self.vd = (torch.from_numpy(a).to(dev)
                                              for a in self.np_scales)
        self.k = torch.full(wl.k_cache.shape, W.E4M3_NAN_CODE, dtype=torch.uint8, device=dev)
        self.v = torch.full_like(self.k, W.E4M3_NAN_CODE)
        nb, bs, hkv, d = wl.k_cache.shape
        slots = torch.from_numpy(W.history_slots(wl)).to(dev)
        for part in torch.split(slots, 1 << 20):
            pkv.write_fp8(wl.k_cache.view(-1, hkv, d).index_select(0, part),
                          wl.v_cache.view(-1, hkv, d).index_select(0, part), part,
                          self.k, self.v, self.ks, self.vs)
        torch.cuda.synchronize(dev)

    def write(self, k_new, v_new, slots, stream):
        if self.fp8:
            self.pkv.write_fp8(k_new, v_new, slots, self.k, self.v, self.ks, self.vs,
                               stream=stream)
        else:
            self.pkv.write(k_new, v_new, slots, self.k, self.v, stream=stream)

    def attention(self, out, q, bt, cl, qsl, ws, stream, kd=None, vd=None, meta_kw=None):
        mk = self.meta_kw if meta_kw is None else meta_kw
        if self.fp8:
            self.pkv.attention_fp8(out, q, self.k, self.v, bt, cl, qsl, self.wl.scale,
                                   self.kd if kd is None else kd, self.vd if vd is None else vd,
                                   workspace=ws, stream=stream, **mk)
        else:
            self.pkv.attention(out, q, self.k, self.v, bt, cl, qsl, self.wl.scale,
                               workspace=ws, stream=stream, **mk)

    def part_timer(self, s0, s1, stream):
        """A zero-argument call of pkv_attention on sequences [s0, s1) alone
        (the caches already hold this step's tokens) and that part's batch."""
        sub = sub_batch(self.wl, s0, s1)
        mk = dict(self.meta_kw, max_query_len=sub.max_query_len,
                  max_context_len=sub.max_context_len, num_decode_seqs=sub.num_decode_seqs)
        meta = self.pkv.attn_meta(sub.q, sub.block_tables, sub.context_lens, **mk)
        ws = torch.empty(max(self.pkv.workspace_size(self.k, meta), 1), dtype=torch.uint8,
                         device=sub.q.device)
        out = torch.empty_like(sub.q)
        kd = self.kd[s0:s1].contiguous() if self.fp8 else None
        vd = self.vd[s0:s1].contiguous() if self.fp8 else None

        def call():
            self.attention(out, sub.q, sub.block_tables, sub.context_lens, sub.query_start_loc,
                           ws, stream, kd=kd, vd=vd, meta_kw=mk)
        return call, sub

    def step(self, out, ws, stream):
        wl = self.wl
        self.write(wl.k_new, wl.v_new, wl.slot_mapping, stream)
        self.attention(out, wl.q, wl.block_tables, wl.context_lens, wl.query_start_loc, ws,
                       stream)


def run_pkv(args, rank, world, device):
    from paged_kv_cache_43_gb300 import build, pkv
    from paged_kv_cache_43_gb300 import workloads as W

    build.build()
    pkv.load()
    seed = rank_seed(args.workload, rank)
    wl = W.workload(args.workload, device=device, seed=seed, num_seqs=args.num_seqs)
    fp8 = args.kv_dtype == "fp8"
    kv = KVCache(wl, fp8, seed, args.kv_split, args.window)
    if args.profile:
        return profile_only(args, kv)
    attn_b, write_b, kv_b = algorithmic_bytes(wl, args.window, fp8)
    step_b = attn_b + write_b
    out = torch.empty_like(wl.q)
    meta = pkv.attn_meta(wl.q, wl.block_tables, wl.context_lens, **kv.meta_kw)
    ws_n = pkv.workspace_size(kv.k, meta)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    nd = wl.num_seqs if wl.max_query_len <= 1 else wl.num_decode_seqs
    launches_per_step = (1 + (1 if nd > 0 else 0) + (1 if ws_n else 0)
                         + (1 if nd < wl.num_seqs else 0))
    # Oracle inputs are copied from the pristine (pre-step) bf16 pool; for fp8
    # the oracle quantises them itself.
    spot = oracle_sample(wl, [int(np.argmin(wl.ctx_lens)), int(np.argmax(wl.ctx_lens))],
                         fp8=kv.np_scales)
    base_samples = []
    if rank == 0 and not args.no_cpu_baseline:
        perm = np.random.default_rng(0).permutation(wl.num_seqs)[:12]
        base_samples = [oracle_sample(wl, [int(s)], fp8=kv.np_scales) for s in perm]

    def step():
        kv.step(out, ws, stream)

    pkv.get_error(clear=True)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    if pkv.get_error(clear=True):
        raise RuntimeError("device error word set during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(device.index if device.index is not None else 0) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        e0, e1, e2 = ev[i]
        e0.record(stream)
        kv.write(wl.k_new, wl.v_new, wl.slot_mapping, stream)
        e1.record(stream)
        kv.attention(out, wl.q, wl.block_tables, wl.context_lens, wl.query_start_loc, ws, stream)
        e2.record(stream)
    end.record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = start.elapsed_time(end)
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps
    write_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    if pkv.get_error(clear=True):
        raise RuntimeError("device error word set during the timed region")
    # parity spot check on the timed output: a few rows against the oracle
    parity = spot_check(wl, out, spot, args.window)

    total_ms = max_over_ranks(total_ms, world, device)
    ms_per_step = total_ms / args.steps

    # ---- end to end: host buffers in, host result out, same stream
    e2e = end_to_end(kv, args, stream, device, step_b)

    if rank != 0:
        return None
    peak, peak_kind = hbm_peak()
    value = job_throughput(step_b, world, ms_per_step)
    achieved = attn_b / (attn_ms * 1e-3) / 1e9
    # the committed counters were taken on full-attention batches at the
    # automatic split size: none for a window or a forced split
    traffic = (recorded_traffic(wl.name + ("-fp8" if fp8 else ""))
               if not args.window and not args.kv_split else None)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) q/k/v, random block placement)",
        "config": {
            "workload": wl.name,
            "num_seqs": wl.num_seqs, "num_q_heads": wl.num_q_heads,
            "num_kv_heads": wl.num_kv_heads, "head_size": wl.head_size, "block_size": 16,
            "context_lens": f"{int(wl.ctx_lens.min())}..{int(wl.ctx_lens.max())} "
                            f"(mean {wl.ctx_lens.mean():.0f})",
            "max_query_len": wl.max_query_len, "num_tokens": wl.num_tokens,
            "kv_split_tokens": args.kv_split or "auto",
            "sliding_window": args.window or None,
            "kv_cache_dtype": "fp8_e4m3" if fp8 else ("bf16" if wl.dtype == torch.bfloat16
                                                       else "f32"),
            "step": ("pkv_write_fp8 of the new tokens + pkv_attention_fp8" if fp8 else
                     "pkv_write of the new tokens + pkv_attention"),
            "l2": f"inputs larger than L2: {kv_b / 1e9:.2f} GB of K/V read per step, no flush",
            "parallelism": f"replicas x{world} (independent sequence batches)",
        },
        "pct_hbm_peak": round(100.0 * value / world / peak, 1),
        "decode_tokens_per_s": round(world * wl.num_tokens / (ms_per_step * 1e-3), 1),
        "attention_ms": round(attn_ms, 5),
        "write_ms": round(write_ms, 5),
        "roofline": {
            "kernel": ("pkv_attention (split-K decode kernel + combine), CUDA events per call"
                       if wl.num_decode_seqs == wl.num_seqs else
                       "pkv_attention (tcgen05 prefill on the side stream with the split-K "
                       "decode kernel + combine), CUDA events per call on the caller's stream"),
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
            "traffic": traffic,
            "algorithmic_bytes_per_launch": attn_b,
        },
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": e2e,
        "parity_max_abs_err": parity,
    }
    if wl.num_decode_seqs < wl.num_seqs:
        # a batch with prefill rows: its dense contraction bounds it
        line["roofline"] = mixed_roofline(kv, stream, attn_ms, min(args.steps, 200),
                                          args.window)
    if base_samples:
        line["cpu_baseline"] = cpu_baseline(base_samples, wl.name, wl.num_seqs, args.window)
    if (world == 1 and args.workload == 2 and not args.window and not args.kv_split
            and not args.num_seqs and args.kv_dtype == "bf16" and not args.no_per_workload):
        # the other decode and mixed configurations, and the e4m3 cache, each
        # measured briefly on the same GPU (not part of `value`)
        steps = max(50, min(args.steps, 200))
        line["per_workload"] = {
            f"{W.WORKLOAD_NAMES[n]}{'-fp8' if f else ''}": workload_entry(n, f, device, steps, 10)
            for n, f in PER_WORKLOAD}
    return line


def mixed_roofline(kv, stream, attn_ms, steps, window=0):
    """Roofline of a batch with decode and prefill rows: the prefill
    sequences' call timed alone against the tensor peak (it is the dense
    contraction: 4 D flops per row and visible key), the decode sequences'
    call timed alone against the HBM bandwidth, and the whole call against
    max(bytes / bandwidth, flops / tensor peak)."""
    wl = kv.wl
    nd, S = wl.num_decode_seqs, wl.num_seqs
    hbm, hbm_kind = hbm_peak()
    tpk, tpk_kind = tensor_peak(sustained=False)
    pf_call, pf = kv.part_timer(nd, S, stream)
    pf_ms = _time_calls(pf_call, steps, 5, stream)
    pf_flops = attention_flops(wl, range(nd, S), window)
    pf_bytes = algorithmic_bytes(pf, window, kv.fp8)[0]
    res = {
        "kernel": "pkv_prefill_tc_kernel: the prefill sequences' pkv_attention call timed "
                  "alone (CUDA events)",
        "bound": "tensor", "achieved": round(pf_flops / (pf_ms * 1e-3) / 1e12, 1),
        "peak": tpk, "unit": "TFLOP/s",
        "frac": round(pf_flops / (pf_ms * 1e-3) / 1e12 / tpk, 4),
        "peak_kind": tpk_kind, "traffic": None,
        "flops_per_launch": pf_flops, "launch_ms": round(pf_ms, 5),
    }
    total_flops = attention_flops(wl, range(S), window)
    total_bytes = algorithmic_bytes(wl, window, kv.fp8)[0]
    if nd:
        dc_call, dc = kv.part_timer(0, nd, stream)
        dc_ms = _time_calls(dc_call, steps, 5, stream)
        dc_bytes = algorithmic_bytes(dc, window, kv.fp8)[0]
        res["decode_half"] = {
            "kernel": "split-K decode kernel + combine: the decode sequences' call timed alone",
            "bound": "hbm", "achieved": round(dc_bytes / (dc_ms * 1e-3) / 1e9, 1),
            "peak": hbm, "unit": "GB/s", "frac": round(dc_bytes / (dc_ms * 1e-3) / 1e9 / hbm, 4),
            "peak_kind": f"{hbm_kind} hbm_gbs", "launch_ms": round(dc_ms, 5),
            "algorithmic_bytes_per_launch": dc_bytes}
    ideal_ms = max(total_bytes / (hbm * 1e9), total_flops / (tpk * 1e12)) * 1e3
    res["whole_call"] = {
        "attention_ms": round(attn_ms, 5), "ideal_ms": round(ideal_ms, 5),
        "frac": round(ideal_ms / attn_ms, 4),
        "ideal": "max(algorithmic bytes / HBM peak, flops / tensor peak)",
        "algorithmic_bytes": total_bytes, "flops": total_flops}
    return res


def workload_entry(n, fp8, device, steps, warmup):
    """One short measurement of workload n (rank-0 seed, automatic split):
    step time (write + attention), attention time, its roofline (HBM for
    decode batches; tensor for the prefill part of a mixed batch, with the
    decode part's HBM fraction beside it) and a parity spot check."""
    from paged_kv_cache_43_gb300 import pkv
    from paged_kv_cache_43_gb300 import workloads as W
    seed = rank_seed(n, 0)
    wl = W.workload(n, device=device, seed=seed)
    kv = KVCache(wl, fp8, seed, 0, 0)
    attn_b, write_b, kv_b = algorithmic_bytes(wl, 0, fp8)
    out = torch.empty_like(wl.q)
    meta = pkv.attn_meta(wl.q, wl.block_tables, wl.context_lens, **kv.meta_kw)
    ws = torch.empty(max(pkv.workspace_size(kv.k, meta), 1), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    spot = oracle_sample(wl, [int(np.argmin(wl.ctx_lens)), int(np.argmax(wl.ctx_lens))],
                         fp8=kv.np_scales)
    for _ in range(warmup):
        kv.step(out, ws, stream)
    torch.cuda.synchronize(device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e0, e1, e2 in ev:
        e0.record(stream)
        kv.write(wl.k_new, wl.v_new, wl.slot_mapping, stream)
        e1.record(stream)
        kv.attention(out, wl.q, wl.block_tables, wl.context_lens, wl.query_start_loc, ws, stream)
        e2.record(stream)
    torch.cuda.synchronize(device)
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / steps
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    if pkv.get_error(clear=True):
        raise RuntimeError(f"device error word set ({wl.name})")
    parity = spot_check(wl, out, spot)
    peak, peak_kind = hbm_peak()
    entry = {
        "workload": wl.name, "kv_cache_dtype": "fp8_e4m3" if fp8 else "bf16", "steps": steps,
        "ms_per_step": round(step_ms, 5), "attention_ms": round(attn_ms, 5),
        "kv_gbs_step": round((attn_b + write_b) / (step_ms * 1e-3) / 1e9, 1),
        "decode_tokens_per_s": round(wl.num_tokens / (step_ms * 1e-3), 1),
        "parity_max_abs_err": parity,
    }
    if wl.num_decode_seqs < wl.num_seqs:
        entry["roofline"] = mixed_roofline(kv, stream, attn_ms, steps)
    else:
        achieved = attn_b / (attn_ms * 1e-3) / 1e9
        entry["roofline"] = {
            "kernel": "pkv_attention (split-K decode kernel + combine), CUDA events per call",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
            "traffic": recorded_traffic(wl.name + ("-fp8" if fp8 else "")),
            "algorithmic_bytes_per_launch": attn_b}
    del kv, wl, out, ws
    torch.cuda.empty_cache()
    return entry


PER_WORKLOAD = [(3, False), (4, False), (5, False), (2, True), (3, True), (4, True), (5, True)]


def profile_only(args, kv):
    """Warm-up then `steps` plain steps, nothing else: a short, fixed launch
    sequence for ncu captures (not a bench measurement).  --part prefill or
    decode: after one whole step, only that part's attention call (the prefill
    sequences alone launch their CTAs longest first)."""
    from paged_kv_cache_43_gb300 import pkv
    wl = kv.wl
    out = torch.empty_like(wl.q)
    meta = pkv.attn_meta(wl.q, wl.block_tables, wl.context_lens, **kv.meta_kw)
    ws = torch.empty(max(pkv.workspace_size(kv.k, meta), 1), dtype=torch.uint8,
                     device=wl.q.device)
    stream = torch.cuda.current_stream()
    if args.part == "all":
        for _ in range(args.warmup + args.steps):
            kv.step(out, ws, stream)
    else:
        kv.step(out, ws, stream)
        nd = wl.num_decode_seqs
        s0, s1 = (nd, wl.num_seqs) if args.part == "prefill" else (0, nd)
        if s0 == s1:
            raise SystemExit(f"workload {wl.name} has no {args.part} sequences")
        call, _ = kv.part_timer(s0, s1, stream)
        for _ in range(args.warmup + args.steps):
            call()
    torch.cuda.synchronize()
    if pkv.get_error(clear=True):
        raise RuntimeError("device error word set")
    print(json.dumps({"profile_run": wl.name, "kv_cache_dtype": args.kv_dtype, "part": args.part,
                      "num_seqs": wl.num_seqs, "steps": args.warmup + args.steps}), flush=True)
    return None


def spot_check(wl, out, spot, window=0):
    """Max |error| of the timed output rows of the spot sample against the
    oracle (run on the pre-step copy)."""
    exp = oracle_pass(spot, window)
    got = out[torch.tensor(spot["rows"], device=out.device)].float().cpu().numpy()
    err = float(np.abs(got.astype(np.float64) - exp).max())
    if not (err <= (2e-2 if wl.dtype == torch.bfloat16 else 1e-5)):
        raise RuntimeError(f"timed output fails parity: max abs err {err}")
    return err


def end_to_end(kv, args, stream, device, step_bytes):
    """Same metric through the public calls with host-resident step inputs:
    every step copies its inputs -- q, new K/V, slots and metadata (and the
    descales of an e4m3 cache) -- from pinned host memory to the device, runs
    the write and the attention on them, and copies its output back to pinned
    host memory.  A step's inputs sit in one pinned staging buffer and go over
    in one copy.  The copies run on their own streams into double-buffered
    device staging, event-joined with the compute stream, so that step i + 1's
    inputs go up (and step i - 1's output comes down) while step i computes, as
    a serving loop stages its next batch ahead; every copy of the n timed
    steps is inside the timed region."""
    from paged_kv_cache_43_gb300 import pkv
    wl = kv.wl
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens",
             "query_start_loc")
    src = {n: getattr(wl, n) for n in names}
    if kv.fp8:
        src.update(k_descale=kv.kd, v_descale=kv.vd)
    offs, total = {}, 0
    for n, t in src.items():
        nbytes = t.numel() * t.element_size()
        offs[n] = (total, nbytes)
        total += (nbytes + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    for n, t in src.items():
        o, nb = offs[n]
        host_buf[o:o + nb].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]
    dev = [{n: b[o:o + nb].view(src[n].dtype).view(src[n].shape)
            for n, (o, nb) in offs.items()} for b in dev_bufs]
    out_h = [torch.empty(wl.q.shape, dtype=wl.q.dtype).pin_memory() for _ in range(2)]
    out_d = [torch.empty_like(wl.q) for _ in range(2)]
    h2d = sum(nb for _, nb in offs.values())
    d2h = out_h[0].numel() * out_h[0].element_size()
    meta = pkv.attn_meta(wl.q, wl.block_tables, wl.context_lens, **kv.meta_kw)
    ws = torch.empty(max(pkv.workspace_size(kv.k, meta), 1), dtype=torch.uint8,
                     device=device)
    up = torch.cuda.Stream(device)      # host -> device
    down = torch.cuda.Stream(device)    # device -> host
    ev = lambda: torch.cuda.Event()     # noqa: E731
    copied, done, drained = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(n, t_start=None):
        up.wait_stream(stream)
        down.wait_stream(stream)
        with torch.cuda.stream(up):
            dev_bufs[0].copy_(host_buf, non_blocking=True)
            copied[0].record(up)
        for i in range(n):
            b, nb = i % 2, (i + 1) % 2
            if i + 1 < n:   # the next step's inputs, once step i - 1 is done with them
                if i >= 1:
                    up.wait_event(done[nb])
                with torch.cuda.stream(up):
                    dev_bufs[nb].copy_(host_buf, non_blocking=True)
                    copied[nb].record(up)
            stream.wait_event(copied[b])
            if i >= 2:
                stream.wait_event(drained[b])   # step i - 2's output has left out_d[b]
            d = dev[b]
            kv.write(d["k_new"], d["v_new"], d["slot_mapping"], stream)
            kv.attention(out_d[b], d["q"], d["block_tables"], d["context_lens"],
                         d["query_start_loc"], ws, stream, kd=d.get("k_descale"),
                         vd=d.get("v_descale"))
            done[b].record(stream)
            down.wait_event(done[b])
            with torch.cuda.stream(down):
                out_h[b].copy_(out_d[b], non_blocking=True)
                drained[b].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    n = max(args.steps // 4, 10)
    run(3)
    torch.cuda.synchronize(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(n)
    b.record(stream)
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / n
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 5),
            "steps": n, "copies": "each step's inputs H2D and output D2H, on two copy "
                                  "streams overlapping the neighbouring steps' compute"}


def _time_calls(fn, steps, warmup, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_cascade_bench(args, device):
    """Cascade attention against the plain call on two batches whose sequences
    share a prefix: (1) the mixed workload 4, whose first 16 decode sequences
    share 64 blocks (cascade for those 16, pkv_attention for the rest of the
    batch), and (2) a decode batch of 64 sequences sharing a 2048-token prefix
    (suffixes U[128, 2048], 32 q / 8 kv heads, head_size 128).  Reports
    attention time and GB/s over the logical bytes (every sequence's keys) and
    over the unique bytes (the shared prefix counted once)."""
    from paged_kv_cache_43_gb300 import build, pkv
    from paged_kv_cache_43_gb300 import workloads as W
    build.build()
    pkv.load()
    stream = torch.cuda.current_stream(device)
    res = {}

    def kv_bytes(ctx, hkv, d, e=2):
        return int(np.asarray(ctx, np.int64).sum()) * hkv * d * e * 2

    # (2) shared-prefix decode batch
    S, P = 64, 128
    rng = np.random.default_rng(4321)
    ctx = P * 16 + rng.integers(128, 2048, S, endpoint=True)
    wl = W.make_workload(np.ones(S, np.int64), ctx, num_q_heads=32, num_kv_heads=8,
                         head_size=128, seed=4321, device=device, shared_prefix_blocks=P,
                         shared_seqs=tuple(range(S)))
    pkv.write(wl.k_new, wl.v_new, wl.slot_mapping, wl.k_cache, wl.v_cache)
    out = torch.empty_like(wl.q)
    meta = pkv.attn_meta(wl.q, wl.block_tables, wl.context_lens, max_query_len=1,
                         max_context_len=wl.max_context_len)
    ws = torch.empty(max(pkv.workspace_size(wl.k_cache, meta),
                         pkv.cascade_workspace_size(wl.k_cache, meta, P)), dtype=torch.uint8,
                     device=device)
    plain = lambda: pkv.attention(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables,
                                  wl.context_lens, wl.query_start_loc, wl.scale, max_query_len=1,
                                  max_context_len=wl.max_context_len, workspace=ws)
    casc = lambda: pkv.attention_cascade(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables,
                                         wl.context_lens, wl.query_start_loc, wl.scale, P,
                                         max_context_len=wl.max_context_len, workspace=ws)
    logical = kv_bytes(ctx, 8, 128)
    unique = kv_bytes(ctx - P * 16, 8, 128) + kv_bytes([P * 16], 8, 128)
    for name, fn in (("plain", plain), ("cascade", casc)):
        ms = _time_calls(fn, args.steps, args.warmup, stream)
        res[f"shared2048_{name}"] = {"attention_ms": round(ms, 5),
                                     "logical_GBs": round(logical / ms / 1e6, 1),
                                     "unique_GBs": round(unique / ms / 1e6, 1)}
    # the same batch over e4m3 caches (history quantised by pkv_write_fp8, untimed)
    kc = KVCache(wl, True, 4321, 0, 0)
    kc.write(wl.k_new, wl.v_new, wl.slot_mapping, stream)
    plain8 = lambda: pkv.attention_fp8(out, wl.q, kc.k, kc.v, wl.block_tables, wl.context_lens,
                                       wl.query_start_loc, wl.scale, kc.kd, kc.vd,
                                       max_query_len=1, max_context_len=wl.max_context_len,
                                       workspace=ws)
    casc8 = lambda: pkv.attention_cascade_fp8(out, wl.q, kc.k, kc.v, wl.block_tables,
                                              wl.context_lens, wl.query_start_loc, wl.scale, P,
                                              kc.kd, kc.vd, max_context_len=wl.max_context_len,
                                              workspace=ws)
    for name, fn in (("plain", plain8), ("cascade", casc8)):
        ms = _time_calls(fn, args.steps, args.warmup, stream)
        res[f"shared2048_e4m3_{name}"] = {"attention_ms": round(ms, 5),
                                          "logical_GBs": round(logical / 2 / ms / 1e6, 1),
                                          "unique_GBs": round(unique / 2 / ms / 1e6, 1)}
    del wl, out, ws, kc
    # (1) workload 4: cascade for its sharing decode sequences, plain for the rest
    wl = W.workload(4, device=device)
    nsh = len(wl.shared_seqs)
    Pb = wl.shared_prefix_blocks
    pkv.write(wl.k_new, wl.v_new, wl.slot_mapping, wl.k_cache, wl.v_cache)
    out = torch.empty_like(wl.q)
    qsl_rest = (wl.query_start_loc[nsh:] - nsh).contiguous()
    bt_sh, cl_sh, qsl_sh = wl.block_tables[:nsh], wl.context_lens[:nsh], wl.query_start_loc[:nsh + 1]
    bt_rest, cl_rest = wl.block_tables[nsh:], wl.context_lens[nsh:]
    ws = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    ws2 = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    mcl_sh = int(wl.ctx_lens[:nsh].max())
    plain4 = lambda: pkv.attention(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables,
                                   wl.context_lens, wl.query_start_loc, wl.scale,
                                   max_query_len=wl.max_query_len,
                                   max_context_len=wl.max_context_len,
                                   num_decode_seqs=wl.num_decode_seqs, workspace=ws)

    def casc4():
        pkv.attention_cascade(out[:nsh], wl.q[:nsh], wl.k_cache, wl.v_cache, bt_sh, cl_sh, qsl_sh,
                              wl.scale, Pb, max_context_len=mcl_sh, workspace=ws)
        pkv.attention(out[nsh:], wl.q[nsh:], wl.k_cache, wl.v_cache, bt_rest, cl_rest, qsl_rest,
                      wl.scale, max_query_len=wl.max_query_len,
                      max_context_len=wl.max_context_len,
                      num_decode_seqs=wl.num_decode_seqs - nsh, workspace=ws2)
    attn_b, _, _ = algorithmic_bytes(wl)
    shared_dup = (nsh - 1) * Pb * 16 * 8 * 128 * 2 * 2
    wl4_shared = Pb
    for name, fn in (("plain", plain4), ("cascade", casc4)):
        ms = _time_calls(fn, args.steps, args.warmup, stream)
        res[f"mixed4_{name}"] = {"attention_ms": round(ms, 5),
                                 "logical_GBs": round(attn_b / ms / 1e6, 1),
                                 "unique_GBs": round((attn_b - shared_dup) / ms / 1e6, 1)}
    del wl, out, ws, ws2
    # (3) a mixed batch where every sequence shares the prefix (48 decode rows
    # and 4 chunks of 512 tokens after it): one cascade call against one plain
    # call, prefixes of 1024 and 4096 tokens
    for Pb in (64, 256):
        rng = np.random.default_rng(99 + Pb)
        q_lens = np.array([1] * 48 + [512] * 4, np.int64)
        ctx = Pb * 16 + q_lens + rng.integers(0, 2048, 52, endpoint=True)
        wl = W.make_workload(q_lens, ctx, num_q_heads=32, num_kv_heads=8, head_size=128,
                             seed=99 + Pb, device=device, shared_prefix_blocks=Pb,
                             shared_seqs=tuple(range(52)))
        pkv.write(wl.k_new, wl.v_new, wl.slot_mapping, wl.k_cache, wl.v_cache)
        out = torch.empty_like(wl.q)
        kw = dict(max_query_len=wl.max_query_len, max_context_len=wl.max_context_len,
                  num_decode_seqs=48)
        meta = pkv.attn_meta(wl.q, wl.block_tables, wl.context_lens, **kw)
        ws = torch.empty(max(pkv.workspace_size(wl.k_cache, meta),
                             pkv.cascade_workspace_size(wl.k_cache, meta, Pb)),
                         dtype=torch.uint8, device=device)
        plain = lambda: pkv.attention(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables,  # noqa: E731
                                      wl.context_lens, wl.query_start_loc, wl.scale,
                                      workspace=ws, **kw)
        casc = lambda: pkv.attention_cascade(out, wl.q, wl.k_cache, wl.v_cache,  # noqa: E731
                                             wl.block_tables, wl.context_lens,
                                             wl.query_start_loc, wl.scale, Pb, workspace=ws,
                                             **kw)
        flops = sum(int((c - q + np.arange(q) + 1).sum()) for q, c in zip(q_lens, ctx)) * 32 * 512
        for name, fn in (("plain", plain), ("cascade", casc)):
            ms = _time_calls(fn, args.steps, args.warmup, stream)
            res[f"mixed_shared{Pb * 16}_{name}"] = {
                "attention_ms": round(ms, 5), "TFLOPs": round(flops / ms / 1e9, 1),
                "cascade_gate": int(pkv.use_cascade(meta, Pb))}
        del wl, out, ws
    if pkv.get_error(clear=True):
        raise RuntimeError("device error word set")
    return {"metric": "cascade attention vs pkv_attention on shared-prefix batches",
            "unit": "ms / GB/s", "results": res,
            "config": {"shared2048": "64 decode seqs, 2048 shared + U[128,2048] own keys, "
                                     "32q/8kv, D=128 bf16 (and e4m3: GB/s over 1-byte codes)",
                       "mixed4": f"workload 4: cascade for its {nsh} sequences sharing "
                                 f"{wl4_shared} blocks, pkv_attention for the rest",
                       "mixed_sharedP": "48 decode rows + 4 chunks of 512, every sequence "
                                        "sharing P tokens, own keys U[0, 2048] + the chunk; "
                                        "one cascade call vs one plain call (TFLOP/s over "
                                        "4 D flops per row and visible key)"},
            "steps": args.steps, "warmup": args.warmup}


def pool_trace(pool, steps, running=256, prompt=768, shared=512, turnover=16, seed=0):
    """A serving trace on a block pool (the C++ one or the oracle's, same
    interface): `running` requests whose prompts share a `shared`-token system
    prompt decode one token per step; every 16 steps `turnover` of them finish
    and as many new ones are admitted (prefix hits + prefill of the rest).
    The prompts are drawn before the clock starts (they are the trace's
    input); the C++ pool gets numpy arrays, one batched call per decode step
    for the appends and one for the slots, the oracle's pool Python lists and
    one call per request.  Returns (slots allocated, seconds)."""
    rng = np.random.default_rng(seed)
    admissions = running + turnover * (steps // 16)
    system = rng.integers(0, 32000, shared).astype(np.int32)
    own = rng.integers(0, 32000, (admissions, prompt - shared)).astype(np.int32)
    prompts = np.concatenate([np.broadcast_to(system, (admissions, shared)), own], axis=1)
    batched = hasattr(pool, "allocate_slots_batch")
    if not batched:
        prompts = prompts.tolist()
    live, next_id, slots = [], 0, 0

    def admit():
        nonlocal next_id, slots
        rid = next_id
        next_id += 1
        toks = prompts[rid]
        pool.add_request(rid, toks)
        cached = pool.admit(rid)
        s = pool.allocate_slots(rid, prompt - cached)
        slots += len(s)
        live.append(rid)

    t0 = time.perf_counter()
    for _ in range(running):
        admit()
    live_ids = np.asarray(live, dtype=np.int64)
    ones = np.ones(running, dtype=np.int32)
    step_tok = np.empty(running, dtype=np.int32)
    for step in range(steps):
        if batched:
            step_tok.fill(step)
            pool.append_token_batch(live_ids, step_tok)
            s, done = pool.allocate_slots_batch(live_ids, ones)
            assert done == running
            slots += len(s)
        else:
            for rid in live:
                pool.append_token(rid, step)
            for rid in live:
                slots += len(pool.allocate_slots(rid, 1))
        if step % 16 == 15:
            for _ in range(turnover):
                pool.free_request(live.pop(0))
                admit()
            live_ids = np.asarray(live, dtype=np.int64)
    return slots, time.perf_counter() - t0


def run_pool_bench(args):
    """Host block pool on a serving trace: the C++ pool (one batched call per
    decode step) against the oracle's Python pool on a shorter run of the same
    trace."""
    from paged_kv_cache_43_gb300 import build
    from paged_kv_cache_43_gb300 import pool as P
    import oracle.pool as OP
    build.build()
    steps = max(args.steps, 16)
    n = P.BlockPool(65536, 16, True)
    pool_trace(n, 16)                       # warm-up
    n.close()
    n = P.BlockPool(65536, 16, True)
    slots, dt = pool_trace(n, steps)
    cached = n.cached_blocks()
    n.close()
    o_steps = 16
    o_slots, o_dt = pool_trace(OP.Pool(65536, 16, True), o_steps)
    return {
        "metric": "host block pool: slots allocated per second on a decode-loop trace",
        "value": round(slots / dt, 1), "unit": "slots/s", "higher_is_better": True,
        "steps": steps, "ms_per_step": round(dt / steps * 1e3, 4),
        "config": {"workload": "256 running requests, 768-token prompts sharing a 512-token "
                               "system prompt, 16 finish and 16 arrive every 16 steps",
                   "num_blocks": 65536, "block_size": 16, "cached_blocks_at_end": cached},
        "cpu_baseline": {"value": round(o_slots / o_dt, 1), "unit": "slots/s", "cores": 1,
                         "kind": "oracle", "sample": f"the same trace, {o_steps} steps"},
        "data": "synthetic token ids",
    }


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is the oracle's KV write +
    attention on a bounded sample of the same workload (generated on the GPU
    with the same seed, copied to the host), sized so that warm-up + steps
    take about PKV_REFERENCE_BUDGET_S seconds (default 150)."""
    if rank != 0:
        return None
    from paged_kv_cache_43_gb300 import workloads as W
    import oracle
    oracle.build()
    device = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    wl = W.workload(args.workload, device=device)
    budget = float(os.environ.get("PKV_REFERENCE_BUDGET_S", "150"))
    seq = int(np.argsort(wl.ctx_lens)[wl.num_seqs // 2])      # median-length sequence
    scales = None
    if args.kv_dtype == "fp8":    # same scales as the pkv arm's rank 0
        sd = rank_seed(args.workload, 0)
        ks, vs = W.fp8_scales(wl.num_kv_heads, sd), W.fp8_scales(wl.num_kv_heads, sd + 1)
        scales = (ks, vs, np.tile(ks, (wl.num_seqs, 1)), np.tile(vs, (wl.num_seqs, 1)))
    smp = oracle_sample(wl, [seq], fp8=scales)
    t0 = time.perf_counter()
    oracle_pass(smp)
    one = time.perf_counter() - t0
    per_step = budget / max(args.steps + args.warmup, 1)
    hkv = wl.num_kv_heads
    if one > per_step:
        hkv = max(1, int(wl.num_kv_heads * per_step / one))
        smp = oracle_sample(wl, [seq], kv_heads=hkv, fp8=scales)
    for _ in range(args.warmup):
        oracle_pass(smp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(smp)
    dt = time.perf_counter() - t0
    value = sample_bytes(smp) * args.steps / dt / 1e9
    sample = (f"sequence {seq} of {wl.name} ({int(smp['cl'][0])} keys), {hkv} of "
              f"{wl.num_kv_heads} kv heads with their q heads, fp64 KV write + attention"
              + (" over an e4m3 cache" if scales is not None else ""))
    return {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded workload, bounded sample)", "impl": "reference",
        "config": {"workload": wl.name, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--kv-split", type=int, default=0)
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window W (keys per query); 0 = full attention")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="cache storage: the workload's bf16, or e4m3 codes with per-kv-head "
                         "scales (workloads 2-5)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the short per-workload measurements of the default run")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="override the batch size (profiling captures on a smaller case)")
    ap.add_argument("--cascade-bench", action="store_true",
                    help="time cascade attention against pkv_attention on shared-prefix batches")
    ap.add_argument("--pool-bench", action="store_true",
                    help="time the host block pool (C++ vs oracle) on a serving trace; no GPU")
    ap.add_argument("--profile", action="store_true",
                    help="run warmup+steps plain steps only (for ncu), print no bench line")
    ap.add_argument("--part", choices=["all", "prefill", "decode"], default="all",
                    help="--profile: the whole step, or one part's attention call alone")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.kv_dtype == "fp8" and args.workload == 1:
        ap.error("--kv-dtype fp8 needs a bf16 workload (2-5)")
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)

    if args.pool_bench:
        print(json.dumps(run_pool_bench(args)), flush=True)
        return
    if args.cascade_bench:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU")
        print(json.dumps(run_cascade_bench(args, torch.device("cuda", 0))), flush=True)
        return

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    try:
        line = run_pkv(args, rank, world, device)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
