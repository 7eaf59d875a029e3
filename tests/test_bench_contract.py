"""bench.py's command-line contract on the host (no GPU): the reference arm
(the oracle on a bounded sample) prints one JSON line with the keys the
driver reads, the pool benchmark runs, and fewer than 3 warm-up steps are
refused."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(*args, env_extra=None):
    env = dict(os.environ, PKV_REFERENCE_BUDGET_S="3", CUDA_VISIBLE_DEVICES="")
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def last_json(out: str) -> dict:
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert lines, out
    return json.loads(lines[-1])


def test_reference_arm_prints_the_contract_line():
    r = run("--impl", "reference", "--workload", "1", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    d = last_json(r.stdout)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["config"]["workload"]


def test_pool_bench_runs_on_the_host():
    r = run("--pool-bench", "--steps", "32")
    assert r.returncode == 0, r.stderr[-2000:]
    d = last_json(r.stdout)
    assert d["unit"] == "slots/s" and d["value"] > d["cpu_baseline"]["value"] > 0


def test_fewer_than_three_warmup_steps_are_refused():
    r = run("--impl", "reference", "--workload", "1", "--steps", "3", "--warmup", "2")
    assert r.returncode != 0


def test_mixed_batch_parts_and_flops():
    """The bench's split of a mixed batch into its decode and prefill parts
    (views over the same caches) and its flop count (4 D per row and visible
    key, the window capping the keys a row sees)."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_43_gb300 import workloads as W
    wl = W.make_workload([1, 1, 5, 3], [40, 17, 30, 3], num_q_heads=4, num_kv_heads=2,
                         head_size=64, seed=3)
    assert wl.num_decode_seqs == 2
    dec, pf = bench.sub_batch(wl, 0, 2), bench.sub_batch(wl, 2, 4)
    assert dec.num_decode_seqs == 2 and pf.num_decode_seqs == 0
    assert pf.query_start_loc.tolist() == [0, 5, 8] and pf.q.shape[0] == 8
    assert pf.q.data_ptr() == wl.q[2:].data_ptr() and pf.k_cache is wl.k_cache
    assert pf.block_tables.tolist() == wl.block_tables[2:].tolist()
    # rows of seq 2 see 26..30 keys, of seq 3 see 1..3 keys
    keys = sum(range(26, 31)) + sum(range(1, 4))
    assert bench.attention_flops(wl, [2, 3]) == keys * 4 * 4 * 64
    assert bench.attention_flops(wl, [0, 1]) == (40 + 17) * 4 * 4 * 64
    keys_w = sum(min(k, 4) for k in range(26, 31)) + sum(range(1, 4))
    assert bench.attention_flops(wl, [2, 3], window=4) == keys_w * 4 * 4 * 64
    assert np.array_equal(pf.ctx_lens, wl.ctx_lens[2:])
