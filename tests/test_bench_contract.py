"""bench.py's output contract, checked on CPU through its reference arm (the
oracle timed alone): one JSON line with the metric, the value, the unit, the
timing keys, a cpu_baseline block and an e2e block.  Also the per-workload
algorithmic units the roofline divides by, against closed forms."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import kvq_inputs as gen  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["metric"] == bench.METRIC and d["config"]["workload"] == "llama_int4_decode"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["warmup"] >= 3


def test_algorithmic_units_closed_forms():
    # decode: every visible packed row of K and V once + table entries + q + out
    wl = gen.llama_int4(0, num_blocks=20000)
    u = bench.algorithmic_units(wl)
    R = bench.row_bytes(wl.mode, wl.head_dim)
    L = wl.seq_lens.astype(np.int64)
    want = int(L.sum()) * 8 * R * 2 + int(((L + 15) // 16).sum()) * 8 * 4 + 64 * 32 * 128 * (2 + 4)
    assert R == 68 and u["decode"] == want
    # prefill: 4 D flops per causal (query, key) pair per q head
    wl = gen.prefill_int4(0, prefixes=(0, 100), chunk=7, num_blocks=100)
    u = bench.algorithmic_units(wl)
    pairs = sum(7 * p + 7 * 8 // 2 for p in (0, 100))   # n (L - n) + n (n + 1) / 2 per sequence and kv head
    assert u["prefill_flops"] == 4 * 128 * pairs * 8 * 4     # x 8 kv heads x group 4
    # gather: rows in and bf16 rows out, K and V, plus the table entries
    cached = int(wl.seq_lens.sum())
    pages = int(((wl.seq_lens + 15) // 16).sum()) * 8
    assert u["gather"] == cached * 8 * 2 * (68 + 256) + pages * 4 + (wl.batch + 1) * 4 + wl.batch * 4
    # 8-bit token-head rows carry the fp32 scale after the codes
    assert bench.row_bytes(gen.MODE_FP8_TOKEN_HEAD, 128) == 132
