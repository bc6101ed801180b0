"""Benchmark: INT4 paged decode on the Llama-3-8B-like layer.

Workload (the one the headline metric is quoted on): 32 q heads, 8 KV heads,
head_dim 128, bf16 q/k/v, block_size 16, batch 64, context lengths uniform in
[1024, 8192], pages at distinct random blocks of a 200,000-block pool, K/V
~ N(0,1) with 1% of (head, channel) pairs x10, RHT on.  One step = kvq_write
of one new token per sequence + kvq_decode_attn of one query per sequence
(split-KV kernel + merge kernel), i.e. every row of the hot path.

Output: one JSON line on rank 0 with the metric (tokens/s), the roofline of
the dominant kernel (decode attention, HBM-bound), the end-to-end number
through the C ABI with host buffers, the clocks seen during the timed region,
and the CPU oracle's throughput on a bounded sample of the same workload.

`--impl reference` times the CPU oracle alone (the reference arm: a plain,
slow program), on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import kvq_inputs as gen  # noqa: E402

METRIC = "INT4 paged decode tokens/s and effective KV GB/s (% of GB300 HBM peak)"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(wl: gen.Workload) -> dict:
    """Bytes the decode step must move at minimum: every visible packed K and
    V row once (row_bytes each), the block-table entries of the visible pages
    (per kv head), q in and out, plus the write of one token per sequence."""
    R = wl.head_dim // 2 + 4
    Hkv, bs = wl.num_kv_heads, wl.block_size
    ctx = wl.seq_lens.astype(np.int64)
    kv_rows = int(ctx.sum()) * Hkv
    pages = int(((ctx + bs - 1) // bs).sum()) * Hkv
    q_bytes = wl.batch * wl.num_q_heads * wl.head_dim * 2
    out_bytes = wl.batch * wl.num_q_heads * wl.head_dim * 4
    decode = kv_rows * R * 2 + pages * 4 + q_bytes + out_bytes
    write = wl.batch * Hkv * 2 * (wl.head_dim * 2 + R)
    return {"decode": decode, "write": write, "kv_only": kv_rows * R * 2}


def recorded_traffic(src_hash: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_stream_llama_int4.md")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != src_hash:
        return None
    try:
        return float(vals["dram_bytes_per_decode_call"])
    except (KeyError, ValueError):
        return None


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for fn in ("kvq_decode.cu", "kvq_common.cuh", "kvq_internal.h"):
        with open(os.path.join(ROOT, "sub_byte_quantized_write_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm

def setup_gpu(wl, device, want_splits=0):
    import torch
    import sub_byte_quantized_write_gb300 as K
    signs = torch.from_numpy(wl.signs).to(device)
    cache = K.PagedCache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, signs, device)
    table = torch.from_numpy(wl.table).to(device)
    pre = wl.prefix_lens
    pag_pre = K.Paging(torch.from_numpy(pre).to(device), block_tables=table)
    # prefix (untimed): write each sequence's cached tokens, drawn on the device
    B = wl.batch
    chunk = 16
    for b0 in range(0, B, chunk):
        bsel = list(range(b0, min(B, b0 + chunk)))
        ks = [gen.kv_values_device(wl, "k", b, 0, int(pre[b]), device) for b in bsel]
        vs = [gen.kv_values_device(wl, "v", b, 0, int(pre[b]), device) for b in bsel]
        counts = np.zeros(B, np.int32)
        counts[bsel] = pre[bsel]
        cu = torch.from_numpy(wl.cu(counts)).to(device)
        K.kvq_write(cache, pag_pre, torch.cat(ks), torch.cat(vs), cu)
    torch.cuda.synchronize()
    step = {
        "k": torch.cat([gen.kv_values_device(wl, "k", b, int(pre[b]), 1, device) for b in range(B)]).contiguous(),
        "v": torch.cat([gen.kv_values_device(wl, "v", b, int(pre[b]), 1, device) for b in range(B)]).contiguous(),
        "q": gen.q_values_device(wl, device).contiguous(),
        "cu": torch.from_numpy(wl.cu(wl.n_new)).to(device),
        "seq_lens": torch.from_numpy(wl.seq_lens).to(device),
    }
    pag = K.Paging(step["seq_lens"], block_tables=table)
    nbytes, splits = K.kvq_decode_workspace_size(cache, pag, wl.num_q_heads, want_splits)
    step["ws"] = torch.empty(nbytes, dtype=torch.uint8, device=device)
    step["out"] = torch.empty((B, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device=device)
    step["splits"] = splits
    return cache, pag, step


def run_gpu(args, rank, world, local_rank):
    import torch
    import sub_byte_quantized_write_gb300 as K
    device = "cuda:%d" % local_rank
    torch.cuda.set_device(local_rank)
    wl = gen.llama_int4(seed=0, num_blocks=args.pool_blocks)
    cache, pag, st = setup_gpu(wl, device, args.splits)
    scale = 1.0 / math.sqrt(wl.head_dim)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device=device)

    def write_call():
        K.kvq_write(cache, pag, st["k"], st["v"], st["cu"], stream=stream)

    def decode_call():
        K.kvq_decode_attn(cache, pag, st["q"], scale, out=st["out"], workspace=st["ws"],
                          num_splits=st["splits"], stream=stream)

    def step():
        write_call()
        decode_call()

    # the step's two library calls are captured once into CUDA graphs and
    # replayed, so the timed region holds only device work
    with torch.cuda.stream(stream):
        for _ in range(2):
            step()  # first calls set the kernels' shared-memory attributes outside capture
        stream.synchronize()
        g_write, g_decode = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_write, stream=stream):
            write_call()
        with torch.cuda.graph(g_decode, stream=stream):
            decode_call()
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        g_write.replay()
        g_decode.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(float(i))  # packed KV already exceeds L2; flush so no step reuses the last one's lines
                e0, e1, e2 = ev[i]
                e0.record(stream)
                g_write.replay()
                e1.record(stream)
                g_decode.replay()
                e2.record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    dec_ms = [b.elapsed_time(c) for a, b, c in ev]
    wr_ms = [a.elapsed_time(b) for a, b, c in ev]
    ms = sum(step_ms) / len(step_ms)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = world * wl.batch / (ms / 1e3)

    # end to end through the C ABI with host buffers: H2D of the step's
    # inputs from pinned memory, write + decode, D2H of the output
    hk = st["k"].cpu().pin_memory()
    hv = st["v"].cpu().pin_memory()
    hq = st["q"].cpu().pin_memory()
    hcu = st["cu"].cpu().pin_memory()
    hsl = st["seq_lens"].cpu().pin_memory()
    hout = torch.empty_like(st["out"], device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hk, hv, hq, hcu, hsl))
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        # plain library calls (no graph), inputs from pinned host memory
        st["k"].copy_(hk, non_blocking=True)
        st["v"].copy_(hv, non_blocking=True)
        st["q"].copy_(hq, non_blocking=True)
        st["cu"].copy_(hcu, non_blocking=True)
        st["seq_lens"].copy_(hsl, non_blocking=True)
        step()
        hout.copy_(st["out"], non_blocking=True)

    e2e_ms = []
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            e2e_step()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(float(i))
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step()
            c.record(stream)
            c.synchronize()
            e2e_ms.append(a.elapsed_time(c))
    e2e_value = world * wl.batch / (sum(e2e_ms) / len(e2e_ms) / 1e3)

    ab = algorithmic_bytes(wl)
    dec = sum(dec_ms) / len(dec_ms)
    peak, peak_kind = peaks()
    achieved = ab["decode"] / (dec / 1e3) / 1e9
    traffic = recorded_traffic(kernel_source_hash())
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4 codes x fp16 tensor-core math, fp32 accumulate/softmax",
        "data": "synthetic (seeded; K/V ~ N(0,1) with 1% outlier channels x10)",
        "config": {"workload": wl.name, "batch": wl.batch, "num_q_heads": wl.num_q_heads,
                   "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
                   "context": "uniform[1024,8192]", "cached_tokens": int(wl.seq_lens.sum()),
                   "pool_blocks": wl.num_blocks, "rht": True, "decode_workers": st["splits"],
                   "timing": "CUDA graphs of the write call and the decode call, events around each replay",
                   "l2": "flushed between timed steps (256 MB write); packed KV 321 MB also exceeds L2",
                   "parallelism": "replicas only" if world > 1 else "single GPU"},
        "effective_kv_GBps": round(ab["decode"] / (dec / 1e3) / 1e9, 1),
        "decode_ms": round(dec, 5), "write_ms": round(sum(wr_ms) / len(wr_ms), 5),
        "roofline": {"bound": "hbm", "kernel": "decode attention (query prep + stream-K split-KV + merge, one kvq_decode_attn call)",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind + " (copy bandwidth)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of_nominal_8000": round(achieved / 8000.0, 4),
                     "algorithmic_bytes_per_launch": ab["decode"], "traffic": traffic},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(sum(e2e_ms) / len(e2e_ms), 5)},
        "gpu_launches": 4 * args.steps,  # write + (prep, stream, merge) per step
        "clocks": clk.summary(),
    }
    return result, wl


def _oracle_step_setup(wl, sample_seqs):
    """Oracle cache holding the prefixes of the sampled sequences (host values)."""
    import oracle
    oc = oracle.Cache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.signs)
    pre = wl.prefix_lens.copy()
    counts = np.zeros(wl.batch, np.int32)
    counts[sample_seqs] = pre[sample_seqs]
    lens = pre.copy()
    ks = [gen.kv_values_host(wl, "k", int(b), 0, int(pre[b])) for b in sample_seqs]
    vs = [gen.kv_values_host(wl, "v", int(b), 0, int(pre[b])) for b in sample_seqs]
    oracle.write(oc, oracle.Paging(wl.table, False, lens), gen.f32_to_bf16_bits(np.concatenate(ks)),
                 gen.f32_to_bf16_bits(np.concatenate(vs)), wl.cu(counts))
    new_k = gen.f32_to_bf16_bits(np.concatenate([gen.kv_values_host(wl, "k", int(b), int(pre[b]), 1) for b in sample_seqs]))
    new_v = gen.f32_to_bf16_bits(np.concatenate([gen.kv_values_host(wl, "v", int(b), int(pre[b]), 1) for b in sample_seqs]))
    q = gen.f32_to_bf16_bits(gen.q_values_host(wl))
    return oc, new_k, new_v, q


def oracle_step(wl, oc, new_k, new_v, q, sample_seqs, threads):
    import oracle
    counts = np.zeros(wl.batch, np.int32)
    counts[sample_seqs] = 1
    pag = oracle.Paging(wl.table, False, wl.seq_lens)
    oracle.write(oc, pag, new_k, new_v, wl.cu(counts))
    oracle.attention(oc, pag, q, 1.0 / math.sqrt(wl.head_dim), rows=np.asarray(sample_seqs, np.int32),
                     threads=threads)


def cpu_baseline(wl, budget_s=15.0):
    """The CPU oracle, as it stands, on a bounded sample of the workload:
    whole decode steps (write one token + attend with all 32 q heads) of a
    subset of the sequences, repeated until ~budget_s of work."""
    threads = os.cpu_count() or 1
    sample = list(range(0, wl.batch, 4))  # 16 of the 64 sequences
    oc, nk, nv, q = _oracle_step_setup(wl, sample)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(wl, oc, nk, nv, q, sample, threads)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 50:
            break
    dt = time.perf_counter() - t0
    return {"value": round(n * len(sample) / dt, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d decode steps of %d of the 64 sequences (every 4th; write 1 token + attention over the "
                      "cached context, all 32 q heads), %.1f s" % (n, len(sample), dt)}


def run_reference(args):
    """Reference arm: the CPU oracle timed alone on the same workload."""
    wl = gen.llama_int4(seed=0)
    threads = os.cpu_count() or 1
    sample = list(range(0, wl.batch, 16))  # 4 sequences per step
    oc, nk, nv, q = _oracle_step_setup(wl, sample)
    for _ in range(args.warmup):
        oracle_step(wl, oc, nk, nv, q, sample, threads)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(wl, oc, nk, nv, q, sample, threads)
        ts.append(time.perf_counter() - t0)
    ms = 1e3 * sum(ts) / len(ts)
    value = len(sample) / (ms / 1e3)
    desc = "%d of the 64 sequences per step (every 16th): write 1 token + attention, all 32 q heads" % len(sample)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, f32 write (CPU oracle)",
            "data": "synthetic (seeded)", "config": {"workload": wl.name, "batch": wl.batch},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pool-blocks", type=int, default=200000,
                    help="block pool size (the workload's is 200000; smaller pools only for profiling)")
    ap.add_argument("--splits", type=int, default=0, help="decode split count (0 = the library's choice)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    result, wl = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            result["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
