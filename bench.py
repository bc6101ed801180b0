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

Other workloads (`--workload`): the same decode layer at head_dim 64 /
block_size 64, with zero-point-in-scale INT4 rows or with INT8 / FP8
per-token-head rows; the ERNIE-like INT2 decode; the Qwen-like INT8 head-wise
decode with sliding windows; the INT4 chunked prefill (tcgen05); and the
gather-and-dequantise of the chunked-prefill layer's whole cache.

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
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, kind) from the measured-peaks file, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def row_bytes(mode: int, D: int) -> int:
    """Bytes of one cache row: packed codes plus the fp16 scale / zero-point pad (INT8: codes only)."""
    return {gen.MODE_INT4: D // 2 + 4, gen.MODE_INT2: D // 4 + 4, gen.MODE_INT8: D, gen.MODE_INT4_STEGO: D // 2 + 4,
            gen.MODE_INT8_TOKEN_HEAD: D + 4, gen.MODE_FP8_TOKEN_HEAD: D + 4}[mode]


def recorded_units(profile: str, key: str, src_hash: str):
    """A per-launch figure (DRAM bytes) from a committed ncu summary, if that
    summary was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", profile)
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
        return float(vals[key])
    except (KeyError, ValueError):
        return None


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for fn in files:
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
        # The timed region starts once nvidia-smi samples (its start-up
        # otherwise overlaps the first timed steps); at most 5 s.
        t0 = time.time()
        while not self.lines and self.proc.poll() is None and time.time() - t0 < 5.0:
            time.sleep(0.01)
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
# ranks (one process per GPU; replicas: every rank runs the whole workload)

def max_over_ranks(x: float, device) -> float:
    """The largest per-rank value (step time) of the job; the value itself on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, ms_max: float, world: int) -> float:
    """Units of all ranks per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_max / 1e3)


# ---------------------------------------------------------------------------
# workloads

WORKLOADS = {
    # name: (factory, metric, kind)
    "llama_int4": (lambda a: gen.llama_int4(seed=0, num_blocks=a.pool_blocks or 200000), METRIC, "decode"),
    "llama_int4_d64_bs64": (lambda a: gen.llama_int4(seed=0, num_blocks=a.pool_blocks or 50000, head_dim=64,
                                                     block_size=64),
                            "INT4 paged decode (head_dim 64, block_size 64) tokens/s and effective KV GB/s "
                            "(% of GB300 HBM peak)", "decode"),
    "llama_int4_stego": (lambda a: gen.llama_int4(seed=0, num_blocks=a.pool_blocks or 200000,
                                                  mode=gen.MODE_INT4_STEGO),
                         "INT4 (zero point in the fp32 scale) paged decode tokens/s and effective KV GB/s "
                         "(% of GB300 HBM peak)", "decode"),
    "llama_int8_token_head": (lambda a: gen.llama_int4(seed=0, num_blocks=a.pool_blocks or 200000,
                                                       mode=gen.MODE_INT8_TOKEN_HEAD),
                              "INT8 per-token-head paged decode tokens/s and effective KV GB/s "
                              "(% of GB300 HBM peak)", "decode"),
    "llama_fp8_token_head": (lambda a: gen.llama_int4(seed=0, num_blocks=a.pool_blocks or 200000,
                                                      mode=gen.MODE_FP8_TOKEN_HEAD),
                             "FP8 (E4M3) per-token-head paged decode tokens/s and effective KV GB/s "
                             "(% of GB300 HBM peak)", "decode"),
    "ernie_int2": (lambda a: gen.ernie_int2(seed=0, num_blocks=a.pool_blocks or 100000),
                   "INT2 paged decode tokens/s and effective KV GB/s (% of GB300 HBM peak)", "decode"),
    "qwen_int8_headwise": (lambda a: gen.qwen_int8_headwise(seed=0),
                           "INT8 head-wise paged decode tokens/s and effective KV GB/s (% of GB300 HBM peak)",
                           "decode"),
    "prefill_int4": (lambda a: gen.prefill_int4(seed=0, prefixes=tuple(a.prefill_prefixes), chunk=a.prefill_chunk,
                                                num_blocks=a.pool_blocks or 200000),
                     "INT4 chunked-prefill tokens/s (causal attention over the paged cache, % of tensor peak)",
                     "prefill"),
    "gather_int4": (lambda a: gen.prefill_int4(seed=0, prefixes=tuple(a.prefill_prefixes), chunk=a.prefill_chunk,
                                               num_blocks=a.pool_blocks or 200000),
                    "INT4 gather-and-dequantise tokens/s (every cached position of the chunked-prefill layer "
                    "back to dense bf16 K/V, % of GB300 HBM peak)", "gather"),
    "gather_dense_prefill_int4": (lambda a: gen.prefill_int4(seed=0, prefixes=tuple(a.prefill_prefixes),
                                                             chunk=a.prefill_chunk, num_blocks=a.pool_blocks or 200000),
                                  "INT4 chunked-prefill tokens/s through gather + dequantise + dense prefill "
                                  "(% of tensor peak)", "gather_prefill"),
}


def visible_keys(wl, b, h, p):
    """Keys a query at position p of sequence b sees in kv head h."""
    W = 0 if wl.window is None else int(wl.window[h])
    if W > 0 and p - W + 1 > wl.sink:
        return min(wl.sink, p + 1) + W
    return p + 1


def algorithmic_units(wl: gen.Workload) -> dict:
    """Decode: bytes the call must move at minimum (every visible packed K and
    V row once, the table entries of the visible pages per kv head, q in, out
    out).  Prefill: tensor FLOPs of causal attention, 4 D per visible (query,
    key) pair per q head.  Gather: every cached row read once (K and V), its
    page-table entry once per page and kv head, bf16 K/V out.  Write: bf16
    K/V in, packed rows out."""
    R = row_bytes(wl.mode, wl.head_dim)
    Hkv, bs, D, G = wl.num_kv_heads, wl.block_size, wl.head_dim, wl.group
    n_new = int(wl.n_new.sum())
    write = n_new * Hkv * 2 * (D * 2 + R)
    cached = int(wl.seq_lens.sum())
    gather_pages = sum(int((L + bs - 1) // bs) for L in wl.seq_lens) * Hkv
    gather = {"gather": cached * Hkv * 2 * (R + 2 * D) + gather_pages * 4 + (wl.batch + 1) * 4 + wl.batch * 4}
    if wl.step == "decode":
        rows = pages = 0
        for b in range(wl.batch):
            p = int(wl.seq_lens[b]) - 1
            for h in range(Hkv):
                vis = visible_keys(wl, b, h, p)
                rows += vis
                pages += (vis + bs - 1) // bs
        q_bytes = wl.batch * wl.num_q_heads * D * 2
        out_bytes = wl.batch * wl.num_q_heads * D * 4
        return {"decode": rows * R * 2 + pages * 4 + q_bytes + out_bytes, "write": write, "kv_only": rows * R * 2}
    pairs = 0
    for b in range(wl.batch):
        L, n = int(wl.seq_lens[b]), int(wl.n_new[b])
        for h in range(Hkv):
            if wl.window is None or int(wl.window[h]) <= 0:
                pairs += n * (L - n) + n * (n + 1) // 2
            else:
                pairs += sum(visible_keys(wl, b, h, p) for p in range(L - n, L))
    return {"prefill_flops": 4 * D * pairs * G, "write": write, **gather}


def setup_gpu(wl, device, want_splits=0):
    """Cache with every sequence's prefix written (untimed, values drawn on
    the device), plus the step's inputs: the new tokens, the queries and the
    outputs / decode workspace."""
    import torch
    import sub_byte_quantized_write_gb300 as K
    signs = None if wl.signs is None else torch.from_numpy(wl.signs).to(device)
    cache = K.PagedCache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, signs, device)
    table = torch.from_numpy(wl.table).to(device)
    win = None if wl.window is None else torch.from_numpy(wl.window).to(device)

    def paging(lens_t):
        if wl.headwise:
            return K.Paging(lens_t, block_tables_headwise=table, window_per_kv_head=win, sink_size=wl.sink)
        return K.Paging(lens_t, block_tables=table, window_per_kv_head=win, sink_size=wl.sink)

    pre = wl.prefix_lens
    B = wl.batch
    # INT8: the first write defines the channel scales, so the whole prefix goes in one call
    groups = [list(range(B))] if wl.mode == gen.MODE_INT8 else [list(range(b0, min(B, b0 + 16))) for b0 in range(0, B, 16)]
    pag_pre = paging(torch.from_numpy(np.ascontiguousarray(pre, np.int32)).to(device))
    for bsel in groups:
        counts = np.zeros(B, np.int32)
        counts[bsel] = pre[bsel]
        if counts.sum() == 0:
            continue
        ks = torch.cat([gen.kv_values_device(wl, "k", b, 0, int(pre[b]), device) for b in bsel if pre[b] > 0])
        vs = torch.cat([gen.kv_values_device(wl, "v", b, 0, int(pre[b]), device) for b in bsel if pre[b] > 0])
        K.kvq_write(cache, pag_pre, ks, vs, torch.from_numpy(wl.cu(counts)).to(device))
        del ks, vs
    torch.cuda.synchronize()
    step = {
        "k": torch.cat([gen.kv_values_device(wl, "k", b, int(pre[b]), int(wl.n_new[b]), device) for b in range(B)]).contiguous(),
        "v": torch.cat([gen.kv_values_device(wl, "v", b, int(pre[b]), int(wl.n_new[b]), device) for b in range(B)]).contiguous(),
        "q": gen.q_values_device(wl, device).contiguous(),
        "cu": torch.from_numpy(wl.cu(wl.n_new)).to(device),
        "seq_lens": torch.from_numpy(wl.seq_lens).to(device),
    }
    # The inputs a serving step receives from the host live in one device
    # buffer (256-byte aligned parts, the step's tensors rebound as views into
    # it), so that the end-to-end run moves them with one copy per step; q is
    # last, so that a step without queries copies the prefix before it.
    parts, off = [], 0
    for n in ("k", "v", "cu", "seq_lens", "q"):
        nb = step[n].numel() * step[n].element_size()
        parts.append((n, off, nb))
        off = (off + nb + 255) // 256 * 256
    inbuf = torch.empty(off, dtype=torch.uint8, device=device)
    for n, o, nb in parts:
        view = inbuf[o:o + nb].view(step[n].dtype).view(step[n].shape)
        view.copy_(step[n])
        step[n] = view
    step["inbuf"], step["q_off"] = inbuf, parts[-1][1]
    pag = paging(step["seq_lens"])
    step["out"] = torch.empty(tuple(step["q"].shape), dtype=torch.float32, device=device)
    # gather: every cached position of every sequence back to dense bf16 K / V
    step["cu_all"] = torch.from_numpy(wl.cu(wl.seq_lens)).to(device)
    step["n_all"] = int(wl.seq_lens.sum())
    step["splits"] = 0
    if wl.step == "decode":
        nbytes, splits = K.kvq_decode_workspace_size(cache, pag, wl.num_q_heads, want_splits)
        step["ws"] = torch.empty(nbytes, dtype=torch.uint8, device=device)
        step["splits"] = splits
    return cache, pag, step


def run_gpu(args, rank, world, local_rank):
    import torch
    import sub_byte_quantized_write_gb300 as K
    device = "cuda:%d" % local_rank
    torch.cuda.set_device(local_rank)
    factory, metric, kind = WORKLOADS[args.workload]
    wl = factory(args)
    cache, pag, st = setup_gpu(wl, device, args.splits)
    scale = 1.0 / math.sqrt(wl.head_dim)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    scrub = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    scrub_sum = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2(i):
        # No step reuses the previous step's L2 lines: write a buffer twice
        # the L2's size, then read another one as large, so that the timed
        # step starts from a cold L2 holding no dirty line to write back.
        flush.fill_(float(i))
        torch.sum(scrub, dim=0, out=scrub_sum)

    stream = torch.cuda.Stream(device=device)
    max_q = int(wl.n_new.max())

    def write_call():
        K.kvq_write(cache, pag, st["k"], st["v"], st["cu"], stream=stream)

    if kind in ("gather", "gather_prefill"):
        st["gk"] = torch.empty((st["n_all"], wl.num_kv_heads, wl.head_dim), dtype=torch.bfloat16, device=device)
        st["gv"] = torch.empty_like(st["gk"])
    if kind == "gather":
        st["out"] = st["gk"]  # the step's result, read back by the end-to-end run (with gv)

    def dense_call():  # gather_prefill: the dense prefill over the gathered rows
        K.kvq_prefill_dense_attn(st["gk"], st["gv"], st["cu_all"], st["seq_lens"], st["q"], st["cu"], max_q, scale,
                                 out=st["out"], stream=stream)

    def attn_call():
        if kind in ("gather", "gather_prefill"):
            K.kvq_gather(cache, pag, st["cu_all"], st["n_all"], k_out=st["gk"], v_out=st["gv"], stream=stream)
        elif kind == "decode":
            K.kvq_decode_attn(cache, pag, st["q"], scale, out=st["out"], workspace=st["ws"],
                              num_splits=st["splits"], stream=stream)
        else:
            K.kvq_prefill_attn(cache, pag, st["q"], st["cu"], max_q, scale, out=st["out"], stream=stream)

    def step():
        write_call()
        attn_call()
        if kind == "gather_prefill":
            dense_call()

    # decode, token-head modes: the same step as one kvq_write_decode_attn
    # call (the write done by the decode's query-preparation kernel; pools
    # and output identical to the two calls), timed beside the step
    fused = kind == "decode" and wl.mode != gen.MODE_INT8

    def fused_call():
        K.kvq_write_decode_attn(cache, pag, st["k"], st["v"], st["cu"], st["q"], scale, out=st["out"],
                                workspace=st["ws"], num_splits=st["splits"], stream=stream)

    # The step's library calls are captured once into a CUDA graph and
    # replayed, so the timed region holds only device work (re-writing the
    # same new tokens at the same positions is idempotent).  One graph holds
    # the whole step (its kernels chain with programmatic dependent launch);
    # two more hold one call each, for the per-call breakdown and rooflines.
    with torch.cuda.stream(stream):
        for _ in range(2):
            step()  # first calls set the kernels' shared-memory attributes outside capture
            if fused:
                fused_call()
        stream.synchronize()
        g_step, g_write, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        g_dense = torch.cuda.CUDAGraph() if kind == "gather_prefill" else None
        with torch.cuda.graph(g_step, stream=stream):
            step()
        with torch.cuda.graph(g_write, stream=stream):
            write_call()
        with torch.cuda.graph(g_attn, stream=stream):
            attn_call()
        if g_dense is not None:
            with torch.cuda.graph(g_dense, stream=stream):
                dense_call()
        g_fused = torch.cuda.CUDAGraph() if fused else None
        if g_fused is not None:
            with torch.cuda.graph(g_fused, stream=stream):
                fused_call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(args.steps)]
    evf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        # the warm-up replays run right before the timed steps (a GPU left
        # idle before them had made the first timed replays slower)
        for _ in range(args.warmup):
            with torch.cuda.stream(stream):
                flush_l2(1)
            g_step.replay()
            g_write.replay()
            g_attn.replay()
            if g_dense is not None:
                g_dense.replay()
            if g_fused is not None:
                with torch.cuda.stream(stream):
                    flush_l2(1)
                g_fused.replay()
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        with torch.cuda.stream(stream):
            # the K timed steps, each followed, where it exists, by the same
            # step as one fused call (both whole-step variants under the same
            # conditions)
            for i in range(args.steps):
                flush_l2(i)
                a, c = evs[i]
                a.record(stream)
                g_step.replay()
                c.record(stream)
                if g_fused is not None:
                    flush_l2(i)
                    a, c = evf[i]
                    a.record(stream)
                    g_fused.replay()
                    c.record(stream)
            for i in range(args.steps):  # per-call breakdown, same steps replayed call by call
                flush_l2(i)
                e0, e1, e2, e3 = ev[i]
                e0.record(stream)
                g_write.replay()
                e1.record(stream)
                g_attn.replay()
                e2.record(stream)
                if g_dense is not None:
                    g_dense.replay()
                e3.record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(c) for a, c in evs]
    att_ms = [b.elapsed_time(c) for a, b, c, d in ev]
    wr_ms = [a.elapsed_time(b) for a, b, c, d in ev]
    dense_ms = [c.elapsed_time(d) for a, b, c, d in ev]
    fused_ms = [a.elapsed_time(c) for a, c in evf] if g_fused is not None else []
    ms = max_over_ranks(sum(step_ms) / len(step_ms), device)
    tokens = {"decode": wl.batch, "prefill": int(wl.n_new.sum()), "gather": st["n_all"],
              "gather_prefill": int(wl.n_new.sum())}[kind]
    value = whole_job_rate(tokens, ms, world)

    # end to end through the C ABI with host buffers: H2D of the step's
    # inputs (new K / V rows, their positions, the lengths and the queries)
    # from one pinned buffer, write + attention, D2H of the output
    nin = st["q_off"] if kind == "gather" else st["inbuf"].numel()  # the gather step takes no queries
    hin = st["inbuf"][:nin].cpu().pin_memory()
    hout = torch.empty_like(st["out"], device="cpu").pin_memory()
    hout_v = torch.empty_like(st["gv"], device="cpu").pin_memory() if kind == "gather" else None
    h2d = nin
    d2h = hout.numel() * hout.element_size() + (hout_v.numel() * hout_v.element_size() if kind == "gather" else 0)

    def e2e_step():
        # plain library calls (no graph), inputs from pinned host memory
        st["inbuf"][:nin].copy_(hin, non_blocking=True)
        step()
        hout.copy_(st["out"], non_blocking=True)
        if kind == "gather":
            hout_v.copy_(st["gv"], non_blocking=True)

    e2e_ms = []
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2(1)
            e2e_step()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2(i)
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_step()
            c.record(stream)
            c.synchronize()
            e2e_ms.append(a.elapsed_time(c))
    e2e_value = whole_job_rate(tokens, max_over_ranks(sum(e2e_ms) / len(e2e_ms), device), world)

    units = algorithmic_units(wl)
    att = sum(att_ms) / len(att_ms)
    hbm, tensor, peak_kind = peaks()
    cfg = {"workload": {"gather": "gather_", "gather_prefill": "gather_dense_"}.get(kind, "") + wl.name,
           "batch": wl.batch, "num_q_heads": wl.num_q_heads,
           "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
           "mode": {0: "int4", 1: "int2", 2: "int8", 3: "int4_stego", 4: "int8_token_head",
                    5: "fp8_token_head"}[wl.mode], "headwise_table": bool(wl.headwise),
           "cached_tokens": int(wl.seq_lens.sum()), "new_tokens_per_step": int(wl.n_new.sum()),
           "pool_blocks": wl.num_blocks, "rht": wl.signs is not None,
           "timing": "one CUDA graph per step (write + attention call), events around each replay; "
                     "per-call graphs for the breakdown",
           "l2": "flushed between timed steps (256 MB written, then 256 MB of another buffer read: cold and clean)",
           "parallelism": "replicas only" if world > 1 else "single GPU"}
    if args.workload.startswith("llama_int4"):
        cfg["context"] = "uniform[1024,8192]"
    if kind == "gather":
        achieved = units["gather"] / (att / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "gather_kernel (one kvq_gather call: every cached row, dequantised, "
                                          "inverse RHT, bf16 out)",
                "achieved": round(achieved, 1), "peak": hbm, "peak_kind": peak_kind + " (copy bandwidth)",
                "unit": "GB/s", "frac": round(achieved / hbm, 4), "algorithmic_bytes_per_launch": units["gather"],
                "traffic": recorded_units("gather_%s.md" % args.workload, "dram_bytes_per_gather_call",
                                          kernel_source_hash(("kvq_write.cu", "kvq_common.cuh", "kvq_internal.h", "kvq_api.cu")))}
        extra = {"gather_ms": round(att, 5), "gathered_tokens_per_step": st["n_all"]}
        launches = 2  # write + gather
        dtype = "u4 codes -> fp32 dequantise + inverse RHT -> bf16"
    elif kind == "gather_prefill":
        dense = sum(dense_ms) / len(dense_ms)
        achieved = units["prefill_flops"] / (dense / 1e3) / 1e12
        traffic = recorded_units("prefill_tc_%s.md" % args.workload, "dram_bytes_per_prefill_call",
                                 kernel_source_hash(("kvq_prefill_tc.cu", "kvq_tc.cuh", "kvq_common.cuh",
                                                     "kvq_internal.h", "kvq_api.cu")))
        roof = {"bound": "tensor", "kernel": "prefill_tc_kernel over dense bf16 rows (one kvq_prefill_dense_attn call)",
                "achieved": round(achieved, 2), "peak": tensor,
                "peak_kind": peak_kind + " (cuBLAS bf16 burst; kind::f16 fp16 runs at the bf16 rate)",
                "unit": "TFLOP/s", "frac": round(achieved / tensor, 4), "executed_tflops": round(2 * achieved, 2),
                "algorithmic_flops_per_launch": units["prefill_flops"], "traffic": traffic}
        extra = {"gather_ms": round(att, 5), "dense_prefill_ms": round(dense, 5),
                 "gathered_tokens_per_step": st["n_all"]}
        launches = 3  # write + gather + dense prefill
        dtype = "u4 codes -> bf16 rows (gather) -> fp16 x fp16 (q hi+lo) tcgen05 math, fp32 TMEM accumulate/softmax"
    elif kind == "decode":
        cfg["decode_workers"] = st["splits"]
        achieved = units["decode"] / (att / 1e3) / 1e9
        traffic = recorded_units("decode_stream_%s.md" % args.workload, "dram_bytes_per_decode_call",
                                 kernel_source_hash(("kvq_decode.cu", "kvq_common.cuh", "kvq_internal.h", "kvq_api.cu")))
        roof = {"bound": "hbm", "kernel": "decode attention (query prep + stream-K split-KV + merge, "
                                          "one kvq_decode_attn call)",
                "achieved": round(achieved, 1), "peak": hbm, "peak_kind": peak_kind + " (copy bandwidth)",
                "unit": "GB/s", "frac": round(achieved / hbm, 4), "frac_of_nominal_8000": round(achieved / 8000.0, 4),
                "algorithmic_bytes_per_launch": units["decode"], "traffic": traffic}
        extra = {"effective_kv_GBps": round(achieved, 1), "decode_ms": round(att, 5)}
        if fused_ms:
            extra["fused_write_decode_step_ms"] = round(sum(fused_ms) / len(fused_ms), 5)
        launches = 4  # write + (prep, stream, merge)
        dtype = {0: "u4", 1: "u2", 2: "s8", 3: "u4", 4: "s8", 5: "e4m3"}[wl.mode] + " codes x fp16 tensor-core math, fp32 accumulate/softmax"
    else:
        achieved = units["prefill_flops"] / (att / 1e3) / 1e12
        traffic = recorded_units("prefill_tc_%s.md" % args.workload, "dram_bytes_per_prefill_call",
                                 kernel_source_hash(("kvq_prefill_tc.cu", "kvq_tc.cuh", "kvq_common.cuh",
                                                     "kvq_internal.h", "kvq_api.cu")))
        roof = {"bound": "tensor", "kernel": "prefill_tc_kernel (tcgen05, one kvq_prefill_attn call)",
                "achieved": round(achieved, 2), "peak": tensor,
                "peak_kind": peak_kind + " (cuBLAS bf16 burst; kind::f16 fp16 runs at the bf16 rate)",
                "unit": "TFLOP/s", "frac": round(achieved / tensor, 4),
                "executed_tflops": round(2 * achieved, 2),
                "algorithmic_flops_per_launch": units["prefill_flops"], "traffic": traffic}
        extra = {"prefill_ms": round(att, 5)}
        launches = 2  # write + prefill
        dtype = "u4 codes x fp16 (hi+lo) tcgen05 math, fp32 TMEM accumulate/softmax"
    if wl.mode == gen.MODE_INT8:
        launches += 1  # INT8 write: channel-amax kernel (returns at once once the scales exist) + quantise kernel
    wr = sum(wr_ms) / len(wr_ms)
    write_gbs = units["write"] / (wr / 1e3) / 1e9
    write_roof = {"bound": "hbm", "kernel": "kvq_write (RHT, scale / zero point, codes, pack, scatter)",
                  "achieved": round(write_gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(write_gbs / hbm, 4),
                  "algorithmic_bytes_per_launch": units["write"],
                  "note": "bf16 K/V in + packed rows out; a 1-token decode write is launch-latency bound"}
    result = {
        "metric": metric, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded; K/V ~ N(0,1)%s)" % (", 1% outlier channels x10" if args.workload.startswith("llama") or args.workload in ("prefill_int4", "gather_int4", "gather_dense_prefill_int4") else ""),
        "config": cfg, **extra, "write_ms": round(wr, 5),
        "roofline": roof,
        "write_roofline": write_roof,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(sum(e2e_ms) / len(e2e_ms), 5)},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    return result, wl


def _oracle_paging(wl, lens):
    import oracle
    return oracle.Paging(wl.table, wl.headwise, np.ascontiguousarray(lens, np.int32), wl.window, wl.sink)


def _oracle_step_setup(wl, sample_seqs):
    """Oracle cache holding the prefixes of the sampled sequences (host values),
    and the step's host inputs (bf16 bits) for those sequences."""
    import oracle
    oc = oracle.Cache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.signs)
    pre = wl.prefix_lens.copy()
    counts = np.zeros(wl.batch, np.int32)
    counts[sample_seqs] = pre[sample_seqs]
    ks = [gen.kv_values_host(wl, "k", int(b), 0, int(pre[b])) for b in sample_seqs if pre[b] > 0]
    vs = [gen.kv_values_host(wl, "v", int(b), 0, int(pre[b])) for b in sample_seqs if pre[b] > 0]
    if ks:
        oracle.write(oc, _oracle_paging(wl, pre), gen.f32_to_bf16_bits(np.concatenate(ks)),
                     gen.f32_to_bf16_bits(np.concatenate(vs)), wl.cu(counts))
    nk = gen.f32_to_bf16_bits(np.concatenate([gen.kv_values_host(wl, "k", int(b), int(pre[b]), int(wl.n_new[b]))
                                              for b in sample_seqs]))
    nv = gen.f32_to_bf16_bits(np.concatenate([gen.kv_values_host(wl, "v", int(b), int(pre[b]), int(wl.n_new[b]))
                                              for b in sample_seqs]))
    q = gen.f32_to_bf16_bits(gen.q_values_host(wl))
    return oc, nk, nv, q


def oracle_step(wl, oc, new_k, new_v, q, sample_seqs, threads, rows=None, kind=None):
    """One step of the oracle on the sampled sequences: write their new
    tokens, then attention (decode: their one query each; prefill: the
    sampled query rows `rows` of the chunk) or, for the gather workload, the
    gather of their whole contexts."""
    import oracle
    counts = np.zeros(wl.batch, np.int32)
    counts[sample_seqs] = wl.n_new[sample_seqs]
    pag = _oracle_paging(wl, wl.seq_lens)
    oracle.write(oc, pag, new_k, new_v, wl.cu(counts))
    scale = 1.0 / math.sqrt(wl.head_dim)
    if kind == "gather":
        counts = np.zeros(wl.batch, np.int32)
        counts[sample_seqs] = wl.seq_lens[sample_seqs]
        oracle.gather(oc, pag, wl.cu(counts))
    elif kind == "gather_prefill":
        lens = np.zeros(wl.batch, np.int32)
        lens[sample_seqs] = wl.seq_lens[sample_seqs]
        cu_kv = wl.cu(lens)
        k, v, _ = oracle.gather(oc, pag, cu_kv)
        kb, vb = gen.f32_to_bf16_bits(k.astype(np.float32)), gen.f32_to_bf16_bits(v.astype(np.float32))
        dpag = oracle.Paging(np.zeros((wl.batch, 1), np.int32), False, lens, wl.window, wl.sink)
        oracle.dense_attention(kb, vb, cu_kv, dpag, q, scale, wl.cu(wl.n_new), rows=rows, threads=threads)
    elif wl.step == "decode":
        oracle.attention(oc, pag, q, scale, rows=np.asarray(sample_seqs, np.int32), threads=threads)
    else:
        oracle.attention(oc, pag, q, scale, cu_q=wl.cu(wl.n_new), rows=rows, threads=threads)


def _prefill_rows(wl, per_seq):
    """per_seq query rows of each sequence's chunk, evenly spaced (the last
    row of each chunk, the one that sees the most keys, included)."""
    cu = wl.cu(wl.n_new)
    rows = []
    for b in range(wl.batch):
        n = int(wl.n_new[b])
        for i in range(per_seq):
            rows.append(int(cu[b]) + (n - 1) - (i * n) // per_seq)
    return np.asarray(sorted(rows), np.int32)


def cpu_baseline(wl, budget_s=15.0, kind=None):
    """The CPU oracle, as it stands, on a bounded sample of the workload,
    repeated until ~budget_s of work.  Decode: whole steps (write one token +
    attend with every q head) of a subset of the sequences.  Prefill: the
    write of the whole chunk + attention of a few query rows per sequence."""
    threads = os.cpu_count() or 1
    if kind == "gather":
        sample = [0, 1, 2]  # the three shorter contexts
        rows = None
        per_step = int(wl.seq_lens[sample].sum())
    elif wl.step == "decode":
        sample = list(range(0, wl.batch, 4))
        rows = None
        per_step = len(sample)
    elif kind == "gather_prefill":
        sample = list(range(wl.batch))
        rows = _prefill_rows(wl, 4)
        per_step = len(rows)
    else:
        sample = list(range(wl.batch))
        rows = _prefill_rows(wl, 4)
        per_step = len(rows)
    oc, nk, nv, q = _oracle_step_setup(wl, sample)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(wl, oc, nk, nv, q, sample, threads, rows, kind)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 50:
            break
    dt = time.perf_counter() - t0
    if kind == "gather":
        desc = ("%d steps of: write of the chunks of sequences %s + gather of their whole contexts (%d positions, "
                "K and V, all %d kv heads; the oracle's gather is single-threaded), %.1f s"
                % (n, sample, per_step, wl.num_kv_heads, dt))
        threads = 1
    elif kind == "gather_prefill":
        desc = ("%d steps of: write of the %d-token chunk + gather of every cached position (single-threaded) + "
                "dense attention of %d query rows (4 per sequence, all %d q heads), %.1f s; tokens/s counts the "
                "attended rows" % (n, int(wl.n_new.sum()), per_step, wl.num_q_heads, dt))
    elif wl.step == "decode":
        desc = ("%d decode steps of %d of the %d sequences (every 4th; write 1 token + attention over the cached "
                "context, all %d q heads), %.1f s" % (n, len(sample), wl.batch, wl.num_q_heads, dt))
    else:
        desc = ("%d steps of: write of the %d-token chunk + attention of %d query rows (4 per sequence, all %d q "
                "heads), %.1f s; tokens/s counts the attended rows" % (n, int(wl.n_new.sum()), per_step,
                                                                       wl.num_q_heads, dt))
    return {"value": round(n * per_step / dt, 2), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}


def run_reference(args):
    """Reference arm: the CPU oracle timed alone on the same workload (a
    bounded sample of it per step)."""
    factory, metric, kind = WORKLOADS[args.workload]
    wl = factory(args)
    threads = os.cpu_count() or 1
    if kind == "gather":
        sample = [0, 1, 2]
        rows = None
        per_step = int(wl.seq_lens[sample].sum())
        desc = ("sequences %s per step: write of their chunks + gather of their whole contexts (%d positions, K and "
                "V, all %d kv heads; single-threaded oracle)" % (sample, per_step, wl.num_kv_heads))
        threads = 1
    elif kind == "gather_prefill":
        sample = list(range(wl.batch))
        rows = _prefill_rows(wl, 1)
        per_step = len(rows)
        desc = ("write of the %d-token chunk + gather of every cached position + dense attention of the last query "
                "row of each sequence, all %d q heads" % (int(wl.n_new.sum()), wl.num_q_heads))
    elif kind == "decode":
        sample = list(range(0, wl.batch, 16))
        rows = None
        per_step = len(sample)
        desc = "%d of the %d sequences per step (every 16th): write 1 token + attention, all %d q heads" % (
            per_step, wl.batch, wl.num_q_heads)
    else:
        sample = list(range(wl.batch))
        rows = _prefill_rows(wl, 1)
        per_step = len(rows)
        desc = ("write of the %d-token chunk + attention of the last query row of each sequence, all %d q heads"
                % (int(wl.n_new.sum()), wl.num_q_heads))
    oc, nk, nv, q = _oracle_step_setup(wl, sample)
    for _ in range(args.warmup):
        oracle_step(wl, oc, nk, nv, q, sample, threads, rows, kind)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(wl, oc, nk, nv, q, sample, threads, rows, kind)
        ts.append(time.perf_counter() - t0)
    ms = 1e3 * sum(ts) / len(ts)
    value = per_step / (ms / 1e3)
    return {"impl": "reference", "metric": metric, "value": round(value, 3), "unit": UNIT, "n_gpus": 0,
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
    ap.add_argument("--workload", default="llama_int4", choices=sorted(WORKLOADS),
                    help="llama_int4 (the headline decode workload), llama_int4_d64_bs64, llama_int4_stego, "
                         "llama_int8_token_head, llama_fp8_token_head, ernie_int2, qwen_int8_headwise, prefill_int4, "
                         "gather_int4, gather_dense_prefill_int4")
    ap.add_argument("--pool-blocks", type=int, default=0,
                    help="block pool size (0 = the workload's own; smaller pools only for profiling)")
    ap.add_argument("--prefill-prefixes", type=int, nargs="+", default=[0, 4096, 16384, 61440],
                    help="cached prefix per sequence of the prefill workload")
    ap.add_argument("--prefill-chunk", type=int, default=2048, help="new tokens per sequence of the prefill workload")
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
            result["cpu_baseline"] = cpu_baseline(wl, kind=WORKLOADS[args.workload][2])
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
