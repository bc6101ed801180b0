"""Seeded synthetic workloads for the paged low-bit KV cache.

This module only DRAWS inputs: random K/V/q values, sign vectors, sequence
lengths and block tables.  It holds none of the quantisation or attention
arithmetic, so both the CPU oracle (``oracle/``) and the CUDA library can be
fed from it without sharing any of the method's code.

Shapes and distributions follow the five workloads the pages' problem
statement describes (tiny INT4 parity case; INT4 decode on a Llama-3-8B-like
layer; dynamic INT2 decode on an ERNIE-4.5-21B-A3B-like layer; INT4 chunked
prefill; INT8 per-channel with head-wise sliding-window tables).  They are
synthetic stand-ins: no model weights or datasets are involved.

Random streams
  * structure (signs, outlier channels, lengths, tables): numpy PCG64 seeded
    with ``[seed, 0]``, drawn in a fixed order per workload;
  * token values: one stream per (tensor, sequence), so any sequence can be
    regenerated alone; on the host numpy PCG64 ``[seed, tag, b]``, on a CUDA
    device a torch generator seeded with a mix of the same three numbers.
    Host and device streams differ; a test uses one of them for both sides.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

MODE_INT4 = 0
MODE_INT2 = 1
MODE_INT8 = 2
MODE_INT4_STEGO = 3  # INT4 with the zero point in the low 4 bits of an fp32 scale
MODE_INT8_TOKEN_HEAD = 4  # symmetric INT8, one fp32 scale per (token, kv head)
MODE_FP8_TOKEN_HEAD = 5  # FP8 E4M3 codes, one fp32 scale per (token, kv head)

_TAG_K, _TAG_V, _TAG_Q = 11, 13, 17


@dataclasses.dataclass
class Workload:
    name: str
    mode: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # "f32" or "bf16" for q/k/v
    num_blocks: int
    max_blocks: int
    seq_lens: np.ndarray            # int32 [B], tokens cached after the step
    n_new: np.ndarray               # int32 [B], tokens written (and queried, for prefill) by the step
    table: np.ndarray               # int32 [B, max_blocks] or [B*Hkv, max_blocks]
    headwise: bool
    window: Optional[np.ndarray]    # int32 [Hkv] or None
    sink: int
    signs: Optional[np.ndarray]     # int8 [D] of +-1, or None (RHT off)
    step: str                       # "decode" or "prefill"
    q_std: float
    outliers_k: tuple               # (heads int array, channels int array, factor)
    outliers_v: tuple
    seed: int

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def prefix_lens(self) -> np.ndarray:
        return (self.seq_lens - self.n_new).astype(np.int32)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def cu(self, counts: np.ndarray) -> np.ndarray:
        out = np.zeros(len(counts) + 1, dtype=np.int32)
        out[1:] = np.cumsum(counts)
        return out

    def uniform_table_equivalent(self) -> np.ndarray:
        """Row b of head 0 of a head-wise table (used when all heads agree)."""
        if not self.headwise:
            return self.table
        return self.table.reshape(self.batch, self.num_kv_heads, self.max_blocks)[:, 0, :].copy()


# ----------------------------------------------------------------------------
# structure draws

def _structure_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, 0]))


def _draw_signs(rng, d):
    return np.where(rng.integers(0, 2, size=d) == 1, 1, -1).astype(np.int8)


def _draw_outliers(rng, hkv, d, count, factor):
    flat = rng.choice(hkv * d, size=count, replace=False)
    return (flat // d).astype(np.int64), (flat % d).astype(np.int64), float(factor)


def _draw_outliers_per_head(rng, hkv, d, per_head, factor):
    heads, chans = [], []
    for h in range(hkv):
        c = rng.choice(d, size=per_head, replace=False)
        heads += [h] * per_head
        chans += list(c)
    return np.array(heads, np.int64), np.array(chans, np.int64), float(factor)


def _tables_from_pool(rng, seq_lens, bs, max_blocks, num_blocks):
    need = [(int(L) + bs - 1) // bs for L in seq_lens]
    total = sum(need)
    if total > num_blocks:
        raise ValueError("pool too small")
    picks = rng.choice(num_blocks, size=total, replace=False).astype(np.int32)
    table = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = picks[o:o + n]
        o += n
    return table


_NO_OUTLIERS = (np.zeros(0, np.int64), np.zeros(0, np.int64), 1.0)


def tiny_int4(seed: int = 0) -> Workload:
    """Tiny INT4 per-token-head parity case: B=2, Hq=4, Hkv=2, D=64, bs=16,
    contexts 37 and 100 placed by a random permutation of a 16-block pool,
    fp32 K/V ~ N(0,1) with 2 outlier channels per head (x20), q ~ N(0,1);
    the step writes all 137 tokens and then decodes."""
    rng = _structure_rng(seed)
    D, Hkv, bs = 64, 2, 16
    signs = _draw_signs(rng, D)
    ok = _draw_outliers_per_head(rng, Hkv, D, 2, 20.0)
    ov = _draw_outliers_per_head(rng, Hkv, D, 2, 20.0)
    perm = rng.permutation(16).astype(np.int32)
    seq_lens = np.array([37, 100], dtype=np.int32)
    max_blocks = 8
    table = np.full((2, max_blocks), -1, dtype=np.int32)
    table[0, :3] = perm[:3]
    table[1, :7] = perm[3:10]
    return Workload("tiny_int4", MODE_INT4, 4, Hkv, D, bs, "f32", 16, max_blocks,
                    seq_lens, seq_lens.copy(), table, False, None, 0, signs, "decode",
                    1.0, ok, ov, seed)


def llama_int4(seed: int = 0, batch: int = 64, ctx_lo: int = 1024, ctx_hi: int = 8192,
               num_blocks: int = 200000, head_dim: int = 128, block_size: int = 16,
               mode: int = MODE_INT4) -> Workload:
    """INT4 per-token-head decode, Llama-3-8B-like layer: Hq=32, Hkv=8, D=128,
    bf16, bs=16, contexts uniform in [ctx_lo, ctx_hi], pages at distinct random
    blocks of the pool, K/V ~ N(0,1) with 1% of (head, channel) pairs x10, RHT
    on, one new token per sequence per step.  `head_dim` / `block_size` give
    the same layer at D = 64 and bs = 32 or 64; `mode` MODE_INT4_STEGO the
    same cache with the zero point carried in the fp32 scale, and
    MODE_INT8_TOKEN_HEAD / MODE_FP8_TOKEN_HEAD the same layer in 8-bit rows."""
    rng = _structure_rng(seed)
    D, Hkv, bs = head_dim, 8, block_size
    signs = _draw_signs(rng, D)
    n_out = int(round(0.01 * Hkv * D))
    ok = _draw_outliers(rng, Hkv, D, n_out, 10.0)
    ov = _draw_outliers(rng, Hkv, D, n_out, 10.0)
    seq_lens = rng.integers(ctx_lo, ctx_hi + 1, size=batch).astype(np.int32)
    max_blocks = (ctx_hi + bs - 1) // bs
    table = _tables_from_pool(rng, seq_lens, bs, max_blocks, num_blocks)
    name = "llama_int4_decode" if (D, bs) == (128, 16) else "llama_int4_d%d_bs%d_decode" % (D, bs)
    tag = {MODE_INT4_STEGO: "int4_stego", MODE_INT8_TOKEN_HEAD: "int8_token_head", MODE_FP8_TOKEN_HEAD: "fp8_token_head"}
    if mode in tag:
        name = name.replace("int4", tag[mode])
    return Workload(name, mode, 32, Hkv, D, bs, "bf16", num_blocks,
                    max_blocks, seq_lens, np.ones(batch, np.int32), table, False, None, 0,
                    signs, "decode", 1.0, ok, ov, seed)


def ernie_int2(seed: int = 0, batch: int = 96, median: int = 16384, sigma: float = 0.5,
               lo: int = 512, hi: int = 131072, num_blocks: int = 100000) -> Workload:
    """Dynamic INT2 decode, ERNIE-4.5-21B-A3B-like layer: Hq=20, Hkv=4, D=128,
    bf16, bs=64, 4 codes per byte, contexts log-normal (median 16k, sigma 0.5)
    clipped to [512, 131072], pool of 100000 blocks, K/V ~ N(0,1),
    q ~ N(0,1)/sqrt(128), RHT on."""
    rng = _structure_rng(seed)
    D, Hkv, bs = 128, 4, 64
    signs = _draw_signs(rng, D)
    raw = rng.lognormal(mean=math.log(median), sigma=sigma, size=batch)
    seq_lens = np.clip(np.rint(raw), lo, hi).astype(np.int32)
    max_blocks = (hi + bs - 1) // bs
    table = _tables_from_pool(rng, seq_lens, bs, max_blocks, num_blocks)
    return Workload("ernie_int2_decode", MODE_INT2, 20, Hkv, D, bs, "bf16", num_blocks,
                    max_blocks, seq_lens, np.ones(batch, np.int32), table, False, None, 0,
                    signs, "decode", 1.0 / math.sqrt(128.0), _NO_OUTLIERS, _NO_OUTLIERS, seed)


def prefill_int4(seed: int = 0, prefixes=(0, 4096, 16384, 61440), chunk: int = 2048,
                 num_blocks: int = 200000) -> Workload:
    """INT4 chunked-prefill append on the Llama-like layer: an 8192-token chunk
    split over 4 sequences (2048 each) whose caches already hold 0 / 4k / 16k /
    60k tokens; outlier channels as in the decode workload."""
    rng = _structure_rng(seed)
    D, Hkv, bs = 128, 8, 16
    signs = _draw_signs(rng, D)
    n_out = int(round(0.01 * Hkv * D))
    ok = _draw_outliers(rng, Hkv, D, n_out, 10.0)
    ov = _draw_outliers(rng, Hkv, D, n_out, 10.0)
    pre = np.array(prefixes, dtype=np.int32)
    n_new = np.full(len(pre), chunk, dtype=np.int32)
    seq_lens = pre + n_new
    max_blocks = int((seq_lens.max() + bs - 1) // bs)
    table = _tables_from_pool(rng, seq_lens, bs, max_blocks, num_blocks)
    return Workload("prefill_int4", MODE_INT4, 32, Hkv, D, bs, "bf16", num_blocks,
                    max_blocks, seq_lens, n_new, table, False, None, 0, signs, "prefill",
                    1.0, ok, ov, seed)


def qwen_int8_headwise(seed: int = 0, batch: int = 32, context: int = 32768,
                       window: int = 4096, sink: int = 4, swa_heads=(4, 5, 6, 7),
                       headwise: bool = True) -> Workload:
    """Dynamic per-channel INT8 K/V with head-wise tables, Qwen2.5-14B-like:
    Hq=40, Hkv=8, D=128, bf16, bs=64, batch 32 at context 32768.  Heads 0-3
    full; heads in `swa_heads` keep the last `window` tokens plus `sink` sink
    tokens, and the blocks holding neither are -1 in their table rows.  The
    prefix (context - 1 tokens) defines the channel scales; the step writes one
    token and decodes at `context`."""
    rng = _structure_rng(seed)
    D, Hkv, bs = 128, 8, 64
    seq_lens = np.full(batch, context, dtype=np.int32)
    nb_seq = (context + bs - 1) // bs
    max_blocks = nb_seq
    num_blocks = batch * nb_seq
    win = np.zeros(Hkv, dtype=np.int32)
    for h in swa_heads:
        win[h] = window
    table = np.full((batch * Hkv, max_blocks), -1, dtype=np.int32)
    for h in range(Hkv):
        perm = rng.permutation(num_blocks).astype(np.int32)
        for b in range(batch):
            table[b * Hkv + h, :] = perm[b * nb_seq:(b + 1) * nb_seq]
    # evict blocks that hold neither sink tokens nor window tokens of the
    # decode query at position context - 1
    p = context - 1
    first_win_block = (p - window + 1) // bs if window > 0 else 0
    last_sink_block = (sink - 1) // bs if sink > 0 else -1
    for h in swa_heads:
        for b in range(batch):
            for blk in range(max_blocks):
                if blk > last_sink_block and blk < first_win_block:
                    table[b * Hkv + h, blk] = -1
    wl = Workload("qwen_int8_headwise", MODE_INT8, 40, Hkv, D, bs, "bf16", num_blocks,
                  max_blocks, seq_lens, np.ones(batch, np.int32), table, True, win, sink,
                  None, "decode", 1.0, _NO_OUTLIERS, _NO_OUTLIERS, seed)
    if not headwise:
        wl.table = wl.table.reshape(batch, Hkv, max_blocks)[:, 0, :].copy()
        wl.headwise = False
    return wl


# ----------------------------------------------------------------------------
# token values

def _mix(seed: int, tag: int, b: int) -> int:
    x = (seed * 0x9E3779B1 + tag * 0x85EBCA77 + b * 0xC2B2AE3D + 0x27D4EB2F) & 0xFFFFFFFFFFFF
    return int(x)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _apply_outliers(x, outl, layout_heads_axis=1):
    heads, chans, factor = outl
    if len(heads):
        x[:, heads, chans] *= factor
    return x


def kv_values_host(wl: Workload, which: str, b: int, start: int, count: int) -> np.ndarray:
    """fp32 [count, Hkv, D] values of K (`which`='k') or V for positions
    start..start+count-1 of sequence b, already rounded to the workload dtype."""
    tag = _TAG_K if which == "k" else _TAG_V
    rng = np.random.Generator(np.random.PCG64([wl.seed, tag, b]))
    total = int(wl.seq_lens[b])
    full = rng.standard_normal((total, wl.num_kv_heads, wl.head_dim), dtype=np.float32)
    x = full[start:start + count].copy()
    _apply_outliers(x, wl.outliers_k if which == "k" else wl.outliers_v)
    if wl.dtype == "bf16":
        x = bf16_bits_to_f32(f32_to_bf16_bits(x))
    return x


def q_values_host(wl: Workload) -> np.ndarray:
    """fp32 q rows, rounded to the workload dtype: [B, Hq, D] for decode,
    [sum(n_new), Hq, D] for prefill (row order = sequence order)."""
    rows = wl.batch if wl.step == "decode" else int(wl.n_new.sum())
    rng = np.random.Generator(np.random.PCG64([wl.seed, _TAG_Q, 0]))
    q = rng.standard_normal((rows, wl.num_q_heads, wl.head_dim), dtype=np.float32) * np.float32(wl.q_std)
    if wl.dtype == "bf16":
        q = bf16_bits_to_f32(f32_to_bf16_bits(q))
    return q.astype(np.float32)


def kv_values_device(wl: Workload, which: str, b: int, start: int, count: int, device="cuda"):
    """Same role as kv_values_host but drawn by torch on a CUDA device (a
    different stream of numbers); returns a tensor of the workload dtype."""
    import torch
    tag = _TAG_K if which == "k" else _TAG_V
    g = torch.Generator(device=device)
    g.manual_seed(_mix(wl.seed, tag, b))
    total = int(wl.seq_lens[b])
    full = torch.randn((total, wl.num_kv_heads, wl.head_dim), generator=g, device=device,
                       dtype=torch.float32)
    x = full[start:start + count].clone()
    heads, chans, factor = wl.outliers_k if which == "k" else wl.outliers_v
    if len(heads):
        hi = torch.as_tensor(heads, device=device)
        ci = torch.as_tensor(chans, device=device)
        x[:, hi, ci] *= factor
    if wl.dtype == "bf16":
        return x.to(torch.bfloat16)
    return x


def q_values_device(wl: Workload, device="cuda"):
    import torch
    rows = wl.batch if wl.step == "decode" else int(wl.n_new.sum())
    g = torch.Generator(device=device)
    g.manual_seed(_mix(wl.seed, _TAG_Q, 0))
    q = torch.randn((rows, wl.num_q_heads, wl.head_dim), generator=g, device=device,
                    dtype=torch.float32) * wl.q_std
    return q.to(torch.bfloat16) if wl.dtype == "bf16" else q


def describe(wl: Workload) -> dict:
    return {
        "workload": wl.name, "mode": ["int4", "int2", "int8"][wl.mode],
        "batch": wl.batch, "num_q_heads": wl.num_q_heads, "num_kv_heads": wl.num_kv_heads,
        "head_dim": wl.head_dim, "block_size": wl.block_size, "dtype": wl.dtype,
        "num_blocks": wl.num_blocks, "cached_tokens": int(wl.seq_lens.sum()),
        "headwise": wl.headwise, "rht": wl.signs is not None, "step": wl.step,
    }


def custom(mode: int, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int, dtype: str,
           seq_lens, n_new, num_blocks: Optional[int] = None, headwise: bool = False, window=None,
           sink: int = 0, rht: bool = True, seed: int = 0, step: str = "decode", q_std: float = 1.0,
           outlier_frac: float = 0.01, outlier_factor: float = 10.0, evict_outside_window: bool = False,
           max_blocks: Optional[int] = None) -> Workload:
    """A small workload of arbitrary shape for parity tests: pages drawn at
    distinct random blocks (per kv head for head-wise tables), optional
    outlier channels, optional eviction (-1) of blocks that hold neither sink
    nor window keys of the last query of each sequence."""
    rng = _structure_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    n_new = np.asarray(n_new, dtype=np.int32)
    B = len(seq_lens)
    bs, Hkv, D = block_size, num_kv_heads, head_dim
    signs = _draw_signs(rng, D) if (rht and mode != MODE_INT8) else None
    n_out = int(round(outlier_frac * Hkv * D))
    ok = _draw_outliers(rng, Hkv, D, n_out, outlier_factor) if n_out else _NO_OUTLIERS
    ov = _draw_outliers(rng, Hkv, D, n_out, outlier_factor) if n_out else _NO_OUTLIERS
    need = int(((seq_lens + bs - 1) // bs).sum())
    if max_blocks is None:
        max_blocks = int((seq_lens.max() + bs - 1) // bs)
    if num_blocks is None:
        num_blocks = need + 7
    win = None if window is None else np.asarray(window, dtype=np.int32)
    if headwise:
        table = np.full((B * Hkv, max_blocks), -1, dtype=np.int32)
        for h in range(Hkv):
            t = _tables_from_pool(rng, seq_lens, bs, max_blocks, num_blocks)
            for b in range(B):
                table[b * Hkv + h] = t[b]
        if evict_outside_window and win is not None:
            for b in range(B):
                p = int(seq_lens[b]) - 1
                for h in range(Hkv):
                    if win[h] <= 0:
                        continue
                    lo_blk = (p - int(win[h]) + 1) // bs
                    hi_sink = (sink - 1) // bs if sink > 0 else -1
                    for blk in range(max_blocks):
                        if hi_sink < blk < lo_blk:
                            table[b * Hkv + h, blk] = -1
    else:
        table = _tables_from_pool(rng, seq_lens, bs, max_blocks, num_blocks)
    return Workload("custom", mode, num_q_heads, Hkv, D, bs, dtype, num_blocks, max_blocks, seq_lens, n_new,
                    table, headwise, win, sink, signs, step, q_std, ok, ov, seed)
