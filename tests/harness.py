"""Test harness: run one workload through the CUDA library and through the
CPU oracle from the same seeded inputs, and compare.

Inputs come from ``kvq_inputs`` only; the oracle never sees an output of the
CUDA path (the comparison reads both sides' results, nothing flows from one
side into the other).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import kvq_inputs as gen
import oracle

ATOL = 2e-3  # maximum absolute error on attention outputs (fp32)


def kvq():
    import sub_byte_quantized_write_gb300 as m
    return m


def to_dev_input(x32: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """fp32 values already on the bf16 grid -> device tensor of that dtype."""
    if dtype == "bf16":
        bits = gen.f32_to_bf16_bits(x32)
        return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(device)


def to_orc_input(x32: np.ndarray, dtype: str) -> np.ndarray:
    return gen.f32_to_bf16_bits(x32) if dtype == "bf16" else np.ascontiguousarray(x32, dtype=np.float32)


@dataclass
class Case:
    wl: gen.Workload
    gcache: object
    gpag_prefix: object
    gpag: object
    ocache: oracle.Cache
    opag_prefix: oracle.Paging
    opag: oracle.Paging
    k_new: np.ndarray
    v_new: np.ndarray
    k_pre: Optional[np.ndarray]
    v_pre: Optional[np.ndarray]
    dev_err: torch.Tensor


def build_case(wl: gen.Workload, fill: int = 0xA5, table: Optional[np.ndarray] = None,
               headwise: Optional[bool] = None, device="cuda") -> Case:
    """Allocate both caches, generate the prefix and step tokens, and run the
    prefix write on both sides (the step write is run by write_step)."""
    K = kvq()
    table = wl.table if table is None else table
    headwise = wl.headwise if headwise is None else headwise
    signs_t = None if wl.signs is None else torch.from_numpy(wl.signs).to(device)
    gcache = K.PagedCache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, signs_t, device)
    gcache.k_pages.fill_(fill)
    gcache.v_pages.fill_(fill)
    ocache = oracle.Cache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.signs, fill)
    t_dev = torch.from_numpy(table).to(device)
    win_dev = None if wl.window is None else torch.from_numpy(wl.window).to(device)
    pre = wl.prefix_lens

    def gpag(lens):
        lt = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).to(device)
        if headwise:
            return K.Paging(lt, block_tables_headwise=t_dev, window_per_kv_head=win_dev, sink_size=wl.sink)
        return K.Paging(lt, block_tables=t_dev, window_per_kv_head=win_dev, sink_size=wl.sink)

    def opag(lens):
        return oracle.Paging(table, headwise, lens, wl.window, wl.sink)

    B = wl.batch
    k_pre = v_pre = None
    if pre.sum() > 0:
        k_pre = np.concatenate([gen.kv_values_host(wl, "k", b, 0, int(pre[b])) for b in range(B)])
        v_pre = np.concatenate([gen.kv_values_host(wl, "v", b, 0, int(pre[b])) for b in range(B)])
    k_new = np.concatenate([gen.kv_values_host(wl, "k", b, int(pre[b]), int(wl.n_new[b])) for b in range(B)])
    v_new = np.concatenate([gen.kv_values_host(wl, "v", b, int(pre[b]), int(wl.n_new[b])) for b in range(B)])
    dev_err = torch.zeros(1, dtype=torch.int32, device=device)
    c = Case(wl, gcache, gpag(pre), gpag(wl.seq_lens), ocache, opag(pre), opag(wl.seq_lens), k_new, v_new,
             k_pre, v_pre, dev_err)
    if k_pre is not None:
        cu = torch.from_numpy(wl.cu(pre)).to(device)
        K.kvq_write(gcache, c.gpag_prefix, to_dev_input(k_pre, wl.dtype), to_dev_input(v_pre, wl.dtype), cu,
                    dev_error=dev_err)
        assert oracle.write(ocache, c.opag_prefix, to_orc_input(k_pre, wl.dtype), to_orc_input(v_pre, wl.dtype),
                            wl.cu(pre)) == 0
    return c


def write_step(c: Case, device="cuda"):
    K = kvq()
    wl = c.wl
    cu = torch.from_numpy(wl.cu(wl.n_new)).to(device)
    K.kvq_write(c.gcache, c.gpag, to_dev_input(c.k_new, wl.dtype), to_dev_input(c.v_new, wl.dtype), cu,
                dev_error=c.dev_err)
    err = oracle.write(c.ocache, c.opag, to_orc_input(c.k_new, wl.dtype), to_orc_input(c.v_new, wl.dtype),
                       wl.cu(wl.n_new))
    assert err == 0


def assert_pools_equal(c: Case):
    torch.cuda.synchronize()
    gk = c.gcache.k_pages.cpu().numpy()
    gv = c.gcache.v_pages.cpu().numpy()
    for name, g, o in (("K", gk, c.ocache.k), ("V", gv, c.ocache.v)):
        if not np.array_equal(g, o):
            bad = np.argwhere(g != o)
            raise AssertionError("%s pool differs at %d bytes, first %s: gpu %d oracle %d"
                                 % (name, len(bad), tuple(bad[0]), g[tuple(bad[0])], o[tuple(bad[0])]))
    if c.wl.mode == gen.MODE_INT8:
        ga = c.gcache.ch_amax.cpu().numpy()
        assert np.array_equal(ga, c.ocache.amax), "channel amax differs"
        assert int(c.gcache.ch_amax_ready.cpu()[0]) == 1
    assert int(c.dev_err.cpu()[0]) == 0


def q_host(wl):
    return gen.q_values_host(wl)


def decode_gpu(c: Case, q32: np.ndarray, num_splits=0, paging=None, cache=None):
    K = kvq()
    wl = c.wl
    out = K.kvq_decode_attn(cache or c.gcache, paging or c.gpag, to_dev_input(q32, wl.dtype),
                            1.0 / math.sqrt(wl.head_dim), num_splits=num_splits, dev_error=c.dev_err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def decode_oracle(c: Case, q32: np.ndarray, rows=None):
    wl = c.wl
    out, err = oracle.attention(c.ocache, c.opag, to_orc_input(q32, wl.dtype), 1.0 / math.sqrt(wl.head_dim),
                                rows=rows)
    assert err == 0
    return out


def prefill_gpu(c: Case, q32: np.ndarray, scale: Optional[float] = None):
    K = kvq()
    wl = c.wl
    cu = torch.from_numpy(wl.cu(wl.n_new)).to("cuda")
    scale = 1.0 / math.sqrt(wl.head_dim) if scale is None else scale
    out = K.kvq_prefill_attn(c.gcache, c.gpag, to_dev_input(q32, wl.dtype), cu, int(wl.n_new.max()),
                             scale, dev_error=c.dev_err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def prefill_oracle(c: Case, q32: np.ndarray, rows=None, scale: Optional[float] = None):
    wl = c.wl
    scale = 1.0 / math.sqrt(wl.head_dim) if scale is None else scale
    out, err = oracle.attention(c.ocache, c.opag, to_orc_input(q32, wl.dtype), scale,
                                cu_q=wl.cu(wl.n_new), rows=rows)
    assert err == 0
    return out


def max_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(gpu.astype(np.float64) - ref)))
