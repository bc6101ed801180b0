"""kvq_prefill_attn on the GPU against the CPU oracle."""
import numpy as np
import pytest
import torch

import kvq_inputs as gen
from harness import (ATOL, assert_pools_equal, build_case, decode_gpu, kvq, max_err, prefill_gpu, prefill_oracle,
                     q_host, write_step)

pytestmark = pytest.mark.gpu


def _run(wl, rows=None):
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)
    q = q_host(wl)
    g = prefill_gpu(c, q)
    o = prefill_oracle(c, q, rows=rows)
    gg = g if rows is None else g[rows]
    e = max_err(gg, o)
    worst = np.unravel_index(np.argmax(np.abs(gg.astype(np.float64) - o)), o.shape)
    assert e <= ATOL, "max abs err %.3g at (row, head, dim) %s" % (e, worst)
    assert int(c.dev_err.item()) == 0
    return c, q, g


def test_prefill_reduced_chunked_append():
    _run(gen.prefill_int4(0, prefixes=(0, 100, 700, 1500), chunk=130, num_blocks=1000))


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8, gen.MODE_INT4_STEGO,
                                  gen.MODE_INT8_TOKEN_HEAD, gen.MODE_FP8_TOKEN_HEAD])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 5])
def test_prefill_modes_dims_groups(mode, D, group):
    Hkv = 2
    wl = gen.custom(mode, Hkv * group, Hkv, D, 16, "bf16", seq_lens=[70, 200, 15], n_new=[70, 77, 15],
                    step="prefill", seed=group + D + mode, outlier_frac=0.02)
    _run(wl)


def test_prefill_sliding_window_headwise():
    wl = gen.custom(gen.MODE_INT8, 10, 2, 128, 64, "bf16", seq_lens=[900, 400], n_new=[200, 150],
                    headwise=True, window=[0, 128], sink=4, step="prefill", seed=9)
    _run(wl)


def test_prefill_single_query_equals_decode():
    wl = gen.custom(gen.MODE_INT4, 16, 4, 128, 16, "bf16", seq_lens=[900, 77], n_new=[1, 1], seed=15)
    c = build_case(wl)
    write_step(c)
    q = q_host(wl)
    gd = decode_gpu(c, q)
    gp = prefill_gpu(c, q)
    # Same fold and the same fp16 hi/lo operands on both paths; they differ
    # only in fp32 summation order (32-key mma.sync tiles vs 64-key tcgen05
    # tiles with a tensor-core accumulation order), i.e. a few ulps of
    # outputs of size ~1 summed over ~1e3 keys.
    assert np.max(np.abs(gd - gp)) <= 5e-5


def test_prefill_full_size_sampled_rows():
    """Chunk of 8192 tokens over 4 sequences with 0 / 4k / 16k / 60k cached
    tokens (the prefill workload at full size), sampled query rows against the
    oracle."""
    wl = gen.prefill_int4(0)
    rows = np.array([0, 1, 2047, 2048, 3000, 4095, 4096, 6000, 6143, 6144, 7000, 8191], dtype=np.int32)
    _run(wl, rows=rows)
