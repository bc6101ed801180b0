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
    c, q, g = _run(gen.prefill_int4(0, prefixes=(0, 100, 700, 1500), chunk=130, num_blocks=1000))
    # a second call on the same inputs returns the same bits: the two softmax
    # halves of a row merge in a fixed order
    assert np.array_equal(g, prefill_gpu(c, q))


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


ALL_MODES = [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8, gen.MODE_INT4_STEGO, gen.MODE_INT8_TOKEN_HEAD,
             gen.MODE_FP8_TOKEN_HEAD]
EVICT_CASES = ([(m, D, 16) for m in ALL_MODES for D in (64, 128)]
               + [(gen.MODE_INT4, 64, 64), (gen.MODE_INT4, 128, 64), (gen.MODE_INT8, 64, 64), (gen.MODE_INT8, 128, 64)])


def _evicted_workload(mode, D, bs, seed):
    """Head-wise tables with -1 blocks: head 0 full, head 1 a 64-token window
    plus 4 sinks.  Blocks are evicted outside the window of each sequence's
    LAST query, so the chunk's first queries (hundreds of positions earlier)
    have their own window keys in -1 blocks and see only the sinks plus
    whatever survives: a skip that consulted the wrong query, or a leak of a
    -1 page, changes their rows.  The same block index is -1 for head 1 and
    live for head 0."""
    wl = gen.custom(mode, 8, 2, D, bs, "bf16", seq_lens=[900, 300, 75], n_new=[400, 300, 60], headwise=True,
                    window=[0, 64], sink=4, evict_outside_window=True, step="prefill", seed=seed,
                    outlier_frac=0.02)
    t = wl.table.reshape(wl.batch, wl.num_kv_heads, -1)
    assert (t[:, 1] == -1).any() and not (t[0, 0, :900 // bs] == -1).any()
    return wl


@pytest.mark.parametrize("mode,D,bs", EVICT_CASES)
def test_prefill_evicted_headwise_blocks(mode, D, bs):
    """The paged prefill over head-wise tables whose -1 entries mark evicted
    sliding-window blocks (FastDeploy PR #7718, PR2-only delta and Correctness
    gates: a -1 block contributes nothing and is never addressed)."""
    _run(_evicted_workload(mode, D, bs, seed=40 + mode + D + bs))


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT8, gen.MODE_FP8_TOKEN_HEAD])
def test_prefill_evicted_pages_never_read(mode):
    """Garbage in every page that no table row of its head references (0x7F:
    a NaN scale pad for INT4, the E4M3 NaN byte for FP8) leaves the prefill's
    output bits unchanged."""
    wl = _evicted_workload(mode, 128, 16, seed=77 + mode)
    c, q, g0 = _run(wl)
    Hkv = wl.num_kv_heads
    rows = wl.table.reshape(wl.batch, Hkv, -1)
    for h in range(Hkv):
        live = set(int(x) for x in rows[:, h].ravel() if x >= 0)
        dead = [b for b in range(wl.num_blocks) if b not in live]
        assert dead
        idx = torch.tensor(dead, dtype=torch.long, device="cuda")
        c.gcache.k_pages[idx, h] = 0x7F
        c.gcache.v_pages[idx, h] = 0x7F
    g1 = prefill_gpu(c, q)
    assert np.array_equal(g0, g1)


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT8_TOKEN_HEAD])
def test_prefill_negative_softmax_scale(mode):
    """softmax(scale * q.k) with scale < 0 (the kernel flips the query's sign
    and uses |scale|) against the oracle's definition."""
    wl = gen.custom(mode, 8, 2, 128, 16, "bf16", seq_lens=[300, 90], n_new=[120, 90], step="prefill", seed=51)
    c = build_case(wl)
    write_step(c)
    q = q_host(wl)
    scale = -0.6 / np.sqrt(wl.head_dim)
    g = prefill_gpu(c, q, scale=scale)
    o = prefill_oracle(c, q, scale=scale)
    assert max_err(g, o) <= ATOL
    assert int(c.dev_err.item()) == 0


def test_prefill_flags_bad_block_id_and_short_table():
    """Device-side contract violations on the read path: a table entry past
    the pool is skipped (that block's keys contribute nothing) and sets
    KVQ_DEVERR_BLOCK_RANGE; a seq_len past max_blocks * block_size drops the
    keys beyond the table and sets KVQ_DEVERR_TABLE_RANGE.  The oracle skips
    the same keys and reports the same bits."""
    import oracle
    from harness import to_dev_input, to_orc_input
    K = kvq()
    wl = gen.custom(gen.MODE_INT4, 8, 2, 128, 16, "bf16", seq_lens=[300, 150], n_new=[40, 30], step="prefill",
                    seed=52)
    c = build_case(wl)
    write_step(c)
    q = q_host(wl)
    scale = 1.0 / np.sqrt(wl.head_dim)
    cu = torch.from_numpy(wl.cu(wl.n_new)).cuda()
    # (1) block 3 of sequence 0 points past the pool
    bad = wl.table.copy()
    bad[0, 3] = wl.num_blocks + 9
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pag = K.Paging(torch.from_numpy(wl.seq_lens).cuda(), block_tables=torch.from_numpy(bad).cuda())
    g = K.kvq_prefill_attn(c.gcache, pag, to_dev_input(q, wl.dtype), cu, 40, scale,
                           dev_error=err)
    torch.cuda.synchronize()
    o, oerr = oracle.attention(c.ocache, oracle.Paging(bad, False, wl.seq_lens), to_orc_input(q, wl.dtype), scale,
                               cu_q=wl.cu(wl.n_new))
    assert oerr == K.KVQ_DEVERR_BLOCK_RANGE and int(err.item()) == K.KVQ_DEVERR_BLOCK_RANGE
    assert max_err(g.cpu().numpy(), o) <= ATOL
    # (2) a table two blocks short of sequence 0's length
    short = np.ascontiguousarray(wl.table[:, :wl.table.shape[1] - 2])
    err.zero_()
    pag = K.Paging(torch.from_numpy(wl.seq_lens).cuda(), block_tables=torch.from_numpy(short).cuda())
    g = K.kvq_prefill_attn(c.gcache, pag, to_dev_input(q, wl.dtype), cu, 40, scale,
                           dev_error=err)
    torch.cuda.synchronize()
    o, oerr = oracle.attention(c.ocache, oracle.Paging(short, False, wl.seq_lens), to_orc_input(q, wl.dtype), scale,
                               cu_q=wl.cu(wl.n_new))
    assert oerr == K.KVQ_DEVERR_TABLE_RANGE and int(err.item()) == K.KVQ_DEVERR_TABLE_RANGE
    assert np.all(np.isfinite(g.cpu().numpy()))
    assert max_err(g.cpu().numpy(), o) <= ATOL
