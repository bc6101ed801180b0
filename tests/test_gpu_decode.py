"""kvq_decode_attn on the GPU against the CPU oracle (max abs error 2e-3 in
fp32), plus metamorphic checks that need no oracle."""
import math

import numpy as np
import pytest
import torch

import kvq_inputs as gen
import oracle
from harness import (ATOL, assert_pools_equal, build_case, decode_gpu, decode_oracle, kvq, max_err, q_host,
                     to_dev_input, to_orc_input,
                     write_step)

pytestmark = pytest.mark.gpu


def _run(wl, splits=0, check_pool=True):
    c = build_case(wl)
    write_step(c)
    if check_pool:
        assert_pools_equal(c)
    q = q_host(wl)
    g = decode_gpu(c, q, num_splits=splits)
    o = decode_oracle(c, q)
    e = max_err(g, o)
    assert e <= ATOL, "max abs err %.3g" % e
    assert int(c.dev_err.item()) == 0
    return c, q, g, e


def test_decode_tiny_workload():
    _run(gen.tiny_int4(0))


def test_decode_llama_like_reduced():
    _run(gen.llama_int4(0, batch=6, ctx_lo=100, ctx_hi=2100, num_blocks=4000))


def test_decode_ernie_int2_reduced():
    _run(gen.ernie_int2(0, batch=5, median=1500, lo=64, hi=4000, num_blocks=1000))


def test_decode_qwen_int8_headwise_reduced():
    _run(gen.qwen_int8_headwise(0, batch=2, context=3000, window=700, sink=4))


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8, gen.MODE_INT4_STEGO,
                                  gen.MODE_INT8_TOKEN_HEAD, gen.MODE_FP8_TOKEN_HEAD])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 5, 8])
def test_decode_modes_dims_groups(mode, D, group):
    Hkv = 2
    wl = gen.custom(mode, Hkv * group, Hkv, D, 32, "bf16", seq_lens=[1, 31, 33, 250, 700], n_new=[1] * 5,
                    seed=7 * group + D + mode, outlier_frac=0.02)
    _run(wl)


@pytest.mark.parametrize("bs", [16, 64])
def test_decode_sliding_window_sentinels(bs):
    wl = gen.custom(gen.MODE_INT4, 8, 2, 128, bs, "bf16", seq_lens=[1500, 900, 40], n_new=[1, 1, 1],
                    headwise=True, window=[0, 300], sink=4, evict_outside_window=True, seed=21)
    _run(wl)


def test_decode_window_without_eviction():
    wl = gen.custom(gen.MODE_INT2, 10, 2, 128, 16, "f32", seq_lens=[700, 90], n_new=[1, 1],
                    window=[100, 33], sink=7, seed=8)
    _run(wl)


def test_decode_split_count_invariance():
    wl = gen.custom(gen.MODE_INT4, 16, 4, 128, 16, "bf16", seq_lens=[3000, 2000, 17], n_new=[1, 1, 1], seed=4)
    c, q, g0, _ = _run(wl)
    for s in (1, 3, 50):
        g = decode_gpu(c, q, num_splits=s)
        assert np.max(np.abs(g - g0)) <= 1e-5


def test_decode_headwise_identical_rows_bit_identical_to_uniform():
    """A head-wise table whose rows all equal the uniform row must give the
    very same output bits as the uniform table (legacy path unchanged)."""
    wl = gen.custom(gen.MODE_INT4, 16, 4, 128, 16, "bf16", seq_lens=[800, 333], n_new=[1, 1], seed=12)
    c = build_case(wl)
    write_step(c)
    q = q_host(wl)
    g_uni = decode_gpu(c, q)
    K = kvq()
    hw = np.repeat(wl.table, wl.num_kv_heads, axis=0)
    pag = K.Paging(torch.from_numpy(wl.seq_lens).cuda(), block_tables_headwise=torch.from_numpy(hw).cuda())
    g_hw = decode_gpu(c, q, paging=pag)
    assert np.array_equal(g_uni, g_hw)


def test_decode_evicted_pages_never_read():
    """Garbage in -1 pages must not change the result."""
    wl = gen.custom(gen.MODE_INT4, 8, 2, 128, 16, "bf16", seq_lens=[1200], n_new=[1], headwise=True,
                    window=[0, 200], sink=4, evict_outside_window=True, seed=30)
    c = build_case(wl)
    write_step(c)
    q = q_host(wl)
    g0 = decode_gpu(c, q)
    Hkv = wl.num_kv_heads
    rows = wl.table.reshape(wl.batch, Hkv, -1)
    for h in range(Hkv):
        live = set(int(x) for x in rows[:, h].ravel() if x >= 0)
        for b in range(wl.num_blocks):
            if b not in live:  # this head's page of block b is referenced by no row of head h
                c.gcache.k_pages[b, h] = 0x77
                c.gcache.v_pages[b, h] = 0x77
    g1 = decode_gpu(c, q)
    assert np.array_equal(g0, g1)


@pytest.mark.parametrize("batch", [17, 20])
def test_decode_pair_count_not_a_multiple_of_the_scan_width(batch):
    """136 or 160 (sequence, kv head) pairs: the stream kernel's prefix scan of
    the pairs' tile counts runs on 128 threads, so each scanning thread owns two
    pairs and the last ones own none.  Parity with the oracle, and a second call
    on the same inputs returns the same bits (the slices and the merge order are
    fixed, not scheduled)."""
    c, q, g, _ = _run(gen.llama_int4(0, batch=batch, ctx_lo=100, ctx_hi=1500, num_blocks=4000))
    assert np.array_equal(g, decode_gpu(c, q))


def test_decode_empty_and_zero_length():
    wl = gen.custom(gen.MODE_INT4, 4, 2, 64, 16, "f32", seq_lens=[5, 9], n_new=[1, 1], seed=2)
    c = build_case(wl)
    write_step(c)
    K = kvq()
    pag = K.Paging(torch.tensor([0, 9], dtype=torch.int32, device="cuda"),
                   block_tables=torch.from_numpy(wl.table).cuda())
    q = q_host(wl)
    g = decode_gpu(c, q, paging=pag)
    assert np.all(g[0] == 0.0)


def test_decode_full_size_llama_sampled():
    """The benchmark's workload at full size (64 sequences, 200k-block pool),
    in the launch configuration the bench times; sampled sequences checked
    against the oracle, the whole pool compared byte for byte."""
    wl = gen.llama_int4(0)
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)
    q = q_host(wl)
    g = decode_gpu(c, q)
    rows = np.array([0, 17, 31, 63], dtype=np.int32)
    o = decode_oracle(c, q, rows=rows)
    assert max_err(g[rows], o) <= ATOL
    assert np.all(np.isfinite(g))


def _full_size_sampled(wl, sample):
    """Full-size workload in the bench's launch configuration with only the
    sampled sequences known to the oracle: the GPU cache holds every sequence
    (host values for the sampled ones, device values for the rest); the
    sampled prefixes go first, in a call of their own, so that an INT8 first
    write defines the channel scales from the same tokens on both sides; the
    oracle writes only the sampled sequences.  Checks the sampled sequences'
    outputs against the oracle and their pages byte for byte."""
    K = kvq()
    dev = "cuda"
    B, pre = wl.batch, wl.prefix_lens
    sample = np.asarray(sample, dtype=np.int32)
    rest = np.setdiff1d(np.arange(B, dtype=np.int32), sample)
    signs_t = None if wl.signs is None else torch.from_numpy(wl.signs).to(dev)
    gc = K.PagedCache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, signs_t, dev)
    oc = oracle.Cache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.signs, 0)
    gc.k_pages.zero_()
    gc.v_pages.zero_()
    t_dev = torch.from_numpy(wl.table).to(dev)
    win = None if wl.window is None else torch.from_numpy(wl.window).to(dev)

    def gpag(lens):
        lt = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).to(dev)
        if wl.headwise:
            return K.Paging(lt, block_tables_headwise=t_dev, window_per_kv_head=win, sink_size=wl.sink)
        return K.Paging(lt, block_tables=t_dev, window_per_kv_head=win, sink_size=wl.sink)

    opag = lambda lens: oracle.Paging(wl.table, wl.headwise, np.ascontiguousarray(lens, np.int32), wl.window, wl.sink)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # 1) the sampled prefixes (host values), first on both sides
    counts = np.zeros(B, np.int32)
    counts[sample] = pre[sample]
    ks = np.concatenate([gen.kv_values_host(wl, "k", int(b), 0, int(pre[b])) for b in sample])
    vs = np.concatenate([gen.kv_values_host(wl, "v", int(b), 0, int(pre[b])) for b in sample])
    K.kvq_write(gc, gpag(pre), to_dev_input(ks, wl.dtype), to_dev_input(vs, wl.dtype),
                torch.from_numpy(wl.cu(counts)).to(dev), dev_error=err)
    assert oracle.write(oc, opag(pre), to_orc_input(ks, wl.dtype), to_orc_input(vs, wl.dtype), wl.cu(counts)) == 0
    del ks, vs
    # 2) the other prefixes, GPU only (device values), in groups of 16 sequences
    for g0 in range(0, len(rest), 16):
        grp = rest[g0:g0 + 16]
        counts = np.zeros(B, np.int32)
        counts[grp] = pre[grp]
        if counts.sum() == 0:
            continue
        kd = torch.cat([gen.kv_values_device(wl, "k", int(b), 0, int(pre[b]), dev) for b in grp if pre[b] > 0])
        vd = torch.cat([gen.kv_values_device(wl, "v", int(b), 0, int(pre[b]), dev) for b in grp if pre[b] > 0])
        K.kvq_write(gc, gpag(pre), kd, vd, torch.from_numpy(wl.cu(counts)).to(dev), dev_error=err)
        del kd, vd
    # 3) the step: one new token per sequence (host values for the sampled ones)
    parts_k, parts_v = [], []
    for b in range(B):
        if b in set(sample.tolist()):
            parts_k.append(to_dev_input(gen.kv_values_host(wl, "k", b, int(pre[b]), 1), wl.dtype))
            parts_v.append(to_dev_input(gen.kv_values_host(wl, "v", b, int(pre[b]), 1), wl.dtype))
        else:
            parts_k.append(gen.kv_values_device(wl, "k", b, int(pre[b]), 1, dev))
            parts_v.append(gen.kv_values_device(wl, "v", b, int(pre[b]), 1, dev))
    K.kvq_write(gc, gpag(wl.seq_lens), torch.cat(parts_k), torch.cat(parts_v),
                torch.from_numpy(wl.cu(wl.n_new)).to(dev), dev_error=err)
    counts = np.zeros(B, np.int32)
    counts[sample] = 1
    nk = np.concatenate([gen.kv_values_host(wl, "k", int(b), int(pre[b]), 1) for b in sample])
    nv = np.concatenate([gen.kv_values_host(wl, "v", int(b), int(pre[b]), 1) for b in sample])
    assert oracle.write(oc, opag(wl.seq_lens), to_orc_input(nk, wl.dtype), to_orc_input(nv, wl.dtype),
                        wl.cu(counts)) == 0
    # decode every sequence; compare the sampled ones
    q = q_host(wl)
    out = K.kvq_decode_attn(gc, gpag(wl.seq_lens), to_dev_input(q, wl.dtype), 1.0 / math.sqrt(wl.head_dim),
                            dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g = out.cpu().numpy()
    assert np.all(np.isfinite(g))
    o, oerr = oracle.attention(oc, opag(wl.seq_lens), to_orc_input(q, wl.dtype), 1.0 / math.sqrt(wl.head_dim),
                               rows=sample)
    assert oerr == 0
    assert max_err(g[sample], o) <= ATOL
    # the sampled sequences' pages, byte for byte
    gk, gv = gc.k_pages.cpu().numpy(), gc.v_pages.cpu().numpy()
    Hkv = wl.num_kv_heads
    for b in sample.tolist():
        nblk = (int(wl.seq_lens[b]) + wl.block_size - 1) // wl.block_size
        for h in range(Hkv):
            row = wl.table[b * Hkv + h] if wl.headwise else wl.table[b]
            for blk in row[:nblk]:
                if blk < 0:
                    continue
                assert np.array_equal(gk[blk, h], oc.k[blk, h]), "K page %d head %d differs" % (blk, h)
                assert np.array_equal(gv[blk, h], oc.v[blk, h]), "V page %d head %d differs" % (blk, h)
    if wl.mode == gen.MODE_INT8:
        assert np.array_equal(gc.ch_amax.cpu().numpy(), oc.amax)


def test_decode_full_size_ernie_int2_sampled():
    """Config 3 at full size: 96 sequences, log-normal contexts up to 128k,
    100k-block pool, INT2 with RHT."""
    _full_size_sampled(gen.ernie_int2(0), [0, 41, 95])


def test_decode_full_size_qwen_int8_headwise_sampled():
    """Config 5 at full size: 32 sequences at context 32768, INT8 channel
    scales from the first write, head-wise tables with -1 outside the sink
    and window of heads 4-7."""
    _full_size_sampled(gen.qwen_int8_headwise(0), [0, 19])


@pytest.mark.parametrize("mode", [gen.MODE_INT4_STEGO, gen.MODE_INT8_TOKEN_HEAD, gen.MODE_FP8_TOKEN_HEAD])
def test_decode_full_size_llama_other_rows_sampled(mode):
    """The Llama-like decode layer at full size (64 sequences, contexts up to
    8192, 200k-block pool) in the other row formats: INT4 with the zero point
    in the scale, INT8 and FP8 with one scale per token-head."""
    _full_size_sampled(gen.llama_int4(0, mode=mode), [0, 33, 63])


@pytest.mark.parametrize("group", [1, 4])
def test_decode_int4_d64_bs64(group):
    """INT4 decode at head_dim 64 / block_size 64: the Llama-like layer at the
    benchmark's reduced shape (group 4), and one kv head per q head."""
    if group == 4:
        wl = gen.llama_int4(0, head_dim=64, block_size=64, batch=6, ctx_lo=100, ctx_hi=2100, num_blocks=4000)
    else:
        wl = gen.custom(gen.MODE_INT4, 4, 4, 64, 64, "bf16", seq_lens=[1, 63, 64, 65, 1500], n_new=[1] * 5,
                        seed=19)
    _run(wl)


def test_decode_full_size_llama_d64_bs64_sampled():
    """The head_dim 64 / block_size 64 decode workload exactly as benchmarked
    (64 sequences, contexts up to 8192, 50k-block pool)."""
    _full_size_sampled(gen.llama_int4(0, num_blocks=50000, head_dim=64, block_size=64), [0, 33, 63])


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8_TOKEN_HEAD])
def test_decode_flags_bad_block_id_and_short_table(mode):
    """Device-side contract violations on the decode path: a table entry past
    the pool is skipped and sets KVQ_DEVERR_BLOCK_RANGE; a seq_len past
    max_blocks * block_size drops the keys beyond the table and sets
    KVQ_DEVERR_TABLE_RANGE.  The oracle skips the same keys and reports the
    same bits; the outputs agree within the usual bound."""
    K = kvq()
    wl = gen.custom(mode, 8, 2, 128, 16, "bf16", seq_lens=[700, 300, 50], n_new=[1, 1, 1], seed=23 + mode)
    c = build_case(wl)
    write_step(c)
    q = q_host(wl)
    scale = 1.0 / math.sqrt(wl.head_dim)
    bad = wl.table.copy()
    bad[0, 5] = wl.num_blocks + 1
    bad[1, 0] = 1 << 30
    short = np.ascontiguousarray(wl.table[:, :wl.table.shape[1] - 3])
    for table, bit in ((bad, K.KVQ_DEVERR_BLOCK_RANGE), (short, K.KVQ_DEVERR_TABLE_RANGE)):
        for splits in (0, 7):
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            pag = K.Paging(torch.from_numpy(wl.seq_lens).cuda(), block_tables=torch.from_numpy(table).cuda())
            g = K.kvq_decode_attn(c.gcache, pag, to_dev_input(q, wl.dtype), scale, num_splits=splits,
                                  dev_error=err)
            torch.cuda.synchronize()
            o, oerr = oracle.attention(c.ocache, oracle.Paging(table, False, wl.seq_lens), to_orc_input(q, wl.dtype),
                                       scale)
            assert oerr == bit and int(err.item()) == bit
            g = g.cpu().numpy()
            assert np.all(np.isfinite(g))
            assert max_err(g, o) <= ATOL
