"""kvq_write_decode_attn (the step's write done by the decode's query
preparation) against kvq_write followed by kvq_decode_attn: the same pages
byte for byte, the same output bits, the same error bits; and the output
against the oracle."""
import math

import numpy as np
import pytest
import torch

import kvq_inputs as gen
import oracle
from harness import ATOL, build_case, kvq, max_err, q_host, to_dev_input, to_orc_input

pytestmark = pytest.mark.gpu

MODES = [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT4_STEGO, gen.MODE_INT8_TOKEN_HEAD, gen.MODE_FP8_TOKEN_HEAD]


def _two_caches(wl):
    """Two GPU caches in the same state after the prefix write."""
    c = build_case(wl)
    K = kvq()
    twin = K.PagedCache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, c.gcache.rht_signs,
                        "cuda")
    twin.k_pages.copy_(c.gcache.k_pages)
    twin.v_pages.copy_(c.gcache.v_pages)
    return c, twin


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("D,bs,headwise", [(128, 16, False), (64, 64, True), (128, 32, True)])
def test_fused_write_decode_equals_write_then_decode(mode, D, bs, headwise):
    K = kvq()
    kw = dict(headwise=True, window=[0, 96], sink=4, evict_outside_window=True) if headwise else {}
    wl = gen.custom(mode, 8, 2, D, bs, "bf16", seq_lens=[700, 130, 3, 400], n_new=[1, 3, 2, 1],
                    seed=90 + mode + D + bs, outlier_frac=0.02, **kw)
    c, twin = _two_caches(wl)
    q = q_host(wl)
    qd = to_dev_input(q, wl.dtype)
    scale = 1.0 / math.sqrt(D)
    cu = torch.from_numpy(wl.cu(wl.n_new)).cuda()
    kn, vn = to_dev_input(c.k_new, wl.dtype), to_dev_input(c.v_new, wl.dtype)
    err_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    err_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.kvq_write(c.gcache, c.gpag, kn, vn, cu, dev_error=err_a)
    out_a = K.kvq_decode_attn(c.gcache, c.gpag, qd, scale, dev_error=err_a)
    out_b = K.kvq_write_decode_attn(twin, c.gpag, kn, vn, cu, qd, scale, dev_error=err_b)
    torch.cuda.synchronize()
    assert torch.equal(twin.k_pages, c.gcache.k_pages) and torch.equal(twin.v_pages, c.gcache.v_pages)
    assert torch.equal(out_a, out_b)
    assert int(err_a.item()) == int(err_b.item()) == 0
    # and the oracle, with its own write of the same tokens
    assert oracle.write(c.ocache, c.opag, to_orc_input(c.k_new, wl.dtype), to_orc_input(c.v_new, wl.dtype),
                        wl.cu(wl.n_new)) == 0
    assert np.array_equal(twin.k_pages.cpu().numpy(), c.ocache.k)
    assert np.array_equal(twin.v_pages.cpu().numpy(), c.ocache.v)
    o, oerr = oracle.attention(c.ocache, c.opag, to_orc_input(q, wl.dtype), scale)
    assert oerr == 0
    assert max_err(out_b.cpu().numpy(), o) <= ATOL


def test_fused_write_decode_error_bits():
    """A destination past the pool and a table shorter than the sequence:
    the fused call skips the same rows and sets the same bits."""
    K = kvq()
    wl = gen.custom(gen.MODE_INT4, 8, 2, 128, 16, "bf16", seq_lens=[300, 100], n_new=[1, 1], seed=97)
    c, twin = _two_caches(wl)
    bad = wl.table.copy()
    last = (int(wl.seq_lens[0]) - 1) // 16
    bad[0, last] = wl.num_blocks + 5
    pag = K.Paging(torch.from_numpy(wl.seq_lens).cuda(), block_tables=torch.from_numpy(bad).cuda())
    q = to_dev_input(q_host(wl), wl.dtype)
    cu = torch.from_numpy(wl.cu(wl.n_new)).cuda()
    kn, vn = to_dev_input(c.k_new, wl.dtype), to_dev_input(c.v_new, wl.dtype)
    err_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    err_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.kvq_write(c.gcache, pag, kn, vn, cu, dev_error=err_a)
    out_a = K.kvq_decode_attn(c.gcache, pag, q, 0.1, dev_error=err_a)
    out_b = K.kvq_write_decode_attn(twin, pag, kn, vn, cu, q, 0.1, dev_error=err_b)
    torch.cuda.synchronize()
    assert int(err_a.item()) == int(err_b.item()) == K.KVQ_DEVERR_BLOCK_RANGE
    assert torch.equal(twin.k_pages, c.gcache.k_pages) and torch.equal(out_a, out_b)
