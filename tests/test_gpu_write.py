"""kvq_write on the GPU against the CPU oracle: packed pages and INT8 channel
state must match byte for byte; pages the write must not touch (pre-filled
with 0xA5) must stay untouched."""
import numpy as np
import pytest

import kvq_inputs as gen
from harness import assert_pools_equal, build_case, write_step

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8, gen.MODE_INT4_STEGO,
                                  gen.MODE_INT8_TOKEN_HEAD, gen.MODE_FP8_TOKEN_HEAD])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_write_bit_exact(mode, D, bs, dtype):
    wl = gen.custom(mode, 8, 2, D, bs, dtype, seq_lens=[1, 37, 130, 64], n_new=[1, 5, 70, 64],
                    seed=3 + mode + D + bs, outlier_frac=0.02, outlier_factor=20.0)
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8, gen.MODE_INT4_STEGO,
                                  gen.MODE_INT8_TOKEN_HEAD, gen.MODE_FP8_TOKEN_HEAD])
def test_write_headwise_with_sentinels(mode):
    wl = gen.custom(mode, 10, 2, 128, 16, "bf16", seq_lens=[300, 210], n_new=[300, 210], headwise=True,
                    window=[0, 64], sink=4, evict_outside_window=True, seed=11)
    assert (wl.table == -1).any()
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)


def test_write_rht_off_and_no_outliers():
    wl = gen.custom(gen.MODE_INT4, 4, 4, 64, 16, "f32", seq_lens=[20, 33], n_new=[20, 33], rht=False,
                    outlier_frac=0.0, seed=5)
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)


def test_write_tiny_workload():
    wl = gen.tiny_int4(0)
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)


def test_write_edge_rows_constant_and_huge():
    """Constant rows (zero scale) and rows whose range overflows fp16
    (saturated scale) are both defined bit for bit."""
    import torch
    from harness import kvq, to_dev_input
    import oracle
    K = kvq()
    D, bs = 64, 16
    x = np.zeros((4, 1, D), np.float32)
    x[0] = 3.0
    x[1, 0, :] = np.linspace(-1e6, 1e6, D)
    x[2, 0, :] = -0.0
    x[3, 0, ::2] = 1e-30
    table = np.array([[0]], np.int32)
    lens = np.array([4], np.int32)
    for mode in (gen.MODE_INT4, gen.MODE_INT2):
        g = K.PagedCache(mode, 1, 1, bs, D, None)
        o = oracle.Cache(mode, 1, 1, bs, D)
        pag = K.Paging(torch.from_numpy(lens).cuda(), block_tables=torch.from_numpy(table).cuda())
        K.kvq_write(g, pag, to_dev_input(x, "f32"), to_dev_input(x, "f32"),
                    torch.tensor([0, 4], dtype=torch.int32, device="cuda"))
        oracle.write(o, oracle.Paging(table, False, lens), x, x, np.array([0, 4], np.int32))
        torch.cuda.synchronize()
        assert np.array_equal(g.k_pages.cpu().numpy(), o.k)


def test_write_flags_bad_block_ids():
    import torch
    from harness import kvq, to_dev_input
    K = kvq()
    g = K.PagedCache(gen.MODE_INT4, 2, 1, 16, 64, None)
    g.k_pages.fill_(0xA5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = to_dev_input(np.ones((3, 1, 64), np.float32), "f32")
    pag = K.Paging(torch.tensor([3], dtype=torch.int32, device="cuda"),
                   block_tables=torch.tensor([[7]], dtype=torch.int32, device="cuda"))
    K.kvq_write(g, pag, x, x, torch.tensor([0, 3], dtype=torch.int32, device="cuda"), dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & K.KVQ_DEVERR_BLOCK_RANGE
    assert bool((g.k_pages == 0xA5).all())
    err.zero_()
    pag2 = K.Paging(torch.tensor([2], dtype=torch.int32, device="cuda"),
                    block_tables=torch.tensor([[0]], dtype=torch.int32, device="cuda"))
    K.kvq_write(g, pag2, x, x, torch.tensor([0, 3], dtype=torch.int32, device="cuda"), dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & K.KVQ_DEVERR_SEQ_LEN


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT4_STEGO, gen.MODE_INT8_TOKEN_HEAD,
                                  gen.MODE_FP8_TOKEN_HEAD])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_write_long_chunk_bit_exact(mode, D, dtype):
    """Writes of 512 tokens or more take the batched kernel (four tokens per
    warp); a ragged count, a one-token sequence and evicted head-wise pages."""
    wl = gen.custom(mode, 4, 2, D, 16, dtype, seq_lens=[700, 300, 5], n_new=[650, 3, 1], headwise=True,
                    window=[0, 64], sink=4, evict_outside_window=True, seed=31 + mode + D)
    assert int(wl.n_new.sum()) >= 512 and int(wl.n_new.sum()) % 4 != 0 and (wl.table == -1).any()
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)
