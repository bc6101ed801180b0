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


def _write_rows_both_sides(mode, x, signs=None, bs=16):
    """Write the rows x [T, D] (one kv head, one sequence, fp32) through the
    library and through the oracle; return both K pools after asserting they
    are equal byte for byte (V gets -x)."""
    import torch
    import oracle
    from harness import kvq, to_dev_input
    K = kvq()
    T, D = x.shape
    nb = (T + bs - 1) // bs
    table = np.arange(nb, dtype=np.int32)[None, :]
    lens = np.array([T], np.int32)
    g = K.PagedCache(mode, nb, 1, bs, D, None if signs is None else torch.from_numpy(signs).cuda())
    g.k_pages.fill_(0xA5)
    g.v_pages.fill_(0xA5)
    o = oracle.Cache(mode, nb, 1, bs, D, signs, 0xA5)
    pag = K.Paging(torch.from_numpy(lens).cuda(), block_tables=torch.from_numpy(table).cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xk = np.ascontiguousarray(x[:, None, :], np.float32)
    xv = np.ascontiguousarray(-x[:, None, :], np.float32)
    K.kvq_write(g, pag, to_dev_input(xk, "f32"), to_dev_input(xv, "f32"),
                torch.tensor([0, T], dtype=torch.int32, device="cuda"), dev_error=err)
    assert oracle.write(o, oracle.Paging(table, False, lens), xk, xv, np.array([0, T], np.int32)) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    gk, gv = g.k_pages.cpu().numpy(), g.v_pages.cpu().numpy()
    assert np.array_equal(gk, o.k) and np.array_equal(gv, o.v)
    if mode == gen.MODE_INT8:
        assert np.array_equal(g.ch_amax.cpu().numpy(), o.amax)
    return gk[:, 0].reshape(nb * bs, -1)[:T]


@pytest.mark.parametrize("bits,D,rht", [(4, 64, False), (4, 128, True), (2, 64, False), (2, 128, True)])
def test_write_ties_round_half_to_even_asymmetric(bits, D, rht):
    """Elements at M + (k + 1/2) S get the even code on the GPU as in the
    oracle (hand-worked codes in tests/tie_rows.py), RHT off and on."""
    import oracle
    import tie_rows
    mode = gen.MODE_INT4 if bits == 4 else gen.MODE_INT2
    y, codes = tie_rows.asym_row(bits, D)
    signs = None
    x = y
    if rht:
        rng = np.random.default_rng(71 + D)
        signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8)
        x = tie_rows.pre_rotate(y, signs)
    rows = _write_rows_both_sides(mode, np.stack([x, x[::-1].copy()]), signs)
    data = D * bits // 8
    assert np.array_equal(oracle.unpack_codes(mode, rows[0, :data], D), codes)


@pytest.mark.parametrize("D", [64, 128])
def test_write_ties_round_half_to_even_stego(D):
    import oracle
    import tie_rows
    x, codes = tie_rows.stego_row(D)
    rows = _write_rows_both_sides(gen.MODE_INT4_STEGO, x[None, :])
    assert rows[0, D // 2:D // 2 + 4].tolist() == tie_rows.STEGO_PAD
    assert np.array_equal(oracle.unpack_codes(gen.MODE_INT4_STEGO, rows[0, :D // 2], D), codes)


def test_write_ties_round_half_to_even_int8_channel():
    import tie_rows
    D = 64
    x, codes = tie_rows.int8_channel_tokens(D)
    rows = _write_rows_both_sides(gen.MODE_INT8, x)
    assert np.array_equal(rows.view(np.int8).astype(np.int64), codes)


def test_write_ties_round_half_to_even_byte_token_head():
    """The 8-bit token-head rows whose scale is exactly 1: INT8 ties 0.5, 1.5,
    2.5, -2.5 and E4M3 ties 17 and 19 (spacing 2 in [16, 32))."""
    D = 64
    x = np.zeros((2, D), np.float32)
    x[0, :8] = [127, -63.5, 0.5, 1.5, 2.5, -2.5, -127, 3.0]
    x[1, :8] = [127, -0.5, -1.5, 63.5, 64.5, 4.5, 5.5, 6.5]
    rows = _write_rows_both_sides(gen.MODE_INT8_TOKEN_HEAD, x)
    assert rows[0, :8].view(np.int8).tolist() == [127, -64, 0, 2, 2, -2, -127, 3]
    assert rows[1, :8].view(np.int8).tolist() == [127, 0, -2, 64, 64, 4, 6, 6]
    assert rows[0, D:].tolist() == [0x00, 0x00, 0x80, 0x3F]
    x = np.zeros((1, D), np.float32)
    x[0, :10] = [448, 1.0, 0.5, -2.0, 17.0, 19.0, 2.0 ** -9, 3 * 2.0 ** -10, -0.0, -448]
    rows = _write_rows_both_sides(gen.MODE_FP8_TOKEN_HEAD, x)
    assert rows[0, :10].tolist() == [0x7E, 0x38, 0x30, 0xC0, 0x58, 0x5A, 0x01, 0x02, 0x80, 0xFE]
