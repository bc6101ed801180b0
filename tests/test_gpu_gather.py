"""kvq_gather on the GPU against the CPU oracle: rows read back through the
table, dequantised and mapped through the inverse RHT to dense K / V.

Tolerance (fp32 output): the dequantised value is one fp32 rounding away from
the exact one, and each of the log2(D) butterfly stages rounds partial sums no
larger than D max|x| of the row, so |gpu - oracle| <= 2^-22 D max|x_row|
(2x margin).  bf16 output adds half a bf16 spacing, 2^-8 |x|.  Rows the
table marks -1 must be exact zeros, and rows the mode represents exactly
must come back exactly.
"""
import math

import numpy as np
import pytest
import torch

import kvq_inputs as gen
import oracle
from harness import assert_pools_equal, build_case, kvq, write_step

pytestmark = pytest.mark.gpu

ALL_MODES = [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8, gen.MODE_INT4_STEGO, gen.MODE_INT8_TOKEN_HEAD,
             gen.MODE_FP8_TOKEN_HEAD]


def _gather_gpu(c, counts, out_dtype):
    K = kvq()
    cu = c.wl.cu(counts)
    k, v = K.kvq_gather(c.gcache, c.gpag, torch.from_numpy(cu).cuda(), int(cu[-1]), out_dtype=out_dtype,
                        dev_error=c.dev_err)
    torch.cuda.synchronize()
    assert int(c.dev_err.cpu()[0]) == 0
    return k.float().cpu().numpy().astype(np.float64), v.float().cpu().numpy().astype(np.float64)


def _assert_close(g, o, bf16):
    D = o.shape[-1]
    scale = np.abs(o).max(axis=-1, keepdims=True)
    bound = 2.0 ** -22 * D * scale
    if bf16:
        bound = bound + np.abs(o) * 2.0 ** -8
    bad = np.abs(g - o) > bound
    assert not bad.any(), "%d elements outside the bound, first at %s: gpu %r oracle %r" % (
        bad.sum(), tuple(np.argwhere(bad)[0]), g[bad][0], o[bad][0])


def _check_case(c, counts):
    ok_, ov, err = oracle.gather(c.ocache, c.opag, c.wl.cu(counts))
    assert err == 0
    for dt in (torch.float32, torch.bfloat16):
        gk, gv = _gather_gpu(c, counts, dt)
        _assert_close(gk, ok_, dt == torch.bfloat16)
        _assert_close(gv, ov, dt == torch.bfloat16)
    return ok_


@pytest.mark.parametrize("mode", ALL_MODES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 64])
def test_gather_modes_dims(mode, D, bs):
    wl = gen.custom(mode, 8, 2, D, bs, "bf16", seq_lens=[1, 37, 130, 64], n_new=[1, 5, 70, 64],
                    seed=5 + mode + D + bs, outlier_frac=0.02, outlier_factor=20.0)
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)
    _check_case(c, wl.seq_lens)                     # whole sequences
    _check_case(c, np.array([0, 3, 70, 1], np.int32))  # the last few positions of each


@pytest.mark.parametrize("mode", ALL_MODES)
def test_gather_headwise_sentinels_give_zero_rows(mode):
    wl = gen.custom(mode, 10, 2, 128, 16, "bf16", seq_lens=[300, 210], n_new=[300, 210], headwise=True,
                    window=[0, 64], sink=4, evict_outside_window=True, seed=13)
    assert (wl.table == -1).any()
    c = build_case(wl)
    write_step(c)
    ok_ = _check_case(c, wl.seq_lens)
    assert (np.abs(ok_).max(axis=-1) == 0).any()    # some rows were evicted


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT4_STEGO, gen.MODE_INT8_TOKEN_HEAD,
                                  gen.MODE_FP8_TOKEN_HEAD])
def test_gather_representable_rows_round_trip_exactly(mode):
    """Rows whose RHT is a grid row of the mode: written and gathered on the
    GPU, they come back bit for bit (fp32 output)."""
    from test_oracle_pins import _rotated_grid_rows
    K = kvq()
    rng = np.random.default_rng(71 + mode)
    D, bs, Hkv, T = 128, 16, 2, 50
    signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8)
    x = _rotated_grid_rows(rng, T * Hkv, D, mode, signs).reshape(T, Hkv, D)
    w = _rotated_grid_rows(rng, T * Hkv, D, mode, signs).reshape(T, Hkv, D)
    gc = K.PagedCache(mode, 8, Hkv, bs, D, torch.from_numpy(signs).cuda())
    table = torch.tensor([[5, 0, 7, 2]], dtype=torch.int32, device="cuda")
    pag = K.Paging(torch.tensor([T], dtype=torch.int32, device="cuda"), block_tables=table)
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.kvq_write(gc, pag, torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(), cu, dev_error=err)
    k, v = K.kvq_gather(gc, pag, cu, T, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(k.cpu().numpy(), x) and np.array_equal(v.cpu().numpy(), w)


def test_gather_flags_rows_it_cannot_locate():
    """More tokens than the sequence holds: error bit, zero rows."""
    K = kvq()
    wl = gen.custom(gen.MODE_INT4, 4, 2, 64, 16, "f32", seq_lens=[20], n_new=[20], seed=3)
    c = build_case(wl)
    write_step(c)
    pag = K.Paging(torch.tensor([5], dtype=torch.int32, device="cuda"), block_tables=torch.from_numpy(wl.table).cuda())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k, _ = K.kvq_gather(c.gcache, pag, torch.tensor([0, 8], dtype=torch.int32, device="cuda"), 8, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == K.KVQ_DEVERR_SEQ_LEN
    assert float(k.abs().max()) == 0.0


def test_gather_full_size_llama_sampled():
    """The Llama-like INT4 cache at full size (64 sequences, 200k-block pool):
    every sequence gathered in one call to bf16, as the bench times it;
    sampled sequences compared with the oracle."""
    K = kvq()
    wl = gen.llama_int4(0)
    c = build_case(wl)
    write_step(c)
    cu = wl.cu(wl.seq_lens)
    k, v = K.kvq_gather(c.gcache, c.gpag, torch.from_numpy(cu).cuda(), int(cu[-1]), out_dtype=torch.bfloat16,
                        dev_error=c.dev_err)
    torch.cuda.synchronize()
    assert int(c.dev_err.cpu()[0]) == 0
    sample = [0, 17, 63]
    counts = np.zeros(wl.batch, np.int32)
    counts[sample] = wl.seq_lens[sample]
    ok_, ov, err = oracle.gather(c.ocache, c.opag, wl.cu(counts))
    assert err == 0
    gk = torch.cat([k[int(cu[b]):int(cu[b + 1])] for b in sample]).float().cpu().numpy().astype(np.float64)
    gv = torch.cat([v[int(cu[b]):int(cu[b + 1])] for b in sample]).float().cpu().numpy().astype(np.float64)
    _assert_close(gk, ok_, True)
    _assert_close(gv, ov, True)


def test_gather_flags_bad_block_id_and_short_table():
    """A table entry past the pool and a position past max_blocks * block_size
    give zero rows and KVQ_DEVERR_BLOCK_RANGE / KVQ_DEVERR_TABLE_RANGE, as in
    the oracle; every other row is gathered as usual."""
    K = kvq()
    wl = gen.custom(gen.MODE_INT4, 4, 2, 64, 16, "f32", seq_lens=[100, 60], n_new=[100, 60], seed=13)
    c = build_case(wl)
    write_step(c)
    cu = wl.cu(wl.seq_lens)
    for kind, table, bit in (("block", None, K.KVQ_DEVERR_BLOCK_RANGE), ("short", None, K.KVQ_DEVERR_TABLE_RANGE)):
        if kind == "block":
            table = wl.table.copy()
            table[1, 2] = wl.num_blocks + 3
        else:
            table = np.ascontiguousarray(wl.table[:, :wl.table.shape[1] - 2])
        pag = K.Paging(torch.from_numpy(wl.seq_lens).cuda(), block_tables=torch.from_numpy(table).cuda())
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        k, v = K.kvq_gather(c.gcache, pag, torch.from_numpy(cu).cuda(), int(cu[-1]), dev_error=err)
        torch.cuda.synchronize()
        ok_, ov, oerr = oracle.gather(c.ocache, oracle.Paging(table, False, wl.seq_lens), cu)
        assert oerr == bit and int(err.item()) == bit
        gk = k.cpu().numpy().astype(np.float64)
        gv = v.cpu().numpy().astype(np.float64)
        zero = np.all(ok_ == 0.0, axis=(1, 2))
        assert zero.sum() >= 16 and np.all(gk[zero] == 0.0) and np.all(gv[zero] == 0.0)
        _assert_close(gk, ok_, False)
        _assert_close(gv, ov, False)
