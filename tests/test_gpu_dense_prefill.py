"""kvq_prefill_dense_attn (the tcgen05 prefill over dense bf16 K / V rows) on
the GPU against the CPU oracle's dense attention, alone and after kvq_gather
(the gather-then-dense-prefill strategy).  Same 2e-3 bound as the paged
attention: the rows reach the tensor cores exactly (bf16 values are fp16
values), the query is split into two fp16 terms and P s into two."""
import math

import numpy as np
import pytest
import torch

import kvq_inputs as gen
import oracle
from harness import ATOL, build_case, kvq, max_err, to_dev_input, to_orc_input, write_step

pytestmark = pytest.mark.gpu


def _dense_paging_orc(seq_lens, window=None, sink=0):
    B = len(seq_lens)
    return oracle.Paging(np.zeros((B, 1), np.int32), False, np.asarray(seq_lens, np.int32), window, sink)


def _run_dense(k_bits, v_bits, seq_lens, n_new, q32, Hkv, window=None, sink=0):
    """GPU and oracle dense prefill over bf16 rows (bit patterns) of every
    sequence's whole context, queries = the last n_b positions."""
    K = kvq()
    L = np.asarray(seq_lens, np.int32)
    n = np.asarray(n_new, np.int32)
    cu_kv = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    cu_q = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    D = q32.shape[-1]
    scale = 1.0 / math.sqrt(D)
    kd = torch.from_numpy(k_bits.view(np.int16)).cuda().view(torch.bfloat16)
    vd = torch.from_numpy(v_bits.view(np.int16)).cuda().view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    win_t = None if window is None else torch.from_numpy(np.asarray(window, np.int32)).cuda()
    out = K.kvq_prefill_dense_attn(kd, vd, torch.from_numpy(cu_kv).cuda(), torch.from_numpy(L).cuda(),
                                   to_dev_input(q32, "bf16"), torch.from_numpy(cu_q).cuda(), int(n.max()), scale,
                                   window_per_kv_head=win_t, sink_size=sink, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o, oerr = oracle.dense_attention(k_bits, v_bits, cu_kv, _dense_paging_orc(L, window, sink),
                                     to_orc_input(q32, "bf16"), scale, cu_q)
    assert oerr == 0
    return out.cpu().numpy(), o


def _bf16_rows(rng, rows, Hkv, D, outliers=True):
    x = rng.standard_normal((rows, Hkv, D)).astype(np.float32)
    if outliers:
        x[:, :, rng.integers(0, D, 2)] *= 10.0
    return gen.f32_to_bf16_bits(x)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 5, 8])
def test_dense_prefill_dims_groups(D, group):
    rng = np.random.default_rng(91 + D + group)
    Hkv = 2
    L, n = [70, 200, 15], [70, 77, 15]
    k = _bf16_rows(rng, sum(L), Hkv, D)
    v = _bf16_rows(rng, sum(L), Hkv, D)
    q = rng.standard_normal((sum(n), Hkv * group, D)).astype(np.float32)
    g, o = _run_dense(k, v, L, n, q, Hkv)
    assert max_err(g, o) <= ATOL
    assert np.all(np.isfinite(g))


def test_dense_prefill_window_and_sink():
    rng = np.random.default_rng(97)
    D, Hkv, G = 128, 2, 5
    L, n = [900, 400], [200, 150]
    k = _bf16_rows(rng, sum(L), Hkv, D)
    v = _bf16_rows(rng, sum(L), Hkv, D)
    q = rng.standard_normal((sum(n), Hkv * G, D)).astype(np.float32)
    g, o = _run_dense(k, v, L, n, q, Hkv, window=[0, 128], sink=4)
    assert max_err(g, o) <= ATOL


def test_dense_prefill_short_cu_kv_is_flagged():
    """A sequence whose dense rows are fewer than its length is skipped with
    the error bit; the others are computed."""
    K = kvq()
    rng = np.random.default_rng(99)
    D, Hkv = 64, 1
    k = torch.from_numpy(_bf16_rows(rng, 40, Hkv, D).view(np.int16)).cuda().view(torch.bfloat16)
    cu_kv = torch.tensor([0, 20, 30], dtype=torch.int32, device="cuda")       # sequence 1 holds 10 < 20 rows
    L = torch.tensor([20, 20], dtype=torch.int32, device="cuda")
    q = torch.zeros((4, 1, D), dtype=torch.bfloat16, device="cuda")
    cu_q = torch.tensor([0, 2, 4], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = K.kvq_prefill_dense_attn(k, k, cu_kv, L, q, cu_q, 2, 0.125, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == K.KVQ_DEVERR_SEQ_LEN
    assert np.all(np.isfinite(out[:2].cpu().numpy()))


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_FP8_TOKEN_HEAD])
def test_gather_then_dense_prefill(mode):
    """Write the chunk, gather every sequence's whole context to bf16, then
    the dense prefill of the chunk's queries; the oracle gathers, rounds to
    bf16 and attends on its own."""
    K = kvq()
    wl = gen.custom(mode, 8, 2, 128, 16, "bf16", seq_lens=[300, 150], n_new=[200, 150], step="prefill",
                    seed=17 + mode, outlier_frac=0.02)
    c = build_case(wl)
    write_step(c)
    cu_all = wl.cu(wl.seq_lens)
    n_all = int(cu_all[-1])
    gk, gv = K.kvq_gather(c.gcache, c.gpag, torch.from_numpy(cu_all).cuda(), n_all, out_dtype=torch.bfloat16,
                          dev_error=c.dev_err)
    q = gen.q_values_host(wl)
    cu_q = wl.cu(wl.n_new)
    out = K.kvq_prefill_dense_attn(gk, gv, torch.from_numpy(cu_all).cuda(), torch.from_numpy(wl.seq_lens).cuda(),
                                   to_dev_input(q, wl.dtype), torch.from_numpy(cu_q).cuda(), int(wl.n_new.max()),
                                   1.0 / math.sqrt(wl.head_dim), dev_error=c.dev_err)
    torch.cuda.synchronize()
    assert int(c.dev_err.cpu()[0]) == 0
    ok_, ov, err = oracle.gather(c.ocache, c.opag, cu_all)
    assert err == 0
    kb = gen.f32_to_bf16_bits(ok_.astype(np.float32))
    vb = gen.f32_to_bf16_bits(ov.astype(np.float32))
    o, oerr = oracle.dense_attention(kb, vb, cu_all, _dense_paging_orc(wl.seq_lens), to_orc_input(q, wl.dtype),
                                     1.0 / math.sqrt(wl.head_dim), cu_q)
    assert oerr == 0
    assert max_err(out.cpu().numpy(), o) <= ATOL


def test_gather_then_dense_prefill_full_size_sampled():
    """The chunked-prefill workload at full size (8192-token chunk over
    prefixes 0 / 4k / 16k / 60k), gathered and attended as the bench times
    it; sampled query rows against the oracle's own gather and attention."""
    K = kvq()
    wl = gen.prefill_int4(0)
    c = build_case(wl)
    write_step(c)
    cu_all = wl.cu(wl.seq_lens)
    gk, gv = K.kvq_gather(c.gcache, c.gpag, torch.from_numpy(cu_all).cuda(), int(cu_all[-1]),
                          out_dtype=torch.bfloat16, dev_error=c.dev_err)
    q = gen.q_values_host(wl)
    cu_q = wl.cu(wl.n_new)
    out = K.kvq_prefill_dense_attn(gk, gv, torch.from_numpy(cu_all).cuda(), torch.from_numpy(wl.seq_lens).cuda(),
                                   to_dev_input(q, wl.dtype), torch.from_numpy(cu_q).cuda(), int(wl.n_new.max()),
                                   1.0 / math.sqrt(wl.head_dim), dev_error=c.dev_err)
    torch.cuda.synchronize()
    assert int(c.dev_err.cpu()[0]) == 0
    rows = np.array([0, 2047, 2048 + 1000, 3 * 2048 + 2047], np.int32)
    ok_, ov, err = oracle.gather(c.ocache, c.opag, cu_all)
    assert err == 0
    kb = gen.f32_to_bf16_bits(ok_.astype(np.float32))
    vb = gen.f32_to_bf16_bits(ov.astype(np.float32))
    del ok_, ov
    o, oerr = oracle.dense_attention(kb, vb, cu_all, _dense_paging_orc(wl.seq_lens), to_orc_input(q, wl.dtype),
                                     1.0 / math.sqrt(wl.head_dim), cu_q, rows=rows)
    assert oerr == 0
    assert max_err(out.cpu().numpy()[rows], o) <= ATOL


@pytest.mark.parametrize("mode", [gen.MODE_INT4, gen.MODE_INT8_TOKEN_HEAD])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gather_full_precision_chunk_then_dense_prefill(mode, out_dtype):
    """The prefill variant that attends to the current chunk as given: the
    prefix gathered from the cache, the chunk's rows taken from the write's
    own inputs (kvq_gather_chunk), then the dense prefill; the oracle does
    the same on its own."""
    K = kvq()
    wl = gen.custom(mode, 8, 2, 128, 16, "bf16", seq_lens=[300, 150], n_new=[200, 150], step="prefill",
                    seed=23 + mode, outlier_frac=0.02)
    c = build_case(wl)
    write_step(c)
    cu_all = wl.cu(wl.seq_lens)
    cu_new = wl.cu(wl.n_new)
    kc, vc = to_dev_input(c.k_new, wl.dtype), to_dev_input(c.v_new, wl.dtype)
    gk, gv = K.kvq_gather(c.gcache, c.gpag, torch.from_numpy(cu_all).cuda(), int(cu_all[-1]), out_dtype=out_dtype,
                          dev_error=c.dev_err, k_chunk=kc, v_chunk=vc, cu_chunk=torch.from_numpy(cu_new).cuda())
    torch.cuda.synchronize()
    assert int(c.dev_err.cpu()[0]) == 0
    ok_, ov, err = oracle.gather_chunk(c.ocache, c.opag, cu_all, to_orc_input(c.k_new, wl.dtype),
                                       to_orc_input(c.v_new, wl.dtype), cu_new)
    assert err == 0
    # the chunk rows are copied exactly; the rest within the gather bound
    g = gk.float().cpu().numpy().astype(np.float64)
    for b in range(wl.batch):
        L, m = int(wl.seq_lens[b]), int(wl.n_new[b])
        rows = slice(int(cu_all[b]) + L - m, int(cu_all[b + 1]))
        assert np.array_equal(g[rows], ok_[rows])
    bound = 2.0 ** -22 * 128 * np.abs(ok_).max(axis=-1, keepdims=True) + (np.abs(ok_) * 2.0 ** -8 if out_dtype == torch.bfloat16 else 0)
    assert np.all(np.abs(g - ok_) <= bound)
    if out_dtype != torch.bfloat16:
        return
    q = gen.q_values_host(wl)
    out = K.kvq_prefill_dense_attn(gk, gv, torch.from_numpy(cu_all).cuda(), torch.from_numpy(wl.seq_lens).cuda(),
                                   to_dev_input(q, wl.dtype), torch.from_numpy(cu_new).cuda(), int(wl.n_new.max()),
                                   1.0 / math.sqrt(wl.head_dim), dev_error=c.dev_err)
    torch.cuda.synchronize()
    kb = gen.f32_to_bf16_bits(ok_.astype(np.float32))
    vb = gen.f32_to_bf16_bits(ov.astype(np.float32))
    o, oerr = oracle.dense_attention(kb, vb, cu_all, _dense_paging_orc(wl.seq_lens), to_orc_input(q, wl.dtype),
                                     1.0 / math.sqrt(wl.head_dim), cu_new)
    assert oerr == 0
    assert max_err(out.cpu().numpy(), o) <= ATOL
