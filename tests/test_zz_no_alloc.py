"""kvq_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory (e.g. a plugin inside a framework that owns all device
memory, or a path that must not pay an allocation's synchronisation).  It
must give the same output as kvq_decode_attn with a caller workspace, call
after call, while its partials live in the library's one static scratch
array.  This file is collected last so that a failure here does not hide the
other tests' results."""
import ctypes
import math

import numpy as np
import pytest
import torch

import kvq_inputs as gen
from harness import ATOL, build_case, kvq, q_host, to_dev_input, write_step

pytestmark = pytest.mark.gpu


def _noalloc_via_c_abi(K, cache, paging, q, scale, out, num_splits=0):
    cs, ps = cache.struct(), paging.struct()
    st = K.lib().kvq_decode_attn_noalloc(ctypes.byref(cs), ctypes.byref(ps), q.data_ptr(), K.KVQ_BF16
                                         if q.dtype == torch.bfloat16 else K.KVQ_F32, q.shape[1],
                                         ctypes.c_float(scale), out.data_ptr(), num_splits, None,
                                         torch.cuda.current_stream().cuda_stream)
    return st


def test_noalloc_decode_matches_workspace_decode_twice():
    K = kvq()
    wl = gen.llama_int4(0, batch=8, ctx_lo=200, ctx_hi=3000, num_blocks=3000)
    c = build_case(wl)
    write_step(c)
    q = to_dev_input(q_host(wl), wl.dtype)
    scale = 1.0 / math.sqrt(wl.head_dim)
    ref = K.kvq_decode_attn(c.gcache, c.gpag, q, scale)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_via_c_abi(K, c.gcache, c.gpag, q, scale, out) == K.KVQ_OK
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert float((out - ref).abs().max()) <= ATOL
    # a second, differently shaped call reuses the same scratch
    wl2 = gen.custom(gen.MODE_INT2, 10, 2, 128, 64, "bf16", seq_lens=[900, 40, 2500], n_new=[1, 1, 1], seed=3)
    c2 = build_case(wl2)
    write_step(c2)
    q2 = to_dev_input(q_host(wl2), wl2.dtype)
    ref2 = K.kvq_decode_attn(c2.gcache, c2.gpag, q2, scale)
    out2 = torch.empty_like(ref2)
    assert _noalloc_via_c_abi(K, c2.gcache, c2.gpag, q2, scale, out2) == K.KVQ_OK
    torch.cuda.synchronize()
    assert float((out2 - ref2).abs().max()) <= ATOL


def test_noalloc_forced_split_count_matches_workspace_decode():
    """A forced split count (num_splits > 0) takes the same clamping and the
    same partial-record layout in the static scratch as in a caller
    workspace: two calls in a row against kvq_decode_attn with that count."""
    K = kvq()
    wl = gen.custom(gen.MODE_INT4, 16, 4, 128, 16, "bf16", seq_lens=[3000, 2000, 17], n_new=[1, 1, 1], seed=4)
    c = build_case(wl)
    write_step(c)
    q = to_dev_input(q_host(wl), wl.dtype)
    scale = 1.0 / math.sqrt(wl.head_dim)
    for splits in (4, 4, 50):
        ref = K.kvq_decode_attn(c.gcache, c.gpag, q, scale, num_splits=splits)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_via_c_abi(K, c.gcache, c.gpag, q, scale, out, num_splits=splits) == K.KVQ_OK
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert float((out - ref).abs().max()) <= ATOL


def test_noalloc_rejects_oversized_calls():
    """A batch large enough that its partials and query images exceed the
    static scratch is refused before any launch."""
    K = kvq()
    B, Hkv, Hq = 4096, 8, 64
    wl = gen.custom(gen.MODE_INT4, Hq, Hkv, 128, 16, "bf16", seq_lens=[16] * 4, n_new=[1] * 4, seed=1)
    c = build_case(wl)
    big = K.Paging(torch.full((B,), 16, dtype=torch.int32, device="cuda"),
                   block_tables=torch.zeros((B, 1), dtype=torch.int32, device="cuda"))
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    need, _ = K.kvq_decode_workspace_size(c.gcache, big, Hq)
    assert need > (32 << 20)
    assert _noalloc_via_c_abi(K, c.gcache, big, q, 0.1, out) == K.KVQ_ERR_WORKSPACE
    assert b"static scratch" in K.lib().kvq_last_error()
