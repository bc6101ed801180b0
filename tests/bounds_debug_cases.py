"""Parity cases run through libkvq_debug.so (KVQ_BOUNDS_CHECK=1): the same
kernels with device-side checks on every index they compute against its
buffer (stream-K record indices, query-image and tile-start indices, table
indices, page-chunk offsets, destination rows, prefill query and output rows).
Each case must match the oracle as the release library does and leave the
KVQ_DEVERR_BOUNDS bit clear.  Run by tests/test_gpu_bounds_debug.py in a
child process (the library is chosen when the package is imported)."""
import math
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import kvq_inputs as gen  # noqa: E402
import oracle  # noqa: E402
from harness import (ATOL, assert_pools_equal, build_case, decode_gpu, decode_oracle, kvq, max_err,  # noqa: E402
                     prefill_gpu, prefill_oracle, q_host, to_dev_input, to_orc_input, write_step)

K = kvq()
assert K.BOUNDS_CHECK and K.LIB_NAME == "libkvq_debug.so", "the debug library is not loaded"
MODES = [gen.MODE_INT4, gen.MODE_INT2, gen.MODE_INT8, gen.MODE_INT4_STEGO, gen.MODE_INT8_TOKEN_HEAD,
         gen.MODE_FP8_TOKEN_HEAD]
done = []


def clear(c):
    e = int(c.dev_err.item())
    assert e & K.KVQ_DEVERR_BOUNDS == 0, "bounds check failed (dev_error %d)" % e
    assert e == 0, "dev_error %d" % e


def decode_case(wl, splits=0):
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)
    q = q_host(wl)
    g = decode_gpu(c, q, num_splits=splits)
    assert max_err(g, decode_oracle(c, q)) <= ATOL
    clear(c)


def prefill_case(wl):
    c = build_case(wl)
    write_step(c)
    assert_pools_equal(c)
    q = q_host(wl)
    assert max_err(prefill_gpu(c, q), prefill_oracle(c, q)) <= ATOL
    clear(c)


# decode: every mode, both head sizes, GQA groups 1 / 4 / 5 (one and two MMA N-tiles)
for mode in MODES:
    for D in (64, 128):
        for group in (1, 4, 5):
            decode_case(gen.custom(mode, 2 * group, 2, D, 16, "bf16", seq_lens=[300, 1000, 17], n_new=[1, 1, 1],
                                   seed=mode + D + group, outlier_frac=0.02))
    done.append("decode mode %d" % mode)
# head-wise tables with evicted blocks, window + sink; 64-row pages at D = 64; forced split counts
decode_case(gen.custom(gen.MODE_INT4, 8, 2, 128, 16, "bf16", seq_lens=[900, 300, 75], n_new=[1, 1, 1], headwise=True,
                       window=[0, 64], sink=4, evict_outside_window=True, seed=3))
decode_case(gen.custom(gen.MODE_INT4, 16, 4, 64, 64, "bf16", seq_lens=[2100, 100, 640], n_new=[1, 1, 1], seed=4))
for s in (1, 3, 50):
    decode_case(gen.custom(gen.MODE_INT2, 10, 2, 128, 64, "bf16", seq_lens=[3000, 70], n_new=[1, 1], seed=5), splits=s)
done.append("decode head-wise / D64 bs64 / forced splits")

# the Llama-like decode layer at full size (64 sequences, 8 kv heads), sampled rows
wl = gen.llama_int4(0, num_blocks=40000)
c = build_case(wl)
write_step(c)
q = q_host(wl)
g = decode_gpu(c, q)
rows = np.array([0, 17, 40, 63])
o, err = oracle.attention(c.ocache, c.opag, to_orc_input(q, wl.dtype), 1.0 / math.sqrt(wl.head_dim), rows=rows)
assert err == 0 and max_err(g[rows], o) <= ATOL
clear(c)
done.append("full-size decode")

# fused write + decode and the allocation-free decode
wl = gen.custom(gen.MODE_INT4, 8, 2, 128, 16, "bf16", seq_lens=[700, 130, 3, 400], n_new=[1, 3, 2, 1], seed=6)
c = build_case(wl)
qd = to_dev_input(q_host(wl), wl.dtype)
cu = torch.from_numpy(wl.cu(wl.n_new)).cuda()
out = K.kvq_write_decode_attn(c.gcache, c.gpag, to_dev_input(c.k_new, wl.dtype), to_dev_input(c.v_new, wl.dtype), cu,
                              qd, 1 / math.sqrt(128), dev_error=c.dev_err)
out2 = K.kvq_decode_attn_noalloc(c.gcache, c.gpag, qd, 1 / math.sqrt(128), dev_error=c.dev_err)
torch.cuda.synchronize()
assert oracle.write(c.ocache, c.opag, to_orc_input(c.k_new, wl.dtype), to_orc_input(c.v_new, wl.dtype),
                    wl.cu(wl.n_new)) == 0
assert_pools_equal(c)
o = decode_oracle(c, q_host(wl))
assert max_err(out.cpu().numpy(), o) <= ATOL and max_err(out2.cpu().numpy(), o) <= ATOL
clear(c)
done.append("fused write + decode, no-alloc decode")

# prefill: every mode, both head sizes, head-wise eviction; the chunk write of 8192 tokens (batched write)
for mode in MODES:
    for D in (64, 128):
        prefill_case(gen.custom(mode, 10, 2, D, 16, "bf16", seq_lens=[70, 200, 15], n_new=[70, 77, 15], step="prefill",
                                seed=10 + mode + D, outlier_frac=0.02))
prefill_case(gen.custom(gen.MODE_INT8, 8, 2, 128, 16, "bf16", seq_lens=[900, 300, 75], n_new=[400, 300, 60],
                        headwise=True, window=[0, 64], sink=4, evict_outside_window=True, step="prefill", seed=11))
wl = gen.prefill_int4(0, prefixes=(0, 300, 4000, 100), chunk=2048, num_blocks=2000)
c = build_case(wl)
write_step(c)
assert_pools_equal(c)
clear(c)
done.append("prefill, batched chunk write")

# gather (dense bf16 rows of every cached position) and the dense prefill over them
wl = gen.custom(gen.MODE_INT4, 8, 2, 128, 16, "bf16", seq_lens=[300, 90], n_new=[120, 90], step="prefill", seed=12)
c = build_case(wl)
write_step(c)
cu_all = torch.from_numpy(wl.cu(wl.seq_lens)).cuda()
n_all = int(wl.seq_lens.sum())
kd, vd = K.kvq_gather(c.gcache, c.gpag, cu_all, n_all, out_dtype=torch.float32, dev_error=c.dev_err)
ko, vo, gerr = oracle.gather(c.ocache, c.opag, wl.cu(wl.seq_lens))
assert gerr == 0
# fp32 rows against the oracle's doubles: a few ulps of the largest magnitude
for g_, o_ in ((kd, ko), (vd, vo)):
    assert np.max(np.abs(g_.cpu().numpy() - o_)) <= 2.0 ** -20 * 128 * max(1.0, float(np.max(np.abs(o_))))
kb, vb = K.kvq_gather(c.gcache, c.gpag, cu_all, n_all, out_dtype=torch.bfloat16, dev_error=c.dev_err)
q = q_host(wl)
cu = torch.from_numpy(wl.cu(wl.n_new)).cuda()
g = K.kvq_prefill_dense_attn(kb, vb, cu_all, c.gpag.seq_lens, to_dev_input(q, wl.dtype), cu, int(wl.n_new.max()),
                             1 / math.sqrt(128), dev_error=c.dev_err)
torch.cuda.synchronize()
# the dense oracle over the same bf16 rows (the oracle's own gather, rounded to bf16)
kbits = gen.f32_to_bf16_bits(ko.astype(np.float32))
vbits = gen.f32_to_bf16_bits(vo.astype(np.float32))
o, oerr = oracle.dense_attention(kbits, vbits, wl.cu(wl.seq_lens), oracle.Paging(np.zeros((wl.batch, 1), np.int32), False, wl.seq_lens),
                                 to_orc_input(q, wl.dtype), 1 / math.sqrt(128), wl.cu(wl.n_new))
assert oerr == 0 and max_err(g.cpu().numpy(), o) <= ATOL
clear(c)
done.append("gather, dense prefill")

# a contract violation still reports its own bit, not a bounds failure
wl = gen.custom(gen.MODE_INT4, 8, 2, 128, 16, "bf16", seq_lens=[300, 100], n_new=[1, 1], seed=13)
c = build_case(wl)
write_step(c)
bad = wl.table.copy()
bad[0, 3] = wl.num_blocks + 9
pag = K.Paging(torch.from_numpy(wl.seq_lens).cuda(), block_tables=torch.from_numpy(bad).cuda())
K.kvq_decode_attn(c.gcache, pag, to_dev_input(q_host(wl), wl.dtype), 0.1, dev_error=c.dev_err)
torch.cuda.synchronize()
assert int(c.dev_err.item()) == K.KVQ_DEVERR_BLOCK_RANGE
done.append("block id past the pool")

print("BOUNDS-DEBUG OK:", "; ".join(done))
