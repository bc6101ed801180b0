"""Host-only checks of the C ABI: the library loads, exports every function
include/kvq.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:kvq_status|int32_t|const char\*)\s+(kvq_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def K():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "kvq_build_lib", os.path.join(ROOT, "sub_byte_quantized_write_gb300", "build_lib.py"))
    build_lib = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build_lib)
    build_lib.build()
    import sub_byte_quantized_write_gb300 as m
    return m


def test_header_declares_the_three_calls():
    names = _declared_functions()
    for n in ("kvq_write", "kvq_decode_attn", "kvq_prefill_attn", "kvq_gather", "kvq_gather_chunk",
              "kvq_prefill_dense_attn",
              "kvq_decode_workspace_size", "kvq_row_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(K):
    lib = ctypes.CDLL(K.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(lib, n), n
    assert lib.kvq_abi_version() == 1


def test_debug_library_exports_every_declared_symbol(K):
    """libkvq_debug.so (the -DKVQ_BOUNDS_CHECK build of the same sources)
    loads and exports the same calls."""
    path = os.path.join(os.path.dirname(K.LIB_PATH), "libkvq_debug.so")
    if not os.path.exists(path):
        pytest.skip("libkvq_debug.so not built")
    lib = ctypes.CDLL(path)
    for n in _declared_functions():
        assert hasattr(lib, n), n
    assert lib.kvq_abi_version() == 1


def test_row_bytes(K):
    assert K.kvq_row_bytes(K.KVQ_INT4_TOKEN_HEAD, 128) == 68
    assert K.kvq_row_bytes(K.KVQ_INT4_TOKEN_HEAD, 64) == 36
    assert K.kvq_row_bytes(K.KVQ_INT2_TOKEN_HEAD, 128) == 36
    assert K.kvq_row_bytes(K.KVQ_INT8_CHANNEL, 128) == 128
    assert K.kvq_row_bytes(K.KVQ_INT4_STEGO, 128) == 68   # same row as INT4: the pad holds the fp32 scale
    assert K.kvq_row_bytes(K.KVQ_INT8_TOKEN_HEAD, 128) == 132   # code bytes + fp32 scale
    assert K.kvq_row_bytes(K.KVQ_FP8_TOKEN_HEAD, 64) == 68
    assert K.kvq_row_bytes(K.KVQ_INT4_TOKEN_HEAD, 80) == 0


def _cache(K, **kw):
    base = dict(k_pages=4096, v_pages=8192, num_blocks=10, num_kv_heads=2, block_size=16, head_dim=128,
                mode=K.KVQ_INT4_TOKEN_HEAD, rht_signs=None, ch_amax=None, ch_amax_ready=None)
    base.update(kw)
    return K.KvqCache(**base)


def _paging(K, **kw):
    base = dict(block_tables=4096, block_tables_headwise=None, max_blocks=4, batch=2, seq_lens=4096,
                window_per_kv_head=None, sink_size=0)
    base.update(kw)
    return K.KvqPaging(**base)


def test_host_validation_statuses(K):
    L = K.lib()
    bref = ctypes.byref
    n, s = ctypes.c_size_t(0), ctypes.c_int32(0)
    # workspace sizing is pure host arithmetic
    assert L.kvq_decode_workspace_size(bref(_cache(K)), bref(_paging(K)), 8, 0, bref(n), bref(s)) == K.KVQ_OK
    assert n.value > 0 and s.value >= 1
    assert L.kvq_decode_workspace_size(bref(_cache(K)), bref(_paging(K)), 7, 0, bref(n), bref(s)) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_write(None, bref(_paging(K)), 16, 16, 1, 16, 1, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_write(bref(_cache(K, head_dim=96)), bref(_paging(K)), 16, 16, 1, 16, 1, None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_write(bref(_cache(K, block_size=8)), bref(_paging(K)), 16, 16, 1, 16, 1, None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_write(bref(_cache(K, k_pages=4097)), bref(_paging(K)), 16, 16, 1, 16, 1, None, None) == K.KVQ_ERR_INVALID_ARG
    both = _paging(K, block_tables_headwise=4096)
    assert L.kvq_write(bref(_cache(K)), bref(both), 16, 16, 1, 16, 1, None, None) == K.KVQ_ERR_INVALID_ARG
    neither = _paging(K, block_tables=None)
    assert L.kvq_write(bref(_cache(K)), bref(neither), 16, 16, 1, 16, 1, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_write(bref(_cache(K, mode=K.KVQ_INT8_CHANNEL)), bref(_paging(K)), 16, 16, 1, 16, 1, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_write(bref(_cache(K)), bref(_paging(K)), 16, 16, 7, 16, 1, None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_write(bref(_cache(K)), bref(_paging(K)), 16, 16, 1, 16, 0, None, None) == K.KVQ_OK  # no-op
    # Hq not a multiple of Hkv (GQA divisibility), too small workspace, group > 8
    assert L.kvq_decode_attn(bref(_cache(K)), bref(_paging(K)), 256, 1, 5, 0.1, 256, 256, 1 << 20, 0, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attn(bref(_cache(K)), bref(_paging(K)), 256, 1, 8, 0.1, 256, 256, 16, 0, None, None) == K.KVQ_ERR_WORKSPACE
    assert L.kvq_decode_attn(bref(_cache(K)), bref(_paging(K)), 256, 1, 18, 0.1, 256, 256, 1 << 30, 0, None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_prefill_attn(bref(_cache(K)), bref(_paging(K)), 256, 1, 8, None, 4, 4, 0.1, 256, None, None) == K.KVQ_ERR_INVALID_ARG
    assert b"cu_q" in L.kvq_last_error()
    # gather: NULL outputs, unsupported output type, misaligned output, empty call
    assert L.kvq_gather(bref(_cache(K)), bref(_paging(K)), 256, 4, None, 512, 0, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_gather(bref(_cache(K)), bref(_paging(K)), 256, 4, 512, 512, 7, None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_gather(bref(_cache(K)), bref(_paging(K)), 256, 4, 520, 512, 0, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_gather(bref(_cache(K)), bref(_paging(K)), 256, 0, None, None, 0, None, None) == K.KVQ_OK
    # gather with a chunk: k_chunk without v_chunk, and a bad chunk dtype
    assert L.kvq_gather_chunk(bref(_cache(K)), bref(_paging(K)), 256, 4, 512, None, 0, 256, 512, 512, 0,
                              None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_gather_chunk(bref(_cache(K)), bref(_paging(K)), 256, 4, 512, 512, 5, 256, 512, 512, 0,
                              None, None) == K.KVQ_ERR_UNSUPPORTED
    # dense prefill: a block table is refused, so are a bad head_dim and a group above 8
    assert L.kvq_prefill_dense_attn(512, 512, 256, 64, 2, 128, bref(_paging(K)), 256, 1, 8, 256, 4, 4, 0.1, 256,
                                    None, None) == K.KVQ_ERR_INVALID_ARG
    none = _paging(K)
    none.block_tables = None
    assert L.kvq_prefill_dense_attn(512, 512, 256, 64, 2, 96, bref(none), 256, 1, 8, 256, 4, 4, 0.1, 256,
                                    None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_prefill_dense_attn(512, 512, 256, 64, 2, 128, bref(none), 256, 1, 18, 256, 4, 4, 0.1, 256,
                                    None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_prefill_dense_attn(512, 512, 256, 0, 2, 128, bref(none), 256, 1, 8, 256, 4, 4, 0.1, 256,
                                    None, None) == K.KVQ_ERR_INVALID_ARG


def test_prefill_grid_limits_are_checked_on_the_host(K):
    """The prefill grid is (query tiles, kv heads, sequences): a kv-head count
    beyond the launch's y limit is refused before any launch, and the
    query-tile count is computed in 64 bits (INT32_MAX queries per sequence
    neither wraps nor reaches a launch here, because the kv-head check
    fails first)."""
    L = K.lib()
    bref = ctypes.byref
    big = _cache(K, num_kv_heads=70000)
    assert L.kvq_prefill_attn(bref(big), bref(_paging(K)), 256, 1, 70000, 256, 4, 0x7FFFFFFF, 0.1, 256,
                              None, None) == K.KVQ_ERR_UNSUPPORTED
    assert b"num_kv_heads" in L.kvq_last_error()
    none = _paging(K)
    none.block_tables = None
    assert L.kvq_prefill_dense_attn(512, 512, 256, 64, 70000, 128, bref(none), 256, 1, 70000, 256, 4, 4, 0.1, 256,
                                    None, None) == K.KVQ_ERR_UNSUPPORTED


def test_fused_write_decode_host_validation(K):
    """kvq_write_decode_attn refuses INT8 per-channel caches (their first
    write takes channel maxima over every token) and NULL write inputs."""
    L = K.lib()
    bref = ctypes.byref
    int8 = _cache(K, mode=K.KVQ_INT8_CHANNEL, ch_amax=4096, ch_amax_ready=4096)
    assert L.kvq_write_decode_attn(bref(int8), bref(_paging(K)), 4096, 4096, 1, 4096, 2, 256, 1, 8, 0.1, 256,
                                   256, 1 << 20, 0, None, None) == K.KVQ_ERR_UNSUPPORTED
    assert L.kvq_write_decode_attn(bref(_cache(K)), bref(_paging(K)), None, 4096, 1, 4096, 2, 256, 1, 8, 0.1, 256,
                                   256, 1 << 20, 0, None, None) == K.KVQ_ERR_INVALID_ARG
    assert L.kvq_write_decode_attn(bref(_cache(K)), bref(_paging(K)), 4096, 4096, 7, 4096, 2, 256, 1, 8, 0.1, 256,
                                   256, 1 << 20, 0, None, None) == K.KVQ_ERR_UNSUPPORTED
