"""Python binding of libkvq: a paged KV cache in dynamic low-bit form on GB300.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, turned into raw pointers and handed to the C ABI declared in
``include/kvq.h``.  Every step of the write and attention paths runs in the
library's CUDA kernels; there is no fallback.  If ``libkvq.so`` has not been
built, importing this package raises ImportError.

Names mirror the C calls: ``kvq_write``, ``kvq_gather``, ``kvq_prefill_dense_attn``, ``kvq_decode_attn``,
``kvq_write_decode_attn``,
``kvq_decode_attn_noalloc``, ``kvq_prefill_attn``, ``kvq_decode_workspace_size``,
``kvq_row_bytes``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVQ_BOUNDS_CHECK=1 loads the debug library: the same kernels with device-side
# bounds checks on their computed indices (a failure sets KVQ_DEVERR_BOUNDS).
BOUNDS_CHECK = os.environ.get("KVQ_BOUNDS_CHECK", "0") == "1"
LIB_NAME = "libkvq_debug.so" if BOUNDS_CHECK else "libkvq.so"
LIB_PATH = os.path.join(_HERE, LIB_NAME)

if not os.path.exists(LIB_PATH):
    raise ImportError("%s is not built: run `python sub_byte_quantized_write_gb300/build_lib.py` "
                      "(or __graft_entry__.build()) first" % LIB_NAME)

_lib = ctypes.CDLL(LIB_PATH)

KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CUDA, KVQ_ERR_WORKSPACE = 0, 1, 2, 3, 4
KVQ_INT4_TOKEN_HEAD, KVQ_INT2_TOKEN_HEAD, KVQ_INT8_CHANNEL, KVQ_INT4_STEGO = 0, 1, 2, 3
KVQ_INT8_TOKEN_HEAD, KVQ_FP8_TOKEN_HEAD = 4, 5
KVQ_F32, KVQ_BF16 = 0, 1
KVQ_DEVERR_BLOCK_RANGE, KVQ_DEVERR_TABLE_RANGE, KVQ_DEVERR_SEQ_LEN, KVQ_DEVERR_TIMEOUT = 1, 2, 4, 8
KVQ_DEVERR_BOUNDS = 16  # debug library only


class KvqCache(ctypes.Structure):
    _fields_ = [("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("rht_signs", ctypes.c_void_p),
                ("ch_amax", ctypes.c_void_p), ("ch_amax_ready", ctypes.c_void_p)]


class KvqPaging(ctypes.Structure):
    _fields_ = [("block_tables", ctypes.c_void_p), ("block_tables_headwise", ctypes.c_void_p),
                ("max_blocks", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("window_per_kv_head", ctypes.c_void_p),
                ("sink_size", ctypes.c_int32)]


_P, _I = ctypes.c_void_p, ctypes.c_int32
_CP, _PP = ctypes.POINTER(KvqCache), ctypes.POINTER(KvqPaging)
_lib.kvq_row_bytes.argtypes, _lib.kvq_row_bytes.restype = [_I, _I], _I
_lib.kvq_abi_version.argtypes, _lib.kvq_abi_version.restype = [], _I
_lib.kvq_status_string.argtypes, _lib.kvq_status_string.restype = [_I], ctypes.c_char_p
_lib.kvq_last_error.argtypes, _lib.kvq_last_error.restype = [], ctypes.c_char_p
_lib.kvq_write.argtypes = [_CP, _PP, _P, _P, _I, _P, _I, _P, _P]
_lib.kvq_write.restype = _I
_lib.kvq_gather.argtypes = [_CP, _PP, _P, _I, _P, _P, _I, _P, _P]
_lib.kvq_gather.restype = _I
_lib.kvq_gather_chunk.argtypes = [_CP, _PP, _P, _I, _P, _P, _I, _P, _P, _P, _I, _P, _P]
_lib.kvq_gather_chunk.restype = _I
_lib.kvq_decode_workspace_size.argtypes = [_CP, _PP, _I, _I, ctypes.POINTER(ctypes.c_size_t),
                                           ctypes.POINTER(ctypes.c_int32)]
_lib.kvq_decode_workspace_size.restype = _I
_lib.kvq_decode_attn.argtypes = [_CP, _PP, _P, _I, _I, ctypes.c_float, _P, _P, ctypes.c_size_t, _I, _P, _P]
_lib.kvq_decode_attn.restype = _I
_lib.kvq_write_decode_attn.argtypes = [_CP, _PP, _P, _P, _I, _P, _I, _P, _I, _I, ctypes.c_float, _P, _P,
                                       ctypes.c_size_t, _I, _P, _P]
_lib.kvq_write_decode_attn.restype = _I
_lib.kvq_decode_attn_noalloc.argtypes = [_CP, _PP, _P, _I, _I, ctypes.c_float, _P, _I, _P, _P]
_lib.kvq_decode_attn_noalloc.restype = _I
_lib.kvq_prefill_attn.argtypes = [_CP, _PP, _P, _I, _I, _P, _I, _I, ctypes.c_float, _P, _P, _P]
_lib.kvq_prefill_attn.restype = _I
_lib.kvq_prefill_dense_attn.argtypes = [_P, _P, _P, _I, _I, _I, _PP, _P, _I, _I, _P, _I, _I, ctypes.c_float, _P, _P,
                                        _P]
_lib.kvq_prefill_dense_attn.restype = _I


class KvqError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__("%s: %s" % (_lib.kvq_status_string(status).decode(), _lib.kvq_last_error().decode()))


def _check(status: int):
    if status != KVQ_OK:
        raise KvqError(status)


def lib() -> ctypes.CDLL:
    return _lib


def kvq_row_bytes(mode: int, head_dim: int) -> int:
    return _lib.kvq_row_bytes(mode, head_dim)


def _dev_ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _qdtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KVQ_F32
    if t.dtype == torch.bfloat16:
        return KVQ_BF16
    raise ValueError("q/k/v must be float32 or bfloat16")


class PagedCache:
    """One layer's paged cache: uint8 K and V pools of shape
    [num_blocks, num_kv_heads, block_size, row_bytes] (allocated here, as
    torch.uint8, unless given), the RHT sign vector and, for INT8, the
    per-channel amax state."""

    def __init__(self, mode: int, num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
                 rht_signs: Optional[torch.Tensor] = None, device="cuda", k_pages=None, v_pages=None,
                 ch_amax=None, ch_amax_ready=None):
        self.mode, self.num_blocks, self.num_kv_heads = mode, num_blocks, num_kv_heads
        self.block_size, self.head_dim = block_size, head_dim
        self.row_bytes = kvq_row_bytes(mode, head_dim)
        if self.row_bytes == 0:
            raise ValueError("unsupported mode/head_dim")
        shape = (num_blocks, num_kv_heads, block_size, self.row_bytes)
        self.k_pages = k_pages if k_pages is not None else torch.zeros(shape, dtype=torch.uint8, device=device)
        self.v_pages = v_pages if v_pages is not None else torch.zeros(shape, dtype=torch.uint8, device=device)
        self.rht_signs = rht_signs
        if mode == KVQ_INT8_CHANNEL:
            self.ch_amax = ch_amax if ch_amax is not None else torch.zeros(
                (2, num_kv_heads, head_dim), dtype=torch.float32, device=device)
            self.ch_amax_ready = ch_amax_ready if ch_amax_ready is not None else torch.zeros(
                1, dtype=torch.int32, device=device)
        else:
            self.ch_amax = None
            self.ch_amax_ready = None

    def struct(self) -> KvqCache:
        return KvqCache(_dev_ptr(self.k_pages, torch.uint8, "k_pages"), _dev_ptr(self.v_pages, torch.uint8, "v_pages"),
                        self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim, self.mode,
                        _dev_ptr(self.rht_signs, torch.int8, "rht_signs"),
                        _dev_ptr(self.ch_amax, torch.float32, "ch_amax"),
                        _dev_ptr(self.ch_amax_ready, torch.int32, "ch_amax_ready"))


class Paging:
    """Block table (uniform [batch, max_blocks] or head-wise
    [batch * num_kv_heads, max_blocks], int32, -1 = evicted), seq_lens [batch]
    and the optional per-kv-head sliding window plus sink size."""

    def __init__(self, seq_lens: torch.Tensor, block_tables: Optional[torch.Tensor] = None,
                 block_tables_headwise: Optional[torch.Tensor] = None,
                 window_per_kv_head: Optional[torch.Tensor] = None, sink_size: int = 0):
        self.seq_lens = seq_lens
        self.block_tables = block_tables
        self.block_tables_headwise = block_tables_headwise
        self.window_per_kv_head = window_per_kv_head
        self.sink_size = int(sink_size)
        t = block_tables if block_tables is not None else block_tables_headwise
        self.max_blocks = 0 if t is None else int(t.shape[1])

    def struct(self) -> KvqPaging:
        return KvqPaging(_dev_ptr(self.block_tables, torch.int32, "block_tables"),
                         _dev_ptr(self.block_tables_headwise, torch.int32, "block_tables_headwise"),
                         self.max_blocks, int(self.seq_lens.shape[0]),
                         _dev_ptr(self.seq_lens, torch.int32, "seq_lens"),
                         _dev_ptr(self.window_per_kv_head, torch.int32, "window_per_kv_head"),
                         self.sink_size)


def kvq_write(cache: PagedCache, paging: Paging, k: torch.Tensor, v: torch.Tensor,
              cu_new_tokens: torch.Tensor, dev_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """Quantise k, v [num_tokens, num_kv_heads, head_dim] and scatter them into the pages."""
    if k.shape != v.shape or k.dtype != v.dtype:
        raise ValueError("k and v must have the same shape and dtype")
    cs, ps = cache.struct(), paging.struct()
    _check(_lib.kvq_write(ctypes.byref(cs), ctypes.byref(ps), _dev_ptr(k, name="k"), _dev_ptr(v, name="v"),
                          _qdtype(k), _dev_ptr(cu_new_tokens, torch.int32, "cu_new_tokens"), int(k.shape[0]),
                          _dev_ptr(dev_error, torch.int32, "dev_error"), _stream_ptr(stream)))


def kvq_gather(cache: PagedCache, paging: Paging, cu_tokens: torch.Tensor, num_tokens: int,
               out_dtype: torch.dtype = torch.float32, k_out: Optional[torch.Tensor] = None,
               v_out: Optional[torch.Tensor] = None, dev_error: Optional[torch.Tensor] = None, stream=None,
               k_chunk: Optional[torch.Tensor] = None, v_chunk: Optional[torch.Tensor] = None,
               cu_chunk: Optional[torch.Tensor] = None):
    """Dense dequantised (k, v) [num_tokens, num_kv_heads, head_dim] of the
    positions cu_tokens names (kvq_write's position map); -1 rows are zeros.
    With k_chunk / v_chunk / cu_chunk (kvq_gather_chunk) the last positions
    of each sequence come from those full-precision rows instead."""
    shape = (num_tokens, cache.num_kv_heads, cache.head_dim)
    dev = cache.k_pages.device
    if k_out is None:
        k_out = torch.empty(shape, dtype=out_dtype, device=dev)
    if v_out is None:
        v_out = torch.empty(shape, dtype=out_dtype, device=dev)
    if k_out.dtype != v_out.dtype:
        raise ValueError("k_out and v_out must have the same dtype")
    cs, ps = cache.struct(), paging.struct()
    if k_chunk is None:
        _check(_lib.kvq_gather(ctypes.byref(cs), ctypes.byref(ps), _dev_ptr(cu_tokens, torch.int32, "cu_tokens"),
                               int(num_tokens), _dev_ptr(k_out, name="k_out"), _dev_ptr(v_out, name="v_out"),
                               _qdtype(k_out), _dev_ptr(dev_error, torch.int32, "dev_error"), _stream_ptr(stream)))
    else:
        if v_chunk is None or k_chunk.dtype != v_chunk.dtype:
            raise ValueError("k_chunk and v_chunk must be given together, with one dtype")
        _check(_lib.kvq_gather_chunk(ctypes.byref(cs), ctypes.byref(ps),
                                     _dev_ptr(cu_tokens, torch.int32, "cu_tokens"), int(num_tokens),
                                     _dev_ptr(k_chunk, name="k_chunk"), _dev_ptr(v_chunk, name="v_chunk"),
                                     _qdtype(k_chunk), _dev_ptr(cu_chunk, torch.int32, "cu_chunk"),
                                     _dev_ptr(k_out, name="k_out"), _dev_ptr(v_out, name="v_out"), _qdtype(k_out),
                                     _dev_ptr(dev_error, torch.int32, "dev_error"), _stream_ptr(stream)))
    return k_out, v_out


def kvq_decode_workspace_size(cache: PagedCache, paging: Paging, num_q_heads: int, num_splits: int = 0):
    """(bytes, splits) the decode call needs for its split-KV partials."""
    cs, ps = cache.struct(), paging.struct()
    nbytes, splits = ctypes.c_size_t(0), ctypes.c_int32(0)
    _check(_lib.kvq_decode_workspace_size(ctypes.byref(cs), ctypes.byref(ps), num_q_heads, num_splits,
                                          ctypes.byref(nbytes), ctypes.byref(splits)))
    return nbytes.value, splits.value


def kvq_decode_attn(cache: PagedCache, paging: Paging, q: torch.Tensor, softmax_scale: float,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    num_splits: int = 0, dev_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention of q [batch, num_q_heads, head_dim]; returns fp32 out."""
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes, _ = kvq_decode_workspace_size(cache, paging, Hq, num_splits)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    cs, ps = cache.struct(), paging.struct()
    _check(_lib.kvq_decode_attn(ctypes.byref(cs), ctypes.byref(ps), _dev_ptr(q, name="q"), _qdtype(q), Hq,
                                float(softmax_scale), _dev_ptr(out, torch.float32, "out"),
                                _dev_ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(),
                                num_splits, _dev_ptr(dev_error, torch.int32, "dev_error"), _stream_ptr(stream)))
    return out


def kvq_write_decode_attn(cache: PagedCache, paging: Paging, k: torch.Tensor, v: torch.Tensor,
                          cu_new_tokens: torch.Tensor, q: torch.Tensor, softmax_scale: float,
                          out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                          num_splits: int = 0, dev_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One decode step in one call: kvq_write of k, v [num_tokens, num_kv_heads, head_dim] (the step's new
    tokens), then decode attention of q [batch, num_q_heads, head_dim]; returns fp32 out.  The pages and
    the output are those of kvq_write followed by kvq_decode_attn."""
    if k.shape != v.shape or k.dtype != v.dtype:
        raise ValueError("k and v must have the same shape and dtype")
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes, _ = kvq_decode_workspace_size(cache, paging, Hq, num_splits)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    cs, ps = cache.struct(), paging.struct()
    _check(_lib.kvq_write_decode_attn(ctypes.byref(cs), ctypes.byref(ps), _dev_ptr(k, name="k"), _dev_ptr(v, name="v"),
                                      _qdtype(k), _dev_ptr(cu_new_tokens, torch.int32, "cu_new_tokens"),
                                      int(k.shape[0]), _dev_ptr(q, name="q"), _qdtype(q), Hq, float(softmax_scale),
                                      _dev_ptr(out, torch.float32, "out"), _dev_ptr(workspace, torch.uint8, "workspace"),
                                      workspace.numel(), int(num_splits), _dev_ptr(dev_error, torch.int32, "dev_error"),
                                      _stream_ptr(stream)))
    return out


def kvq_decode_attn_noalloc(cache: PagedCache, paging: Paging, q: torch.Tensor, softmax_scale: float,
                            out: Optional[torch.Tensor] = None, num_splits: int = 0,
                            dev_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """kvq_decode_attn without a caller workspace: for callers that cannot
    allocate device memory at call time.  Uses the library's one static
    device scratch array (KVQ_NOALLOC_SCRATCH_BYTES per GPU); calls that
    overlap on the GPU race on it, so serialise them.  The first call on a
    device must come before any stream capture."""
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    cs, ps = cache.struct(), paging.struct()
    _check(_lib.kvq_decode_attn_noalloc(ctypes.byref(cs), ctypes.byref(ps), _dev_ptr(q, name="q"), _qdtype(q), Hq,
                                        float(softmax_scale), _dev_ptr(out, torch.float32, "out"), num_splits,
                                        _dev_ptr(dev_error, torch.int32, "dev_error"), _stream_ptr(stream)))
    return out


def kvq_prefill_attn(cache: PagedCache, paging: Paging, q: torch.Tensor, cu_q: torch.Tensor, max_q_per_seq: int,
                     softmax_scale: float, out: Optional[torch.Tensor] = None,
                     dev_error: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal chunked-prefill attention of q [total_q, num_q_heads, head_dim]; returns fp32 out."""
    T, Hq, D = q.shape
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=q.device)
    cs, ps = cache.struct(), paging.struct()
    _check(_lib.kvq_prefill_attn(ctypes.byref(cs), ctypes.byref(ps), _dev_ptr(q, name="q"), _qdtype(q), Hq,
                                 _dev_ptr(cu_q, torch.int32, "cu_q"), T, int(max_q_per_seq), float(softmax_scale),
                                 _dev_ptr(out, torch.float32, "out"), _dev_ptr(dev_error, torch.int32, "dev_error"),
                                 _stream_ptr(stream)))
    return out


def kvq_prefill_dense_attn(k: torch.Tensor, v: torch.Tensor, cu_kv: torch.Tensor, seq_lens: torch.Tensor,
                           q: torch.Tensor, cu_q: torch.Tensor, max_q_per_seq: int, softmax_scale: float,
                           window_per_kv_head: Optional[torch.Tensor] = None, sink_size: int = 0,
                           out: Optional[torch.Tensor] = None, dev_error: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """Causal chunked-prefill attention of q [total_q, num_q_heads, head_dim]
    over dense bf16 k, v [rows, num_kv_heads, head_dim] (sequence b's key j at
    row cu_kv[b] + j, e.g. kvq_gather's output); returns fp32 out."""
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16 or k.shape != v.shape:
        raise ValueError("k and v must be bfloat16 tensors of one shape")
    T, Hq, D = q.shape
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.float32, device=q.device)
    ps = KvqPaging(None, None, 0, int(seq_lens.shape[0]), _dev_ptr(seq_lens, torch.int32, "seq_lens"),
                   _dev_ptr(window_per_kv_head, torch.int32, "window_per_kv_head"), int(sink_size))
    _check(_lib.kvq_prefill_dense_attn(_dev_ptr(k, name="k"), _dev_ptr(v, name="v"),
                                       _dev_ptr(cu_kv, torch.int32, "cu_kv"), int(k.shape[0]), int(k.shape[1]),
                                       int(k.shape[2]),
                                       ctypes.byref(ps), _dev_ptr(q, name="q"), _qdtype(q), Hq,
                                       _dev_ptr(cu_q, torch.int32, "cu_q"), T, int(max_q_per_seq),
                                       float(softmax_scale), _dev_ptr(out, torch.float32, "out"),
                                       _dev_ptr(dev_error, torch.int32, "dev_error"), _stream_ptr(stream)))
    return out
