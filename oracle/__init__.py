"""CPU oracle of the paged low-bit KV cache (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The library under ``sub_byte_quantized_write_gb300``
never does: the two share no code, and the oracle never sees an output of the
CUDA path.

The arithmetic lives in ``kvq_oracle.cpp`` (plain C++, fp32 write path in a
fixed order, double-precision attention); this module compiles it with g++
and marshals numpy arrays through ctypes.

Parity status: every exported function is pinned by ``tests/test_oracle_pins.py``
(closed forms, library routines, brute force and worked examples); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_INT4, MODE_INT2, MODE_INT8, MODE_INT4_STEGO = 0, 1, 2, 3
MODE_INT8_TOKEN_HEAD, MODE_FP8_TOKEN_HEAD = 4, 5
DT_F32, DT_BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source (idempotent)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class OrcCache(ctypes.Structure):
    _fields_ = [("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("signs", ctypes.c_void_p),
                ("ch_amax", ctypes.c_void_p), ("ch_ready", ctypes.c_void_p)]


class OrcPaging(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("headwise", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("window", ctypes.c_void_p),
                ("sink", ctypes.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
            L.orc_row_bytes.argtypes, L.orc_row_bytes.restype = [I, I], I
            L.orc_f16_round.argtypes, L.orc_f16_round.restype = [F], ctypes.c_uint16
            L.orc_f16_saturate.argtypes, L.orc_f16_saturate.restype = [F], ctypes.c_uint16
            L.orc_f16_decode.argtypes, L.orc_f16_decode.restype = [ctypes.c_uint16], F
            L.orc_rht_forward.argtypes, L.orc_rht_forward.restype = [P, I, P], None
            L.orc_pack_codes.argtypes, L.orc_pack_codes.restype = [I, P, I, P], None
            L.orc_unpack_codes.argtypes, L.orc_unpack_codes.restype = [I, P, I, P], None
            L.orc_signed_code.argtypes, L.orc_signed_code.restype = [I, I], I
            L.orc_e4m3_decode.argtypes, L.orc_e4m3_decode.restype = [ctypes.c_uint8], ctypes.c_double
            L.orc_e4m3_round.argtypes, L.orc_e4m3_round.restype = [F], ctypes.c_uint8
            L.orc_quant_row.argtypes, L.orc_quant_row.restype = [I, P, I, P, P], None
            L.orc_dequant_row.argtypes, L.orc_dequant_row.restype = [I, P, I, P, P, P], None
            L.orc_write.argtypes = [ctypes.POINTER(OrcCache), ctypes.POINTER(OrcPaging), P, P, I, P, I]
            L.orc_write.restype = I
            L.orc_attention.argtypes = [ctypes.POINTER(OrcCache), ctypes.POINTER(OrcPaging), P, I, I,
                                        P, I, F, P, I, P, I]
            L.orc_attention.restype = I
            L.orc_gather.argtypes = [ctypes.POINTER(OrcCache), ctypes.POINTER(OrcPaging), P, I, P, P]
            L.orc_gather.restype = I
            L.orc_gather_chunk.argtypes = [ctypes.POINTER(OrcCache), ctypes.POINTER(OrcPaging), P, I, P, P, I, P, P, P]
            L.orc_gather_chunk.restype = I
            L.orc_dense_attention.argtypes = [P, P, I, P, ctypes.POINTER(OrcPaging), I, I, P, I, I, P, I, F, P, I,
                                              P, I]
            L.orc_dense_attention.restype = I
            L.orc_rounding_mode_is_nearest.argtypes, L.orc_rounding_mode_is_nearest.restype = [], I
            _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def row_bytes(mode: int, head_dim: int) -> int:
    return lib().orc_row_bytes(mode, head_dim)


def f16_round(x: float) -> int:
    return lib().orc_f16_round(float(x))


def f16_saturate(x: float) -> int:
    return lib().orc_f16_saturate(float(x))


def f16_decode(h: int) -> float:
    return lib().orc_f16_decode(int(h))


def rht_forward(x: np.ndarray, signs: Optional[np.ndarray]) -> np.ndarray:
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    s = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    lib().orc_rht_forward(_ptr(y), y.shape[-1], _ptr(s))
    return y


def pack_codes(mode: int, codes: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(codes, dtype=np.uint8)
    D = u.shape[0]
    out = np.zeros(row_bytes(mode, D) - (0 if mode == MODE_INT8 else 4), dtype=np.uint8)
    lib().orc_pack_codes(mode, _ptr(u), D, _ptr(out))
    return out


def unpack_codes(mode: int, data: np.ndarray, D: int) -> np.ndarray:
    b = np.ascontiguousarray(data, dtype=np.uint8)
    u = np.zeros(D, dtype=np.uint8)
    lib().orc_unpack_codes(mode, _ptr(b), D, _ptr(u))
    return u


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e4m3_round(x: float) -> int:
    return lib().orc_e4m3_round(float(x))


def signed_code(mode: int, u: int) -> int:
    return lib().orc_signed_code(mode, int(u))


def quant_row(mode: int, x: np.ndarray, signs: Optional[np.ndarray]) -> np.ndarray:
    xx = np.ascontiguousarray(x, dtype=np.float32)
    D = xx.shape[0]
    row = np.zeros(row_bytes(mode, D), dtype=np.uint8)
    s = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    lib().orc_quant_row(mode, _ptr(xx), D, _ptr(s), _ptr(row))
    return row


def dequant_row(mode: int, row: np.ndarray, D: int, signs: Optional[np.ndarray] = None,
                amax: Optional[np.ndarray] = None) -> np.ndarray:
    r = np.ascontiguousarray(row, dtype=np.uint8)
    out = np.zeros(D, dtype=np.float64)
    s = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    a = None if amax is None else np.ascontiguousarray(amax, dtype=np.float32)
    lib().orc_dequant_row(mode, _ptr(r), D, _ptr(s), _ptr(a), _ptr(out))
    return out


class Cache:
    """Host-memory paged cache mirroring the library's layout
    [num_blocks][num_kv_heads][block_size][row_bytes], separate K and V."""

    def __init__(self, mode, num_blocks, num_kv_heads, block_size, head_dim, signs=None, fill=0):
        self.mode, self.num_blocks, self.num_kv_heads = mode, num_blocks, num_kv_heads
        self.block_size, self.head_dim = block_size, head_dim
        self.R = row_bytes(mode, head_dim)
        shape = (num_blocks, num_kv_heads, block_size, self.R)
        self.k = np.full(shape, fill, dtype=np.uint8)
        self.v = np.full(shape, fill, dtype=np.uint8)
        self.signs = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
        self.amax = np.zeros((2, num_kv_heads, head_dim), dtype=np.float32)
        self.ready = np.zeros(1, dtype=np.int32)

    def struct(self) -> OrcCache:
        return OrcCache(self.k.ctypes.data, self.v.ctypes.data, self.num_blocks, self.num_kv_heads,
                        self.block_size, self.head_dim, self.mode,
                        None if self.signs is None else self.signs.ctypes.data,
                        self.amax.ctypes.data if self.mode == MODE_INT8 else None,
                        self.ready.ctypes.data)


class Paging:
    def __init__(self, table, headwise, seq_lens, window=None, sink=0):
        self.table = np.ascontiguousarray(table, dtype=np.int32)
        self.headwise = bool(headwise)
        self.seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        self.window = None if window is None else np.ascontiguousarray(window, dtype=np.int32)
        self.sink = int(sink)

    def struct(self) -> OrcPaging:
        return OrcPaging(self.table.ctypes.data, int(self.headwise), self.table.shape[1],
                         self.seq_lens.shape[0], self.seq_lens.ctypes.data,
                         None if self.window is None else self.window.ctypes.data, self.sink)


def _input(x: np.ndarray):
    """Accept fp32 values or bf16 bit patterns (uint16)."""
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), DT_BF16
    return np.ascontiguousarray(x, dtype=np.float32), DT_F32


def write(cache: Cache, paging: Paging, k: np.ndarray, v: np.ndarray, cu_new: np.ndarray) -> int:
    kk, dt = _input(k)
    vv, dt2 = _input(v)
    assert dt == dt2
    cu = np.ascontiguousarray(cu_new, dtype=np.int32)
    cs, ps = cache.struct(), paging.struct()
    return lib().orc_write(ctypes.byref(cs), ctypes.byref(ps), _ptr(kk), _ptr(vv), dt, _ptr(cu),
                           int(kk.shape[0]))


def gather(cache: Cache, paging: Paging, cu_tokens: np.ndarray):
    """Dequantised K and V (double [num_tokens, Hkv, D]) of the positions the
    cu map names, and the error bits."""
    cu = np.ascontiguousarray(cu_tokens, dtype=np.int32)
    n = int(cu[-1])
    k = np.zeros((n, cache.num_kv_heads, cache.head_dim), dtype=np.float64)
    v = np.zeros_like(k)
    cs, ps = cache.struct(), paging.struct()
    err = lib().orc_gather(ctypes.byref(cs), ctypes.byref(ps), _ptr(cu), n, _ptr(k), _ptr(v))
    return k, v, err


def gather_chunk(cache: Cache, paging: Paging, cu_tokens: np.ndarray, k_chunk: np.ndarray, v_chunk: np.ndarray,
                 cu_chunk: np.ndarray):
    """gather() with the last m_b positions of each sequence taken from the
    full-precision chunk rows k_chunk / v_chunk (fp32 values or bf16 bits),
    sequence b's at rows cu_chunk[b] ..; returns (k, v, error bits)."""
    cu = np.ascontiguousarray(cu_tokens, dtype=np.int32)
    cc = np.ascontiguousarray(cu_chunk, dtype=np.int32)
    kk, dt = _input(k_chunk)
    vv, dt2 = _input(v_chunk)
    assert dt == dt2
    n = int(cu[-1])
    k = np.zeros((n, cache.num_kv_heads, cache.head_dim), dtype=np.float64)
    v = np.zeros_like(k)
    cs, ps = cache.struct(), paging.struct()
    err = lib().orc_gather_chunk(ctypes.byref(cs), ctypes.byref(ps), _ptr(cu), n, _ptr(kk), _ptr(vv), dt, _ptr(cc),
                                 _ptr(k), _ptr(v))
    return k, v, err


def attention(cache: Cache, paging: Paging, q: np.ndarray, scale: float, cu_q=None, rows=None,
              threads: Optional[int] = None):
    """Returns (out double [n_rows, Hq, D], error bits)."""
    qq, dt = _input(q)
    total_q, Hq, D = qq.shape
    cu = None if cu_q is None else np.ascontiguousarray(cu_q, dtype=np.int32)
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n_rows = total_q if sel is None else sel.shape[0]
    out = np.zeros((n_rows, Hq, D), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    cs, ps = cache.struct(), paging.struct()
    err = lib().orc_attention(ctypes.byref(cs), ctypes.byref(ps), _ptr(qq), dt, Hq, _ptr(cu), total_q,
                              float(scale), _ptr(sel), n_rows, _ptr(out), int(threads))
    return out, err


def dense_attention(k: np.ndarray, v: np.ndarray, cu_kv: np.ndarray, paging: Paging, q: np.ndarray, scale: float,
                    cu_q: np.ndarray, rows=None, threads: Optional[int] = None):
    """Attention over dense K / V [rows, Hkv, D] (fp32 values or bf16 bits):
    sequence b's key j is row cu_kv[b] + j.  Returns (out double
    [n_rows, Hq, D], error bits)."""
    kk, kdt = _input(k)
    vv, vdt = _input(v)
    assert kdt == vdt
    qq, dt = _input(q)
    total_q, Hq, D = qq.shape
    Hkv = kk.shape[1]
    cu = np.ascontiguousarray(cu_kv, dtype=np.int32)
    cq = np.ascontiguousarray(cu_q, dtype=np.int32)
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n_rows = total_q if sel is None else sel.shape[0]
    out = np.zeros((n_rows, Hq, D), dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    ps = paging.struct()
    err = lib().orc_dense_attention(_ptr(kk), _ptr(vv), kdt, _ptr(cu), ctypes.byref(ps), Hkv, D, _ptr(qq), dt, Hq,
                                    _ptr(cq), total_q, float(scale), _ptr(sel), n_rows, _ptr(out), int(threads))
    return out, err
