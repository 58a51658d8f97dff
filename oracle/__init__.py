"""fp64 CPU oracle for absorbed-MLA decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library (``mla_latent_kv_15_gb300``) and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, explicit
threads); this module compiles it with gcc and wraps it with ctypes.  The
compute-friendly (expanded MHA) path used to pin the absorbed path is in
``expanded.py``.  Function-by-function citations are in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CACHE_BF16 = 0
CACHE_E4M3 = 1
LKV = 512
DQK = 576


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no fast-math, no FMA contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                            "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, dbl, flt = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
        lib.oracle_bf16_to_f64.restype = dbl
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_to_f64.restype = dbl
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        lib.oracle_f32_to_e4m3.argtypes = [flt]
        for name in ("oracle_decode_bf16_array", "oracle_decode_e4m3_array", "oracle_encode_e4m3_array"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [P, P, i64]
        lib.oracle_cache_write.restype = i32
        lib.oracle_cache_write.argtypes = [P, P, P, i64, P, i64, i32, i32, flt]
        lib.oracle_decode.restype = i32
        lib.oracle_decode.argtypes = [P, P, i64, i32, i32, dbl, P, i32, P, P, i32, i32, dbl,
                                      P, i64, i64, i64, P, P, i32]
        lib.oracle_merge.restype = None
        lib.oracle_merge.argtypes = [P, P, P, P, i64, i32, P, P]
        lib.oracle_gather_cache.restype = i32
        lib.oracle_gather_cache.argtypes = [P, i64, i32, i32, flt, P, i32, P, P, i32, P, i64]
        lib.oracle_num_cores.restype = i32
        lib.oracle_num_cores.argtypes = []
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_cores() -> int:
    return int(_load().oracle_num_cores())


# ------------------------------------------------------------------ formats

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_bf16_array(_ptr(bits), _ptr(out), bits.size)
    return out


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _load().oracle_decode_e4m3_array(_ptr(codes), _ptr(out), codes.size)
    return out


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_encode_e4m3_array(_ptr(x), _ptr(out), x.size)
    return out


def quantize_fp8(x_bf16_bits: np.ndarray, scale: float) -> np.ndarray:
    """scaled_fp8_quant with a static per-tensor scale (common.py,
    MLACommonImpl.forward, decode branch with an fp8 cache: the absorbed query
    and q_pe are quantised with layer._q_scale): code = e4m3(float32(x) /
    float32(scale)), the divide correctly rounded in float32, then the OCP
    E4M3 encoding (nearest even, finite overflow saturated) -- the same rule
    as the cache write."""
    x = bf16_to_f64(np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)).astype(np.float32)
    return f32_to_e4m3(x / np.float32(scale))


# -------------------------------------------------------------- cache write

def cache_write(kv_c: np.ndarray, k_pe: np.ndarray, slot_mapping: np.ndarray, cache: np.ndarray,
                page_size: int, cache_dtype: int, kv_scale: float = 1.0) -> None:
    """In-place write of new latent rows into ``cache`` ([num_blocks, page, 576];
    uint16 bf16 bits or uint8 e4m3 codes)."""
    kv_c = np.ascontiguousarray(kv_c, dtype=np.uint16)
    k_pe = np.ascontiguousarray(k_pe, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    want = np.uint16 if cache_dtype == CACHE_BF16 else np.uint8
    assert cache.dtype == want and cache.flags["C_CONTIGUOUS"]
    rc = _load().oracle_cache_write(_ptr(kv_c), _ptr(k_pe), _ptr(slots), slots.size, _ptr(cache),
                                    cache.shape[0], page_size, cache_dtype, float(kv_scale))
    if rc != 0:
        raise ValueError("oracle_cache_write: slot out of range")


# ----------------------------------------------------------- context gather

def gather_cache(cache: np.ndarray, page_size: int, cache_dtype: int, kv_scale: float, block_table: np.ndarray,
                 cu_seq_lens: np.ndarray, seq_starts, dst_rows: int) -> np.ndarray:
    """gather_and_maybe_dequant_cache: bf16 bits [dst_rows, 576]; rows past
    cu_seq_lens[-1] are left zero."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seq_lens, dtype=np.int32)
    st = None if seq_starts is None else np.ascontiguousarray(seq_starts, dtype=np.int32)
    dst = np.zeros((dst_rows, DQK), dtype=np.uint16)
    rc = _load().oracle_gather_cache(_ptr(cache), cache.shape[0], page_size, cache_dtype, float(kv_scale),
                                     _ptr(bt), bt.shape[1], _ptr(cu), _ptr(st) if st is not None else None,
                                     cu.size - 1, _ptr(dst), dst_rows)
    if rc != 0:
        raise ValueError("oracle_gather_cache: position, page or destination row out of range")
    return dst


# ------------------------------------------------------------------- decode

def decode(q: np.ndarray, cache: np.ndarray, page_size: int, cache_dtype: int, kv_scale: float,
           block_table: np.ndarray, seq_lens: np.ndarray, query_start_loc: np.ndarray,
           num_heads: int, scale: float, rows=None, key_begin: int = 0, key_end: int = -1,
           nthreads: int = 0):
    """Attention of query rows (flattened ``t*N + h``; default all) in fp64.

    ``q`` is float64 [T, N, 576] (``[q_abs | q_pe]``).  Returns
    ``(out [nrows, 512], lse [nrows], threads_used)``.
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    T = q.shape[0]
    assert q.shape[1:] == (num_heads, DQK)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    if rows is None:
        rows_arr = np.arange(T * num_heads, dtype=np.int64)
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows_arr.size
    out = np.zeros((n, LKV), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    if n == 0:
        return out, lse, 0
    used = _load().oracle_decode(_ptr(q), _ptr(cache), cache.shape[0], page_size, cache_dtype,
                                 float(kv_scale), _ptr(bt), bt.shape[1], _ptr(sl), _ptr(qsl),
                                 sl.size, num_heads, float(scale), _ptr(rows_arr), n,
                                 int(key_begin), int(key_end), _ptr(out), _ptr(lse), int(nthreads))
    if used < 0:
        raise ValueError("oracle_decode: bad argument or page out of range")
    return out, lse, used


def merge(o_a, lse_a, o_b, lse_b):
    """merge_attn_states of two partials in fp64: returns (out, lse)."""
    o_a = np.ascontiguousarray(o_a, dtype=np.float64)
    o_b = np.ascontiguousarray(o_b, dtype=np.float64)
    lse_a = np.ascontiguousarray(lse_a, dtype=np.float64)
    lse_b = np.ascontiguousarray(lse_b, dtype=np.float64)
    rows, dim = o_a.shape
    out = np.empty_like(o_a)
    lse = np.empty(rows, dtype=np.float64)
    _load().oracle_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, dim, _ptr(out), _ptr(lse))
    return out, lse


# ------------------------------------------------------- whole-case helpers

def prepare_cache(case, with_new_rows: bool = True) -> np.ndarray:
    """The cache the decode of ``case`` reads, built on the host by the oracle:
    the drawn pool (quantised by the oracle's cache write for an fp8 cache),
    then the step's new rows written at ``slot_mapping``."""
    if case.cache_dtype == "bf16":
        cache = case.pool.copy()
        dt = CACHE_BF16
    else:
        cache = np.zeros(case.pool.shape, dtype=np.uint8)
        slots = case.referenced_slots
        flat = case.pool.reshape(-1, DQK)
        cache_write(flat[slots, :LKV], flat[slots, LKV:], slots, cache, case.page_size,
                    CACHE_E4M3, case.kv_scale)
        dt = CACHE_E4M3
    if with_new_rows:
        cache_write(case.new_kv_c, case.new_k_pe, case.slot_mapping, cache, case.page_size, dt,
                    case.kv_scale)
    return cache


def decode_case(case, cache: np.ndarray, rows=None, key_begin: int = 0, key_end: int = -1,
                nthreads: int = 0):
    """oracle decode of a ``synth.DecodeCase`` against ``cache`` (see prepare_cache)."""
    q = np.concatenate([bf16_to_f64(case.q_abs), bf16_to_f64(case.q_pe)], axis=-1)
    dt = CACHE_BF16 if case.cache_dtype == "bf16" else CACHE_E4M3
    return decode(q, cache, case.page_size, dt, case.kv_scale, case.block_table, case.seq_lens,
                  case.query_start_loc, case.num_heads, case.scale, rows=rows,
                  key_begin=key_begin, key_end=key_end, nthreads=nthreads)
