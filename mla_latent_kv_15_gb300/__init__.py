"""Python binding of libmla.so: absorbed MLA decode over a paged latent KV cache
on GB300 (sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels,
reached through its C ABI (``include/mla.h``) with ctypes.  PyTorch provides
device memory and streams.  There is no fallback: if ``libmla.so`` is missing
or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla.so")

MLA_OK = 0
MLA_BF16 = 0
MLA_FP8_E4M3 = 1
MLA_FP32 = 2
DEVERR_TIMEOUT = 1
DEVERR_BAD_SEQ_LEN = 2
DEVERR_BAD_BLOCK = 4
DEVERR_BAD_QSL = 8
LKV = 512
ROPE = 64
DQK = 576

C_ABI_SYMBOLS = ("mla_cache_write", "mla_decode_workspace_size", "mla_decode", "mla_decode_status",
                 "mla_merge_states", "mla_last_error", "mla_device_sm_count", "mla_set_decode_timing_events",
                 "mla_decode_no_alloc", "mla_q_absorb", "mla_v_up_proj", "mla_proj_status",
                 "mla_gather_cache", "mla_quantize_fp8", "mla_decode_fp8q", "mla_set_decode_wait_test",
                 "mla_decode_no_alloc_status", "mla_decode_step", "mla_decode_fp8q_step")
NO_ALLOC_SCRATCH_BYTES = 96 << 20

_lib = None


class MLAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmla.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.mla_cache_write.restype = i32
    lib.mla_cache_write.argtypes = [P, P, P, i64, P, i64, i32, i32, f32, P]
    lib.mla_decode_workspace_size.restype = sz
    lib.mla_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.mla_decode.restype = i32
    lib.mla_decode.argtypes = [P, P, P, i64, i32, i32, f32, P, i32, P, i32, P, i32, i32, f32, i32, P, P, P, sz, P]
    lib.mla_decode_status.restype = i32
    lib.mla_decode_status.argtypes = [P, ctypes.POINTER(ctypes.c_int), P]
    lib.mla_merge_states.restype = i32
    lib.mla_merge_states.argtypes = [P, P, P, P, i64, i32, i32, P, P, P]
    lib.mla_last_error.restype = ctypes.c_char_p
    lib.mla_last_error.argtypes = []
    lib.mla_device_sm_count.restype = i32
    lib.mla_device_sm_count.argtypes = []
    lib.mla_set_decode_timing_events.restype = i32
    lib.mla_set_decode_timing_events.argtypes = [P, P]
    lib.mla_decode_no_alloc.restype = i32
    lib.mla_decode_no_alloc.argtypes = [P, P, P, i64, i32, i32, f32, P, i32, P, i32, P, i32, i32, f32, i32, P, P, P]
    lib.mla_q_absorb.restype = i32
    lib.mla_q_absorb.argtypes = [P, i64, P, i64, i32, i32, P, P]
    lib.mla_v_up_proj.restype = i32
    lib.mla_v_up_proj.argtypes = [P, P, i64, i32, i32, P, P]
    lib.mla_decode_fp8q.restype = i32
    lib.mla_decode_fp8q.argtypes = [P, f32, P, i64, i32, f32, P, i32, P, i32, P, i32, i32, f32, i32, P, P, P, sz, P]
    lib.mla_quantize_fp8.restype = i32
    lib.mla_quantize_fp8.argtypes = [P, i64, i64, i32, f32, P, i64, P]
    lib.mla_gather_cache.restype = i32
    lib.mla_gather_cache.argtypes = [P, i64, i32, i32, f32, P, i32, P, P, i32, P, i64, P, P]
    lib.mla_proj_status.restype = i32
    lib.mla_proj_status.argtypes = [ctypes.POINTER(ctypes.c_int), i32, P]
    lib.mla_set_decode_wait_test.restype = i32
    lib.mla_set_decode_wait_test.argtypes = [i32, ctypes.c_ulonglong]
    lib.mla_decode_no_alloc_status.restype = i32
    lib.mla_decode_no_alloc_status.argtypes = [ctypes.POINTER(ctypes.c_int), i32, P]
    lib.mla_decode_fp8q_step.restype = i32
    lib.mla_decode_fp8q_step.argtypes = [P, P, P, i64, P, P, f32, P, P, i64, i32, f32, P, i32, P, i32, P, i32, i32, f32,
                                         i32, P, P, P, sz, P]
    lib.mla_decode_step.restype = i32
    lib.mla_decode_step.argtypes = [P, P, P, i64, P, P, P, i64, i32, i32, f32, P, i32, P, i32, P, i32, i32, f32, i32,
                                    P, P, P, sz, P]
    _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != MLA_OK:
        raise MLAError(rc, load().mla_last_error().decode())


def _ptr(t):
    """Device address of a CUDA tensor (None passes NULL).  Every tensor the
    library reads or writes lives on the GPU: a host tensor is refused here,
    before its address could reach a kernel."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(cache):
    import torch
    if cache.dtype == torch.bfloat16:
        return MLA_BF16
    if cache.dtype in (torch.float8_e4m3fn, torch.uint8):
        return MLA_FP8_E4M3
    raise TypeError(f"cache dtype {cache.dtype} is neither bf16 nor float8_e4m3fn")


def _dense(t, name: str, dtypes, shape=None, dims=None):
    """Refuse a tensor the library would misread: the C ABI takes dense
    row-major tensors of fixed element types.  ``shape`` entries of None
    match any size; ``dims`` checks only the rank."""
    import torch
    if not isinstance(dtypes, tuple):
        dtypes = (dtypes,)
    if t.dtype not in dtypes:
        want = " or ".join(str(d).replace("torch.", "") for d in dtypes)
        raise ValueError(f"{name} must be {want}, got {str(t.dtype).replace('torch.', '')}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions, got shape {tuple(t.shape)}")
    if shape is not None:
        if t.dim() != len(shape) or any(w is not None and int(n) != w for n, w in zip(t.shape, shape)):
            exp = "[" + ", ".join("*" if w is None else str(w) for w in shape) + "]"
            raise ValueError(f"{name} must have shape {exp}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (dense rows), got strides {t.stride()}")
    del torch


def _cache_checked(cache, name="cache"):
    import torch
    _dense(cache, name, (torch.bfloat16, torch.float8_e4m3fn, torch.uint8), dims=3)
    if cache.shape[2] != DQK:
        raise ValueError(f"cache rows must be {DQK} wide, got {cache.shape[2]}")
    return cache.shape


def cache_write(kv_c, k_pe, slot_mapping, cache, kv_scale: float = 1.0, stream=None) -> None:
    """concat_and_cache_mla: cache[num_blocks, page, 576] (bf16 or float8_e4m3fn)."""
    import torch
    nb, ps, _ = _cache_checked(cache)
    _dense(slot_mapping, "slot_mapping", torch.int64, dims=1)
    T = slot_mapping.numel()
    _dense(kv_c, "kv_c", torch.bfloat16, (T, LKV))
    _dense(k_pe, "k_pe", torch.bfloat16, (T, ROPE))
    _check(load().mla_cache_write(_ptr(kv_c), _ptr(k_pe), _ptr(slot_mapping), slot_mapping.numel(), _ptr(cache),
                                  nb, ps, _dtype_code(cache), float(kv_scale), _stream(stream)))


def decode_workspace_size(batch: int, total_q: int, num_heads: int, max_splits: int = 0) -> int:
    return int(load().mla_decode_workspace_size(batch, total_q, num_heads, max_splits))


def decode(q_abs, q_pe, cache, block_table, seq_lens, out, workspace, *, scale: float,
           query_start_loc=None, lse=None, num_splits: int = 0, kv_scale: float = 1.0, stream=None) -> None:
    """Absorbed MLA decode (forward_mqa) into ``out`` [T, N, 512] bf16 and ``lse`` [T, N] fp32."""
    T, N, _ = q_abs.shape
    nb, ps, _ = _decode_checked(q_abs, q_pe, cache, block_table, seq_lens, out, query_start_loc, lse)
    _dense(workspace, "workspace", (workspace.dtype,))
    B = seq_lens.numel()
    _check(load().mla_decode(_ptr(q_abs), _ptr(q_pe), _ptr(cache), nb, ps, _dtype_code(cache), float(kv_scale),
                             _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, _ptr(query_start_loc),
                             T, N, float(scale), int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)))


def decode_step(kv_c, k_pe, slot_mapping, q_abs, q_pe, cache, block_table, seq_lens, out, workspace, *,
                scale: float, query_start_loc=None, lse=None, num_splits: int = 0, kv_scale: float = 1.0,
                stream=None) -> None:
    """cache_write(kv_c, k_pe, slot_mapping, cache) then decode(...) in one
    call: the new rows are written by extra blocks of the scheduler's launch."""
    import torch
    T, N, _ = q_abs.shape
    nb, ps, _ = _decode_checked(q_abs, q_pe, cache, block_table, seq_lens, out, query_start_loc, lse)
    _dense(slot_mapping, "slot_mapping", torch.int64, dims=1)
    W = slot_mapping.numel()
    _dense(kv_c, "kv_c", torch.bfloat16, (W, LKV))
    _dense(k_pe, "k_pe", torch.bfloat16, (W, ROPE))
    _dense(workspace, "workspace", (workspace.dtype,))
    B = seq_lens.numel()
    _check(load().mla_decode_step(_ptr(kv_c), _ptr(k_pe), _ptr(slot_mapping), W, _ptr(q_abs), _ptr(q_pe),
                                  _ptr(cache), nb, ps, _dtype_code(cache), float(kv_scale), _ptr(block_table),
                                  block_table.shape[1], _ptr(seq_lens), B, _ptr(query_start_loc), T, N, float(scale),
                                  int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def decode_fp8q_step(kv_c, k_pe, slot_mapping, q_abs, q_pe, q_scale: float, q_fp8, cache, block_table, seq_lens,
                     out, workspace, *, scale: float, query_start_loc=None, lse=None, num_splits: int = 0,
                     kv_scale: float = 1.0, stream=None) -> None:
    """cache_write, quantize_fp8 of q_abs and q_pe into ``q_fp8`` [T, N, 576]
    ([q_abs | q_pe] e4m3 rows, written by this call) and decode_fp8q in one
    call: the rows and the codes are written by extra blocks of the
    scheduler's launch."""
    import torch
    _dense(q_abs, "q_abs", torch.bfloat16, (None, None, LKV))
    T, N, _ = q_abs.shape
    _dense(q_pe, "q_pe", torch.bfloat16, (T, N, ROPE))
    nb, ps, _ = _decode_checked(None, None, cache, block_table, seq_lens, out, query_start_loc, lse, q8=q_fp8)
    if tuple(q_fp8.shape[:2]) != (T, N):
        raise ValueError(f"q_fp8 must have shape [{T}, {N}, {DQK}], got {tuple(q_fp8.shape)}")
    _dense(slot_mapping, "slot_mapping", torch.int64, dims=1)
    W = slot_mapping.numel()
    _dense(kv_c, "kv_c", torch.bfloat16, (W, LKV))
    _dense(k_pe, "k_pe", torch.bfloat16, (W, ROPE))
    _dense(workspace, "workspace", (workspace.dtype,))
    B = seq_lens.numel()
    _check(load().mla_decode_fp8q_step(_ptr(kv_c), _ptr(k_pe), _ptr(slot_mapping), W, _ptr(q_abs), _ptr(q_pe),
                                       float(q_scale), _ptr(q_fp8), _ptr(cache), nb, ps, float(kv_scale),
                                       _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
                                       _ptr(query_start_loc), T, N, float(scale), int(num_splits), _ptr(out),
                                       _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))


def _decode_checked(q_abs, q_pe, cache, block_table, seq_lens, out, query_start_loc, lse, q8=None):
    """Validate the dense tensors of a decode call; returns the cache shape."""
    import torch
    if q8 is None:
        _dense(q_abs, "q_abs", torch.bfloat16, (None, None, LKV))
        T, N, _ = q_abs.shape
        _dense(q_pe, "q_pe", torch.bfloat16, (T, N, ROPE))
    else:
        _dense(q8, "q_fp8", (torch.uint8, torch.float8_e4m3fn), (None, None, DQK))
        T, N, _ = q8.shape
    shape = _cache_checked(cache)
    _dense(block_table, "block_table", torch.int32, dims=2)
    _dense(seq_lens, "seq_lens", torch.int32, dims=1)
    B = seq_lens.numel()
    if block_table.shape[0] != B:
        raise ValueError(f"block_table must have one row per request ({B}), got {block_table.shape[0]}")
    if query_start_loc is not None:
        _dense(query_start_loc, "query_start_loc", torch.int32, (B + 1,))
    _dense(out, "out", torch.bfloat16, (T, N, LKV))
    if lse is not None:
        _dense(lse, "lse", torch.float32, (T, N))
    return shape


def decode_no_alloc(q_abs, q_pe, cache, block_table, seq_lens, out, *, scale: float, query_start_loc=None,
                    lse=None, num_splits: int = 0, kv_scale: float = 1.0, stream=None) -> None:
    """decode() for callers that cannot allocate: the split-KV scratch is the
    library's own fixed 96 MiB device array (shared by all calls; calls that
    overlap on the GPU race).  Batches needing more scratch raise MLAError."""
    T, N, _ = q_abs.shape
    nb, ps, _ = _decode_checked(q_abs, q_pe, cache, block_table, seq_lens, out, query_start_loc, lse)
    B = seq_lens.numel()
    _check(load().mla_decode_no_alloc(_ptr(q_abs), _ptr(q_pe), _ptr(cache), nb, ps, _dtype_code(cache),
                                      float(kv_scale), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B,
                                      _ptr(query_start_loc), T, N, float(scale), int(num_splits), _ptr(out),
                                      _ptr(lse), _stream(stream)))


def decode_fp8q(q_fp8, q_scale: float, cache, block_table, seq_lens, out, workspace, *, scale: float,
                query_start_loc=None, lse=None, num_splits: int = 0, kv_scale: float = 1.0, stream=None) -> None:
    """decode() with an e4m3 query ``q_fp8`` [T, N, 576] (quantised with
    q_scale) over an e4m3 cache: fp8 x fp8 score MMAs."""
    T, N, _ = q_fp8.shape
    nb, ps, _ = _decode_checked(None, None, cache, block_table, seq_lens, out, query_start_loc, lse, q8=q_fp8)
    _dense(workspace, "workspace", (workspace.dtype,))
    B = seq_lens.numel()
    _check(load().mla_decode_fp8q(_ptr(q_fp8), float(q_scale), _ptr(cache), nb, ps, float(kv_scale),
                                  _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, _ptr(query_start_loc),
                                  T, N, float(scale), int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def decode_status(workspace, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(load().mla_decode_status(_ptr(workspace), ctypes.byref(st), _stream(stream)))
    return st.value


def decode_no_alloc_status(clear: bool = False, stream=None) -> int:
    """Device error word of the last decode_no_alloc on the current device
    (OR of the DEVERR_* bits); optionally cleared afterwards."""
    st = ctypes.c_int(0)
    _check(load().mla_decode_no_alloc_status(ctypes.byref(st), int(clear), _stream(stream)))
    return st.value


def set_decode_wait_test(skip_first_tile: bool = False, wait_limit_ns: int = 0) -> None:
    """Test aid for the bounded on-chip waits: later decodes of this thread
    run with every wait bounded by ``wait_limit_ns`` (0: the default 1 s) and,
    with ``skip_first_tile``, one CTA never loads its first cache tile, so a
    wait for it runs out and the device error word gets DEVERR_TIMEOUT."""
    _check(load().mla_set_decode_wait_test(int(bool(skip_first_tile)), int(wait_limit_ns)))


def merge_states(o_a, lse_a, o_b, lse_b, out, lse_out=None, stream=None) -> None:
    """merge_attn_states of two partials (rows x dim, bf16 or fp32)."""
    import torch
    _dense(lse_a, "lse_a", torch.float32, dims=1)
    rows = lse_a.numel()
    _dense(o_a, "o_a", (torch.bfloat16, torch.float32))
    dim = o_a.numel() // max(rows, 1)
    if rows > 0 and (o_a.numel() != rows * dim or o_a.shape[0] != rows):
        raise ValueError(f"o_a must hold one row per LSE entry ({rows}), got shape {tuple(o_a.shape)}")
    _dense(o_b, "o_b", o_a.dtype, tuple(o_a.shape))
    _dense(out, "out", o_a.dtype, tuple(o_a.shape))
    _dense(lse_b, "lse_b", torch.float32, (rows,))
    if lse_out is not None:
        _dense(lse_out, "lse_out", torch.float32, (rows,))
    code = MLA_BF16 if o_a.dtype == torch.bfloat16 else MLA_FP32
    _check(load().mla_merge_states(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, dim, code, _ptr(out),
                                   _ptr(lse_out), _stream(stream)))


def q_absorb(q_nope, w_uk_t, ql_nope, stream=None) -> None:
    """ql_nope[t, n, :] = q_nope[t, n, :] @ w_uk_t[n] (bf16; w_uk_t [N, P, 512]).
    ``q_nope`` [T, N, P] may be a column slice of a wider tensor (for example
    ``q[..., :128]`` of q = [q_nope | q_pe]): its last dimension must be
    contiguous and the (t, n) rows equally spaced."""
    import torch
    T, N, P_ = q_nope.shape
    if q_nope.dtype != torch.bfloat16:
        raise ValueError(f"q_nope must be bfloat16, got {q_nope.dtype}")
    if q_nope.stride(2) != 1 or q_nope.stride(0) != N * q_nope.stride(1):
        raise ValueError("q_nope rows must be equally spaced with a contiguous last dimension")
    _dense(w_uk_t, "w_uk_t", torch.bfloat16, (N, P_, LKV))
    _dense(ql_nope, "ql_nope", torch.bfloat16, (T, N, LKV))
    _check(load().mla_q_absorb(_ptr(q_nope), q_nope.stride(1), _ptr(w_uk_t), T, N, P_, _ptr(ql_nope),
                               _stream(stream)))


def v_up_proj(o_lat, w_uv, out, stream=None) -> None:
    """out[t, n, :] = o_lat[t, n, :] @ w_uv[n] (bf16; w_uv [N, 512, V], out [T, N, V])."""
    import torch
    _dense(o_lat, "o_lat", torch.bfloat16, (None, None, LKV))
    T, N, _ = o_lat.shape
    _dense(w_uv, "w_uv", torch.bfloat16, (N, LKV, None))
    _dense(out, "out", torch.bfloat16, (T, N, w_uv.shape[2]))
    _check(load().mla_v_up_proj(_ptr(o_lat), _ptr(w_uv), T, N, w_uv.shape[2], _ptr(out), _stream(stream)))


def gather_cache(cache, block_table, cu_seq_lens, dst, seq_starts=None, kv_scale: float = 1.0, status=None,
                 stream=None) -> None:
    """gather_and_maybe_dequant_cache: dst [num_tokens, 576] bf16 receives the
    chunk rows of every request (cu_seq_lens [B+1], seq_starts [B] int32)."""
    import torch
    nb, ps, _ = _cache_checked(cache)
    _dense(cu_seq_lens, "cu_seq_lens", torch.int32, dims=1)
    B = cu_seq_lens.numel() - 1
    _dense(block_table, "block_table", torch.int32, dims=2)
    if seq_starts is not None:
        _dense(seq_starts, "seq_starts", torch.int32, (B,))
    _dense(dst, "dst", torch.bfloat16, (None, DQK))
    if status is not None:
        _dense(status, "status", torch.int32, (1,))
    _check(load().mla_gather_cache(_ptr(cache), nb, ps, _dtype_code(cache), float(kv_scale), _ptr(block_table),
                                   block_table.shape[1], _ptr(cu_seq_lens), _ptr(seq_starts), B, _ptr(dst),
                                   dst.shape[0], _ptr(status), _stream(stream)))


def quantize_fp8(x, scale: float, out, stream=None) -> None:
    """scaled_fp8_quant: out = e4m3(x / scale) row by row.  ``x`` (bf16) and
    ``out`` (uint8 or float8_e4m3fn) have the same shape; their last dimension
    is contiguous and may be a column slice of wider rows (e.g. the q_abs and
    q_pe parts of [q_abs | q_pe] rows); 1-D tensors are one row."""
    if tuple(x.shape) != tuple(out.shape):
        raise ValueError("x and out must have the same shape")
    width = x.shape[-1]
    rows = x.numel() // width if width else 0
    xs, os_ = _row_pitch(x), _row_pitch(out)
    _check(load().mla_quantize_fp8(_ptr(x), xs, rows, width, float(scale), _ptr(out), os_, _stream(stream)))


def _row_pitch(t) -> int:
    """Element distance between consecutive rows (the last dimension is a
    row) of a tensor whose rows are equally spaced in memory with a contiguous
    last dimension; dimensions of size 1 may carry any stride.  A tensor of
    one row reports its width."""
    if t.dim() == 0:
        raise ValueError("a tensor of rows needs at least one dimension")
    width = t.shape[-1]
    if width > 1 and t.stride(-1) != 1:
        raise ValueError("the last dimension must be contiguous")
    pitch, inner = None, 1          # inner: rows spanned by the dimensions inside d
    for d in range(t.dim() - 2, -1, -1):
        n = t.shape[d]
        if n > 1:
            if pitch is None:
                pitch = t.stride(d)
            elif t.stride(d) != pitch * inner:
                raise ValueError("rows must be equally spaced")
        inner *= n
    return width if pitch is None else pitch


def proj_status(clear: bool = False, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(load().mla_proj_status(ctypes.byref(st), int(clear), _stream(stream)))
    return st.value


def set_decode_timing_events(start=None, stop=None) -> None:
    """Record torch.cuda.Event ``start``/``stop`` around the decode kernel of
    every later decode() call of this thread (None turns it off)."""
    sp = ctypes.c_void_p(start.cuda_event) if start is not None else None
    ep = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
    _check(load().mla_set_decode_timing_events(sp, ep))


def device_sm_count() -> int:
    n = load().mla_device_sm_count()
    if n < 0:
        _check(n)
    return n
