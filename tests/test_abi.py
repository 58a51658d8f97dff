"""CPU checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mla_latent_kv_15_gb300 import _build
    import mla_latent_kv_15_gb300 as mla
    _build.build()
    return mla.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    return re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("mla_cache_write", "mla_decode", "mla_merge_states", "mla_decode_workspace_size", "mla_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import mla_latent_kv_15_gb300 as mla
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert set(declared_symbols()) == set(mla.C_ABI_SYMBOLS)


def test_workspace_size_grows_with_splits(lib):
    a = lib.mla_decode_workspace_size(64, 64, 128, 0)
    b = lib.mla_decode_workspace_size(64, 64, 128, 16)
    assert 0 < a < b
    assert lib.mla_decode_workspace_size(0, 64, 128, 0) == 0


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)          # never dereferenced: validation fails first
    # num_heads out of range
    rc = lib.mla_decode(fake, fake, fake, 10, 64, 0, 1.0, fake, 4, fake, 2, None, 2, 0, 0.1, 0, fake, None,
                        fake, 1 << 30, None)
    assert rc == -1 and b"num_heads" in lib.mla_last_error()
    # unsupported page size
    rc = lib.mla_decode(fake, fake, fake, 10, 48, 0, 1.0, fake, 4, fake, 2, None, 2, 16, 0.1, 0, fake, None,
                        fake, 1 << 30, None)
    assert rc == -2 and b"page_size" in lib.mla_last_error()
    # misaligned q_abs
    rc = lib.mla_decode(P((1 << 20) + 2), fake, fake, 10, 64, 0, 1.0, fake, 4, fake, 2, None, 2, 16, 0.1, 0, fake,
                        None, fake, 1 << 30, None)
    assert rc == -1 and b"aligned" in lib.mla_last_error()
    # total_q != batch without query_start_loc
    rc = lib.mla_decode(fake, fake, fake, 10, 64, 0, 1.0, fake, 4, fake, 2, None, 3, 16, 0.1, 0, fake, None,
                        fake, 1 << 30, None)
    assert rc == -1
    # workspace too small
    rc = lib.mla_decode(fake, fake, fake, 10, 64, 0, 1.0, fake, 4, fake, 2, None, 2, 16, 0.1, 0, fake, None,
                        P(1 << 24), 16, None)
    assert rc == -4
    # zero softmax scale
    rc = lib.mla_decode(fake, fake, fake, 10, 64, 0, 1.0, fake, 4, fake, 2, None, 2, 16, 0.0, 0, fake, None,
                        fake, 1 << 30, None)
    assert rc == -1 and b"scale" in lib.mla_last_error()
    # fp8 with a bad scale
    rc = lib.mla_cache_write(fake, fake, fake, 4, fake, 10, 64, 1, 0.0, None)
    assert rc == -1 and b"kv_scale" in lib.mla_last_error()
    # merge: bad dim, aliasing LSE
    rc = lib.mla_merge_states(fake, fake, fake, fake, 10, 12, 2, fake, None, None)
    assert rc == -1
    rc = lib.mla_merge_states(fake, P(64), fake, P(128), 10, 512, 2, fake, P(64), None)
    assert rc == -1 and b"alias" in lib.mla_last_error()
    # empty work is a no-op that never touches the device
    assert lib.mla_decode(None, None, None, 1, 64, 0, 1.0, None, 1, None, 0, None, 0, 16, 0.1, 0, None, None,
                          None, 0, None) == 0
    assert lib.mla_cache_write(None, None, None, 0, None, 1, 64, 0, 1.0, None) == 0
    assert lib.mla_last_error() == b""


def test_projection_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    x, w, y = P(1 << 20), P(1 << 28), P(1 << 32)       # never dereferenced
    # unsupported widths
    assert lib.mla_v_up_proj(x, w, 4, 2, 96, y, None) == -2 and b"v_head_dim" in lib.mla_last_error()
    assert lib.mla_q_absorb(x, 128, w, 4, 2, 100, y, None) == -2 and b"nope_dim" in lib.mla_last_error()
    # row stride below the width or not a multiple of 8
    assert lib.mla_q_absorb(x, 64, w, 4, 2, 128, y, None) == -1 and b"q_row_stride" in lib.mla_last_error()
    assert lib.mla_q_absorb(x, 196, w, 4, 2, 128, y, None) == -1
    # head count, misalignment, null pointers, overlap of input and output
    assert lib.mla_v_up_proj(x, w, 4, 0, 128, y, None) == -1 and b"num_heads" in lib.mla_last_error()
    assert lib.mla_v_up_proj(P((1 << 20) + 8), w, 4, 2, 128, y, None) == -1
    assert lib.mla_v_up_proj(None, w, 4, 2, 128, y, None) == -1
    assert lib.mla_v_up_proj(x, w, 4, 2, 128, P((1 << 20) + 64), None) == -1 and b"overlap" in lib.mla_last_error()
    assert lib.mla_q_absorb(x, 192, w, -1, 2, 128, y, None) == -1
    # empty batch is a no-op that touches nothing
    assert lib.mla_v_up_proj(None, None, 0, 2, 128, None, None) == 0
    assert lib.mla_q_absorb(None, 128, None, 0, 2, 128, None, None) == 0
    assert lib.mla_last_error() == b""
    assert lib.mla_proj_status(None, 0, None) == -1


def test_quantize_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    x, o = P(1 << 20), P(1 << 24)
    assert lib.mla_quantize_fp8(x, 64, 10, 64, 0.0, o, 64, None) == -1 and b"scale" in lib.mla_last_error()
    assert lib.mla_quantize_fp8(x, 64, -1, 64, 1.0, o, 64, None) == -1
    assert lib.mla_quantize_fp8(x, 64, 10, 60, 1.0, o, 64, None) == -1 and b"width" in lib.mla_last_error()
    assert lib.mla_quantize_fp8(x, 32, 10, 64, 1.0, o, 64, None) == -1 and b"stride" in lib.mla_last_error()
    assert lib.mla_quantize_fp8(P((1 << 20) + 8), 64, 10, 64, 1.0, o, 64, None) == -1
    assert lib.mla_quantize_fp8(None, 64, 10, 64, 1.0, o, 64, None) == -1
    assert lib.mla_quantize_fp8(None, 64, 0, 64, 1.0, None, 64, None) == 0


def test_gather_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    c, bt, cu, d = P(1 << 20), P(1 << 24), P(1 << 26), P(1 << 28)    # never dereferenced
    assert lib.mla_gather_cache(c, 10, 64, 3, 1.0, bt, 4, cu, None, 2, d, 100, None, None) == -1
    assert b"cache_dtype" in lib.mla_last_error()
    assert lib.mla_gather_cache(c, 10, 0, 0, 1.0, bt, 4, cu, None, 2, d, 100, None, None) == -1
    assert lib.mla_gather_cache(c, 10, 64, 1, 0.0, bt, 4, cu, None, 2, d, 100, None, None) == -1
    assert b"kv_scale" in lib.mla_last_error()
    assert lib.mla_gather_cache(c, 10, 64, 0, 1.0, bt, 4, None, None, 2, d, 100, None, None) == -1
    assert lib.mla_gather_cache(P((1 << 20) + 8), 10, 64, 0, 1.0, bt, 4, cu, None, 2, d, 100, None, None) == -1
    assert lib.mla_gather_cache(c, 10, 64, 0, 1.0, bt, 4, cu, None, 2, d, 100, P((1 << 20) + 2), None) == -1
    assert lib.mla_gather_cache(c, 10, 64, 0, 1.0, bt, 4, cu, None, 2, d, -1, None, None) == -1
    # nothing to gather: no-op
    assert lib.mla_gather_cache(None, 0, 0, 0, 0.0, None, 0, None, None, 0, None, 0, None, None) == 0
    assert lib.mla_last_error() == b""


def test_product_fails_loudly_without_library(tmp_path):
    """No fallback: a missing library is an ImportError, not a CPU path."""
    import mla_latent_kv_15_gb300 as mla
    saved = mla._lib
    mla._lib = None
    try:
        with pytest.raises(ImportError):
            mla.load(str(tmp_path / "missing.so"))
    finally:
        mla._lib = saved


def test_row_pitch_of_strided_tensors():
    """The binding's row pitch (host logic of mla_quantize_fp8's wrapper):
    column slices of wider rows, size-1 dimensions with any stride, and the
    layouts it must refuse."""
    import torch
    from mla_latent_kv_15_gb300 import _row_pitch
    q8 = torch.empty((7, 16, 576), dtype=torch.uint8)
    assert _row_pitch(q8) == 576
    assert _row_pitch(q8[..., :512]) == 576 and _row_pitch(q8[..., 512:]) == 576
    assert _row_pitch(q8[3]) == 576 and _row_pitch(q8[3, 5]) == 576        # one row: its width
    assert _row_pitch(torch.empty((5, 1, 64)).transpose(0, 1)) == 64      # size-1 dim, any stride
    assert _row_pitch(torch.empty((1, 1, 64))) == 64
    assert _row_pitch(q8[:, :1, :512]) == 16 * 576                        # one head of each token
    with pytest.raises(ValueError):
        _row_pitch(q8[::2])                                                # gaps between tokens
    with pytest.raises(ValueError):
        _row_pitch(q8.transpose(1, 2))                                     # non-contiguous rows
    with pytest.raises(ValueError):
        _row_pitch(torch.empty(()))


def test_binding_refuses_host_tensors_and_bad_cache_width():
    """The binding hands the library device addresses only: host tensors and
    caches of the wrong row width are refused before any call."""
    import torch
    import mla_latent_kv_15_gb300 as mla
    with pytest.raises(ValueError, match="CUDA tensor"):
        mla._ptr(torch.empty(4))
    assert mla._ptr(None) is None
    with pytest.raises(ValueError, match="576"):
        mla.cache_write(None, None, None, torch.empty((2, 64, 512), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="576"):
        mla.gather_cache(torch.empty((2, 64, 512), dtype=torch.bfloat16), None, torch.zeros(2), None)


def test_fp8_query_decode_validation_rejects_before_launch(lib):
    """mla_decode_fp8q refuses bad scales, a misaligned or missing query and a
    short workspace on the host; an empty batch is a no-op."""
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def call(q=fake, q_scale=0.5, kv_scale=0.01, batch=2, total_q=2, ws_bytes=1 << 30):
        return lib.mla_decode_fp8q(q, q_scale, fake, 10, 64, kv_scale, fake, 4, fake, batch, None, total_q, 16,
                                   0.1, 0, fake, None, fake, ws_bytes, None)

    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert call(q_scale=bad) == -1 and b"q_scale" in lib.mla_last_error()
    assert call(kv_scale=0.0) == -1
    assert call(q_scale=1e-30, kv_scale=1e-30) == -1 and b"normal" in lib.mla_last_error()
    assert call(q=P((1 << 20) + 8)) == -1 and b"aligned" in lib.mla_last_error()
    assert call(q=None) == -1 and b"null" in lib.mla_last_error()
    assert call(ws_bytes=16) != 0 and b"workspace" in lib.mla_last_error()
    assert call(batch=0, total_q=0) == 0


def test_step_validation_rejects_before_launch(lib):
    """mla_decode_step and mla_decode_fp8q_step check the write's and the
    decode's arguments on the host before anything is launched; with no
    query rows and no new rows they are no-ops."""
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def step(kv=fake, n_new=4, cache_dtype=0, kv_scale=1.0, num_heads=16, page_size=64, batch=2, total_q=2):
        return lib.mla_decode_step(kv, fake, fake, n_new, fake, fake, fake, 10, page_size, cache_dtype, kv_scale,
                                   fake, 4, fake, batch, None, total_q, num_heads, 0.1, 0, fake, None, fake,
                                   1 << 30, None)

    assert step(n_new=-1) == -1 and b"num_tokens" in lib.mla_last_error()
    assert step(kv=P((1 << 20) + 4)) == -1 and b"aligned" in lib.mla_last_error()
    assert step(cache_dtype=1, kv_scale=0.0) == -1 and b"kv_scale" in lib.mla_last_error()
    assert step(num_heads=0) == -1 and b"num_heads" in lib.mla_last_error()
    assert step(page_size=48) == -2 and b"page_size" in lib.mla_last_error()
    assert step(n_new=0, batch=0, total_q=0) == 0

    def step8(q8=fake, q_scale=0.5, n_new=4, batch=2, total_q=2):
        return lib.mla_decode_fp8q_step(fake, fake, fake, n_new, fake, fake, q_scale, q8, fake, 10, 64, 0.01, fake,
                                        4, fake, batch, None, total_q, 16, 0.1, 0, fake, None, fake, 1 << 30, None)

    assert step8(q_scale=0.0) == -1 and b"q_scale" in lib.mla_last_error()
    assert step8(q8=None) == -1 and b"null" in lib.mla_last_error()
    assert step8(q8=P((1 << 20) + 8)) == -1 and b"aligned" in lib.mla_last_error()
    assert step8(n_new=0, batch=0, total_q=0) == 0


def test_binding_refuses_layouts_the_kernels_would_misread():
    """The kernels read dense rows of fixed element types; the binding refuses
    column slices, transposed views and wrong integer widths before any call
    (host tensors suffice: the checks come before any device address)."""
    import torch
    import mla_latent_kv_15_gb300 as mla
    cache = torch.empty((4, 64, 576), dtype=torch.bfloat16)
    proj = torch.empty((8, 640), dtype=torch.bfloat16)          # a [T, 576 + 64] projection output
    kv_c_slice = proj[:, :512]                                  # column slice: rows 640 apart
    k_pe = torch.empty((8, 64), dtype=torch.bfloat16)
    slots64 = torch.arange(8, dtype=torch.int64)
    with pytest.raises(ValueError, match="kv_c must be contiguous"):
        mla.cache_write(kv_c_slice, k_pe, slots64, cache)
    with pytest.raises(ValueError, match="slot_mapping must be int64"):
        mla.cache_write(torch.empty((8, 512), dtype=torch.bfloat16), k_pe, slots64.to(torch.int32), cache)
    with pytest.raises(ValueError, match="k_pe must have shape"):
        mla.cache_write(torch.empty((8, 512), dtype=torch.bfloat16), k_pe[:4], slots64, cache)
    with pytest.raises(ValueError, match="kv_c must be bfloat16"):
        mla.cache_write(torch.empty((8, 512), dtype=torch.float16), k_pe, slots64, cache)

    T, N, B = 4, 16, 4
    q_abs = torch.empty((T, N, 512), dtype=torch.bfloat16)
    q_pe = torch.empty((T, N, 64), dtype=torch.bfloat16)
    bt = torch.zeros((B, 2), dtype=torch.int32)
    sl = torch.ones(B, dtype=torch.int32)
    out = torch.empty((T, N, 512), dtype=torch.bfloat16)
    ws = torch.empty(1 << 20, dtype=torch.uint8)
    ok = dict(q_abs=q_abs, q_pe=q_pe, cache=cache, block_table=bt, seq_lens=sl, out=out, workspace=ws)

    def call(**over):
        kw = dict(ok)
        kw.update(over)
        mla.decode(kw["q_abs"], kw["q_pe"], kw["cache"], kw["block_table"], kw["seq_lens"], kw["out"],
                   kw["workspace"], scale=0.07, lse=kw.get("lse"), query_start_loc=kw.get("qsl"))

    with pytest.raises(ValueError, match="q_abs must be contiguous"):
        call(q_abs=torch.empty((N, T, 512), dtype=torch.bfloat16).transpose(0, 1))   # a bmm's [N, T, L] output
    with pytest.raises(ValueError, match="q_pe must have shape"):
        call(q_pe=torch.empty((T, N, 32), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="block_table must be int32"):
        call(block_table=bt.to(torch.int64))
    with pytest.raises(ValueError, match="seq_lens must be int32"):
        call(seq_lens=sl.to(torch.int64))
    with pytest.raises(ValueError, match="query_start_loc must have shape"):
        call(qsl=torch.zeros(B, dtype=torch.int32))
    with pytest.raises(ValueError, match="out must be bfloat16"):
        call(out=torch.empty((T, N, 512), dtype=torch.float32))
    with pytest.raises(ValueError, match="lse must be float32"):
        call(lse=torch.empty((T, N), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="cache rows must be 576"):
        call(cache=torch.empty((4, 64, 512), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="cache must be"):
        call(cache=torch.empty((4, 64, 576), dtype=torch.float32))
    # a well-formed call gets past every check (and then needs the device)
    with pytest.raises(ValueError, match="CUDA tensor"):
        call()
    # merge: mismatched partner shapes and LSE dtype
    o = torch.empty((10, 512), dtype=torch.float32)
    l32 = torch.empty(10, dtype=torch.float32)
    with pytest.raises(ValueError, match="o_b must have shape"):
        mla.merge_states(o, l32, torch.empty((10, 256), dtype=torch.float32), l32, o)
    with pytest.raises(ValueError, match="lse_b must be float32"):
        mla.merge_states(o, l32, o, l32.double(), o)
