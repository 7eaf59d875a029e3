"""Thin ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every step of the path runs in the CUDA kernels behind the C ABI; this module
only checks tensor shapes/dtypes, fills the descriptor structs and passes data
pointers and the current CUDA stream.  If the library cannot be loaded the
calls raise: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_lock = threading.Lock()
_lib = None

PKV_F32, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
# FP8 caches hold e4m3 codes; either dtype may carry them.
FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn)
ERR_SLOT = 1 << 0
ERR_BLOCK_ID = 1 << 1
ERR_CONTEXT_LEN = 1 << 2
ERR_QUERY_LEN = 1 << 3
ERR_DECODE_QLEN = 1 << 4
ERR_TIMEOUT = 1 << 5
EXPORTED = ("pkv_write", "pkv_write_fp8", "pkv_attention_workspace_size", "pkv_attention",
            "pkv_attention_fp8", "pkv_attention_static_scratch",
            "pkv_attention_cascade_workspace_size", "pkv_attention_cascade",
            "pkv_attention_cascade_fp8", "pkv_use_cascade",
            "pkv_get_error", "pkv_status_string", "pkv_last_cuda_error",
            "pkv_last_cuda_error_string", "pkv_debug_wait_test")
STATIC_SCRATCH_BYTES = 64 << 20


class PkvError(RuntimeError):
    pass


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_size", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class AttnMeta(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("block_table_stride", ctypes.c_int32),
                ("max_query_len", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
                ("num_decode_seqs", ctypes.c_int32), ("sliding_window", ctypes.c_int32),
                ("kv_split_tokens", ctypes.c_int32)]


def library_path() -> str:
    from . import build as _b
    return _b.LIB_PATH


def load(path: str | None = None):
    """Load libpkv.so (built by ``paged_kv_cache_43_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or library_path()
        if not os.path.exists(path):
            raise PkvError(f"libpkv.so not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i32, i64p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
        lib.pkv_write.restype = ctypes.c_int
        lib.pkv_write.argtypes = [vp, vp, i64p, i32, vp, vp, ctypes.POINTER(CacheDesc), vp]
        lib.pkv_attention_workspace_size.restype = ctypes.c_size_t
        lib.pkv_attention_workspace_size.argtypes = [ctypes.POINTER(CacheDesc),
                                                     ctypes.POINTER(AttnMeta)]
        lib.pkv_attention.restype = ctypes.c_int
        lib.pkv_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                      ctypes.POINTER(CacheDesc), ctypes.POINTER(AttnMeta),
                                      vp, ctypes.c_size_t, vp]
        lib.pkv_write_fp8.restype = ctypes.c_int
        lib.pkv_write_fp8.argtypes = [vp, vp, i64p, i32, vp, vp, vp, vp,
                                      ctypes.POINTER(CacheDesc), vp]
        lib.pkv_attention_fp8.restype = ctypes.c_int
        lib.pkv_attention_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                          ctypes.POINTER(CacheDesc), ctypes.POINTER(AttnMeta),
                                          vp, ctypes.c_size_t, vp]
        lib.pkv_attention_cascade_workspace_size.restype = ctypes.c_size_t
        lib.pkv_attention_cascade_workspace_size.argtypes = [ctypes.POINTER(CacheDesc),
                                                             ctypes.POINTER(AttnMeta), i32]
        lib.pkv_attention_cascade.restype = ctypes.c_int
        lib.pkv_attention_cascade.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, i32,
                                              ctypes.POINTER(CacheDesc), ctypes.POINTER(AttnMeta),
                                              vp, ctypes.c_size_t, vp]
        lib.pkv_attention_cascade_fp8.restype = ctypes.c_int
        lib.pkv_attention_cascade_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, i32,
                                                  vp, vp, ctypes.POINTER(CacheDesc),
                                                  ctypes.POINTER(AttnMeta), vp, ctypes.c_size_t,
                                                  vp]
        lib.pkv_use_cascade.restype = ctypes.c_int
        lib.pkv_use_cascade.argtypes = [ctypes.POINTER(AttnMeta), i32]
        lib.pkv_attention_static_scratch.restype = ctypes.c_int
        lib.pkv_attention_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                                     ctypes.POINTER(CacheDesc),
                                                     ctypes.POINTER(AttnMeta), vp]
        lib.pkv_get_error.restype = ctypes.c_int
        lib.pkv_get_error.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_last_cuda_error.restype = ctypes.c_int
        lib.pkv_last_cuda_error.argtypes = []
        lib.pkv_last_cuda_error_string.restype = ctypes.c_char_p
        lib.pkv_last_cuda_error_string.argtypes = []
        lib.pkv_debug_wait_test.restype = ctypes.c_int
        lib.pkv_debug_wait_test.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        lib = load()
        msg = f"pkv status {status}: {lib.pkv_status_string(status).decode()}"
        if status == -7:   # PKV_E_CUDA: say which CUDA error
            msg += f" ({lib.pkv_last_cuda_error_string().decode()})"
        raise PkvError(msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    if t.dtype == torch.float32:
        return PKV_F32
    if t.dtype in FP8_DTYPES:
        return PKV_FP8_E4M3
    raise PkvError(f"unsupported dtype {t.dtype}")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    nb, bs, hkv, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d, _dtype_code(k_cache))


def _require(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not t.is_cuda:
        raise PkvError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PkvError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PkvError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise PkvError(f"{name} must have {ndim} dims")


def write(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """pkv_write: scatter k/v [T, Hkv, D] into the caches at slot_mapping[T]."""
    lib = load()
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n, dtype=k_cache.dtype)
    _require(slot_mapping, "slot_mapping", dtype=torch.int64, ndim=1)
    T = slot_mapping.shape[0]
    if k.shape[0] < T or v.shape[0] < T:
        raise PkvError("k/v have fewer rows than slot_mapping")
    desc = cache_desc(k_cache)
    _check(lib.pkv_write(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                         k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                         _stream(stream)))


def write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None) -> None:
    """pkv_write_fp8: quantise bf16 k/v [T, Hkv, D] with the per-kv-head
    scales (fp32 [Hkv]) into the e4m3 caches at slot_mapping[T]."""
    lib = load()
    for t, n in ((k, "k"), (v, "v")):
        _require(t, n, dtype=torch.bfloat16)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n)
        if t.dtype not in FP8_DTYPES:
            raise PkvError(f"{n} must hold e4m3 codes (uint8 or float8_e4m3fn)")
    hkv = k_cache.shape[2]
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _require(t, n, dtype=torch.float32, ndim=1)
        if t.shape[0] != hkv:
            raise PkvError(f"{n} must have num_kv_heads entries")
    _require(slot_mapping, "slot_mapping", dtype=torch.int64, ndim=1)
    T = slot_mapping.shape[0]
    if k.shape[0] < T or v.shape[0] < T:
        raise PkvError("k/v have fewer rows than slot_mapping")
    desc = cache_desc(k_cache)
    _check(lib.pkv_write_fp8(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                             k_cache.data_ptr(), v_cache.data_ptr(), k_scale.data_ptr(),
                             v_scale.data_ptr(), ctypes.byref(desc), _stream(stream)))


def attn_meta(q, block_tables, context_lens, *, max_query_len, max_context_len,
              num_decode_seqs=-1, kv_split_tokens=0, sliding_window=0) -> AttnMeta:
    return AttnMeta(int(context_lens.shape[0]), int(q.shape[0]), int(q.shape[1]),
                    int(block_tables.shape[1]), int(max_query_len), int(max_context_len),
                    int(num_decode_seqs), int(sliding_window), int(kv_split_tokens))


def workspace_size(k_cache, meta: AttnMeta) -> int:
    desc = cache_desc(k_cache)
    n = load().pkv_attention_workspace_size(ctypes.byref(desc), ctypes.byref(meta))
    if n == ctypes.c_size_t(-1).value:
        raise PkvError("invalid attention description")
    return int(n)


def attention(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale,
              *, max_query_len, max_context_len, num_decode_seqs=-1, kv_split_tokens=0,
              sliding_window=0, workspace=None, stream=None) -> None:
    """pkv_attention into ``out`` [T, Hq, D].  ``workspace`` (uint8 CUDA tensor)
    is allocated here when not given and the batch needs split-K scratch."""
    lib = load()
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n, dtype=k_cache.dtype)
    _require(block_tables, "block_tables", dtype=torch.int32, ndim=2)
    _require(context_lens, "context_lens", dtype=torch.int32, ndim=1)
    _require(query_start_loc, "query_start_loc", dtype=torch.int32, ndim=1)
    if out.shape != q.shape:
        raise PkvError("out and q must have the same shape")
    meta = attn_meta(q, block_tables, context_lens, max_query_len=max_query_len,
                     max_context_len=max_context_len, num_decode_seqs=num_decode_seqs,
                     kv_split_tokens=kv_split_tokens, sliding_window=sliding_window)
    desc = cache_desc(k_cache)
    need = workspace_size(k_cache, meta)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.pkv_attention(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(),
                             v_cache.data_ptr(), block_tables.data_ptr(),
                             context_lens.data_ptr(), query_start_loc.data_ptr(),
                             float(scale), ctypes.byref(desc), ctypes.byref(meta),
                             ws_ptr, ws_bytes, _stream(stream)))


def attention_fp8(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale,
                  k_descale, v_descale, *, max_query_len, max_context_len, num_decode_seqs=-1,
                  kv_split_tokens=0, sliding_window=0, workspace=None, stream=None) -> None:
    """pkv_attention_fp8 into ``out`` [T, Hq, D] (bf16) over e4m3 caches;
    ``k_descale``/``v_descale`` fp32 [num_seqs, Hkv]."""
    lib = load()
    for t, n in ((out, "out"), (q, "q")):
        _require(t, n, dtype=torch.bfloat16)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n)
        if t.dtype not in FP8_DTYPES:
            raise PkvError(f"{n} must hold e4m3 codes (uint8 or float8_e4m3fn)")
    _require(block_tables, "block_tables", dtype=torch.int32, ndim=2)
    _require(context_lens, "context_lens", dtype=torch.int32, ndim=1)
    _require(query_start_loc, "query_start_loc", dtype=torch.int32, ndim=1)
    for t, n in ((k_descale, "k_descale"), (v_descale, "v_descale")):
        _require(t, n, dtype=torch.float32, ndim=2)
        if tuple(t.shape) != (context_lens.shape[0], k_cache.shape[2]):
            raise PkvError(f"{n} must be [num_seqs, num_kv_heads]")
    if out.shape != q.shape:
        raise PkvError("out and q must have the same shape")
    meta = attn_meta(q, block_tables, context_lens, max_query_len=max_query_len,
                     max_context_len=max_context_len, num_decode_seqs=num_decode_seqs,
                     kv_split_tokens=kv_split_tokens, sliding_window=sliding_window)
    desc = cache_desc(k_cache)
    need = workspace_size(k_cache, meta)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.pkv_attention_fp8(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(),
                                 v_cache.data_ptr(), block_tables.data_ptr(),
                                 context_lens.data_ptr(), query_start_loc.data_ptr(),
                                 float(scale), k_descale.data_ptr(), v_descale.data_ptr(),
                                 ctypes.byref(desc), ctypes.byref(meta), ws_ptr, ws_bytes,
                                 _stream(stream)))


def cascade_workspace_size(k_cache, meta: AttnMeta, common_prefix_blocks: int) -> int:
    desc = cache_desc(k_cache)
    n = load().pkv_attention_cascade_workspace_size(ctypes.byref(desc), ctypes.byref(meta),
                                                    int(common_prefix_blocks))
    if n == ctypes.c_size_t(-1).value:
        raise PkvError("invalid cascade description")
    return int(n)


def use_cascade(meta: AttnMeta, common_prefix_blocks: int) -> bool:
    """The cascade gate (>= 256 shared tokens, >= 8 sequences, no window,
    decode rows)."""
    return bool(load().pkv_use_cascade(ctypes.byref(meta), int(common_prefix_blocks)))


def attention_cascade(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale,
                      common_prefix_blocks, *, max_context_len, max_query_len=1,
                      num_decode_seqs=-1, kv_split_tokens=0, workspace=None,
                      stream=None) -> None:
    """pkv_attention_cascade: a batch (decode rows, then chunked-prefill
    sequences) whose sequences share their first ``common_prefix_blocks``
    blocks; same result as attention()."""
    lib = load()
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n, dtype=k_cache.dtype)
    _require(block_tables, "block_tables", dtype=torch.int32, ndim=2)
    _require(context_lens, "context_lens", dtype=torch.int32, ndim=1)
    _require(query_start_loc, "query_start_loc", dtype=torch.int32, ndim=1)
    meta = attn_meta(q, block_tables, context_lens, max_query_len=max_query_len,
                     max_context_len=max_context_len, num_decode_seqs=num_decode_seqs,
                     kv_split_tokens=kv_split_tokens)
    desc = cache_desc(k_cache)
    if workspace is None:
        need = cascade_workspace_size(k_cache, meta, common_prefix_blocks)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(lib.pkv_attention_cascade(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(),
                                     v_cache.data_ptr(), block_tables.data_ptr(),
                                     context_lens.data_ptr(), query_start_loc.data_ptr(),
                                     float(scale), int(common_prefix_blocks), ctypes.byref(desc),
                                     ctypes.byref(meta), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def attention_cascade_fp8(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                          scale, common_prefix_blocks, k_descale, v_descale, *, max_context_len,
                          max_query_len=1, num_decode_seqs=-1, kv_split_tokens=0,
                          workspace=None, stream=None) -> None:
    """pkv_attention_cascade_fp8: attention_cascade over e4m3 caches with the
    descales of attention_fp8."""
    lib = load()
    for t, n in ((out, "out"), (q, "q")):
        _require(t, n, dtype=torch.bfloat16)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n)
        if t.dtype not in FP8_DTYPES:
            raise PkvError(f"{n} must hold e4m3 codes (uint8 or float8_e4m3fn)")
    _require(block_tables, "block_tables", dtype=torch.int32, ndim=2)
    _require(context_lens, "context_lens", dtype=torch.int32, ndim=1)
    _require(query_start_loc, "query_start_loc", dtype=torch.int32, ndim=1)
    for t, n in ((k_descale, "k_descale"), (v_descale, "v_descale")):
        _require(t, n, dtype=torch.float32, ndim=2)
        if tuple(t.shape) != (context_lens.shape[0], k_cache.shape[2]):
            raise PkvError(f"{n} must be [num_seqs, num_kv_heads]")
    meta = attn_meta(q, block_tables, context_lens, max_query_len=max_query_len,
                     max_context_len=max_context_len, num_decode_seqs=num_decode_seqs,
                     kv_split_tokens=kv_split_tokens)
    desc = cache_desc(k_cache)
    if workspace is None:
        need = cascade_workspace_size(k_cache, meta, common_prefix_blocks)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(lib.pkv_attention_cascade_fp8(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(),
                                         v_cache.data_ptr(), block_tables.data_ptr(),
                                         context_lens.data_ptr(), query_start_loc.data_ptr(),
                                         float(scale), int(common_prefix_blocks),
                                         k_descale.data_ptr(), v_descale.data_ptr(),
                                         ctypes.byref(desc), ctypes.byref(meta),
                                         workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream)))


def attention_static_scratch(out, q, k_cache, v_cache, block_tables, context_lens,
                             query_start_loc, scale, *, max_query_len, max_context_len,
                             num_decode_seqs=-1, kv_split_tokens=0, sliding_window=0,
                             stream=None) -> int:
    """pkv_attention_static_scratch: pkv_attention with the split-K workspace
    taken from the library's own fixed device array (no allocation anywhere).
    Returns the C status (0 = enqueued; PKV_E_WORKSPACE = batch needs more than
    STATIC_SCRATCH_BYTES)."""
    lib = load()
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n, dtype=k_cache.dtype)
    _require(block_tables, "block_tables", dtype=torch.int32, ndim=2)
    _require(context_lens, "context_lens", dtype=torch.int32, ndim=1)
    _require(query_start_loc, "query_start_loc", dtype=torch.int32, ndim=1)
    meta = attn_meta(q, block_tables, context_lens, max_query_len=max_query_len,
                     max_context_len=max_context_len, num_decode_seqs=num_decode_seqs,
                     kv_split_tokens=kv_split_tokens, sliding_window=sliding_window)
    desc = cache_desc(k_cache)
    return int(lib.pkv_attention_static_scratch(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), context_lens.data_ptr(), query_start_loc.data_ptr(),
        float(scale), ctypes.byref(desc), ctypes.byref(meta), _stream(stream)))


def get_error(clear: bool = True) -> int:
    """Device error word (PKV_ERR_* bits); synchronises the device."""
    bits = ctypes.c_int32(0)
    _check(load().pkv_get_error(ctypes.byref(bits), int(clear)))
    return int(bits.value)


def debug_wait_test(enable: bool) -> None:
    """Test hook of the timeout path (pkv_debug_wait_test): while enabled,
    decode and tcgen05 prefill launches wait at most 20 us and withhold their
    first key block, so their waits run out and PKV_ERR_TIMEOUT is set."""
    _check(load().pkv_debug_wait_test(1 if enable else 0))


def status_string(status: int) -> str:
    return load().pkv_status_string(status).decode()


def run_step(wl, out, workspace=None, kv_split_tokens=0, sliding_window=0, stream=None) -> None:
    """One pass of the hot path over a workload: the KV write of this step's
    tokens, then attention over the updated cache."""
    write(wl.k_new, wl.v_new, wl.slot_mapping, wl.k_cache, wl.v_cache, stream=stream)
    attention(out, wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens,
              wl.query_start_loc, wl.scale, max_query_len=wl.max_query_len,
              max_context_len=wl.max_context_len, num_decode_seqs=wl.num_decode_seqs,
              kv_split_tokens=kv_split_tokens, sliding_window=sliding_window,
              workspace=workspace, stream=stream)
