"""CPU oracle for the paged KV-cache write and PagedAttention (fp64).

TEST INFRASTRUCTURE ONLY.  The product path never imports, links or calls
anything in this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` do.  It shares no code with the CUDA library
in ``paged_kv_cache_43_gb300``; the two meet only through the seeded inputs of
``paged_kv_cache_43_gb300.workloads``.

Two independent implementations live here:

* ``pkv_oracle.c`` (loaded through ctypes): walks each sequence's block table
  key by key and accumulates in fp64, OpenMP-parallel over (row, head).
* ``brute.py``: numpy, densifies each sequence's keys first and applies a
  plain softmax; for tiny inputs only.

Sources are the pages "Implémentation du cœur du moteur d'inférence haute
performance vLLM" (AiReadCodeBooks), ch. 5 and ch. 6, and "Khám phá vLLM: Giải
phẫu hệ thống suy luận LLM thông lượng cao" (KV cache manager note,
allocate_slots); each function cites its section.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, FP8 = 0, 1, 2


class OrcProblem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p),
        ("context_lens", ctypes.c_void_p),
        ("query_start_loc", ctypes.c_void_p),
        ("bt_stride", ctypes.c_int64),
        ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("window", ctypes.c_int32),
        ("k_descale", ctypes.c_void_p),
        ("v_descale", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``_build/liboracle.so`` (gcc -O2, OpenMP,
    no fast-math).  Returns the library path."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.orc_write.restype = ctypes.c_int64
        lib.orc_write.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_int32]
        lib.orc_row_state.restype = ctypes.c_int
        lib.orc_row_state.argtypes = [ctypes.POINTER(OrcProblem), ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                      ctypes.c_int64, ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
        lib.orc_merge.restype = None
        lib.orc_merge.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
        lib.orc_attention.restype = ctypes.c_int32
        lib.orc_attention.argtypes = [ctypes.POINTER(OrcProblem), ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_int32]
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_write_fp8.restype = ctypes.c_int64
        lib.orc_write_fp8.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        lib.orc_max_threads.restype = ctypes.c_int32
        lib.orc_max_threads.argtypes = []
        _lib = lib
    return _lib


def _raw(a: np.ndarray) -> np.ndarray:
    """A C-contiguous numpy array (bit patterns untouched)."""
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def dtype_code(arr: np.ndarray) -> int:
    """Storage code of a cache/query array: float32 -> F32, uint16 (bf16 bit
    patterns) -> BF16, uint8 (e4m3 codes) -> FP8."""
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.uint8:
        return FP8
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits), got {arr.dtype}")


def e4m3_decode(code: int) -> float:
    """Value of one e4m3 code (FP8 KV cache, ch. 6 capability matrix)."""
    return float(_load().orc_e4m3_decode(int(code)))


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code of an fp32 value (ties to even, clamped to 448)."""
    return int(_load().orc_e4m3_encode(float(x)))


def write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale) -> int:
    """FP8 KV write: k/v bf16 bits (uint16) [T, Hkv, D] quantised to e4m3 codes
    with per-kv-head scales (encode(k / scale) in fp32) into uint8 caches
    [NB, bs, Hkv, D], in place.  Returns the number of out-of-range slots."""
    lib = _load()
    k, v = _raw(np.asarray(k, np.uint16)), _raw(np.asarray(v, np.uint16))
    slots = _raw(np.asarray(slot_mapping, dtype=np.int64))
    ks = _raw(np.asarray(k_scale, np.float32))
    vs = _raw(np.asarray(v_scale, np.float32))
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    nb, bs, hkv, d = k_cache.shape
    return int(lib.orc_write_fp8(_ptr(k), _ptr(v), _ptr(slots), slots.shape[0], _ptr(k_cache),
                                 _ptr(v_cache), nb, bs, hkv, d, _ptr(ks), _ptr(vs)))


def write(k, v, slot_mapping, k_cache, v_cache) -> int:
    """KV-cache write ("Écriture du KV cache", ch. 6 of the vLLM core book;
    -1 padding of slot_mapping, ch. 5): copies row t of ``k``/``v`` into cache
    row ``slot_mapping[t]`` for every slot >= 0, in place.  ``k``/``v`` are
    [T, Hkv, D], caches [NB, bs, Hkv, D], all float32 or uint16 (bf16 bits).
    Returns the number of out-of-range slots (skipped)."""
    lib = _load()
    k, v = _raw(k), _raw(v)
    slots = _raw(np.asarray(slot_mapping, dtype=np.int64))
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    nb, bs, hkv, d = k_cache.shape
    return int(lib.orc_write(_ptr(k), _ptr(v), _ptr(slots), slots.shape[0],
                             _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d,
                             k_cache.dtype.itemsize))


class Problem:
    """Keeps the numpy buffers of one attention problem alive for ctypes."""

    def __init__(self, q, k_cache, v_cache, block_tables, context_lens,
                 query_start_loc, scale, window: int = 0, k_descale=None, v_descale=None):
        self.q = _raw(q)
        self.k_cache = _raw(k_cache)
        self.v_cache = _raw(v_cache)
        self.block_tables = _raw(np.asarray(block_tables, dtype=np.int32))
        self.context_lens = _raw(np.asarray(context_lens, dtype=np.int32))
        self.query_start_loc = _raw(np.asarray(query_start_loc, dtype=np.int32))
        code = dtype_code(self.k_cache)
        assert code == dtype_code(self.v_cache)
        assert dtype_code(self.q) == (BF16 if code == FP8 else code)
        self.k_descale = self.v_descale = None
        if code == FP8:
            self.k_descale = _raw(np.asarray(k_descale, np.float32))
            self.v_descale = _raw(np.asarray(v_descale, np.float32))
        nb, bs, hkv, d = self.k_cache.shape
        self.num_tokens, hq, dq = self.q.shape
        assert dq == d and hq % hkv == 0
        s = self.context_lens.shape[0]
        assert self.query_start_loc.shape[0] == s + 1
        self.shape = dict(S=s, Hq=hq, Hkv=hkv, D=d, bs=bs, NB=nb)
        self.c = OrcProblem(
            _ptr(self.q), _ptr(self.k_cache), _ptr(self.v_cache),
            _ptr(self.block_tables), _ptr(self.context_lens), _ptr(self.query_start_loc),
            self.block_tables.shape[1] if self.block_tables.ndim == 2 else 0,
            s, hq, hkv, d, bs, nb, code, float(scale), int(window),
            _ptr(self.k_descale) if self.k_descale is not None else None,
            _ptr(self.v_descale) if self.v_descale is not None else None)


def attention(q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
              scale, nthreads: int = 0, window: int = 0, k_descale=None, v_descale=None):
    """Exact paged attention in fp64 (ch. 6 "Structure des métadonnées",
    "Flux des paramètres du chemin non-cascadé", "Branche de masque"); with
    ``window`` W > 0 a query at position pos sees keys pos - W < p <= pos.
    With uint8 (e4m3) caches, q is bf16 and K/V are decode(code) times
    ``k_descale`` / ``v_descale`` [num_seqs, num_kv_heads].

    Returns ``(out, seq_status)``: ``out`` is float64 [T, Hq, D]; rows of a
    sequence with status 1 (metadata error) are zero, status 2 (block id out of
    range) NaN."""
    lib = _load()
    P = Problem(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, window,
                k_descale, v_descale)
    out = np.zeros((P.num_tokens, P.shape["Hq"], P.shape["D"]), dtype=np.float64)
    status = np.zeros(P.shape["S"], dtype=np.int32)
    lib.orc_attention(ctypes.byref(P.c), _ptr(out), _ptr(status), int(nthreads))
    return out, status


def row_state(problem: Problem, s: int, hq: int, j: int, p_lo: int = 0,
              p_hi: int = 2**62):
    """Unnormalised softmax state (m, l, acc[D]) of one query row over the
    visible keys in [p_lo, p_hi): the per-split partial of the split buffer
    (ch. 6 "build() étape par étape", fourth step)."""
    lib = _load()
    m = ctypes.c_double()
    l = ctypes.c_double()
    acc = np.zeros(problem.shape["D"], dtype=np.float64)
    st = lib.orc_row_state(ctypes.byref(problem.c), s, hq, j, p_lo, p_hi,
                           ctypes.byref(m), ctypes.byref(l), _ptr(acc))
    return st, m.value, l.value, acc


def merge(ms, ls, accs):
    """Merge partial states into one normalised row (merge_attn_states of the
    ch. 6 sequence diagram)."""
    lib = _load()
    m = _raw(np.asarray(ms, dtype=np.float64))
    l = _raw(np.asarray(ls, dtype=np.float64))
    a = _raw(np.asarray(accs, dtype=np.float64))
    n, d = a.shape
    out = np.zeros(d, dtype=np.float64)
    lib.orc_merge(n, _ptr(m), _ptr(l), _ptr(a), d, _ptr(out))
    return out


def cascade(problem: Problem, prefix_len: int):
    """Cascade attention of a batch whose sequences share their first
    ``prefix_len`` keys ("Implémentation du cœur ... vLLM", ch. 6: the cascade
    branch runs a prefix call over every query token of the batch and a suffix
    call over each sequence's own keys, and merges them with
    merge_attn_states): per (query row, q head), the state over the shared
    keys [0, prefix_len) — the same physical blocks in every sequence's table,
    the caller's contract — and the state over the row's own visible keys
    from prefix_len on (causal inside a chunk), merged.  float64 [T, Hq, D].
    Every query row must sit after the prefix (position >= prefix_len): then
    all shared keys are visible to it and the split is exact."""
    sh = problem.shape
    out = np.zeros((problem.num_tokens, sh["Hq"], sh["D"]), dtype=np.float64)
    for s in range(sh["S"]):
        q0 = int(problem.query_start_loc[s])
        qn = int(problem.query_start_loc[s + 1]) - q0
        L = int(problem.context_lens[s])
        assert L - qn >= prefix_len, "a query row inside the shared prefix"
        for j in range(qn):
            for hq in range(sh["Hq"]):
                st0, m0, l0, a0 = row_state(problem, s, hq, j, 0, prefix_len)
                st1, m1, l1, a1 = row_state(problem, s, hq, j, prefix_len)
                assert st0 == 0 and st1 == 0
                out[q0 + j, hq] = merge([m0, m1], [l0, l1], [a0, a1])
    return out


def max_threads() -> int:
    return int(_load().orc_max_threads())
