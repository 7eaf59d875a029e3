"""ctypes binding of the host block pool (include/pkv_pool.h): argument
marshalling only; the pool itself is the C++ in csrc/pkv_pool.cpp, inside
libpkv.so.  Host memory only: these calls need no GPU."""
from __future__ import annotations

import ctypes

import numpy as np

from . import pkv

NO_SPACE = 1
E_REQUEST = -10
EXPORTED = ("pkv_pool_create", "pkv_pool_destroy", "pkv_pool_num_free", "pkv_pool_null_block",
            "pkv_pool_num_cached", "pkv_pool_add_request", "pkv_pool_append_tokens",
            "pkv_pool_append_token_batch",
            "pkv_pool_admit", "pkv_pool_allocate_slots", "pkv_pool_allocate_slots_batch",
            "pkv_pool_free_request",
            "pkv_pool_block_table", "pkv_pool_build_block_tables", "pkv_pool_num_computed",
            "pkv_pool_block_state", "pkv_pool_free_queue")

_sigs_done = False


def _lib():
    global _sigs_done
    lib = pkv.load()
    if not _sigs_done:
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        P32, P64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
        sig = {
            "pkv_pool_create": (vp, [i32, i32, i32]),
            "pkv_pool_destroy": (None, [vp]),
            "pkv_pool_num_free": (i32, [vp]),
            "pkv_pool_null_block": (i32, [vp]),
            "pkv_pool_num_cached": (i32, [vp]),
            "pkv_pool_add_request": (ctypes.c_int, [vp, i64, P32, i32]),
            "pkv_pool_append_tokens": (ctypes.c_int, [vp, i64, P32, i32]),
            "pkv_pool_append_token_batch": (ctypes.c_int, [vp, P64, P32, i32]),
            "pkv_pool_admit": (ctypes.c_int, [vp, i64, P32]),
            "pkv_pool_allocate_slots": (ctypes.c_int, [vp, i64, i32, i32, P64]),
            "pkv_pool_allocate_slots_batch": (ctypes.c_int, [vp, P64, P32, i32, i32, P64, P32]),
            "pkv_pool_free_request": (ctypes.c_int, [vp, i64]),
            "pkv_pool_block_table": (ctypes.c_int, [vp, i64, P32, i32, P32]),
            "pkv_pool_build_block_tables": (ctypes.c_int, [vp, P64, i32, P32, i32]),
            "pkv_pool_num_computed": (ctypes.c_int, [vp, i64, P32]),
            "pkv_pool_block_state": (ctypes.c_int, [vp, i32, P32, ctypes.POINTER(ctypes.c_uint64), P32]),
            "pkv_pool_free_queue": (ctypes.c_int, [vp, P32, i32, P32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _sigs_done = True
    return lib


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


class BlockPool:
    """The C++ pool.  Request ids are ints (int64)."""

    def __init__(self, num_blocks: int, block_size: int = 16, caching: bool = True):
        self._lib = _lib()
        self._p = self._lib.pkv_pool_create(int(num_blocks), int(block_size), int(bool(caching)))
        if not self._p:
            raise pkv.PkvError("pkv_pool_create failed")
        self.block_size = block_size

    def close(self):
        if self._p:
            self._lib.pkv_pool_destroy(self._p)
            self._p = None

    def __del__(self):
        self.close()

    def _check(self, st):
        if st < 0:
            raise pkv.PkvError(f"pool status {st}")
        return st

    @property
    def null_block(self) -> int:
        return int(self._lib.pkv_pool_null_block(self._p))

    def num_free(self) -> int:
        return int(self._lib.pkv_pool_num_free(self._p))

    def cached_blocks(self) -> int:
        return int(self._lib.pkv_pool_num_cached(self._p))

    def add_request(self, req_id: int, tokens):
        a, ptr = _i32(tokens)
        self._check(self._lib.pkv_pool_add_request(self._p, int(req_id), ptr, a.size))

    def append_token(self, req_id: int, token: int):
        self.append_tokens(req_id, [token])

    def append_tokens(self, req_id: int, tokens):
        a, ptr = _i32(tokens)
        self._check(self._lib.pkv_pool_append_tokens(self._p, int(req_id), ptr, a.size))

    def append_token_batch(self, req_ids, tokens):
        ids = np.ascontiguousarray(req_ids, dtype=np.int64)
        t, tp = _i32(tokens)
        self._check(self._lib.pkv_pool_append_token_batch(
            self._p, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), tp, ids.size))

    def admit(self, req_id: int) -> int:
        n = ctypes.c_int32(0)
        self._check(self._lib.pkv_pool_admit(self._p, int(req_id), ctypes.byref(n)))
        return int(n.value)

    def allocate_slots(self, req_id: int, num_new_tokens: int, window: int = 0):
        """np.int64 slots of the new positions, or None when the pool is short."""
        out = np.empty(max(int(num_new_tokens), 1), dtype=np.int64)
        st = self._check(self._lib.pkv_pool_allocate_slots(
            self._p, int(req_id), int(num_new_tokens), int(window),
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
        return None if st == NO_SPACE else out[:num_new_tokens]

    def allocate_slots_batch(self, req_ids, num_new_tokens, window: int = 0):
        """(slots of the served requests, packed; number of requests served)"""
        ids = np.ascontiguousarray(req_ids, dtype=np.int64)
        nn = np.ascontiguousarray(num_new_tokens, dtype=np.int32)
        out = np.empty(max(int(nn.sum()), 1), dtype=np.int64)
        done = ctypes.c_int32(0)
        self._check(self._lib.pkv_pool_allocate_slots_batch(
            self._p, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            nn.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ids.size, int(window),
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ctypes.byref(done)))
        return out[:int(nn[:done.value].sum())], int(done.value)

    def free_request(self, req_id: int):
        self._check(self._lib.pkv_pool_free_request(self._p, int(req_id)))

    def block_table(self, req_id: int):
        n = ctypes.c_int32(0)
        self._check(self._lib.pkv_pool_block_table(self._p, int(req_id), None, 0, ctypes.byref(n)))
        row = np.empty(max(n.value, 1), dtype=np.int32)
        self._check(self._lib.pkv_pool_block_table(
            self._p, int(req_id), row.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n.value,
            ctypes.byref(n)))
        return [int(x) for x in row[:n.value]]

    def block_tables(self, req_ids, stride: int) -> np.ndarray:
        ids = np.ascontiguousarray(req_ids, dtype=np.int64)
        out = np.empty((ids.size, stride), dtype=np.int32)
        self._check(self._lib.pkv_pool_build_block_tables(
            self._p, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ids.size,
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(stride)))
        return out

    def num_computed(self, req_id: int) -> int:
        n = ctypes.c_int32(0)
        self._check(self._lib.pkv_pool_num_computed(self._p, int(req_id), ctypes.byref(n)))
        return int(n.value)

    def block_state(self, block: int):
        """(ref count, hash or None)"""
        r, h, has = ctypes.c_int32(0), ctypes.c_uint64(0), ctypes.c_int32(0)
        self._check(self._lib.pkv_pool_block_state(self._p, int(block), ctypes.byref(r),
                                                   ctypes.byref(h), ctypes.byref(has)))
        return int(r.value), (int(h.value) if has.value else None)

    def free_queue(self):
        n = ctypes.c_int32(0)
        self._check(self._lib.pkv_pool_free_queue(self._p, None, 0, ctypes.byref(n)))
        out = np.empty(max(n.value, 1), dtype=np.int32)
        self._check(self._lib.pkv_pool_free_queue(
            self._p, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n.value, ctypes.byref(n)))
        return [int(x) for x in out[:n.value]]
