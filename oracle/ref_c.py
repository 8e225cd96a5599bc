"""ctypes wrapper of the C oracle (``ibp_ref.c``) -- TEST INFRASTRUCTURE ONLY.

Arrays are numpy; every call is a thin marshalling of the C function of the
same name.  ``build()`` compiles the oracle with gcc (OpenMP over rows only).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ibp_ref.c")
_LIB = os.path.join(_HERE, "libibp_ref.so")
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_i64p = ctypes.POINTER(ctypes.c_int64)
_intp = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile ibp_ref.c into libibp_ref.so beside it (plain -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-Wall", "-Wextra", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def bind(L):
    """Declare the argument and return types of the oracle's functions on a
    loaded copy of it (the test suite also loads deliberately broken builds)."""
    L.ibp_ref_build_meta.argtypes = [_u8p, ctypes.c_uint64, ctypes.c_uint32, _i64p,
                                     ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                     _u32p, _u32p]
    L.ibp_ref_build_meta.restype = ctypes.c_int
    L.ibp_ref_compress_row.argtypes = [_u8p, ctypes.c_uint32, ctypes.c_uint32, _u32p, _u32p,
                                       _u8p, _intp, _u64p]
    L.ibp_ref_compress_row.restype = ctypes.c_uint32
    L.ibp_ref_decompress_row.argtypes = [_u8p, ctypes.c_uint32, ctypes.c_int, ctypes.c_uint32,
                                         ctypes.c_uint32, _u32p, _u32p, _u8p]
    L.ibp_ref_decompress_row.restype = ctypes.c_int
    L.ibp_ref_compress_batch.argtypes = [_u8p, ctypes.c_uint64, ctypes.c_uint64, _i64p, _u8p,
                                         ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                         _u32p, _u32p, _u32p, _u32p, ctypes.c_int]
    L.ibp_ref_compress_batch.restype = ctypes.c_uint64
    L.ibp_ref_decompress_batch.argtypes = [_u8p, _u64p, ctypes.c_uint64, ctypes.c_uint32,
                                           _u32p, _i64p, ctypes.c_uint64, ctypes.c_uint32,
                                           ctypes.c_uint32, _u32p, _u32p, _u8p,
                                           ctypes.c_uint64, ctypes.c_int]
    L.ibp_ref_decompress_batch.restype = ctypes.c_uint64
    L.ibp_ref_max_threads.argtypes = []
    L.ibp_ref_max_threads.restype = ctypes.c_int
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = bind(ctypes.CDLL(_LIB))
    return _lib


def _p(a: Optional[np.ndarray], t):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(t)


def _bytes2d(rows: np.ndarray) -> np.ndarray:
    rows = np.ascontiguousarray(rows)
    return rows.reshape(rows.shape[0], -1).view(np.uint8)


def build_meta(rows: np.ndarray, num: int, den: int,
               sample_ids: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Mask, Bitval (uint32[W]) from rows [N, R bytes] (any dtype) and optional sample ids."""
    b = _bytes2d(rows)
    R = b.shape[1]
    n = b.shape[0] if sample_ids is None else len(sample_ids)
    ids = None if sample_ids is None else np.ascontiguousarray(sample_ids, dtype=np.int64)
    mask = np.zeros(R // 4, np.uint32)
    bitval = np.zeros(R // 4, np.uint32)
    st = lib().ibp_ref_build_meta(_p(b, _u8p), R, R, _p(ids, _i64p), n, num, den,
                                  _p(mask, _u32p), _p(bitval, _u32p))
    if st != 0:
        raise ValueError("ibp_ref_build_meta: invalid arguments (status %d)" % st)
    return mask, bitval


def compress_row(row: bytes, C: int, mask: np.ndarray, bitval: np.ndarray):
    """(stored bytes, is_raw, stream bits) of one row."""
    r = np.frombuffer(bytes(row), np.uint8).copy()
    out = np.zeros(len(r), np.uint8)
    raw = ctypes.c_int(0)
    bits = ctypes.c_uint64(0)
    st = lib().ibp_ref_compress_row(_p(r, _u8p), len(r), C, _p(mask, _u32p), _p(bitval, _u32p),
                                    _p(out, _u8p), ctypes.byref(raw), ctypes.byref(bits))
    if st == 0:
        raise ValueError("ibp_ref_compress_row: bad geometry")
    return out[:st].tobytes(), bool(raw.value), int(bits.value)


def decompress_row(stored: bytes, is_raw: bool, R: int, C: int, mask: np.ndarray,
                   bitval: np.ndarray):
    """R bytes, or None if the stream is corrupt."""
    s = np.frombuffer(bytes(stored), np.uint8).copy()
    if len(s) == 0:
        s = np.zeros(4, np.uint8)
        n = 0
    else:
        n = len(s)
    out = np.zeros(R, np.uint8)
    st = lib().ibp_ref_decompress_row(_p(s, _u8p), n, int(is_raw), R, C, _p(mask, _u32p),
                                      _p(bitval, _u32p), _p(out, _u8p))
    return None if st != 0 else out.tobytes()


def compress_batch(rows: np.ndarray, C: int, mask: np.ndarray, bitval: np.ndarray,
                   slots: np.ndarray, bitmap: np.ndarray, slot_ids: Optional[np.ndarray] = None,
                   nthreads: int = 1) -> np.ndarray:
    """Compress rows [n, R] into slots [N, S] (uint8), updating bitmap (uint32).

    Returns the stored byte count of each row."""
    b = _bytes2d(rows)
    n, R = b.shape
    assert slots.dtype == np.uint8 and slots.ndim == 2 and slots.flags["C_CONTIGUOUS"]
    ids = None if slot_ids is None else np.ascontiguousarray(slot_ids, dtype=np.int64)
    stored = np.zeros(n, np.uint32)
    bad = lib().ibp_ref_compress_batch(_p(b, _u8p), R, n, _p(ids, _i64p), _p(slots, _u8p),
                                       slots.shape[1], R, C, _p(mask, _u32p), _p(bitval, _u32p),
                                       _p(bitmap, _u32p), _p(stored, _u32p), nthreads)
    if bad:
        raise ValueError("ibp_ref_compress_batch: %d rows failed" % bad)
    return stored


def decompress_batch(src: np.ndarray, bitmap: np.ndarray, R: int, C: int, mask: np.ndarray,
                     bitval: np.ndarray, ids: Optional[np.ndarray] = None, n: Optional[int] = None,
                     offsets: Optional[np.ndarray] = None, slot_stride: int = 0,
                     avail: Optional[int] = None, out: Optional[np.ndarray] = None,
                     nthreads: int = 1) -> Tuple[np.ndarray, int]:
    """Decompress rows ids (or 0..n-1) of a slot store / packed cache.

    Returns (out [n, R] uint8, number of corrupt rows)."""
    src = np.ascontiguousarray(src).reshape(-1).view(np.uint8)
    idv = None if ids is None else np.ascontiguousarray(ids, dtype=np.int64)
    cnt = len(idv) if idv is not None else int(n)
    if out is None:
        out = np.zeros((cnt, R), np.uint8)
    offs = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.uint64)
    av = int(avail if avail is not None else (slot_stride if slot_stride else R))
    bad = lib().ibp_ref_decompress_batch(_p(src, _u8p), _p(offs, _u64p), slot_stride, av,
                                         _p(bitmap, _u32p), _p(idv, _i64p), cnt, R, C,
                                         _p(mask, _u32p), _p(bitval, _u32p), _p(out, _u8p),
                                         out.strides[0], nthreads)
    return out, int(bad)


def max_threads() -> int:
    return int(lib().ibp_ref_max_threads())


def pack_slots(slots: np.ndarray, stored: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Packed cache layout (System Integration: compressed GPU cache): row i's
    stored bytes at offsets[i] = sum_{i'<i} roundup(stored[i'], 16); offsets has
    n+1 entries, the last being the total.  Returns (packed uint8, offsets uint64)."""
    sizes = (stored.astype(np.uint64) + np.uint64(15)) & ~np.uint64(15)
    offsets = np.zeros(len(stored) + 1, np.uint64)
    offsets[1:] = np.cumsum(sizes)
    packed = np.zeros(int(offsets[-1]), np.uint8)
    for i in range(len(stored)):
        packed[int(offsets[i]):int(offsets[i]) + int(stored[i])] = slots[i, :int(stored[i])]
    return packed, offsets
