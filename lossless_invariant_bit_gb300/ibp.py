"""Thin ctypes binding of libibp.so (declared in include/ibp.h).

Every function has the name of the C entry point it calls and only marshals
arguments: buffers may be torch tensors (device or pinned host), numpy arrays
(host-only calls) or raw integer addresses; ``stream`` defaults to torch's
current CUDA stream.  A non-OK status raises ``IbpError``.  There is no
fallback: if the library has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libibp.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "ibp.h")

IBP_OK, IBP_EINVAL, IBP_EALIGN, IBP_ERANGE, IBP_ECORRUPT, IBP_ENOMEM, IBP_ECUDA, IBP_ETIMEOUT = \
    range(8)
STATUS_NAMES = ["IBP_OK", "IBP_EINVAL", "IBP_EALIGN", "IBP_ERANGE", "IBP_ECORRUPT",
                "IBP_ENOMEM", "IBP_ECUDA", "IBP_ETIMEOUT"]


class IbpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s" % (where, _lib_handle().ibp_status_str(int(status)).decode()))


class ibp_store_info(ctypes.Structure):
    _fields_ = [("row_bytes", ctypes.c_uint32), ("chunk_bytes", ctypes.c_uint32),
                ("n_chunks", ctypes.c_uint32), ("min_bits", ctypes.c_uint32),
                ("n_rows", ctypes.c_uint64), ("slot_bytes", ctypes.c_uint64),
                ("meta_valid", ctypes.c_uint32), ("max_runs", ctypes.c_uint32)]


_lib = None
_P = ctypes.c_void_p
_U32 = ctypes.c_uint32
_U64 = ctypes.c_uint64
_ST = ctypes.c_int

_SIGS = {
    "ibp_store_create": [ctypes.POINTER(ctypes.c_void_p), _U32, _U32, _U64, _U64],
    "ibp_store_destroy": [_P],
    "ibp_store_get_info": [_P, ctypes.POINTER(ibp_store_info)],
    "ibp_build_meta": [_P, _P, _U64, _P, _U64, _U32, _U32, _P],
    "ibp_build_meta_tuned": [_P, _P, _U64, _P, _U64, _P, _P, _U32, _P, _P, _P],
    "ibp_build_meta_noalloc": [_P, _U64, _U32, _P, _U64, _U32, _U32, _P, _P, _P],
    "ibp_compress": [_P, _P, _P, _U64, _P, _U64, _P, _P],
    "ibp_decompress": [_P, _P, _P, _P, _U64, _P],
    "ibp_gather_decompress": [_P, _P, _P, _P, _P, _U64, _P],
    "ibp_gather_decompress_strided": [_P, _P, _U64, _P, _P, _P, _U64, _P],
    "ibp_pack": [_P, _P, _P, _P, _P, _U64, _P],
    "ibp_gather_decompress_cached": [_P, _P, _U64, _P, _P, _U64, _P, _P, _U64, _P],
    "ibp_gather_decompress_ordered": [_P, _P, _U64, _P, _P, _P, _U64, _P, _U64, _P],
    "ibp_store_set_lengths": [_P, _P],
    "ibp_group_gather_decompress_ordered": [_P, _P, _U64, _P, _U64, _P, _U64, _P],
    "ibp_group_order_plan": [_P, _P, _U64, _P, _U64, _P],
    "ibp_group_gather_decompress_planned": [_P, _P, _U64, _P, _U64, _P, _U64, _P],
    "ibp_gather_decompress_split": [_P, _P, _U64, _U64, _U64, _U64, _P, _P, _P, _U64, _P],
    "ibp_group_create": [ctypes.POINTER(ctypes.c_void_p), _P, _P, _U32],
    "ibp_group_destroy": [_P],
    "ibp_group_gather_decompress": [_P, _P, _U64, _P, _U64, _P],
    "ibp_meta_get": [_P, _P, _P],
    "ibp_meta_set": [_P, _P, _P],
    "ibp_bitmap_get": [_P, _P],
    "ibp_bitmap_set": [_P, _P],
    "ibp_stream_status": [_P, _P, ctypes.POINTER(ctypes.c_int), ctypes.c_int],
    "ibp_link_copy": [_P, _P, _U64, _P],
    "ibp_gather_copy": [_P, _P, _U64, _U32, _P, _U64, _U64, _P],
    "ibp_gather_copy_dma": [_P, _P, _U64, _U32, _P, _U64, _U64, _P],
    "ibp_gather_copy_staged": [_P, _P, _U64, _U32, _P, _U64, _U64, _P, _P],
    "ibp_project_compress": [_P, _P, _U64, _U64, _P, _P, _U32, _P, _P, _P, _P, _P, _U64, _P],
}


def library_path() -> str:
    return LIB_PATH


def _lib_handle():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libibp.so is not built (%s); run lossless_invariant_bit_gb300.build.build() "
                "-- there is no CPU fallback" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _ST
        L.ibp_status_str.argtypes = [_ST]
        L.ibp_status_str.restype = ctypes.c_char_p
        _lib = L
    return _lib


def declared_symbols() -> list:
    """Names of the entry points include/ibp.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^IBP_API\s+[\w\s\*]+?\b(ibp_\w+)\s*\(", text, flags=re.M)))


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError("cannot take the address of %r" % type(x))


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str) -> None:
    if st != IBP_OK:
        raise IbpError(st, where)


# ---------------------------------------------------------------- entry points
def ibp_store_create(row_bytes: int, chunk_bytes: int, n_rows: int, slot_bytes: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(_lib_handle().ibp_store_create(ctypes.byref(h), row_bytes, chunk_bytes, n_rows,
                                          slot_bytes), "ibp_store_create")
    return h.value


def ibp_store_destroy(store: int) -> None:
    _check(_lib_handle().ibp_store_destroy(store), "ibp_store_destroy")


def ibp_store_get_info(store: int) -> ibp_store_info:
    info = ibp_store_info()
    _check(_lib_handle().ibp_store_get_info(store, ctypes.byref(info)), "ibp_store_get_info")
    return info


def ibp_build_meta(store: int, rows, row_stride: int, sample_ids, n: int, thr_num: int,
                   thr_den: int, stream=None) -> None:
    _check(_lib_handle().ibp_build_meta(store, _ptr(rows), row_stride, _ptr(sample_ids), n,
                                        thr_num, thr_den, _stream(stream)), "ibp_build_meta")


def ibp_build_meta_tuned(store: int, rows, row_stride: int, sample_ids, n: int, thr_num,
                         thr_den, chosen_out=None, sizes_out=None, stream=None) -> None:
    """thr_num / thr_den: sequences of candidate thresholds (host)."""
    k = len(thr_num)
    num = (ctypes.c_uint32 * k)(*[int(v) for v in thr_num])
    den = (ctypes.c_uint32 * k)(*[int(v) for v in thr_den])
    _check(_lib_handle().ibp_build_meta_tuned(store, _ptr(rows), row_stride, _ptr(sample_ids), n,
                                              ctypes.cast(num, ctypes.c_void_p),
                                              ctypes.cast(den, ctypes.c_void_p), k,
                                              _ptr(chosen_out), _ptr(sizes_out), _stream(stream)),
           "ibp_build_meta_tuned")


def ibp_build_meta_noalloc(rows, row_stride: int, row_bytes: int, sample_ids, n: int,
                           thr_num: int, thr_den: int, mask_out, bitval_out, stream=None) -> None:
    """Builder that allocates nothing: Mask/Bitval into the caller's device arrays."""
    _check(_lib_handle().ibp_build_meta_noalloc(_ptr(rows), row_stride, row_bytes,
                                                _ptr(sample_ids), n, thr_num, thr_den,
                                                _ptr(mask_out), _ptr(bitval_out),
                                                _stream(stream)), "ibp_build_meta_noalloc")


def ibp_compress(store: int, dst_slots, src_rows, src_stride: int, slot_ids, n: int,
                 stored_bytes_out=None, stream=None) -> None:
    _check(_lib_handle().ibp_compress(store, _ptr(dst_slots), _ptr(src_rows), src_stride,
                                      _ptr(slot_ids), n, _ptr(stored_bytes_out),
                                      _stream(stream)), "ibp_compress")


def ibp_decompress(store: int, dst, src, offsets, n: int, stream=None) -> None:
    _check(_lib_handle().ibp_decompress(store, _ptr(dst), _ptr(src), _ptr(offsets), n,
                                        _stream(stream)), "ibp_decompress")


def ibp_gather_decompress(store: int, dst, host_or_dev_src, offsets, ids, n: int,
                          stream=None) -> None:
    _check(_lib_handle().ibp_gather_decompress(store, _ptr(dst), _ptr(host_or_dev_src),
                                               _ptr(offsets), _ptr(ids), n, _stream(stream)),
           "ibp_gather_decompress")


def ibp_gather_decompress_strided(store: int, dst, dst_stride_bytes: int, host_or_dev_src,
                                  offsets, ids, n: int, stream=None) -> None:
    _check(_lib_handle().ibp_gather_decompress_strided(store, _ptr(dst), dst_stride_bytes,
                                                       _ptr(host_or_dev_src), _ptr(offsets),
                                                       _ptr(ids), n, _stream(stream)),
           "ibp_gather_decompress_strided")


def ibp_gather_decompress_split(store: int, dst, group_rows: int, group_stride: int,
                                row_stride: int, chunk_stride: int, src, offsets, ids, n: int,
                                stream=None) -> None:
    _check(_lib_handle().ibp_gather_decompress_split(store, _ptr(dst), group_rows, group_stride,
                                                     row_stride, chunk_stride, _ptr(src),
                                                     _ptr(offsets), _ptr(ids), n,
                                                     _stream(stream)),
           "ibp_gather_decompress_split")


def ibp_store_set_lengths(store: int, lengths) -> None:
    """Attach each slot's stored bytes (device uint32/int32 [n_rows]) or detach (None)."""
    _check(_lib_handle().ibp_store_set_lengths(store, _ptr(lengths)), "ibp_store_set_lengths")


def project_workspace_bytes(m: int, row_bytes: int) -> int:
    """IBP_PROJECT_WORKSPACE_BYTES(m, R) of include/ibp.h."""
    m, R = int(m), int(row_bytes)
    return (m * (R // 16) + 255) // 256 * 256 + m * R


def ibp_project_compress(store: int, x, m: int, k_dim: int, w, bias, dtype: int, y, dst_slots,
                         slot_ids, stored_bytes_out, workspace, workspace_bytes: int,
                         stream=None) -> None:
    """Y = X W^T (+ bias) on the tensor cores, each row of Y compressed into
    its slot in the same launch (dtype 0: fp16, 1: bf16)."""
    _check(_lib_handle().ibp_project_compress(store, _ptr(x), m, k_dim, _ptr(w), _ptr(bias),
                                              dtype, _ptr(y), _ptr(dst_slots), _ptr(slot_ids),
                                              _ptr(stored_bytes_out), _ptr(workspace),
                                              workspace_bytes, _stream(stream)),
           "ibp_project_compress")


def order_workspace_bytes(n: int) -> int:
    """Bytes of workspace the ordered gathers need for n ids (items)."""
    return 20 * int(n) + 65536


def ibp_gather_decompress_ordered(store: int, dst, dst_stride_bytes: int, src, offsets, ids,
                                  n: int, workspace, workspace_bytes: int, stream=None) -> None:
    _check(_lib_handle().ibp_gather_decompress_ordered(store, _ptr(dst), dst_stride_bytes,
                                                       _ptr(src), _ptr(offsets), _ptr(ids), n,
                                                       _ptr(workspace), workspace_bytes,
                                                       _stream(stream)),
           "ibp_gather_decompress_ordered")


def ibp_group_gather_decompress_ordered(group: int, dst, dst_row_stride: int, ids, batch: int,
                                        workspace, workspace_bytes: int, stream=None) -> None:
    _check(_lib_handle().ibp_group_gather_decompress_ordered(group, _ptr(dst), dst_row_stride,
                                                             _ptr(ids), batch, _ptr(workspace),
                                                             workspace_bytes, _stream(stream)),
           "ibp_group_gather_decompress_ordered")


def ibp_group_order_plan(group: int, ids, batch: int, workspace, workspace_bytes: int,
                         stream=None) -> None:
    _check(_lib_handle().ibp_group_order_plan(group, _ptr(ids), batch, _ptr(workspace),
                                              workspace_bytes, _stream(stream)),
           "ibp_group_order_plan")


def ibp_group_gather_decompress_planned(group: int, dst, dst_row_stride: int, ids, batch: int,
                                        workspace, workspace_bytes: int, stream=None) -> None:
    _check(_lib_handle().ibp_group_gather_decompress_planned(group, _ptr(dst), dst_row_stride,
                                                             _ptr(ids), batch, _ptr(workspace),
                                                             workspace_bytes, _stream(stream)),
           "ibp_group_gather_decompress_planned")


def ibp_gather_decompress_cached(store: int, dst, dst_stride_bytes: int, host_src, cache_src,
                                 cache_slots: int, cache_map, ids, n: int, stream=None) -> None:
    _check(_lib_handle().ibp_gather_decompress_cached(store, _ptr(dst), dst_stride_bytes,
                                                      _ptr(host_src), _ptr(cache_src), cache_slots,
                                                      _ptr(cache_map), _ptr(ids), n,
                                                      _stream(stream)),
           "ibp_gather_decompress_cached")


def ibp_pack(store: int, dst_packed, offsets_out, src_slots, stored_bytes, n: int,
             stream=None) -> None:
    _check(_lib_handle().ibp_pack(store, _ptr(dst_packed), _ptr(offsets_out), _ptr(src_slots),
                                  _ptr(stored_bytes), n, _stream(stream)), "ibp_pack")


def ibp_group_create(stores, srcs) -> int:
    """stores: sequence of store handles; srcs: their slot buffers (tensors or addresses)."""
    n = len(stores)
    st_arr = (ctypes.c_void_p * n)(*stores)
    src_arr = (ctypes.c_void_p * n)(*[_ptr(x) for x in srcs])
    h = ctypes.c_void_p()
    _check(_lib_handle().ibp_group_create(ctypes.byref(h), ctypes.cast(st_arr, ctypes.c_void_p),
                                          ctypes.cast(src_arr, ctypes.c_void_p), n),
           "ibp_group_create")
    return h.value


def ibp_group_destroy(group: int) -> None:
    _check(_lib_handle().ibp_group_destroy(group), "ibp_group_destroy")


def ibp_group_gather_decompress(group: int, dst, dst_row_stride: int, ids, batch: int,
                                stream=None) -> None:
    _check(_lib_handle().ibp_group_gather_decompress(group, _ptr(dst), dst_row_stride, _ptr(ids),
                                                     batch, _stream(stream)),
           "ibp_group_gather_decompress")


def ibp_meta_get(store: int, mask_host, bitval_host) -> None:
    _check(_lib_handle().ibp_meta_get(store, _ptr(mask_host), _ptr(bitval_host)), "ibp_meta_get")


def ibp_meta_set(store: int, mask_host, bitval_host) -> None:
    _check(_lib_handle().ibp_meta_set(store, _ptr(mask_host), _ptr(bitval_host)), "ibp_meta_set")


def ibp_bitmap_get(store: int, bitmap_host) -> None:
    _check(_lib_handle().ibp_bitmap_get(store, _ptr(bitmap_host)), "ibp_bitmap_get")


def ibp_bitmap_set(store: int, bitmap_host) -> None:
    _check(_lib_handle().ibp_bitmap_set(store, _ptr(bitmap_host)), "ibp_bitmap_set")


def ibp_stream_status(store: int, stream=None, reset: bool = False) -> int:
    out = ctypes.c_int(0)
    _check(_lib_handle().ibp_stream_status(store, _stream(stream), ctypes.byref(out),
                                           int(bool(reset))), "ibp_stream_status")
    return out.value


def ibp_link_copy(dst, src, nbytes: int, stream=None) -> None:
    _check(_lib_handle().ibp_link_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)),
           "ibp_link_copy")


def ibp_gather_copy(dst, src, slot_bytes: int, row_bytes: int, ids, n: int, n_rows: int,
                    stream=None) -> None:
    _check(_lib_handle().ibp_gather_copy(_ptr(dst), _ptr(src), slot_bytes, row_bytes, _ptr(ids),
                                         n, n_rows, _stream(stream)), "ibp_gather_copy")


def ibp_gather_copy_dma(dst, src, slot_bytes: int, row_bytes: int, ids_host, n: int, n_rows: int,
                        stream=None) -> None:
    _check(_lib_handle().ibp_gather_copy_dma(_ptr(dst), _ptr(src), slot_bytes, row_bytes,
                                             _ptr(ids_host), n, n_rows, _stream(stream)),
           "ibp_gather_copy_dma")


def ibp_gather_copy_staged(dst, src, slot_bytes: int, row_bytes: int, ids_host, n: int,
                           n_rows: int, staging_host, stream=None) -> None:
    _check(_lib_handle().ibp_gather_copy_staged(_ptr(dst), _ptr(src), slot_bytes, row_bytes,
                                                _ptr(ids_host), n, n_rows, _ptr(staging_host),
                                                _stream(stream)), "ibp_gather_copy_staged")


def ibp_status_str(status: int) -> str:
    return _lib_handle().ibp_status_str(int(status)).decode()
