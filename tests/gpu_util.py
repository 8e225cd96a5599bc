"""Helpers for the GPU parity tests: stores on cuda:0 and oracle references."""
import numpy as np
import torch

from lossless_invariant_bit_gb300 import ibp
from oracle import ref_c

DEV = torch.device("cuda:0")


class Store:
    """A libibp store with host-side accessors (marshalling only)."""

    def __init__(self, R, C, n_rows, slot=0):
        self.R, self.C, self.n_rows = R, C, n_rows
        self.h = ibp.ibp_store_create(R, C, n_rows, slot)
        self.slot = ibp.ibp_store_get_info(self.h).slot_bytes

    def close(self):
        if self.h:
            ibp.ibp_store_destroy(self.h)
            self.h = None

    def meta(self):
        m = np.zeros(self.R // 4, np.uint32)
        b = np.zeros(self.R // 4, np.uint32)
        ibp.ibp_meta_get(self.h, m, b)
        return m, b

    def set_meta(self, m, b):
        ibp.ibp_meta_set(self.h, np.ascontiguousarray(m, np.uint32),
                         np.ascontiguousarray(b, np.uint32))

    def bitmap(self):
        bm = np.zeros((self.n_rows + 31) // 32, np.uint32)
        ibp.ibp_bitmap_get(self.h, bm)
        return bm

    def set_bitmap(self, bm):
        ibp.ibp_bitmap_set(self.h, np.ascontiguousarray(bm, np.uint32))

    def status(self, reset=True):
        return ibp.ibp_stream_status(self.h, reset=reset)


def _signed(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint64:
        return a.view(np.int64)
    if a.dtype == np.uint32:
        return a.view(np.int32)
    return a


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(_signed(a)).to(DEV)


def to_pinned(a: np.ndarray) -> torch.Tensor:
    a = _signed(a)
    t = torch.empty(a.shape, dtype=torch.from_numpy(a[:0]).dtype, pin_memory=True)
    t.copy_(torch.from_numpy(a))
    return t


def rows_u8(rows: np.ndarray) -> np.ndarray:
    rows = np.ascontiguousarray(rows)
    return rows.reshape(rows.shape[0], -1).view(np.uint8)


def oracle_slots(rows_b, C, mask, bitval, slot):
    """Oracle compression of every row into slots of `slot` bytes."""
    n, R = rows_b.shape
    slots = np.zeros((n, slot), np.uint8)
    bm = np.zeros((n + 31) // 32, np.uint32)
    stored = ref_c.compress_batch(rows_b, C, mask, bitval, slots, bm, nthreads=8)
    return slots, bm, stored


def assert_streams_equal(gpu_slots: np.ndarray, ref_slots: np.ndarray, stored: np.ndarray,
                         rows=None):
    rows = range(len(stored)) if rows is None else rows
    for j, i in enumerate(rows):
        s = int(stored[j])
        if not np.array_equal(gpu_slots[j, :s], ref_slots[j, :s]):
            bad = np.nonzero(gpu_slots[j, :s] != ref_slots[j, :s])[0]
            raise AssertionError("row %d: stored stream differs at bytes %s" % (i, bad[:8]))
