"""The allocation-free builder, ibp_build_meta_noalloc.

It exists for callers that cannot allocate device memory when they build a
Mask/Bitval (code inside another framework's memory pool, or a loop that
cannot afford cudaMalloc's implicit device synchronisation).  Its counters
live in a fixed array of device memory shared by every call, so the GPU test
makes two calls in a row -- different rows, a smaller row after a larger one,
with and without sample ids -- and checks each against the store-based
ibp_build_meta bit for bit.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl


def _store_meta(rows_dev, R, ids_dev, n, num, den):
    st = ibp.ibp_store_create(R, 256, 1)
    try:
        ibp.ibp_build_meta(st, rows_dev, R, ids_dev, n, num, den)
        m = np.zeros(R // 4, np.uint32)
        b = np.zeros(R // 4, np.uint32)
        ibp.ibp_meta_get(st, m, b)
    finally:
        ibp.ibp_store_destroy(st)
    return m, b


@pytest.mark.gpu
def test_noalloc_builder_matches_store_builder_twice():
    dev = torch.device("cuda:0")
    calls = [  # (R, rows, per-mille sample or 0 for all rows, num, den)
        (8192, 3000, 0, 95, 100),
        (512, 20000, 50, 9, 10),
    ]
    for k, (R, n_rows, per_mille, num, den) in enumerate(calls):
        rows = torch.from_numpy(wl.fuzz_rows(n_rows, R, seed=100 + k)).to(dev)
        if per_mille:
            ids = torch.from_numpy(wl.sample_ids(n_rows, per_mille, seed=k)).to(dev)
            n = ids.numel()
        else:
            ids, n = None, n_rows
        mask = torch.full((R // 4,), 0x5A5A5A5A, dtype=torch.int32, device=dev)
        bitval = torch.full((R // 4,), 0x5A5A5A5A, dtype=torch.int32, device=dev)
        ibp.ibp_build_meta_noalloc(rows, R, R, ids, n, num, den, mask, bitval)
        torch.cuda.synchronize()
        m_ref, b_ref = _store_meta(rows, R, ids, n, num, den)
        assert np.array_equal(mask.cpu().numpy().view(np.uint32), m_ref), "call %d mask" % k
        assert np.array_equal(bitval.cpu().numpy().view(np.uint32), b_ref), "call %d bitval" % k


def test_noalloc_builder_rejects_rows_above_its_limit():
    lib = ibp._lib_handle()
    # checked on the host before any device work
    assert lib.ibp_build_meta_noalloc(16, 16384, 16384, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
    assert lib.ibp_build_meta_noalloc(16, 8208, 8208, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
    assert lib.ibp_build_meta_noalloc(None, 512, 512, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
