"""The allocation-free builder, ibp_build_meta_noalloc.

It exists for callers that cannot allocate device memory when they build a
Mask/Bitval (code inside another framework's memory pool, whose allocator
must own every device allocation, or a loop that cannot afford cudaMalloc's
implicit device synchronisation).  Its counters live in a fixed array of
device memory that every call shares and that keeps the previous call's
contents, so the GPU test makes two calls in a row -- different rows, a
smaller row after a larger one, with and without sample ids -- and checks
each against the oracle's builder (and the store-based ibp_build_meta) bit
for bit.

The file name sorts last, so pytest collects it after every other test file:
a run that stops at the first failure (-x) has then run every other test
before this one.  The test itself depends on nothing that ran before it; it
passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
from oracle import ref_c


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
def test_noalloc_builder_matches_oracle_twice():
    dev = torch.device("cuda:0")
    calls = [  # (R, rows, per-mille sample or 0 for all rows, num, den)
        (8192, 3000, 0, 95, 100),
        (512, 20000, 50, 9, 10),
    ]
    for k, (R, n_rows, per_mille, num, den) in enumerate(calls):
        rows_np = wl.fuzz_rows(n_rows, R, seed=100 + k)
        rows = torch.from_numpy(rows_np).to(dev)
        if per_mille:
            ids_np = wl.sample_ids(n_rows, per_mille, seed=k)
            ids = torch.from_numpy(ids_np).to(dev)
            n = ids.numel()
        else:
            ids_np, ids, n = None, None, n_rows
        mask = torch.full((R // 4,), 0x5A5A5A5A, dtype=torch.int32, device=dev)
        bitval = torch.full((R // 4,), 0x5A5A5A5A, dtype=torch.int32, device=dev)
        ibp.ibp_build_meta_noalloc(rows, R, R, ids, n, num, den, mask, bitval)
        torch.cuda.synchronize()
        got_m = mask.cpu().numpy().view(np.uint32)
        got_b = bitval.cpu().numpy().view(np.uint32)
        m_or, b_or = ref_c.build_meta(rows_np, num, den, sample_ids=ids_np)
        assert np.array_equal(got_m, m_or), "call %d mask vs oracle" % k
        assert np.array_equal(got_b, b_or), "call %d bitval vs oracle" % k
        m_st, b_st = _store_meta(rows, R, ids, n, num, den)
        assert np.array_equal(got_m, m_st) and np.array_equal(got_b, b_st), "call %d" % k


def test_noalloc_builder_rejects_bad_arguments_on_the_host():
    """Every check below returns before any device work (the addresses are
    never dereferenced), so this runs without a GPU."""
    lib = ibp._lib_handle()
    # rows above the array's limit, or not a multiple of 16 bytes
    assert lib.ibp_build_meta_noalloc(16, 16384, 16384, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
    assert lib.ibp_build_meta_noalloc(16, 8208, 8208, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
    assert lib.ibp_build_meta_noalloc(16, 520, 520, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
    # missing rows or outputs, no rows, a threshold outside (1/2, 1]
    assert lib.ibp_build_meta_noalloc(None, 512, 512, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
    assert lib.ibp_build_meta_noalloc(16, 512, 512, None, 1, 95, 100, None, 16,
                                      None) == ibp.IBP_EINVAL
    assert lib.ibp_build_meta_noalloc(16, 512, 512, None, 0, 95, 100, 16, 16,
                                      None) == ibp.IBP_EINVAL
    assert lib.ibp_build_meta_noalloc(16, 512, 512, None, 1, 1, 2, 16, 16,
                                      None) == ibp.IBP_EINVAL
    # misaligned rows, row stride, outputs or sample ids
    assert lib.ibp_build_meta_noalloc(24, 512, 512, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EALIGN
    assert lib.ibp_build_meta_noalloc(16, 520, 512, None, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EALIGN
    assert lib.ibp_build_meta_noalloc(16, 512, 512, None, 1, 95, 100, 18, 16,
                                      None) == ibp.IBP_EALIGN
    assert lib.ibp_build_meta_noalloc(16, 512, 512, None, 1, 95, 100, 16, 17,
                                      None) == ibp.IBP_EALIGN
    assert lib.ibp_build_meta_noalloc(16, 512, 512, 20, 1, 95, 100, 16, 16,
                                      None) == ibp.IBP_EALIGN
