"""Parity at the full size of the sparse-GNN workload, in the launch
configuration bench.py times: 2,000,000 x 512 B rows compressed by the GPU
into pinned host slots, gather-decompressed 200,000 uniform ids at a time.

The oracle cannot redo 2M rows bit by bit in seconds, so it checks samples:
the Mask/Bitval from the same 1 % sample ids (all of them), the stored
streams and raw bits of 20,000 sampled slots, and 20,000 sampled output rows
of the gather through the oracle's own decoder; the whole gathered batch is
also compared with the generated rows (decompress(compress(x)) == x).
"""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
from oracle import ref_c
from tests.gpu_util import DEV

pytestmark = pytest.mark.gpu


def test_sparse_gnn_full_size():
    n_rows, dim, R, C = 2_000_000, 128, 512, 1024
    rows = np.empty((n_rows, dim), np.float32)
    wl.sparse_gnn_rows(n_rows, dim, seed=0, out=rows)
    rb = rows.view(np.uint8)
    sample = wl.sample_ids(n_rows, 10, seed=0)
    st = ibp.ibp_store_create(R, C, n_rows, 0)
    try:
        slot = ibp.ibp_store_get_info(st).slot_bytes
        slots = torch.empty((n_rows, slot), dtype=torch.uint8, pin_memory=True)
        d_rows = torch.from_numpy(rb).to(DEV)
        ibp.ibp_build_meta(st, d_rows, R, torch.from_numpy(sample).to(DEV), len(sample), 95, 100)
        stored = torch.empty(n_rows, dtype=torch.int32, device=DEV)
        ibp.ibp_compress(st, slots, d_rows, R, None, n_rows, stored)
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
        del d_rows

        mask = np.zeros(R // 4, np.uint32)
        bitval = np.zeros(R // 4, np.uint32)
        ibp.ibp_meta_get(st, mask, bitval)
        m_ref, b_ref = ref_c.build_meta(rb, 95, 100, sample_ids=sample)
        assert np.array_equal(mask, m_ref) and np.array_equal(bitval, b_ref)

        g = np.random.default_rng(11)
        pick = np.sort(g.choice(n_rows, size=20000, replace=False))
        ref_sl = np.zeros((len(pick), slot), np.uint8)
        ref_bm = np.zeros((len(pick) + 31) // 32, np.uint32)
        ref_st = ref_c.compress_batch(rb[pick], C, m_ref, b_ref, ref_sl, ref_bm, nthreads=8)
        st_gpu = stored.cpu().numpy().astype(np.uint32)
        assert np.array_equal(st_gpu[pick], ref_st)
        sl = slots.numpy()
        for j, i in enumerate(pick):
            s = int(ref_st[j])
            assert np.array_equal(sl[i, :s], ref_sl[j, :s]), i
        bm = np.zeros((n_rows + 31) // 32, np.uint32)
        ibp.ibp_bitmap_get(st, bm)
        raw = np.unpackbits(bm.view(np.uint8), bitorder="little")[:n_rows].astype(bool)
        assert np.array_equal(raw[pick], ref_st == R)
        assert np.array_equal(raw, st_gpu == R)

        ids = wl.uniform_ids(200_000, n_rows, seed=0, batch=0)
        out = torch.empty((len(ids), R), dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress(st, out, slots, None, torch.from_numpy(ids).to(DEV), len(ids))
        assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
        o = out.cpu().numpy()
        assert np.array_equal(o, rb[ids])
        sub = np.sort(g.choice(len(ids), size=20000, replace=False))
        ref_out, bad = ref_c.decompress_batch(sl, bm, R, C, m_ref, b_ref, ids=ids[sub],
                                              slot_stride=slot, nthreads=8)
        assert bad == 0 and np.array_equal(o[sub], ref_out)
    finally:
        ibp.ibp_store_destroy(st)
