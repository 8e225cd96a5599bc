"""Randomised GPU-vs-oracle sweep over geometries, store modes, sources and layouts.

Each case draws a row size (16 B .. 8 KB, multiples of 16), a chunk size
(4 B .. 2 R, multiples of 4), a row count with a ragged tail, a Mask source
(built at a random threshold, or an empty / full / two-run Mask set from the
host), rows with planted structure and misses, and a source (HBM or pinned
host).  The GPU compressor must reproduce the oracle's stored bytes, sizes
and raw bits, and the dense, gather (with duplicates) and packed-cache
decoders must return the rows.
"""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
from oracle import ref_c
from tests.gpu_util import DEV, Store, assert_streams_equal, oracle_slots, to_dev

pytestmark = pytest.mark.gpu


def _case(seed):
    g = np.random.default_rng(1000 + seed)
    R = int(g.choice([16, 32, 48, 112, 256, 512, 528, 1024, 1040, 2048, 4096, 8192]))
    W = R // 4
    C = int(g.choice([4, 8, 12, 16, 64, 100, 256, 1024, 4096, 2 * R]))
    C = min(C, 2 * R)
    while (W + C // 4 - 1) // (C // 4) > 256:  # at most 256 chunks
        C *= 2
    n = int(g.integers(1, 2500 if R <= 2048 else 400))
    rows = wl.fuzz_rows(n, R, seed=seed, tag=3)
    how = g.choice(["build", "build", "empty", "full", "tworun"])
    if how == "build":
        num, den = [(51, 100), (3, 4), (9, 10), (95, 100), (1, 1)][int(g.integers(0, 5))]
        mask, bitval = ref_c.build_meta(rows, num, den)
    elif how == "empty":
        mask = np.zeros(W, np.uint32)
        bitval = np.zeros(W, np.uint32)
    elif how == "full":
        mask = np.full(W, 0xFFFFFFFF, np.uint32)
        bitval = rows[0].view(np.uint32).copy()
    else:
        mask = np.zeros(W, np.uint32)
        for w in range(W):
            a0 = int(g.integers(0, 20))
            keep = ((1 << int(g.integers(1, 9))) - 1) << a0
            if g.random() < 0.5:
                keep |= 1 << 31
            mask[w] = np.uint32(~keep & 0xFFFFFFFF)
        bitval = rows[0].view(np.uint32) & mask
    host = bool(g.random() < 0.5)
    return R, C, n, rows, mask, bitval, host, g


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_compress_decompress_gather(seed):
    R, C, n, rows, mask, bitval, host, g = _case(seed)
    st = Store(R, C, n)
    try:
        st.set_meta(mask, bitval)
        ref_sl, ref_bm, ref_st = oracle_slots(rows, C, mask, bitval, st.slot)
        slots = (torch.zeros((n, st.slot), dtype=torch.uint8, pin_memory=True) if host
                 else torch.zeros((n, st.slot), dtype=torch.uint8, device=DEV))
        stored = torch.zeros(n, dtype=torch.int32, device=DEV)
        ibp.ibp_compress(st.h, slots, to_dev(rows), R, None, n, stored)
        torch.cuda.synchronize()
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(stored.cpu().numpy().astype(np.uint32), ref_st)
        assert np.array_equal(st.bitmap(), ref_bm)
        assert_streams_equal(slots.cpu().numpy(), ref_sl, ref_st)
        # dense decode
        out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
        ibp.ibp_decompress(st.h, out, slots, None, n)
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(out.cpu().numpy(), rows)
        # gather with duplicates, into a strided output
        m = int(g.integers(1, 3 * n + 2))
        ids = g.integers(0, n, size=m).astype(np.int64)
        stride = R + 16 * int(g.integers(0, 3))
        out2 = torch.zeros((m, stride), dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress_strided(st.h, out2, stride, slots, None, to_dev(ids), m)
        assert st.status() == ibp.IBP_OK
        o2 = out2.cpu().numpy()
        assert np.array_equal(o2[:, :R], rows[ids])
        assert np.all(o2[:, R:] == 0)
        # packed HBM cache
        offs = torch.zeros(n + 1, dtype=torch.int64, device=DEV)
        ibp.ibp_pack(st.h, None, offs, slots, stored, n)
        total = int(offs[-1].item())
        cache = torch.zeros(total + R, dtype=torch.uint8, device=DEV)  # R readable bytes past the end
        ibp.ibp_pack(st.h, cache, offs, slots, stored, n)
        out.zero_()
        ibp.ibp_decompress(st.h, out, cache, offs, n)
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(out.cpu().numpy(), rows)
    finally:
        st.close()
