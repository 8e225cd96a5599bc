"""GPU path vs CPU oracle, through the C ABI.  Integer work: bit-exact.

Covered: builder (all rows, sampled ids, host-mapped rows, thresholds),
compressor (stored bytes, sizes, raw bitmap; HBM and host slots), decoder
(dense slots, packed cache, gather with duplicates, strided output, host
source), the pack step, geometry edges (R from 16 B to the 32 KB maximum, C
above R and not dividing R, up to 256 chunks, ragged batch sizes, n = 0 and
1), degenerate metadata (empty Mask, full Mask with rows equal to the
Bitval), and the kernel-detected data errors.
"""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
from oracle import ref_c
from tests.gpu_util import (DEV, Store, assert_streams_equal, oracle_slots, rows_u8, to_dev,
                            to_pinned)

pytestmark = pytest.mark.gpu


@pytest.fixture
def stores():
    made = []

    def make(*a, **k):
        s = Store(*a, **k)
        made.append(s)
        return s

    yield make
    for s in made:
        s.close()


def gpu_compress(st, d_rows, n, slot_ids=None, host=False):
    slots = (torch.zeros((st.n_rows, st.slot), dtype=torch.uint8, pin_memory=True) if host
             else torch.zeros((st.n_rows, st.slot), dtype=torch.uint8, device=DEV))
    stored = torch.zeros(n, dtype=torch.int32, device=DEV)
    ids = None if slot_ids is None else to_dev(slot_ids.astype(np.int64))
    ibp.ibp_compress(st.h, slots, d_rows, d_rows.stride(0) * d_rows.element_size(), ids, n,
                     stored)
    torch.cuda.synchronize()
    return slots, stored.cpu().numpy().astype(np.uint32)


# ---------------------------------------------------------------- builder
@pytest.mark.parametrize("where", ["hbm", "host"])
def test_build_meta_tiny(stores, where):
    rows, _ = wl.tiny_rows(seed=0)
    b = rows_u8(rows)
    st = stores(1024, 256, len(b))
    d = to_dev(b) if where == "hbm" else to_pinned(b)
    ibp.ibp_build_meta(st.h, d, 1024, None, len(b), 95, 100)
    m, bv = st.meta()
    mr, br = ref_c.build_meta(b, 95, 100)
    assert np.array_equal(m, mr) and np.array_equal(bv, br)
    assert np.all(m == 0xFF801FFF) and np.all(bv == 0x3F800000)
    info = ibp.ibp_store_get_info(st.h)
    assert info.meta_valid == 1 and info.min_bits == 4 + 4 * 640 and info.max_runs == 1


@pytest.mark.parametrize("R,num,den,per_mille", [
    (64, 3, 4, 0), (512, 95, 100, 100), (2048, 9, 10, 50), (8192, 999, 1000, 0),
    (32768, 1, 1, 0), (112, 51, 100, 300)])
def test_build_meta_fuzz(stores, R, num, den, per_mille):
    n = 3000 if R <= 8192 else 700
    b = wl.fuzz_rows(n, R, seed=R + num)
    ids = wl.sample_ids(n, per_mille, seed=1) if per_mille else None
    st = stores(R, 256, n)
    d = to_dev(b)
    d_ids = None if ids is None else to_dev(ids)
    ibp.ibp_build_meta(st.h, d, R, d_ids, n if ids is None else len(ids), num, den)
    m, bv = st.meta()
    mr, br = ref_c.build_meta(b, num, den, sample_ids=ids)
    assert np.array_equal(m, mr) and np.array_equal(bv, br)


def test_build_meta_many_rows_spill(stores):
    """More rows per thread than the 8 bit-plane counters hold (255): exercises the spill."""
    n = 400_000
    b = wl.fuzz_rows(n, 64, seed=5)
    st = stores(64, 16, n)
    ibp.ibp_build_meta(st.h, to_dev(b), 64, None, n, 7, 8)
    m, bv = st.meta()
    mr, br = ref_c.build_meta(b, 7, 8)
    assert np.array_equal(m, mr) and np.array_equal(bv, br)


def test_build_meta_rejects_bad_threshold(stores):
    st = stores(64, 16, 4)
    d = torch.zeros((4, 64), dtype=torch.uint8, device=DEV)
    for num, den in [(1, 2), (2, 1), (0, 0)]:
        with pytest.raises(ibp.IbpError) as e:
            ibp.ibp_build_meta(st.h, d, 64, None, 4, num, den)
        assert e.value.status == ibp.IBP_EINVAL


# ---------------------------------------------------------------- compressor + decoder
GEOMS = [(16, 4), (16, 8), (64, 16), (112, 12), (512, 1024), (512, 256), (1024, 256),
         (2048, 1024), (8192, 256), (4096, 4096), (8192, 8192), (32768, 128), (4096, 16),
         (1024, 100)]


@pytest.mark.parametrize("R,C", GEOMS)
def test_compress_and_decompress_fuzz(stores, R, C):
    n = 777 if R <= 8192 else 133  # ragged: not a multiple of the warps per block
    b = wl.fuzz_rows(n, R, seed=R * 7 + C)
    mr, br = ref_c.build_meta(b, 9, 10)
    st = stores(R, C, n)
    st.set_meta(mr, br)
    d = to_dev(b)
    slots, stored = gpu_compress(st, d, n)
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, mr, br, st.slot)
    assert np.array_equal(stored, ref_st)
    assert np.array_equal(st.bitmap(), ref_bm)
    assert_streams_equal(slots.cpu().numpy(), ref_sl, ref_st)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, slots, None, n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)


@pytest.mark.parametrize("R,C", [(1024, 256), (8192, 256), (512, 1024)])
def test_decompress_oracle_streams_from_host(stores, R, C):
    """Decoder input written by the oracle, read zero-copy from pinned host memory."""
    n = 1500
    b = wl.fuzz_rows(n, R, seed=R + 3)
    mr, br = ref_c.build_meta(b, 95, 100)
    st = stores(R, C, n)
    st.set_meta(mr, br)
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, mr, br, st.slot)
    st.set_bitmap(ref_bm)
    src = to_pinned(ref_sl)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, src, None, n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)


def test_compress_into_host_slots_with_ids(stores):
    R, C, N = 512, 256, 4000
    n = 1000
    b = wl.fuzz_rows(n, R, seed=77)
    mr, br = ref_c.build_meta(b, 95, 100)
    st = stores(R, C, N)
    st.set_meta(mr, br)
    slot_ids = np.random.default_rng(3).permutation(N)[:n].astype(np.int64)
    slots, stored = gpu_compress(st, to_dev(b), n, slot_ids=slot_ids, host=True)
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, mr, br, st.slot)
    assert np.array_equal(stored, ref_st)
    sl = slots.numpy()[slot_ids]
    assert_streams_equal(sl, ref_sl, ref_st)
    bm = st.bitmap()
    raw = np.unpackbits(bm.view(np.uint8), bitorder="little")[:N].astype(bool)
    assert np.array_equal(np.nonzero(raw)[0], np.sort(slot_ids[ref_st == R]))
    # gather them back through the host link, duplicates included
    ids = np.concatenate([slot_ids, slot_ids[:300]])
    out = torch.empty((len(ids), R), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress(st.h, out, slots, None, to_dev(ids), len(ids))
    assert st.status() == ibp.IBP_OK
    inv = np.empty(N, np.int64)
    inv[slot_ids] = np.arange(n)
    assert np.array_equal(out.cpu().numpy(), b[inv[ids]])


def test_gather_strided(stores):
    R, C, N, T = 1024, 1024, 5000, 3
    b = wl.fuzz_rows(N, R, seed=8)
    mr, br = ref_c.build_meta(b, 95, 100)
    st = stores(R, C, N)
    st.set_meta(mr, br)
    slots, stored = gpu_compress(st, to_dev(b), N, host=True)
    ids = np.random.default_rng(4).integers(0, N, size=2049)
    out = torch.full((len(ids), T, R), 0xAB, dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress_strided(st.h, out[:, 1], T * R, slots, None, to_dev(ids), len(ids))
    assert st.status() == ibp.IBP_OK
    o = out.cpu().numpy()
    assert np.array_equal(o[:, 1], b[ids])
    assert np.all(o[:, 0] == 0xAB) and np.all(o[:, 2] == 0xAB)


def test_packed_cache_tiny(stores):
    """Cache path: oracle-packed bytes decode on the GPU, and GPU compress + pack
    reproduces the oracle's packed cache and offsets byte for byte."""
    rows, pick = wl.tiny_rows(seed=0)
    b = rows_u8(rows)
    n, R, C = len(b), 1024, 256
    st = stores(R, C, n, R)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, n, 95, 100)
    mr, br = st.meta()
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, mr, br, R)
    packed_ref, offs_ref = ref_c.pack_slots(ref_sl, ref_st)
    assert int(ref_st.sum()) == 1_355_104
    # decode the oracle's cache
    st.set_bitmap(ref_bm)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, to_dev(packed_ref), to_dev(offs_ref[:-1]), n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)
    # GPU compress + pack
    slots, stored = gpu_compress(st, d, n)
    d_stored = to_dev(stored.astype(np.int32))
    offs = torch.zeros(n + 1, dtype=torch.int64, device=DEV)
    ibp.ibp_pack(st.h, None, offs, slots, d_stored, n)
    total = int(offs[-1].item())
    assert total == int(offs_ref[-1])
    packed = torch.zeros(total, dtype=torch.uint8, device=DEV)
    ibp.ibp_pack(st.h, packed, offs, slots, d_stored, n)
    torch.cuda.synchronize()
    assert np.array_equal(offs.cpu().numpy().astype(np.uint64), offs_ref)
    pk = packed.cpu().numpy()
    for i in range(n):
        o, s = int(offs_ref[i]), int(ref_st[i])
        assert np.array_equal(pk[o:o + s], packed_ref[o:o + s]), i


# ---------------------------------------------------------------- degenerate metadata, sizes
def test_empty_mask_all_raw(stores):
    R, C, n = 256, 64, 100
    b = wl.fuzz_rows(n, R, seed=12)
    st = stores(R, C, n)
    slots, stored = gpu_compress(st, to_dev(b), n)  # fresh store: Mask all zero
    assert np.all(stored == R)
    assert np.all(np.unpackbits(st.bitmap().view(np.uint8), bitorder="little")[:n] == 1)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, slots, None, n)
    assert st.status() == ibp.IBP_OK and np.array_equal(out.cpu().numpy(), b)


def test_full_mask_rows_equal_bitval(stores):
    R, C, n = 4096, 256, 64
    bitval = np.random.default_rng(2).integers(0, 1 << 32, size=R // 4, dtype=np.uint64)
    bitval = bitval.astype(np.uint32)
    rows = np.repeat(bitval[None, :], n, axis=0).view(np.uint8)
    st = stores(R, C, n)
    ibp.ibp_build_meta(st.h, to_dev(rows), R, None, n, 95, 100)
    m, bv = st.meta()
    assert np.all(m == 0xFFFFFFFF) and np.array_equal(bv, bitval)
    slots, stored = gpu_compress(st, to_dev(rows), n)
    assert np.all(stored == 4)  # 16 participation bits in one word
    assert np.all(slots.cpu().numpy()[:, :4].view(np.uint32) == 0xFFFF)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, slots, None, n)
    assert np.array_equal(out.cpu().numpy(), rows)


def test_zero_and_one_rows(stores):
    R, C = 512, 256
    b = wl.fuzz_rows(1, R, seed=1)
    st = stores(R, C, 1)
    mr, br = ref_c.build_meta(b, 1, 1)
    st.set_meta(mr, br)
    out = torch.empty((1, R), dtype=torch.uint8, device=DEV)
    d = to_dev(b)
    ibp.ibp_compress(st.h, out, d, R, None, 0)   # n = 0: no-op
    ibp.ibp_decompress(st.h, out, d, None, 0)
    slots, stored = gpu_compress(st, d, 1)
    ibp.ibp_decompress(st.h, out, slots, None, 1)
    assert st.status() == ibp.IBP_OK and np.array_equal(out.cpu().numpy(), b)


# ---------------------------------------------------------------- data errors
def test_out_of_range_ids_flagged_and_zeroed(stores):
    R, C, N = 512, 256, 100
    b = wl.fuzz_rows(N, R, seed=21)
    mr, br = ref_c.build_meta(b, 95, 100)
    st = stores(R, C, N)
    st.set_meta(mr, br)
    slots, _ = gpu_compress(st, to_dev(b), N)
    ids = np.array([0, 5, N, -1, 7], np.int64)
    out = torch.full((len(ids), R), 0x55, dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress(st.h, out, slots, None, to_dev(ids), len(ids))
    assert st.status() == ibp.IBP_ERANGE
    assert st.status() == ibp.IBP_OK  # reset by the previous read
    o = out.cpu().numpy()
    assert np.array_equal(o[[0, 1, 4]], b[[0, 5, 7]])
    assert np.all(o[[2, 3]] == 0)


def test_corrupt_stream_flagged_and_zeroed(stores):
    """A row flagged compressed whose header says every chunk is raw needs more
    than R bytes: the decoder reports it and writes zeros (the stream is built on
    the host; every read stays inside the slot)."""
    R, C, n = 1024, 256, 4
    rows, _ = wl.tiny_rows(seed=0, n_rows=64, raw_frac=0.0)
    b = rows_u8(rows)[:n]
    mr, br = ref_c.build_meta(rows_u8(rows), 95, 100)
    st = stores(R, C, n)
    st.set_meta(mr, br)
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, mr, br, R)
    assert ref_bm.sum() == 0
    ref_sl[2, 0] &= 0xF0  # clear the 4 participation bits of row 2
    st.set_bitmap(ref_bm)
    out = torch.full((n, R), 0x55, dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, to_dev(ref_sl), None, n)
    assert st.status() == ibp.IBP_ECORRUPT
    o = out.cpu().numpy()
    assert np.all(o[2] == 0)
    assert np.array_equal(o[[0, 1, 3]], b[[0, 1, 3]])


def test_misaligned_offset_flagged(stores):
    R, C, n = 512, 256, 3
    b = wl.fuzz_rows(n, R, seed=4)
    st = stores(R, C, n)
    slots, stored = gpu_compress(st, to_dev(b), n)  # all raw (empty Mask)
    flat = slots.reshape(-1)
    offs = np.array([0, 2 * st.slot + 8, st.slot], np.uint64)
    out = torch.full((n, R), 0x55, dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, flat, to_dev(offs), n)
    assert st.status() == ibp.IBP_EALIGN
    o = out.cpu().numpy()
    assert np.array_equal(o[0], b[0]) and np.all(o[1] == 0) and np.array_equal(o[2], b[1])


def test_host_checks_alignment(stores):
    st = stores(512, 256, 8)
    d = torch.zeros(8 * 512 + 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(ibp.IbpError) as e:
        ibp.ibp_decompress(st.h, d[1:], d, None, 1)
    assert e.value.status == ibp.IBP_EALIGN
    with pytest.raises(ibp.IbpError) as e:
        ibp.ibp_decompress(st.h, d, d, None, 9)  # more rows than slots
    assert e.value.status == ibp.IBP_ERANGE


# ---------------------------------------------------------------- copies
def test_link_copy_and_gather_copy():
    n = (1 << 22) + 48
    src = torch.randint(0, 256, (n,), dtype=torch.uint8).pin_memory()
    dst = torch.empty(n, dtype=torch.uint8, device=DEV)
    ibp.ibp_link_copy(dst, src, n)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src)
    R, S, N = 512, 640, 1000
    store = torch.randint(0, 256, (N, S), dtype=torch.uint8).pin_memory()
    ids = torch.tensor([3, 999, 0, 3, 1000, -2], dtype=torch.int64, device=DEV)
    out = torch.full((6, R), 7, dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_copy(out, store, S, R, ids, 6, N)
    o = out.cpu()
    assert torch.equal(o[:4], store[[3, 999, 0, 3], :R])
    assert torch.all(o[4:] == 0)
    # the CPU-initiated baselines: one copy per row, and gather-then-copy
    ids_h = torch.tensor([5, 0, 999, 5, 17], dtype=torch.int64).pin_memory()
    out = torch.zeros((5, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_copy_dma(out, store, S, R, ids_h, 5, N)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), store[[5, 0, 999, 5, 17], :R])
    staging = torch.empty(5 * R, dtype=torch.uint8, pin_memory=True)
    out.zero_()
    ibp.ibp_gather_copy_staged(out, store, S, R, ids_h, 5, N, staging)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), store[[5, 0, 999, 5, 17], :R])
    bad = torch.tensor([1, N], dtype=torch.int64).pin_memory()
    with pytest.raises(ibp.IbpError) as e:
        ibp.ibp_gather_copy_dma(out, store, S, R, bad, 2, N)
    assert e.value.status == ibp.IBP_ERANGE


# ---------------------------------------------------------------- decoder modes
def _two_run_meta(W, seed):
    """Per-word Masks whose kept bits form at most two runs, all different."""
    g = np.random.default_rng(seed)
    mask = np.zeros(W, np.uint32)
    for w in range(W):
        a0, l0 = int(g.integers(0, 20)), int(g.integers(1, 8))
        a1 = int(g.integers(a0 + l0 + 1, 32)) if a0 + l0 + 1 < 32 else 31
        l1 = int(g.integers(0, 32 - a1)) if a1 < 31 else 0
        keep = ((1 << l0) - 1) << a0 | (((1 << l1) - 1) << a1 if l1 else 0)
        mask[w] = np.uint32(~keep & 0xFFFFFFFF)
    bitval = g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32) & mask
    return mask, bitval


@pytest.mark.parametrize("R,C", [(1024, 256), (512, 1024), (2048, 64)])
def test_decoder_two_run_store(stores, R, C):
    n = 3000
    mask, bitval = _two_run_meta(R // 4, seed=R + C)
    g = np.random.default_rng(C)
    rows = (g.integers(0, 1 << 32, size=(n, R // 4), dtype=np.uint64).astype(np.uint32)
            & ~mask) | bitval
    flip = g.random(n) < 0.1  # some rows miss the Bitval in one word: a raw chunk
    rows[flip, g.integers(0, R // 4, size=int(flip.sum()))] ^= mask[0] | 1
    b = rows.view(np.uint8)
    st = stores(R, C, n)
    st.set_meta(mask, bitval)
    assert ibp.ibp_store_get_info(st.h).max_runs <= 2
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, mask, bitval, st.slot)
    slots, stored = gpu_compress(st, to_dev(b), n)
    assert np.array_equal(stored, ref_st)
    assert_streams_equal(slots.cpu().numpy(), ref_sl, ref_st)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, slots, None, n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)


@pytest.mark.parametrize("kind", ["tiny", "fuzz"])
def test_decoder_before_store_properties_reach_host(stores, kind):
    """A decode enqueued right behind the builder, while the GPU is still busy,
    cannot know the store's mode on the host yet: it runs the kernel that reads
    the mode on the device.  Same bytes either way."""
    if kind == "tiny":
        rows, _ = wl.tiny_rows(seed=3)
        b = rows_u8(rows)
        R, C = 1024, 256
    else:
        R, C = 512, 64
        b = wl.fuzz_rows(2000, R, seed=31)
    n = len(b)
    st = stores(R, C, n)
    d = to_dev(b)
    slots = torch.zeros((n, st.slot), dtype=torch.uint8, device=DEV)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)  # keep the stream busy (about 0.1 s)
    ibp.ibp_build_meta(st.h, d, R, None, n, 9, 10)
    ibp.ibp_compress(st.h, slots, d, R, None, n, None)
    ibp.ibp_decompress(st.h, out, slots, None, n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)
    m, bv = st.meta()
    mr, br = ref_c.build_meta(b, 9, 10)
    assert np.array_equal(m, mr) and np.array_equal(bv, br)


# ---------------------------------------------------------------- chunk-aware builder
CANDS = [(9, 10), (95, 100), (99, 100), (999, 1000), (1, 1)]


@pytest.mark.parametrize("kind", ["sparse", "dense", "fuzz", "kv"])
def test_tuned_builder_matches_oracle(stores, kind):
    """The installed Mask is the candidate whose sample would be stored in the
    fewest bytes (first on ties); sizes and choice match the oracle's."""
    if kind == "sparse":
        n, R, C = 60_000, 512, 1024
        b = rows_u8(wl.sparse_gnn_rows(n, seed=5))
        sample = wl.sample_ids(n, 50, seed=5)
    elif kind == "dense":
        n, R, C = 20_000, 512, 256
        b = rows_u8(wl.dense_gnn_rows(n, seed=6))
        sample = wl.sample_ids(n, 100, seed=6)
    elif kind == "kv":
        R, C = 8192, 256
        b = wl.kv_rows(0, 1, 2, range(200)).view(np.uint8).reshape(-1, R)
        n = len(b)
        sample = None
    else:
        n, R, C = 5000, 256, 64
        b = wl.fuzz_rows(n, R, seed=9)
        sample = wl.sample_ids(n, 200, seed=9)
    st = stores(R, C, n)
    d = to_dev(b)
    d_s = None if sample is None else to_dev(sample)
    m_n = n if sample is None else len(sample)
    chosen = torch.zeros(1, dtype=torch.int32, device=DEV)
    sizes = torch.zeros(len(CANDS), dtype=torch.int64, device=DEV)
    ibp.ibp_build_meta_tuned(st.h, d, R, d_s, m_n, [c[0] for c in CANDS], [c[1] for c in CANDS],
                             chosen, sizes)
    assert st.status() == ibp.IBP_OK
    m, bv = st.meta()
    ref_sizes = []
    metas = []
    rows_s = b if sample is None else b[sample]
    for num, den in CANDS:
        mr, br = ref_c.build_meta(b, num, den, sample_ids=sample)
        slots = np.zeros((len(rows_s), R), np.uint8)
        bm = np.zeros((len(rows_s) + 31) // 32, np.uint32)
        stored = ref_c.compress_batch(rows_s, C, mr, br, slots, bm, nthreads=8)
        ref_sizes.append(int(stored.astype(np.int64).sum()))
        metas.append((mr, br))
    best = int(np.argmin(ref_sizes))
    assert sizes.cpu().tolist() == ref_sizes
    assert int(chosen.item()) == best
    assert np.array_equal(m, metas[best][0]) and np.array_equal(bv, metas[best][1])
    if kind == "sparse":  # the rare 1.0 bits leave the Mask: every row packs
        assert CANDS[best] in [(999, 1000), (1, 1)]
    # and the store decodes what it compresses under the chosen Mask
    slots_g, stored_g = gpu_compress(st, d, n)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, slots_g, None, n)
    assert st.status() == ibp.IBP_OK and np.array_equal(out.cpu().numpy(), b)


def test_tuned_builder_rejects_bad_candidates(stores):
    st = stores(64, 16, 4)
    d = torch.zeros((4, 64), dtype=torch.uint8, device=DEV)
    for nums, dens in [([], []), ([1] * 9, [1] * 9), ([1, 1], [2, 1])]:
        with pytest.raises(ibp.IbpError) as e:
            ibp.ibp_build_meta_tuned(st.h, d, 64, None, 4, nums, dens)
        assert e.value.status == ibp.IBP_EINVAL


@pytest.mark.parametrize("kind", ["dense", "sparse999", "tiny"])
def test_compress_uniform_store_matches_oracle(stores, kind):
    """Once the store's properties have reached the host, a uniform store is
    packed by the compressor's uniform form (masks and shifts as launch
    parameters): its bytes must equal the oracle's."""
    if kind == "dense":
        b = rows_u8(wl.dense_gnn_rows(30_000, seed=8))
        R, C, num, den = 512, 256, 95, 100
    elif kind == "sparse999":
        b = rows_u8(wl.sparse_gnn_rows(30_000, seed=8))
        R, C, num, den = 512, 1024, 999, 1000
    else:
        b = rows_u8(wl.tiny_rows(seed=8)[0])
        R, C, num, den = 1024, 256, 95, 100
    n = len(b)
    st = stores(R, C, n)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, n, num, den)
    torch.cuda.synchronize()
    info = ibp.ibp_store_get_info(st.h)
    assert info.max_runs <= 2
    slots, stored = gpu_compress(st, d, n)
    m, bv = st.meta()
    assert len(set(m.tolist())) == 1 and len(set(bv.tolist())) == 1  # uniform
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, m, bv, st.slot)
    assert np.array_equal(stored, ref_st)
    assert np.array_equal(st.bitmap(), ref_bm)
    assert_streams_equal(slots.cpu().numpy(), ref_sl, ref_st)


def test_store_state_save_and_restore(stores):
    """A store's whole state is its Mask/Bitval and raw bitmap: copied out to
    the host and installed into a fresh store, the slots decode the same."""
    R, C, n = 1024, 256, 3000
    rows, _ = wl.tiny_rows(seed=12, n_rows=n)
    b = rows_u8(rows)
    a = stores(R, C, n)
    d = to_dev(b)
    ibp.ibp_build_meta(a.h, d, R, None, n, 95, 100)
    slots, stored = gpu_compress(a, d, n)
    m, bv = a.meta()
    bm = a.bitmap()
    # a new store, the saved state installed from host arrays
    c = stores(R, C, n)
    c.set_meta(m, bv)
    c.set_bitmap(bm)
    info_a, info_c = ibp.ibp_store_get_info(a.h), ibp.ibp_store_get_info(c.h)
    assert (info_a.min_bits, info_a.max_runs) == (info_c.min_bits, info_c.max_runs)
    host_slots = slots.cpu().pin_memory()
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(c.h, out, host_slots, None, n)
    assert c.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)
    with pytest.raises(ibp.IbpError) as e:  # a Bitval bit outside the Mask is refused
        c.set_meta(np.zeros_like(m), np.ones_like(bv))
    assert e.value.status == ibp.IBP_EINVAL


@pytest.mark.parametrize("R,C", [(512, 256), (8192, 256)])
def test_gather_through_hbm_cache_front(stores, R, C):
    """Rows cached in HBM are read from the cache, the rest over the host link,
    in one launch: the output is every requested row either way."""
    N = 4000 if R <= 2048 else 600
    b = (rows_u8(wl.dense_gnn_rows(N, dim=R // 4, seed=13)) if R <= 2048
         else wl.kv_rows(1, 0, 3, range(N // 3)).view(np.uint8).reshape(-1, R)[:N])
    N = len(b)
    st = stores(R, C, N)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, N, 95, 100)
    host = torch.zeros((N, st.slot), dtype=torch.uint8, pin_memory=True)
    ibp.ibp_compress(st.h, host, d, R, None, N, None)
    torch.cuda.synchronize()
    g = np.random.default_rng(R)
    cached = np.sort(g.choice(N, size=N // 3, replace=False))
    cmap = np.full(N, -1, np.int64)
    cmap[cached] = np.arange(len(cached))[::-1]  # cache slots in another order
    cache = torch.zeros((len(cached), st.slot), dtype=torch.uint8, device=DEV)
    cache[torch.from_numpy(cmap[cached])] = host[torch.from_numpy(cached)].to(DEV)
    ids = g.integers(0, N, size=5 * N // 2).astype(np.int64)
    stride = R + 32
    out = torch.zeros((len(ids), stride), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress_cached(st.h, out, stride, host, cache, len(cached), to_dev(cmap),
                                     to_dev(ids), len(ids))
    assert st.status() == ibp.IBP_OK
    o = out.cpu().numpy()
    assert np.array_equal(o[:, :R], b[ids]) and np.all(o[:, R:] == 0)
    # the cache really is read: poison the host copies of the cached rows
    host[torch.from_numpy(cached)] = 0xEE
    out.zero_()
    ibp.ibp_gather_decompress_cached(st.h, out, stride, host, cache, len(cached), to_dev(cmap),
                                     to_dev(ids), len(ids))
    assert st.status() == ibp.IBP_OK
    o = out.cpu().numpy()
    hit = np.isin(ids, cached)
    assert np.array_equal(o[hit, :R], b[ids[hit]])
    # a map entry past the cache's slots is an error, not a read past the cache
    bad = int(cached[0])
    ids[0] = bad
    cmap[bad] = len(cached) + 5
    out.fill_(0x77)
    ibp.ibp_gather_decompress_cached(st.h, out, stride, host, cache, len(cached), to_dev(cmap),
                                     to_dev(ids), len(ids))
    assert st.status() == ibp.IBP_ERANGE
    o = out.cpu().numpy()
    isbad = ids == bad
    assert np.all(o[isbad, :R] == 0)
    hit = np.isin(ids, cached) & ~isbad
    assert np.array_equal(o[hit, :R], b[ids[hit]])


@pytest.mark.parametrize("n", [8192, 8193, 20_000, 3 * 8192 - 1])
def test_pack_offsets_across_tiles(stores, n):
    """The packed-cache offset scan runs in tiles of 8192 rows: offsets over
    several tiles and a ragged last tile equal the oracle's packing, and the
    packed cache decodes to the rows."""
    R, C = 64, 16
    b = wl.fuzz_rows(n, R, seed=n)
    st = stores(R, C, n, R)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, n, 9, 10)
    slots, stored = gpu_compress(st, d, n)
    mr, br = st.meta()
    ref_sl, _, ref_st = oracle_slots(b, C, mr, br, R)
    assert np.array_equal(stored, ref_st)
    _, offs_ref = ref_c.pack_slots(ref_sl, ref_st)
    offs = torch.zeros(n + 1, dtype=torch.int64, device=DEV)
    ibp.ibp_pack(st.h, None, offs, slots, to_dev(stored.astype(np.int32)), n)
    total = int(offs[-1].item())
    assert np.array_equal(offs.cpu().numpy().astype(np.uint64), offs_ref)
    packed = torch.zeros(total + R, dtype=torch.uint8, device=DEV)
    ibp.ibp_pack(st.h, packed, offs, slots, to_dev(stored.astype(np.int32)), n)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, packed, offs, n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)


@pytest.mark.parametrize("R,C,n", [(512, 1024, 5000), (512, 256, 33), (8192, 256, 700),
                                   (400, 100, 1500), (512, 1024, 1)])
def test_ordered_gather_matches_gather(stores, R, C, n):
    """The ordered gather (ids bucketed by address, rows written back to their
    own positions) gives the plain gather's bytes, duplicates, a strided output
    and an out-of-range id included, on the fast and the generic decoders."""
    N = 3000
    b = wl.fuzz_rows(N, R, seed=R + n)
    st = stores(R, C, N)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, N, 9, 10)
    slots, _ = gpu_compress(st, d, N, host=True)
    g = np.random.default_rng(n)
    ids = g.integers(0, N, size=n).astype(np.int64)
    ids[n // 2] = N + 3 if n > 2 else ids[n // 2]
    stride = R + 48
    ref = torch.full((n, stride), 0x5A, dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress_strided(st.h, ref, stride, slots, None, to_dev(ids), n)
    s_ref = st.status()
    out = torch.full((n, stride), 0x5A, dtype=torch.uint8, device=DEV)
    ws = torch.empty(ibp.order_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress_ordered(st.h, out, stride, slots, None, to_dev(ids), n, ws,
                                      ws.numel())
    assert st.status() == s_ref
    assert torch.equal(out, ref)
    ok = (ids >= 0) & (ids < N)
    assert np.array_equal(out.cpu().numpy()[ok, :R], b[ids[ok]])


def test_ordered_gather_checks_its_workspace(stores):
    st = stores(512, 1024, 100)
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    ids = torch.zeros(64, dtype=torch.int64, device=DEV)
    with pytest.raises(ibp.IbpError) as e:
        ibp.ibp_gather_decompress_ordered(st.h, buf, 512, buf, None, ids, 64, buf,
                                          ibp.order_workspace_bytes(64) - 16)
    assert e.value.status == ibp.IBP_EINVAL
    with pytest.raises(ibp.IbpError) as e:
        ibp.ibp_gather_decompress_ordered(st.h, buf, 512, buf, None, ids, 64,
                                          buf.data_ptr() + 8, ibp.order_workspace_bytes(64))
    assert e.value.status == ibp.IBP_EALIGN


@pytest.mark.parametrize("R,C", [(8192, 256), (2048, 256), (1024, 64), (400, 100)])
def test_length_table_changes_nothing_but_fetches(stores, R, C):
    """With the slots' stored sizes attached, gathers from host slots (fast and
    generic decoders; rows with raw chunks) return the same bytes as without;
    wrong entries (too short, too long) still decode correctly."""
    N = 1200 if R >= 2048 else 3000
    b = (wl.kv_rows(0, 1, 2, range(N // 2)).view(np.uint8).reshape(-1, R)[:N] if R == 8192
         else wl.fuzz_rows(N, R, seed=R))
    N = len(b)
    st = stores(R, C, N)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, N, 95, 100)
    slots = torch.zeros((N, st.slot), dtype=torch.uint8, pin_memory=True)
    stored = torch.zeros(N, dtype=torch.int32, device=DEV)
    ibp.ibp_compress(st.h, slots, d, R, None, N, stored)
    torch.cuda.synchronize()
    ids = to_dev(np.random.default_rng(R).integers(0, N, size=2 * N).astype(np.int64))
    ref = torch.empty((2 * N, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress(st.h, ref, slots, None, ids, 2 * N)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(ref.cpu().numpy(), b[ids.cpu().numpy()])
    for lens in (stored, torch.zeros_like(stored), torch.full_like(stored, 1 << 20)):
        ibp.ibp_store_set_lengths(st.h, lens)
        out = torch.empty_like(ref)
        ibp.ibp_gather_decompress(st.h, out, slots, None, ids, 2 * N)
        assert st.status() == ibp.IBP_OK
        assert torch.equal(out, ref)
    ibp.ibp_store_set_lengths(st.h, None)


@pytest.mark.parametrize("keep,pos", [(1, 31), (4, 0), (7, 23), (10, 13), (11, 5)])
def test_uniform_single_run_decoder_with_raw_chunks(stores, keep, pos):
    """Every word keeps one run of `keep` bits at bit `pos` (the uniform,
    single-run store form; runs of up to 10 bits take a 64-bit window of the
    stream per 4 words).  Some rows carry a raw chunk (a word missing its
    Mask) ahead of packed ones, some are raw throughout; decoded from device
    slots, pinned host slots and a packed cache, the rows come back and the
    stored bytes equal the oracle's."""
    R, C, n = 1024, 256, 3000
    W = R // 4
    run = ((1 << keep) - 1) << pos
    rng = np.random.default_rng(keep * 100 + pos)
    mask = np.full(W, ~run & 0xFFFFFFFF, np.uint32)
    bitval = np.full(W, int(rng.integers(0, 1 << 32)) & int(mask[0]), np.uint32)
    rows = (bitval[None, :] | (rng.integers(0, 1 << 32, (n, W), dtype=np.uint32) & run))
    rows = rows.astype(np.uint32)
    for i in range(0, n, 7):  # a raw chunk: one word misses the Mask
        c = int(rng.integers(0, R // C))
        low = int(mask[0]) & -int(mask[0])  # the lowest Mask bit
        rows[i, c * (C // 4) + int(rng.integers(0, C // 4))] ^= np.uint32(low)
    rows[5::97] = rng.integers(0, 1 << 32, rows[5::97].shape, dtype=np.uint32)  # raw rows
    b = rows.view(np.uint8).reshape(n, R)
    st = stores(R, C, n)
    st.set_meta(mask, bitval)
    torch.cuda.synchronize()
    d = to_dev(b)
    slots, stored = gpu_compress(st, d, n)
    ref_sl, ref_bm, ref_st = oracle_slots(b, C, mask, bitval, st.slot)
    assert np.array_equal(stored, ref_st)
    assert_streams_equal(slots.cpu().numpy(), ref_sl, ref_st)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_decompress(st.h, out, slots, None, n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)
    host = to_pinned(slots.cpu().numpy())
    ids = rng.integers(0, n, 5000).astype(np.int64)
    outg = torch.empty((len(ids), R), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress(st.h, outg, host, None, to_dev(ids), len(ids))
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(outg.cpu().numpy(), b[ids])
    packed_ref, offs_ref = ref_c.pack_slots(ref_sl, ref_st)
    cache = to_dev(np.concatenate([packed_ref, np.zeros(R, np.uint8)]))
    out.zero_()
    ibp.ibp_decompress(st.h, out, cache, to_dev(offs_ref[:n]), n)
    assert st.status() == ibp.IBP_OK
    assert np.array_equal(out.cpu().numpy(), b)


def test_ordered_gather_zipf_batch(stores):
    """A Zipf batch (hot rows looked up thousands of times, their bucket's ids
    ranked within each CTA before one atomic per CTA) through the ordered
    gather: the plain gather's bytes and the rows."""
    N, R, C, n = 3000, 512, 256, 20000
    b = wl.fuzz_rows(N, R, seed=77)
    st = stores(R, C, N)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, N, 9, 10)
    slots, _ = gpu_compress(st, d, N, host=True)
    ids = wl.zipf_ids(n, N, alpha=1.2, seed=5)
    assert np.bincount(ids).max() > 2000
    ref = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress(st.h, ref, slots, None, to_dev(ids), n)
    out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
    ws = torch.empty(ibp.order_workspace_bytes(n), dtype=torch.uint8, device=DEV)
    ibp.ibp_gather_decompress_ordered(st.h, out, R, slots, None, to_dev(ids), n, ws, ws.numel())
    assert st.status() == ibp.IBP_OK
    assert torch.equal(out, ref)
    assert np.array_equal(out.cpu().numpy(), b[ids])


def test_packed_cache_tiles_match_the_row_gather(stores):
    """ibp_decompress of a packed HBM cache reads whole tiles of rows with bulk
    copies when the offsets allow it.  Every case must give the bytes and the
    status of the same rows gathered one by one (ids 0..n-1, the fast
    gather), which reads each row within its own stream:
    - offsets in order, over a ragged last tile;
    - a tile whose offsets run backwards;
    - a row whose start is more than R bytes before the next;
    - streams whose header claims more bytes than the row was packed into,
      mid-tile and on a tile's last row (they run into the next row);
    - a header whose stream would exceed R (corrupt)."""
    rows, _ = wl.tiny_rows(seed=9, n_rows=3000, raw_frac=0.02)
    b = rows_u8(rows)
    n, R, C = len(b), 1024, 256
    st = stores(R, C, n)
    d = to_dev(b)
    ibp.ibp_build_meta(st.h, d, R, None, n, 95, 100)
    slots, stored = gpu_compress(st, d, n)
    offs = torch.zeros(n + 1, dtype=torch.int64, device=DEV)
    ibp.ibp_pack(st.h, None, offs, slots, to_dev(stored.astype(np.int32)), n)
    total = int(offs[-1].item())
    cache = torch.zeros(total + 4 * R, dtype=torch.uint8, device=DEV)
    ibp.ibp_pack(st.h, cache, offs, slots, to_dev(stored.astype(np.int32)), n)
    base = offs[:n].cpu().numpy().astype(np.int64)
    assert st.status() == ibp.IBP_OK
    packed_rows = np.flatnonzero(stored == stored[stored < R].min())
    ids = to_dev(np.arange(n, dtype=np.int64))

    def both(o):
        out = torch.full((n, R), 0x5A, dtype=torch.uint8, device=DEV)
        ibp.ibp_decompress(st.h, out, cache, to_dev(o.astype(np.uint64)), n)
        s1 = st.status()
        ref = torch.full((n, R), 0x5A, dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress(st.h, ref, cache, to_dev(o.astype(np.uint64)), ids, n)
        s2 = st.status()
        assert s1 == s2
        assert torch.equal(out, ref)
        return out.cpu().numpy(), s1

    o, s = both(base)
    assert s == ibp.IBP_OK and np.array_equal(o, b)
    back = base.copy()
    back[64:96] = base[64:96][::-1]  # tile 2 backwards
    back[200] = base[900]            # row 200 far from its neighbours
    o, s = both(back)
    assert s == ibp.IBP_OK
    want = np.arange(n)
    want[64:96] = want[64:96][::-1]
    want[200] = 900
    assert np.array_equal(o, b[want])
    # headers of all-packed rows changed: one claims a raw chunk (a longer
    # stream, still below R), one claims every chunk raw (above R: corrupt)
    hdr = cache.view(torch.int32)
    mid, last, bad = packed_rows[packed_rows % 32 == 5][0], packed_rows[packed_rows % 32 == 31][0], \
        packed_rows[packed_rows % 32 == 12][0]
    for r, value in ((mid, 0b1011), (last, 0b0111), (bad, 0)):
        w = int(base[r]) // 4
        hdr[w] = (int(hdr[w].item()) & ~0xF) | value
    o, s = both(base)
    assert s == ibp.IBP_ECORRUPT
    assert not o[bad].any()
    keep = np.ones(n, bool)
    keep[[mid, last, bad]] = False
    assert np.array_equal(o[keep], b[keep])


_WITHHELD_CHILD = r"""
import numpy as np, torch
from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
dev = torch.device("cuda:0")
rows, _ = wl.tiny_rows(seed=3, n_rows=4096)
b = rows.view(np.uint8).reshape(len(rows), -1)
n, R, C = len(b), 1024, 256
st = ibp.ibp_store_create(R, C, n, 0)
d = torch.from_numpy(b).to(dev)
ibp.ibp_build_meta(st, d, R, None, n, 95, 100)
info = ibp.ibp_store_get_info(st)
slots = torch.zeros((n, info.slot_bytes), dtype=torch.uint8, device=dev)
stored = torch.zeros(n, dtype=torch.int32, device=dev)
ibp.ibp_compress(st, slots, d, R, None, n, stored)
offs = torch.zeros(n + 1, dtype=torch.int64, device=dev)
ibp.ibp_pack(st, None, offs, slots, stored, n)
cache = torch.zeros(int(offs[-1].item()) + R, dtype=torch.uint8, device=dev)
ibp.ibp_pack(st, cache, offs, slots, stored, n)
torch.cuda.synchronize()
assert ibp.ibp_stream_status(st, reset=True) == ibp.IBP_OK
out = torch.zeros((n, R), dtype=torch.uint8, device=dev)
ibp.ibp_decompress(st, out, cache, offs, n)          # tile 5 is never released
torch.cuda.synchronize()
print("status", ibp.ibp_stream_status(st, reset=True))
ids = torch.arange(n, dtype=torch.int64, device=dev)  # the ring decoder: no tiles
ibp.ibp_gather_decompress(st, out, cache, offs, ids, n)
torch.cuda.synchronize()
print("after", ibp.ibp_stream_status(st, reset=True), bool(np.array_equal(out.cpu().numpy(), b)))
"""


def test_tile_decoder_wait_gives_up_and_the_context_stays_usable():
    """The tile decoder's waits are bounded.  A test hook
    (IBP_DEBUG_WITHHOLD_TILE, read once per process) makes the producer never
    release one tile: the warps waiting for it give up after ~2 s, the call
    reports IBP_ETIMEOUT, and the next call in the same process decodes every
    row.  Run in a child process so the hook touches no other test."""
    import os
    import subprocess
    import sys
    env = dict(os.environ, IBP_DEBUG_WITHHOLD_TILE="5")
    r = subprocess.run([sys.executable, "-c", _WITHHELD_CHILD], env=env, capture_output=True,
                       text=True, timeout=600,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(l.split(" ", 1) for l in r.stdout.strip().splitlines() if " " in l)
    assert int(lines["status"]) == ibp.IBP_ETIMEOUT
    assert lines["after"] == "%d True" % ibp.IBP_OK
