"""Pins of the CPU oracle to facts other than itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped header
bit, a wrong bit order, Mask and Bitval swapped, an off-by-one chunk bound, a
wrong threshold direction) fails at least one of them:
  * hand-worked examples (tests/golden), derived from the format readings;
  * closed forms of the tiny and sparse workloads;
  * brute force over every (Mask, Bitval) pair on a few free bits: round trip
    and minimality of the encoder over all legal participation vectors;
  * the T = 1 builder against AND over rows of agreement with row 0;
  * the size identity and round trip on random rows with ragged chunks;
  * the pure-Python and the C oracle agreeing bit for bit.
"""
import itertools

import numpy as np
import pytest

from oracle import ibp_ref as py
from oracle import ref_c
from lossless_invariant_bit_gb300 import workloads as wl
from tests import golden_io

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def w2b(words):
    return np.asarray(words, dtype=np.uint32).astype("<u4").tobytes()


def b2w(b):
    return list(np.frombuffer(b, dtype="<u4").astype(np.uint32))


# ------------------------------------------------------------ worked examples
@pytest.mark.parametrize("name", golden_io.names("e1") + golden_io.names("e2") + golden_io.names("e4") + golden_io.names("e5"))
@pytest.mark.parametrize("impl", ["py", "c"])
def test_golden_compress(name, impl):
    g = golden_io.load(name)
    row = w2b(g["row"])
    mask = np.array(g["mask"], np.uint32)
    bitval = np.array(g["bitval"], np.uint32)
    assert py.participation(row, g["C"], list(mask), list(bitval)) == g["p"]
    if impl == "py":
        stored, raw, bits = py.compress(row, g["C"], list(mask), list(bitval))
        back = py.decompress(stored, raw, g["R"], g["C"], list(mask), list(bitval))
    else:
        stored, raw, bits = ref_c.compress_row(row, g["C"], mask, bitval)
        back = ref_c.decompress_row(stored, raw, g["R"], g["C"], mask, bitval)
    assert bits == g["bits"]
    assert int(raw) == g["raw"]
    assert b2w(stored) == g["stored"]
    assert back == row


@pytest.mark.parametrize("name", golden_io.names("e1b"))
def test_golden_prefallback_stream(name):
    """The stream a raw row would have had before the raw decision, rebuilt bit by
    bit from the hand-worked participation vector (its length must also match)."""
    g = golden_io.load(name)
    x = g["row"]
    mask, bitval = g["mask"], g["bitval"]
    p = g["p"]
    bits = list(p)
    for k, pk in enumerate(p):
        for w in range(k * (g["C"] // 4), min((k + 1) * (g["C"] // 4), len(x))):
            for b in range(32):
                if not pk or not (mask[w] >> b) & 1:
                    bits.append((x[w] >> b) & 1)
    words = [0] * ((len(bits) + 31) // 32)
    for s, v in enumerate(bits):
        words[s // 32] |= v << (s % 32)
    assert len(bits) == g["bits"]
    assert words == g["prefallback"]


@pytest.mark.parametrize("name", golden_io.names("e3"))
@pytest.mark.parametrize("impl", ["py", "c"])
def test_golden_build(name, impl):
    g = golden_io.load(name)
    rows = [w2b([r]) for r in g["rows"]]
    if impl == "py":
        m, b = py.build_meta(rows, g["num"], g["den"])
    else:
        arr = np.array(g["rows"], np.uint32).reshape(-1, 1)
        m, b = ref_c.build_meta(arr, g["num"], g["den"])
        m, b = list(m), list(b)
    assert [int(v) for v in m] == g["mask"]
    assert [int(v) for v in b] == g["bitval"]


# ------------------------------------------------------------ closed forms
def test_tiny_closed_form():
    """1 + k/1024 fixes sign, exponent and the low 13 mantissa bits; the 1 % of
    N(0,1) rows cannot move a >= 95 % majority.  keep = 10 bits per word, a
    compressible 1 KB row is 4 + 4*640 = 2564 bits = 81 words = 324 B, and every
    N(0,1) row is raw."""
    rows, pick = wl.tiny_rows(seed=0)
    assert len(pick) == 40
    mask, bitval = ref_c.build_meta(rows, 95, 100)
    assert np.all(mask == 0xFF801FFF)
    assert np.all(bitval == 0x3F800000)
    R, C = 1024, 256
    slots = np.zeros((4096, R), np.uint8)
    bitmap = np.zeros(4096 // 32, np.uint32)
    stored = ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap, nthreads=4)
    expect = np.full(4096, 324, np.uint32)
    expect[pick] = 1024
    assert np.array_equal(stored, expect)
    assert int(stored.sum()) == 1_355_104
    raw = np.unpackbits(bitmap.view(np.uint8), bitorder="little").astype(bool)
    assert np.array_equal(np.nonzero(raw)[0], pick)
    out, bad = ref_c.decompress_batch(slots, bitmap, R, C, mask, bitval, n=4096,
                                      slot_stride=R, nthreads=4)
    assert bad == 0
    assert np.array_equal(out, rows.view(np.uint8).reshape(4096, R))


@pytest.mark.parametrize("num,den", [(95, 100), (999, 1000)])
def test_sparse_closed_form(num, den):
    """Entries are 1.0 (bits 23..29) w.p. 0.01 else 0.0.  At T = 0.95 every bit is
    invariant zero: all-zero rows shrink to one 4-byte word, any other row is raw.
    At T = 0.999 bits 23..29 stay, 1 + 128*7 = 897 bits = 29 words = 116 B per row
    (analysing all rows there: a 1 % sample of 20k rows can miss a column's ones)."""
    n = 20000
    rows = wl.sparse_gnn_rows(n, seed=3)
    ids = wl.sample_ids(n, 10, seed=3) if num == 95 else None
    mask, bitval = ref_c.build_meta(rows, num, den, sample_ids=ids)
    R, C = 512, 1024
    slots = np.zeros((n, R), np.uint8)
    bitmap = np.zeros((n + 31) // 32, np.uint32)
    stored = ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap, nthreads=4)
    if num == 95:
        assert np.all(mask == 0xFFFFFFFF) and np.all(bitval == 0)
        zero = ~rows.any(axis=1)
        assert np.array_equal(stored, np.where(zero, 4, 512).astype(np.uint32))
    else:
        assert np.all(mask == ~np.uint32(0x3F800000)) and np.all(bitval == 0)
        assert np.all(stored == 116)
    out, bad = ref_c.decompress_batch(slots, bitmap, R, C, mask, bitval, n=n, slot_stride=R,
                                      nthreads=4)
    assert bad == 0 and np.array_equal(out, rows.view(np.uint8))


@pytest.mark.parametrize("R,C", [(4096, 256), (4096, 1024), (4096, 4096), (512, 256), (48, 8)])
@pytest.mark.parametrize("k", [0, 1, 5, 16, 28, 32])
@pytest.mark.parametrize("scattered", [False, True])
def test_invariant_rows_closed_form(R, C, k, scattered):
    """Rows with exactly k invariant bits per word (the space-saving sweep's input):
    the builder finds Mask = those bits and Bitval = their values; with k > 0 every
    chunk participates, so a row is nch + W*(32 - k) bits, rounded up to words, and
    raw only if that reaches R; with k = 0 every row is raw."""
    n, W = 400, R // 4
    nch = (W + C // 4 - 1) // (C // 4)
    rows = wl.invariant_rows(n, R, k, scattered, seed=5)
    keep, const = wl.invariant_pattern(W, k, scattered, seed=5)
    mask, bitval = ref_c.build_meta(rows, 95, 100)
    assert np.array_equal(mask, ~keep) and np.array_equal(bitval, const)
    slots = np.zeros((n, R), np.uint8)
    bitmap = np.zeros((n + 31) // 32, np.uint32)
    stored = ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap, nthreads=4)
    want = R if k == 0 else 4 * ((nch + W * (32 - k) + 31) // 32)
    want = R if want >= R else want
    assert np.all(stored == want)
    out, bad = ref_c.decompress_batch(slots, bitmap, R, C, mask, bitval, n=n, slot_stride=R,
                                      nthreads=4)
    assert bad == 0 and np.array_equal(out, rows)


# ------------------------------------------------------------ special cases
def test_mask_zero_all_raw():
    rows = wl.fuzz_rows(64, 64, seed=1)
    W = 16
    mask = np.zeros(W, np.uint32)
    bitval = np.zeros(W, np.uint32)
    for r in rows:
        stored, raw, bits = ref_c.compress_row(r.tobytes(), 16, mask, bitval)
        assert raw and bits == 4 + 512 and stored == r.tobytes()


@pytest.mark.parametrize("R,C", [(64, 16), (128, 4), (4096, 256), (100, 12)])
def test_rows_equal_bitval_full_mask(R, C):
    """Mask = ~0 and every row equal to the Bitval: the stream is nch header ones."""
    W = R // 4
    nch = (W + C // 4 - 1) // (C // 4)
    g = np.random.default_rng(5)
    bitval = g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32)
    mask = np.full(W, 0xFFFFFFFF, np.uint32)
    stored, raw, bits = ref_c.compress_row(bitval.tobytes(), C, mask, bitval)
    assert bits == nch
    nwords = (nch + 31) // 32
    if 4 * nwords >= R:
        assert raw
    else:
        assert not raw
        w = b2w(stored)
        assert len(w) == nwords
        allbits = sum(int(v) << (32 * i) for i, v in enumerate(w))
        assert allbits == (1 << nch) - 1


def test_builder_t1_is_agreement_with_row0():
    rows = wl.fuzz_rows(300, 256, seed=2).view(np.uint32)
    mask, bitval = ref_c.build_meta(rows, 1, 1)
    agree = np.bitwise_and.reduce(~(rows ^ rows[0:1]), axis=0)
    assert np.array_equal(mask, agree)
    assert np.array_equal(bitval, rows[0] & agree)


def test_builder_identical_rows():
    row = np.random.default_rng(9).integers(0, 1 << 32, size=(1, 32), dtype=np.uint64)
    rows = np.repeat(row.astype(np.uint32), 7, axis=0)
    for num, den in [(51, 100), (95, 100), (1, 1)]:
        mask, bitval = ref_c.build_meta(rows, num, den)
        assert np.all(mask == 0xFFFFFFFF) and np.array_equal(bitval, rows[0])


def test_builder_threshold_boundary():
    """20 rows, bit 0 set in exactly 19: 19/20 = 0.95 is invariant at T = 0.95
    (the comparison is >=), not at T = 0.96."""
    rows = np.zeros((20, 1), np.uint32)
    rows[:19, 0] = 1
    m, b = ref_c.build_meta(rows, 95, 100)
    assert m[0] == 0xFFFFFFFF and b[0] == 1
    m, b = ref_c.build_meta(rows, 96, 100)
    assert m[0] == 0xFFFFFFFE and b[0] == 0
    # the same count of zeros is invariant zero
    m, b = ref_c.build_meta(1 - rows, 95, 100)
    assert m[0] == 0xFFFFFFFF and b[0] == 0


@pytest.mark.parametrize("num,den", [(1, 2), (3, 2), (0, 1), (1, 0)])
def test_builder_rejects_bad_threshold(num, den):
    with pytest.raises(ValueError):
        ref_c.build_meta(np.zeros((4, 1), np.uint32), num, den)


# ------------------------------------------------------------ brute force
def _bits_for(p, mask, W, C):
    wpc = C // 4
    nch = (W + wpc - 1) // wpc
    bits = nch
    for k in range(nch):
        for w in range(k * wpc, min((k + 1) * wpc, W)):
            bits += (32 - bin(int(mask[w])).count("1")) if p[k] else 32
    return bits


@pytest.mark.parametrize("W,positions", [
    (1, [0, 5, 13, 22, 30, 31]),
    (2, [1, 31, 32 + 0, 32 + 7, 32 + 23, 32 + 31]),
])
def test_bruteforce_all_mask_bitval_pairs(W, positions):
    """Every (Mask, Bitval) with Bitval inside Mask over the free positions
    (3^6 pairs; the other bits are never invariant).  For each pair: round trip,
    and the encoder's stream is the shortest over all legal participation
    vectors (a chunk may take p = 1 only if it matches)."""
    C = 4
    R = 4 * W
    g = np.random.default_rng(11)
    rows = []
    base = g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32)
    for i in range(6):
        r = base.copy()
        for pos in positions:
            if g.random() < 0.5:
                r[pos // 32] ^= np.uint32(1 << (pos % 32))
        rows.append(r)
    checked = 0
    for states in itertools.product((0, 1, 2), repeat=len(positions)):
        mask = np.zeros(W, np.uint32)
        bitval = np.zeros(W, np.uint32)
        for pos, s in zip(positions, states):
            if s:
                mask[pos // 32] |= np.uint32(1 << (pos % 32))
            if s == 2:
                bitval[pos // 32] |= np.uint32(1 << (pos % 32))
        for r in rows:
            rb = r.tobytes()
            stored, raw, bits = ref_c.compress_row(rb, C, mask, bitval)
            assert ref_c.decompress_row(stored, raw, R, C, mask, bitval) == rb
            nch = W
            best = None
            for p in itertools.product((0, 1), repeat=nch):
                legal = all(
                    (not p[k]) or (int(r[k]) & int(mask[k])) == int(bitval[k]) for k in range(nch))
                if legal:
                    b = _bits_for(p, mask, W, C)
                    best = b if best is None else min(best, b)
            assert bits == best
            checked += 1
    assert checked == 3 ** len(positions) * len(rows)


# ------------------------------------------------------------ invariants
@pytest.mark.parametrize("R,C", [(16, 4), (64, 16), (96, 40), (512, 1024), (1024, 256),
                                 (2048, 1024), (200, 64), (8192, 256)])
def test_roundtrip_and_size_identity(R, C):
    rows = wl.fuzz_rows(200, R, seed=R + C)
    mask, bitval = ref_c.build_meta(rows, 9, 10)
    W = R // 4
    slots = np.zeros((len(rows), ((R + 127) // 128) * 128), np.uint8)
    bitmap = np.zeros((len(rows) + 31) // 32, np.uint32)
    stored = ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap)
    m32 = rows.view(np.uint32)
    wpc = C // 4
    nch = (W + wpc - 1) // wpc
    for i in range(len(rows)):
        p = []
        for k in range(nch):
            ws = range(k * wpc, min((k + 1) * wpc, W))
            keep = sum(32 - bin(int(mask[w])).count("1") for w in ws)
            match = all((int(m32[i, w]) & int(mask[w])) == int(bitval[w]) for w in ws)
            p.append(int(match and keep < 32 * len(ws)))
        bits = _bits_for(p, mask, W, C)
        expect = R if 4 * ((bits + 31) // 32) >= R else 4 * ((bits + 31) // 32)
        assert stored[i] == expect
        is_raw = (bitmap[i // 32] >> (i % 32)) & 1
        assert bool(is_raw) == (expect == R)
    out, bad = ref_c.decompress_batch(slots, bitmap, R, C, mask, bitval, n=len(rows),
                                      slot_stride=slots.shape[1])
    assert bad == 0 and np.array_equal(out, rows)


@pytest.mark.parametrize("R,C", [(16, 4), (64, 16), (96, 40), (40, 8)])
def test_python_and_c_oracles_agree(R, C):
    rows = wl.fuzz_rows(40, R, seed=7 * R + C)
    for num, den in [(3, 4), (9, 10), (1, 1)]:
        mc, bc = ref_c.build_meta(rows, num, den)
        mp, bp = py.build_meta([r.tobytes() for r in rows], num, den)
        assert list(mc) == mp and list(bc) == bp
        for r in rows:
            sc = ref_c.compress_row(r.tobytes(), C, mc, bc)
            sp = py.compress(r.tobytes(), C, mp, bp)
            assert sc == sp


def test_corrupt_stream_detected():
    g = golden_io.load("e2a_compress.txt")
    mask = np.array(g["mask"], np.uint32)
    bitval = np.array(g["bitval"], np.uint32)
    stored = w2b(g["stored"])
    # truncated: one word short
    assert ref_c.decompress_row(stored[:4], False, 16, 4, mask, bitval) is None
    assert py.decompress(stored[:4], False, 16, 4, list(mask), list(bitval)) is None
    # header claiming every chunk raw needs 4 + 128 bits -> would have been a raw row
    bad = w2b([0x0, 0x0, 0x0, 0x0, 0x0])
    assert ref_c.decompress_row(bad, False, 16, 4, mask, bitval) is None
    assert py.decompress(bad, False, 16, 4, list(mask), list(bitval)) is None


def test_pack_slots_layout():
    """The packed cache: every row starts on a 16-byte boundary right after the
    previous row's bytes rounded up, the last offset is the total, and the
    stored bytes (not the rest of the slot) are what is copied; a packed
    cache decodes to the rows."""
    n, R, C = 300, 96, 32
    rows = wl.fuzz_rows(n, R, seed=8)
    mask, bitval = ref_c.build_meta(rows, 9, 10)
    slots = np.full((n, R), 0xAB, np.uint8)
    bitmap = np.zeros((n + 31) // 32, np.uint32)
    stored = ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap, nthreads=2)
    packed, offs = ref_c.pack_slots(slots, stored)
    assert offs[0] == 0 and len(offs) == n + 1
    for i in range(n):
        assert offs[i] % 16 == 0
        assert offs[i + 1] - offs[i] == -(-int(stored[i]) // 16) * 16
        assert np.array_equal(packed[offs[i]:offs[i] + stored[i]], slots[i, :stored[i]])
    assert offs[-1] == len(packed)
    for i in (0, 1, n // 2, n - 1):
        raw = bool((bitmap[i >> 5] >> (i & 31)) & 1)
        got = py.decompress(bytes(packed[offs[i]:offs[i] + stored[i]]), raw, R, C, list(mask),
                            list(bitval))
        assert got == rows[i].tobytes()


def test_packed_cache_golden():
    """Hand-worked packed cache (tests/golden/e6_packed_cache.txt): the
    stored words and raw bits of three rows (both chunks packed, one chunk
    raw, a raw row), and the 16-byte rounded offsets they pack at."""
    g = golden_io.load("e6_packed_cache.txt")
    R, C = g["R"], g["C"]
    mask = np.array(g["mask"], np.uint32)
    bitval = np.array(g["bitval"], np.uint32)
    rows = np.stack([np.array(g["row%d" % i], np.uint32) for i in range(3)]).view(np.uint8)
    slots = np.full((3, R), 0xEE, np.uint8)
    bitmap = np.zeros(1, np.uint32)
    stored = ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap, nthreads=1)
    for i in range(3):
        want = np.array(g["stored%d" % i], np.uint32).view(np.uint8)
        assert int(stored[i]) == len(want), i
        assert np.array_equal(slots[i, :len(want)], want), i
        assert (int(bitmap[0]) >> i) & 1 == g["rawbits"][i], i
        got = py.compress(rows[i].tobytes(), C, list(mask), list(bitval))
        assert got[0] == want.tobytes() and int(got[1]) == g["rawbits"][i], i
    packed, offs = ref_c.pack_slots(slots, stored)
    assert [int(o) for o in offs] == g["offsets"]
    for i in range(3):
        want = np.array(g["stored%d" % i], np.uint32).view(np.uint8)
        assert np.array_equal(packed[offs[i]:offs[i] + len(want)], want), i


def test_id_indexed_paths_match_their_definitions():
    """The id lists of the batch calls mean what they say: a build over sample
    ids is the build over rows[ids] (repeats counted, n = the sample's size),
    compressing into slot ids is compressing in order and moving each slot,
    and a gather is the dense decode indexed by ids."""
    n, R, C = 300, 96, 32
    rows = wl.fuzz_rows(n, R, seed=12)
    g = np.random.default_rng(12)
    ids = g.integers(0, n, size=80).astype(np.int64)  # unsorted, with repeats
    m_s, b_s = ref_c.build_meta(rows, 9, 10, sample_ids=ids)
    m_g, b_g = ref_c.build_meta(rows[ids], 9, 10)
    mp, bp = py.build_meta([rows[i].tobytes() for i in ids], 9, 10)
    assert np.array_equal(m_s, m_g) and np.array_equal(b_s, b_g)
    assert list(m_s) == mp and list(b_s) == bp
    # a bit set in exactly the sampled rows is invariant one over the sample
    # (and would be invariant zero if n counted every stored row)
    marked = np.zeros((200, 4), np.uint32)
    sample = np.arange(0, 200, 10, dtype=np.int64)
    marked[sample, 0] = 1
    m1, b1 = ref_c.build_meta(marked.view(np.uint8), 9, 10, sample_ids=sample)
    assert (m1[0] & 1) and (b1[0] & 1)
    # slot ids: the same stored bytes, sizes and raw bits, at the slots named
    slots = np.zeros((n, R), np.uint8)
    bitmap = np.zeros((n + 31) // 32, np.uint32)
    stored = ref_c.compress_batch(rows, C, m_s, b_s, slots, bitmap)
    perm = g.permutation(2 * n)[:n].astype(np.int64)  # into a store of 2n slots
    slots2 = np.zeros((2 * n, R), np.uint8)
    bitmap2 = np.zeros((2 * n + 31) // 32, np.uint32)
    stored2 = ref_c.compress_batch(rows, C, m_s, b_s, slots2, bitmap2, slot_ids=perm)
    assert np.array_equal(stored2, stored)
    raw = np.unpackbits(bitmap.view(np.uint8), bitorder="little")[:n]
    raw2 = np.unpackbits(bitmap2.view(np.uint8), bitorder="little")[:2 * n]
    assert np.array_equal(raw2[perm], raw)
    assert raw2.sum() == raw.sum()  # no other slot marked
    for i in range(n):
        assert np.array_equal(slots2[perm[i], :stored[i]], slots[i, :stored[i]])
    # gather: the dense decode indexed by ids (repeats included)
    dense, bad = ref_c.decompress_batch(slots, bitmap, R, C, m_s, b_s, n=n, slot_stride=R)
    assert bad == 0 and np.array_equal(dense, rows)
    got, bad = ref_c.decompress_batch(slots2, bitmap2, R, C, m_s, b_s, ids=perm[ids],
                                      slot_stride=R)
    assert bad == 0 and np.array_equal(got, rows[ids])
