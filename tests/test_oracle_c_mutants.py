"""Do the pins catch plausible mistakes in the C oracle?

The GPU parity tests compare the CUDA library with the C oracle
(``oracle/ibp_ref.c``), so its pins must catch slips in it too, not only in
the pure-Python oracle.  Each mutant here is a copy of the C source with one
planted slip (a strict threshold, a dropped invariant-zero rule, sample ids or
slot ids or gather ids ignored, MSB-first packing, a raw tie stored
compressed, a participation rule that ignores the empty-Mask case, a decoder
that forgets the Bitval or an overrun, a raw bit never cleared), compiled with
gcc into a temporary library and loaded in place of the real one.  Every
mutant must fail at least one pin that the real source, compiled the same
way, passes.  All of it runs on the CPU.
"""
import ctypes
import itertools
import os
import subprocess

import numpy as np
import pytest

from lossless_invariant_bit_gb300 import workloads as wl
from oracle import ref_c
from tests import golden_io

SRC = os.path.join(os.path.dirname(ref_c.__file__), "ibp_ref.c")
# the mutants are built beside the tests (a git-ignored folder), one file per
# mutant and process, so parallel runs do not share a library
BUILD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_mutant_build")

MUTANTS = {
    "strict_threshold": ("const int inv1 = o * (uint64_t)den >= (uint64_t)num * n;",
                         "const int inv1 = o * (uint64_t)den > (uint64_t)num * n;"),
    "no_invariant_zero": ("if (inv1 || inv0) m |= 1u << bit;", "if (inv1) m |= 1u << bit;"),
    "sample_ids_ignored": ("const uint64_t r = sample_ids ? (uint64_t)sample_ids[i] : i;",
                           "const uint64_t r = i;"),
    "msb_first": ("if (v) bw->words[bw->pos / 32] |= 1u << (bw->pos % 32);",
                  "if (v) bw->words[bw->pos / 32] |= 1u << (31 - bw->pos % 32);"),
    "raw_tie_compressed": ("if (4 * stored_words >= R) {", "if (4 * stored_words > R) {"),
    "participate_when_empty": ("p[k] = all_match && keep < full;", "p[k] = all_match;"),
    "decoder_drops_bitval": ("v = bit_of(bitval[w], b);", "v = 0;"),
    "decoder_ignores_overrun": ("if (br.overrun) status = IBP_REF_ECORRUPT;",
                                "if (0) status = IBP_REF_ECORRUPT;"),
    # the first occurrence is the loop that writes the slots
    "slot_ids_ignored": ("const uint64_t s = slot_ids ? (uint64_t)slot_ids[i] : i;",
                         "const uint64_t s = i;"),
    "raw_bit_never_cleared": ("bitmap[s / 32] &= ~(1u << (s % 32));", "(void)0;"),
    "gather_ids_ignored": ("const uint64_t id = ids ? (uint64_t)ids[i] : i;",
                           "const uint64_t id = i;"),
    "chunk_one_word_short": ("return e < W ? e : W;", "return e - 1 < W ? e - 1 : W;"),
}


def w2b(words):
    return np.asarray(words, dtype=np.uint32).astype("<u4").tobytes()


def _compile(name, src):
    os.makedirs(BUILD, exist_ok=True)
    stem = os.path.join(BUILD, "%s_%d" % (name, os.getpid()))
    with open(stem + ".c", "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o",
                           stem + ".so", stem + ".c"])
    L = ref_c.bind(ctypes.CDLL(stem + ".so"))
    os.remove(stem + ".c")  # the loaded library stays mapped; its files go
    os.remove(stem + ".so")
    return L


def _c_pins():
    """Run the pins through ``ref_c`` (whatever library it has loaded); return
    the names of those that fail."""
    failed = []

    def check(name, fn):
        try:
            ok = bool(fn())
        except Exception:
            ok = False
        if not ok:
            failed.append(name)

    for name in golden_io.names("e1") + golden_io.names("e2") + golden_io.names("e4") + golden_io.names("e5"):
        g = golden_io.load(name)

        def golden(g=g):
            row = w2b(g["row"])
            mask = np.array(g["mask"], np.uint32)
            bitval = np.array(g["bitval"], np.uint32)
            stored, raw, bits = ref_c.compress_row(row, g["C"], mask, bitval)
            back = ref_c.decompress_row(stored, raw, g["R"], g["C"], mask, bitval)
            return (bits == g["bits"] and int(raw) == g["raw"] and back == row
                    and list(np.frombuffer(stored, "<u4")) == g["stored"])
        check(name, golden)

    for name in golden_io.names("e3"):
        g = golden_io.load(name)

        def golden_build(g=g):
            m, b = ref_c.build_meta(np.array(g["rows"], np.uint32).reshape(-1, 1), g["num"],
                                    g["den"])
            return list(m) == g["mask"] and list(b) == g["bitval"]
        check(name, golden_build)

    def boundary():  # 19 of 20 rows set bit 0: invariant one at T = 0.95
        m, b = ref_c.build_meta(np.array([1] * 19 + [0], np.uint32).reshape(-1, 1), 95, 100)
        return m[0] == 0xFFFFFFFF and b[0] == 1
    check("threshold_boundary", boundary)

    def sampled_build():  # a bit set in exactly the sampled rows: invariant one
        marked = np.zeros((200, 4), np.uint32)
        sample = np.arange(3, 200, 10, dtype=np.int64)
        marked[sample, 0] = 1
        m, b = ref_c.build_meta(marked.view(np.uint8), 9, 10, sample_ids=sample)
        return (m[0] & 1) and (b[0] & 1)
    check("sampled_build", sampled_build)

    n, R, C = 64, 96, 32
    rows = wl.fuzz_rows(n, R, seed=31)
    mask, bitval = ref_c.build_meta(rows, 9, 10)

    def batch_round_trip():  # slots whose raw bits start set
        slots = np.zeros((n, R), np.uint8)
        bitmap = np.full(n // 32, 0xFFFFFFFF, np.uint32)
        stored = ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap)
        raw = np.unpackbits(bitmap.view(np.uint8), bitorder="little")[:n].astype(bool)
        out, bad = ref_c.decompress_batch(slots, bitmap, R, C, mask, bitval, n=n,
                                          slot_stride=R)
        return (bad == 0 and np.array_equal(out, rows) and np.array_equal(raw, stored == R)
                and 0 < raw.sum() < n)
    check("batch_round_trip", batch_round_trip)

    def slot_and_gather_ids():
        perm = np.random.default_rng(31).permutation(n).astype(np.int64)
        slots = np.zeros((n, R), np.uint8)
        bitmap = np.zeros(n // 32, np.uint32)
        ref_c.compress_batch(rows, C, mask, bitval, slots, bitmap, slot_ids=perm)
        # n ids (repeats included), so a mutant that reads slot i stays in bounds
        ids = np.random.default_rng(32).integers(0, n, size=n).astype(np.int64)
        got, bad = ref_c.decompress_batch(slots, bitmap, R, C, mask, bitval, ids=perm[ids],
                                          slot_stride=R)
        return bad == 0 and np.array_equal(got, rows[ids])
    check("slot_and_gather_ids", slot_and_gather_ids)

    def corrupt_detected():  # a compressed stream cut one word short
        g = golden_io.load("e2a_compress.txt")
        stored = w2b(g["stored"])
        return ref_c.decompress_row(stored[:4], False, 16, 4, np.array(g["mask"], np.uint32),
                                    np.array(g["bitval"], np.uint32)) is None
    check("corrupt_detected", corrupt_detected)

    def minimal_streams():  # every (Mask, Bitval) on 4 free bits of a 2-word row, C = 4
        positions = [0, 9, 32 + 3, 32 + 30]
        base = np.random.default_rng(2).integers(0, 1 << 32, size=2,
                                                 dtype=np.uint64).astype(np.uint32)
        for states in itertools.product((0, 1, 2), repeat=len(positions)):
            mk = np.zeros(2, np.uint32)
            bv = np.zeros(2, np.uint32)
            for pos, st in zip(positions, states):
                if st:
                    mk[pos // 32] |= np.uint32(1 << (pos % 32))
                if st == 2:
                    bv[pos // 32] |= np.uint32(1 << (pos % 32))
            for flips in range(4):
                r = base.copy()
                for j, pos in enumerate(positions[:2]):
                    if (flips >> j) & 1:
                        r[pos // 32] ^= np.uint32(1 << (pos % 32))
                stored, raw, bits = ref_c.compress_row(r.tobytes(), 4, mk, bv)
                if ref_c.decompress_row(stored, raw, 8, 4, mk, bv) != r.tobytes():
                    return False
                best = min(2 + sum((32 - bin(int(mk[k])).count("1")) if p[k] else 32
                                   for k in range(2))
                           for p in itertools.product((0, 1), repeat=2)
                           if all((not p[k]) or (int(r[k]) & int(mk[k])) == int(bv[k])
                                  for k in range(2)))
                if bits != best:
                    return False
        return True
    check("minimal_streams", minimal_streams)
    return failed


@pytest.fixture
def swap_library(monkeypatch):
    def use(L):
        monkeypatch.setattr(ref_c, "_lib", L)
    return use


def test_real_c_source_passes_every_pin(swap_library):
    swap_library(_compile("real", open(SRC).read()))
    assert _c_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_c_mutant_is_caught(name, swap_library):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, "mutation anchor missing: %r" % old
    swap_library(_compile(name, src.replace(old, new, 1)))
    failed = _c_pins()
    assert failed, "mutant %s passed every pin" % name
