"""Do the oracle's pins catch plausible mistakes?

Each mutant is a copy of the pure-Python oracle (``oracle/ibp_ref.py``) with
one planted slip -- a dropped header, a wrong bit order, Mask and Bitval
swapped, a strict threshold, an off-by-one chunk bound, a lost raw-row rule,
a participation rule that ignores the empty-Mask case.  Every mutant must
fail at least one pin that the real oracle passes (hand-worked examples,
closed form of the builder, brute-force minimality, round trip).  The mistakes
are planted in the oracle, on the CPU; nothing here touches the GPU library.
"""
import itertools
import types

import numpy as np
import pytest

from oracle import ibp_ref
from tests import golden_io


def w2b(words):
    return np.asarray(words, dtype=np.uint32).astype("<u4").tobytes()


def _clone():
    m = types.ModuleType("ibp_ref_mutant")
    exec(compile(open(ibp_ref.__file__).read(), ibp_ref.__file__, "exec"), m.__dict__)
    return m


def _patch_source(old, new):
    src = open(ibp_ref.__file__).read()
    assert old in src, "mutation anchor missing: %r" % old
    m = types.ModuleType("ibp_ref_mutant")
    exec(compile(src.replace(old, new, 1), ibp_ref.__file__, "exec"), m.__dict__)
    return m


MUTANTS = {
    # the nch participation bits are not written at the stream start
    "no_header": ("    bits: List[int] = list(p)  # header: one participation bit per chunk",
                  "    bits: List[int] = []"),
    # bits packed MSB-first inside each stream word
    "msb_first": ("        out[s // 32] |= v << (s % 32)", "        out[s // 32] |= v << (31 - s % 32)"),
    # invariant value taken from the wrong side of the threshold
    "bitval_inverted": ("            if inv1:\n                b |= 1 << bit",
                        "            if inv0 and not inv1:\n                b |= 1 << bit"),
    # strict comparison at the threshold
    "strict_threshold": ("            inv1 = ones * den >= num * n", "            inv1 = ones * den > num * n"),
    # chunks one word short
    "chunk_off_by_one": ("    return [range(k * wpc, min((k + 1) * wpc, W)) for k in range((W + wpc - 1) // wpc)]",
                         "    return [range(k * wpc, min((k + 1) * wpc - 1, W)) for k in range((W + wpc - 1) // wpc)]"),
    # rows that do not shrink are not stored raw
    "no_raw_fallback": ("    if 4 * nwords >= R:\n        return bytes(row), True, nbits",
                        "    if False:\n        return bytes(row), True, nbits"),
    # a chunk participates whenever it matches, even when it saves nothing
    "participate_when_empty": ("        out.append(1 if (match and keep < 32 * len(ch)) else 0)",
                               "        out.append(1 if match else 0)"),
    # Mask tested against the wrong operand
    "mask_bitval_swapped": ("        match = all((x[w] & mask[w]) == bitval[w] for w in ch)",
                            "        match = all((x[w] & bitval[w]) == mask[w] for w in ch)"),
}


def _pins(m):
    """Run the pins against oracle module `m`; return the names that fail."""
    failed = []
    # hand-worked compression examples
    for name in golden_io.names("e1") + golden_io.names("e2") + golden_io.names("e4") + golden_io.names("e5"):
        g = golden_io.load(name)
        try:
            stored, raw, bits = m.compress(w2b(g["row"]), g["C"], g["mask"], g["bitval"])
            ok = (bits == g["bits"] and int(raw) == g["raw"]
                  and list(np.frombuffer(stored, "<u4")) == g["stored"])
        except Exception:
            ok = False
        if not ok:
            failed.append(name)
    # hand-worked builder examples
    for name in golden_io.names("e3"):
        g = golden_io.load(name)
        try:
            mk, bv = m.build_meta([w2b([r]) for r in g["rows"]], g["num"], g["den"])
            ok = mk == g["mask"] and bv == g["bitval"]
        except Exception:
            ok = False
        if not ok:
            failed.append(name)
    # builder at the threshold boundary: 19 of 20 rows set bit 0, T = 0.95 -> invariant one
    rows = [w2b([1])] * 19 + [w2b([0])]
    try:
        mk, bv = m.build_meta(rows, 95, 100)
        if not (mk[0] == 0xFFFFFFFF and bv[0] == 1):
            failed.append("threshold_boundary")
    except Exception:
        failed.append("threshold_boundary")
    # brute force: round trip and minimality over every (Mask, Bitval) on 4 free bits of a 2-word row
    positions = [0, 9, 32 + 3, 32 + 30]
    g = np.random.default_rng(2)
    base = g.integers(0, 1 << 32, size=2, dtype=np.uint64).astype(np.uint32)
    bad = False
    for states in itertools.product((0, 1, 2), repeat=len(positions)):
        mask = [0, 0]
        bitval = [0, 0]
        for pos, st in zip(positions, states):
            if st:
                mask[pos // 32] |= 1 << (pos % 32)
            if st == 2:
                bitval[pos // 32] |= 1 << (pos % 32)
        for flips in range(4):
            r = base.copy()
            for j, pos in enumerate(positions[:2]):
                if (flips >> j) & 1:
                    r[pos // 32] ^= np.uint32(1 << (pos % 32))
            rb = r.tobytes()
            try:
                stored, raw, bits = m.compress(rb, 4, mask, bitval)
                back = m.decompress(stored, raw, 8, 4, mask, bitval)
            except Exception:
                bad = True
                break
            if back != rb:
                bad = True
                break
            best = None
            for p in itertools.product((0, 1), repeat=2):
                if all((not p[k]) or (int(r[k]) & mask[k]) == bitval[k] for k in range(2)):
                    b = 2 + sum((32 - bin(mask[k]).count("1")) if p[k] else 32 for k in range(2))
                    best = b if best is None else min(best, b)
            if bits != best:
                bad = True
                break
        if bad:
            break
    if bad:
        failed.append("bruteforce")
    return failed


def test_real_oracle_passes_every_pin():
    assert _pins(_clone()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    failed = _pins(_patch_source(old, new))
    assert failed, "mutant %s passed every pin" % name
