"""Invariant Bit Packing (IBP) -- pure-Python oracle for small inputs.

TEST INFRASTRUCTURE ONLY: used by the test suite, the smoke check and the
benchmark's CPU-baseline leg; never by the library.  It is a second,
independent restatement of the same format as ``ibp_ref.c`` (written with
Python integers and lists, no shared code), so that the two oracles and the
pinned examples cross-check one another.

Source: "Reducing the GPU Memory Bottleneck with Lossless Compression for ML
-- Extended" (gist.science explainer), Technical Summary, Methodology > Core
Algorithm (Preprocessing, Compression, Decompression) and System Integration
(in-place buffers, GPU bitmask of compressed tensors); juhe.plus review,
metadata paragraph (uncompressible tensors stay raw).

Format readings (the pages fix the idea, not the bitstream):
  * a row of R bytes = R/4 little-endian uint32 words; row bit j = bit j%32
    of word j//32;
  * bit j is invariant iff ones*den >= num*n or (n-ones)*den >= num*n;
  * chunk k = words [k*wpc, min((k+1)*wpc, W)), wpc = C/4;
  * p_k = 1 iff the chunk matches Bitval on Mask in every word and
    keep_k < 32*|k|;
  * stream = nch participation bits, then per chunk the kept bits (p_k = 1)
    or all bits (p_k = 0), LSB-first into uint32 words;
  * raw row iff 4*ceil(bits/32) >= R.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple


def row_words(row: bytes) -> List[int]:
    """Split R bytes into R/4 little-endian 32-bit words."""
    assert len(row) % 4 == 0
    return [int.from_bytes(row[4 * i: 4 * i + 4], "little") for i in range(len(row) // 4)]


def words_bytes(words: Sequence[int]) -> bytes:
    return b"".join(int(w & 0xFFFFFFFF).to_bytes(4, "little") for w in words)


def chunks(W: int, C: int) -> List[range]:
    """Word ranges of the chunks of a W-word row at chunk size C bytes."""
    wpc = C // 4
    return [range(k * wpc, min((k + 1) * wpc, W)) for k in range((W + wpc - 1) // wpc)]


def build_meta(rows: Sequence[bytes], num: int, den: int) -> Tuple[List[int], List[int]]:
    """Mask and Bitval words from the analysed rows (Core Algorithm, Preprocessing)."""
    n = len(rows)
    assert n >= 1 and 0 < den and 2 * num > den and num <= den
    W = len(rows[0]) // 4
    words = [row_words(r) for r in rows]
    mask, bitval = [], []
    for w in range(W):
        m = b = 0
        for bit in range(32):
            ones = sum((ws[w] >> bit) & 1 for ws in words)
            inv1 = ones * den >= num * n
            inv0 = (n - ones) * den >= num * n
            if inv1 or inv0:
                m |= 1 << bit
            if inv1:
                b |= 1 << bit
        mask.append(m)
        bitval.append(b)
    return mask, bitval


def participation(row: bytes, C: int, mask: Sequence[int], bitval: Sequence[int]) -> List[int]:
    x = row_words(row)
    out = []
    for ch in chunks(len(x), C):
        keep = sum(32 - bin(mask[w]).count("1") for w in ch)
        match = all((x[w] & mask[w]) == bitval[w] for w in ch)
        out.append(1 if (match and keep < 32 * len(ch)) else 0)
    return out


def compress(row: bytes, C: int, mask: Sequence[int], bitval: Sequence[int]
             ) -> Tuple[bytes, bool, int]:
    """Compress one row.  Returns (stored bytes, is_raw, stream bits)."""
    x = row_words(row)
    R = len(row)
    p = participation(row, C, mask, bitval)
    bits: List[int] = list(p)  # header: one participation bit per chunk
    for pk, ch in zip(p, chunks(len(x), C)):
        for w in ch:
            for b in range(32):
                if pk == 0 or not (mask[w] >> b) & 1:
                    bits.append((x[w] >> b) & 1)
    nbits = len(bits)
    nwords = (nbits + 31) // 32
    if 4 * nwords >= R:
        return bytes(row), True, nbits
    out = [0] * nwords
    for s, v in enumerate(bits):
        out[s // 32] |= v << (s % 32)
    return words_bytes(out), False, nbits


def decompress(stored: bytes, is_raw: bool, R: int, C: int, mask: Sequence[int],
               bitval: Sequence[int]) -> Optional[bytes]:
    """Inverse of ``compress``.  Returns None for a corrupt stream."""
    if is_raw:
        return bytes(stored[:R]) if len(stored) >= R else None
    sw = row_words(stored[: len(stored) // 4 * 4])
    avail = 32 * len(sw)
    pos = 0

    def take() -> Optional[int]:
        nonlocal pos
        if pos >= avail:
            return None
        v = (sw[pos // 32] >> (pos % 32)) & 1
        pos += 1
        return v

    W = R // 4
    chs = chunks(W, C)
    p = [take() for _ in chs]
    if any(v is None for v in p):
        return None
    need = len(chs) + sum((32 - bin(mask[w]).count("1")) if pk else 32
                          for pk, ch in zip(p, chs) for w in ch)
    if 4 * ((need + 31) // 32) >= R:
        return None
    out = [0] * W
    for pk, ch in zip(p, chs):
        for w in ch:
            v = 0
            for b in range(32):
                if pk and (mask[w] >> b) & 1:
                    bit = (bitval[w] >> b) & 1
                else:
                    bit = take()
                    if bit is None:
                        return None
                v |= bit << b
            out[w] = v
    return words_bytes(out)
