"""Seeded synthetic inputs for the IBP workloads.

This module only draws random numbers and index lists.  It holds none of the
codec's arithmetic, so both the GPU path and the CPU oracle may be fed from it.
Every generator is block-seeded: rows [b*B, (b+1)*B) come from
``numpy.random.default_rng([seed, tag, b])``, so any block can be regenerated
on its own (used to check sampled rows of full-size stores).

Workloads (shapes and distributions of the pages' evaluation, synthetic
stand-ins for their datasets):
  tiny        4096 x 256 fp32, 1 + k/1024 with k ~ U{0..1023}; 1 % of rows N(0,1)
  sparse GNN  N x 128 fp32, 1.0 with p = 0.01 else 0.0
  dense GNN   N x 128 fp32 ~ N(0, 0.1^2)
  DLRM        tables of N x dim fp32 ~ N(0, 0.01^2), Zipf(1.05) lookups
  KV cache    fp16 K/V rows of 32 heads x 128, N(0,1) x per-channel log-normal
              scale, 2 % outlier channels x 20
  saving      rows with exactly k invariant bits per 32-bit word (space-saving
              sweep): the k high bits, equal in every word, or k scattered
              positions per word with a per-word constant
  weights     bf16 weight matrices ~ N(0, 0.02^2) (rounded to nearest even),
              rows of 4096 values (weight-offload stream)
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np

BLOCK_ROWS = 65536

_TAG = {"tiny": 1, "sparse": 2, "dense": 3, "dlrm": 4, "kv": 5, "ids": 6, "fuzz": 7,
        "saving": 8, "weights": 9}


def _rng(seed: int, tag: str, *more: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), _TAG[tag], *[int(m) for m in more]])


# ---------------------------------------------------------------- rows
def tiny_rows(seed: int = 0, n_rows: int = 4096, dim: int = 256, raw_frac: float = 0.01
              ) -> Tuple[np.ndarray, np.ndarray]:
    """(rows float32 [n_rows, dim], indices of the N(0,1) rows)."""
    g = _rng(seed, "tiny")
    k = g.integers(0, 1024, size=(n_rows, dim))
    rows = (1.0 + k.astype(np.float64) / 1024.0).astype(np.float32)
    n_raw = int(raw_frac * n_rows)
    pick = np.sort(g.choice(n_rows, size=n_raw, replace=False))
    rows[pick] = g.standard_normal((n_raw, dim)).astype(np.float32)
    return rows, pick


def _blocks(n_rows: int, first: int = 0, count: Optional[int] = None):
    count = n_rows - first if count is None else count
    r = first
    end = first + count
    while r < end:
        b = r // BLOCK_ROWS
        lo = r - b * BLOCK_ROWS
        hi = min(BLOCK_ROWS, end - b * BLOCK_ROWS)
        yield b, lo, hi
        r = b * BLOCK_ROWS + hi


def sparse_gnn_rows(n_rows: int, dim: int = 128, p: float = 0.01, seed: int = 0,
                    first: int = 0, count: Optional[int] = None,
                    out: Optional[np.ndarray] = None) -> np.ndarray:
    """Rows [first, first+count) of the sparse feature matrix (1.0 w.p. p else 0.0)."""
    count = n_rows - first if count is None else count
    if out is None:
        out = np.empty((count, dim), np.float32)
    o = 0
    for b, lo, hi in _blocks(n_rows, first, count):
        u = _rng(seed, "sparse", b).random((BLOCK_ROWS, dim), dtype=np.float32)[lo:hi]
        out[o:o + hi - lo] = (u < p).astype(np.float32)
        o += hi - lo
    return out


def dense_gnn_rows(n_rows: int, dim: int = 128, sigma: float = 0.1, seed: int = 0,
                   first: int = 0, count: Optional[int] = None,
                   out: Optional[np.ndarray] = None) -> np.ndarray:
    """Rows [first, first+count) of the dense feature matrix ~ N(0, sigma^2)."""
    count = n_rows - first if count is None else count
    if out is None:
        out = np.empty((count, dim), np.float32)
    o = 0
    for b, lo, hi in _blocks(n_rows, first, count):
        z = _rng(seed, "dense", b).standard_normal((BLOCK_ROWS, dim), dtype=np.float32)[lo:hi]
        out[o:o + hi - lo] = z * np.float32(sigma)
        o += hi - lo
    return out


def dlrm_rows(n_rows: int, dim: int, table: int, sigma: float = 0.01, seed: int = 0,
              first: int = 0, count: Optional[int] = None,
              out: Optional[np.ndarray] = None) -> np.ndarray:
    """Rows of embedding table `table` ~ N(0, sigma^2)."""
    count = n_rows - first if count is None else count
    if out is None:
        out = np.empty((count, dim), np.float32)
    o = 0
    bl = max(1, BLOCK_ROWS * 128 // dim)
    r = first
    end = first + count
    while r < end:
        b = r // bl
        lo = r - b * bl
        hi = min(bl, end - b * bl)
        z = _rng(seed, "dlrm", table, dim, b).standard_normal((bl, dim), dtype=np.float32)[lo:hi]
        out[o:o + hi - lo] = z * np.float32(sigma)
        o += hi - lo
        r = b * bl + hi
    return out


def kv_channel_scales(layer: int, kv: int, channels: int = 4096, sigma: float = 0.5,
                      outlier_frac: float = 0.02, outlier_gain: float = 20.0,
                      seed: int = 0) -> np.ndarray:
    """Per-channel scale s_c = exp(sigma*z_c), with 2 % of channels x outlier_gain."""
    g = _rng(seed, "kv", layer, kv, 1 << 20)
    s = np.exp(sigma * g.standard_normal(channels))
    n_out = int(round(outlier_frac * channels))
    s[g.choice(channels, size=n_out, replace=False)] *= outlier_gain
    return s.astype(np.float32)


def kv_rows(layer: int, kv: int, batch: int, tokens: Sequence[int], channels: int = 4096,
            seed: int = 0, scales: Optional[np.ndarray] = None) -> np.ndarray:
    """fp16 K (kv=0) or V (kv=1) rows [batch, len(tokens), channels] of one layer.

    Token t of sequence b is drawn from its own stream, so any token can be
    regenerated alone."""
    if scales is None:
        scales = kv_channel_scales(layer, kv, channels, seed=seed)
    tokens = list(tokens)
    out = np.empty((batch, len(tokens), channels), np.float16)
    for b in range(batch):
        for i, t in enumerate(tokens):
            z = _rng(seed, "kv", layer, kv, b, t).standard_normal(channels, dtype=np.float32)
            out[b, i] = (z * scales).astype(np.float16)
    return out


# ---------------------------------------------------------------- ids
def splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (Steele, Lea, Flood 2014), vectorised on uint64."""
    with np.errstate(over="ignore"):
        z = (x.astype(np.uint64) + np.uint64(0x9E3779B97F4A7C15))
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def sample_ids(n_rows: int, per_mille: int, seed: int = 0) -> np.ndarray:
    """Rows in the metadata sample: id is in iff splitmix64(seed ^ id) mod 1000 < per_mille."""
    ids = np.arange(n_rows, dtype=np.uint64)
    h = splitmix64(ids ^ np.uint64(seed))
    return np.nonzero(h % np.uint64(1000) < np.uint64(per_mille))[0].astype(np.int64)


def uniform_ids(n: int, n_rows: int, seed: int = 0, batch: int = 0) -> np.ndarray:
    """n row ids ~ U[0, n_rows), with replacement."""
    return _rng(seed, "ids", 1, batch).integers(0, n_rows, size=n, dtype=np.int64)


def two_hop_ids(n_rows: int, seeds: int = 1024, fanout: Tuple[int, int] = (15, 10),
                seed: int = 0, batch: int = 0) -> np.ndarray:
    """Sorted unique ids of a 2-hop sampled mini-batch on a uniform random graph."""
    g = _rng(seed, "ids", 2, batch)
    s = g.integers(0, n_rows, size=seeds, dtype=np.int64)
    h1 = g.integers(0, n_rows, size=seeds * fanout[0], dtype=np.int64)
    h2 = g.integers(0, n_rows, size=seeds * fanout[0] * fanout[1], dtype=np.int64)
    return np.unique(np.concatenate([s, h1, h2]))


def zipf_ids(batch: int, n_rows: int, alpha: float = 1.05, table: int = 0, seed: int = 0
             ) -> np.ndarray:
    """batch ids of a truncated Zipf(alpha) over [1, n_rows] ranks, mapped through a
    seeded permutation of the table's rows (inverse-CDF sampling)."""
    g = _rng(seed, "ids", 3, table)
    ranks = np.arange(1, n_rows + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** -alpha)
    cdf /= cdf[-1]
    r = np.searchsorted(cdf, g.random(batch), side="left")
    r = np.minimum(r, n_rows - 1)
    perm = g.permutation(n_rows)
    return perm[r].astype(np.int64)


def kv_row_ids(batch: int, tokens: int, seq_len: int = 2048) -> np.ndarray:
    """Local ids b*seq_len + t of the first `tokens` tokens of each of `batch` sequences."""
    b = np.arange(batch, dtype=np.int64)[:, None]
    t = np.arange(tokens, dtype=np.int64)[None, :]
    return (b * seq_len + t).reshape(-1)


def fuzz_rows(n: int, R: int, seed: int, tag: int = 0) -> np.ndarray:
    """Random rows [n, R bytes] with a planted bit structure: most bit positions
    constant, a few random, a few rows fully random."""
    g = _rng(seed, "fuzz", tag)
    W = R // 4
    base = g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32)
    vary = g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32)
    vary &= g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32)
    vary &= g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32)
    noise = g.integers(0, 1 << 32, size=(n, W), dtype=np.uint64).astype(np.uint32)
    rows = (base[None, :] & ~vary[None, :]) | (noise & vary[None, :])
    flip = g.random((n, W)) < 0.002
    rows = np.where(flip, noise, rows).astype(np.uint32)
    wild = g.random(n) < 0.05
    rows[wild] = g.integers(0, 1 << 32, size=(int(wild.sum()), W), dtype=np.uint64).astype(np.uint32)
    return rows.view(np.uint8).reshape(n, R)


def invariant_pattern(W: int, k: int, scattered: bool, seed: int = 0
                      ) -> Tuple[np.ndarray, np.ndarray]:
    """(keep, const), u32[W] each: keep marks the 32 - k bits of each word that vary,
    const gives the value of the k others.

    Not scattered: the k high bits of every word are invariant and take the same
    value (fp32 rows of one magnitude class).  Scattered: k distinct random
    positions per word, a random constant per word."""
    assert 0 <= k <= 32
    g = _rng(seed, "saving", k, int(scattered))
    if not scattered:
        inv = 0 if k == 0 else ((0xFFFFFFFF << (32 - k)) & 0xFFFFFFFF)
        keep = np.full(W, (~inv) & 0xFFFFFFFF, np.uint32)
        const = np.full(W, int(g.integers(0, 1 << 32, dtype=np.uint64)) & inv, np.uint32)
        return keep, const
    keep = np.full(W, 0xFFFFFFFF, np.uint32)
    for w in range(W):
        for b in g.choice(32, size=k, replace=False):
            keep[w] &= np.uint32(~(1 << int(b)) & 0xFFFFFFFF)
    const = g.integers(0, 1 << 32, size=W, dtype=np.uint64).astype(np.uint32) & ~keep
    return keep, const


def invariant_rows(n: int, R: int, k: int, scattered: bool, seed: int = 0) -> np.ndarray:
    """Rows [n, R bytes]: random bits where keep is set, const elsewhere."""
    W = R // 4
    keep, const = invariant_pattern(W, k, scattered, seed)
    noise = _rng(seed, "saving", k, int(scattered), 1).integers(
        0, 1 << 32, size=(n, W), dtype=np.uint64).astype(np.uint32)
    return ((noise & keep[None, :]) | const[None, :]).view(np.uint8).reshape(n, R)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_weight_rows(n_rows: int, cols: int = 4096, sigma: float = 0.02, seed: int = 0,
                     matrix: int = 0) -> np.ndarray:
    """Rows [n_rows, cols] of bf16 bit patterns of one weight matrix ~ N(0, sigma^2)."""
    z = _rng(seed, "weights", matrix).standard_normal((n_rows, cols), dtype=np.float32)
    return to_bf16_bits(z * np.float32(sigma))
