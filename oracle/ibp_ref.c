/*
 * Invariant Bit Packing (IBP) -- plain CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * restatement of the IBP format that the GPU library is checked against.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or constant with the CUDA
 * library, and the library never calls it.
 *
 * Everything is done one bit at a time, in the order the method states it:
 *
 *   "Reducing the GPU Memory Bottleneck with Lossless Compression for ML --
 *    Extended" (gist.science explainer), Technical Summary,
 *   Methodology > Core Algorithm:
 *     - Preprocessing: a bit position is invariant when it holds the same
 *       value in at least a fraction T of the analysed tensors; the Mask marks
 *       those positions and the Bitval holds their values.
 *     - Compression: tensors are handled in chunks; a chunk whose invariant
 *       bits equal the Bitval has them removed and the remaining bits shifted
 *       together; each chunk carries a participation bit saying whether it was
 *       compressed or left as it was.
 *     - Decompression: the inverse, re-inserting the invariant bits.
 *   System Integration: in-place compression into fixed-size buffers, and a
 *   GPU bitmask of which tensors are stored compressed.
 *   (juhe.plus review, "metadata" paragraph: a tensor whose compressed form
 *    saves no space is kept in its original form.)
 *
 * Readings taken where the pages leave the bitstream open (each one is a
 * choice, not something the pages fix):
 *   - a row of R bytes is R/4 little-endian 32-bit words; row bit j is bit
 *     (j mod 32) of word floor(j/32); Mask and Bitval have one bit per row
 *     bit position;
 *   - threshold: ones*den >= num*n (invariant one) or
 *     (n-ones)*den >= num*n (invariant zero), exact integer arithmetic,
 *     with 1/2 < num/den <= 1;
 *   - chunk k covers words [k*wpc, min((k+1)*wpc, W)), wpc = C/4;
 *   - a chunk participates (p_k = 1) iff every one of its words matches the
 *     Bitval on the Mask AND removing the invariant bits saves at least one
 *     bit (keep_k < 32*|k|);
 *   - stream: bits LSB-first into 32-bit words; first the nch participation
 *     bits, then chunk by chunk either the non-invariant bits of each word in
 *     ascending bit order (p_k = 1) or all 32 bits of each word (p_k = 0);
 *     unused high bits of the last word are zero;
 *   - a row whose stream needs 4*ceil(bits/32) >= R bytes is stored raw
 *     (its R bytes unchanged) and flagged in the raw bitmap.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IBP_REF_OK 0
#define IBP_REF_EINVAL 1
#define IBP_REF_ECORRUPT 4

/* ---- little-endian word access, independent of host byte order ---- */
static uint32_t load_le32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
         ((uint32_t)p[3] << 24);
}
static void store_le32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)(v & 0xFFu);
  p[1] = (uint8_t)((v >> 8) & 0xFFu);
  p[2] = (uint8_t)((v >> 16) & 0xFFu);
  p[3] = (uint8_t)((v >> 24) & 0xFFu);
}
static int bit_of(uint32_t word, unsigned b) { return (int)((word >> b) & 1u); }

static unsigned count_ones(uint32_t v) {
  unsigned c = 0;
  for (unsigned b = 0; b < 32; ++b) c += (unsigned)bit_of(v, b);
  return c;
}

/* Geometry of a row: W words, wpc words per chunk, nch chunks. */
static int geometry(uint32_t R, uint32_t C, uint32_t* W, uint32_t* wpc, uint32_t* nch) {
  if (R == 0 || C == 0 || (R % 4) != 0 || (C % 4) != 0) return IBP_REF_EINVAL;
  *W = R / 4;
  *wpc = C / 4;
  *nch = (*W + *wpc - 1) / *wpc;
  return IBP_REF_OK;
}
static uint32_t chunk_first(uint32_t k, uint32_t wpc) { return k * wpc; }
static uint32_t chunk_end(uint32_t k, uint32_t wpc, uint32_t W) {
  uint32_t e = (k + 1) * wpc;
  return e < W ? e : W;
}

/* ------------------------------------------------------------------ */
/* Preprocessing: Mask / Bitval from n sample rows.                    */
/* ------------------------------------------------------------------ */
int ibp_ref_build_meta(const uint8_t* rows, uint64_t row_stride, uint32_t R,
                       const int64_t* sample_ids, uint64_t n, uint32_t num, uint32_t den,
                       uint32_t* mask, uint32_t* bitval) {
  if (R == 0 || (R % 4) != 0 || n == 0 || den == 0) return IBP_REF_EINVAL;
  if ((uint64_t)num > (uint64_t)den || 2ull * num <= (uint64_t)den) return IBP_REF_EINVAL;
  const uint32_t W = R / 4;
  const uint64_t nbits = 8ull * R;
  uint64_t* ones = (uint64_t*)calloc(nbits, sizeof(uint64_t));
  if (!ones) return IBP_REF_EINVAL;
  for (uint64_t i = 0; i < n; ++i) {
    const uint64_t r = sample_ids ? (uint64_t)sample_ids[i] : i;
    const uint8_t* row = rows + r * row_stride;
    for (uint64_t j = 0; j < nbits; ++j) {
      const uint32_t word = load_le32(row + 4 * (j / 32));
      ones[j] += (uint64_t)bit_of(word, (unsigned)(j % 32));
    }
  }
  for (uint32_t w = 0; w < W; ++w) {
    uint32_t m = 0, b = 0;
    for (unsigned bit = 0; bit < 32; ++bit) {
      const uint64_t o = ones[32ull * w + bit];
      const int inv1 = o * (uint64_t)den >= (uint64_t)num * n;
      const int inv0 = (n - o) * (uint64_t)den >= (uint64_t)num * n;
      if (inv1 || inv0) m |= 1u << bit;
      if (inv1) b |= 1u << bit;
    }
    mask[w] = m;
    bitval[w] = b;
  }
  free(ones);
  return IBP_REF_OK;
}

/* ------------------------------------------------------------------ */
/* Compression of one row.                                             */
/* ------------------------------------------------------------------ */
typedef struct {
  uint32_t* words;
  uint64_t pos; /* next stream bit */
} bit_writer;

static void put_bit(bit_writer* bw, int v) {
  if (v) bw->words[bw->pos / 32] |= 1u << (bw->pos % 32);
  bw->pos += 1;
}

/* Number of bits a row's stream needs, given its participation vector. */
static uint64_t stream_bits(const int* p, const uint32_t* mask, uint32_t W, uint32_t wpc,
                            uint32_t nch) {
  uint64_t bits = nch;
  for (uint32_t k = 0; k < nch; ++k)
    for (uint32_t w = chunk_first(k, wpc); w < chunk_end(k, wpc, W); ++w)
      bits += p[k] ? (32u - count_ones(mask[w])) : 32u;
  return bits;
}

/*
 * Compress one row of R bytes.  `out` must hold R bytes.  Returns the number
 * of stored bytes (4*stored_words, or R for a raw row); *is_raw gets the raw
 * bitmap bit; *bits_out (optional) the stream length in bits before the raw
 * decision.  Returns 0 on bad geometry.
 */
uint32_t ibp_ref_compress_row(const uint8_t* row, uint32_t R, uint32_t C,
                              const uint32_t* mask, const uint32_t* bitval,
                              uint8_t* out, int* is_raw, uint64_t* bits_out) {
  uint32_t W, wpc, nch;
  if (geometry(R, C, &W, &wpc, &nch) != IBP_REF_OK) return 0;
  int* p = (int*)calloc(nch, sizeof(int));
  uint32_t* words = (uint32_t*)calloc((size_t)W + 2, sizeof(uint32_t));
  /* participation bits */
  for (uint32_t k = 0; k < nch; ++k) {
    uint32_t keep = 0, all_match = 1;
    for (uint32_t w = chunk_first(k, wpc); w < chunk_end(k, wpc, W); ++w) {
      const uint32_t x = load_le32(row + 4 * w);
      keep += 32u - count_ones(mask[w]);
      for (unsigned b = 0; b < 32; ++b)
        if (bit_of(mask[w], b) && bit_of(x, b) != bit_of(bitval[w], b)) all_match = 0;
    }
    const uint32_t full = 32u * (chunk_end(k, wpc, W) - chunk_first(k, wpc));
    p[k] = all_match && keep < full;
  }
  const uint64_t bits = stream_bits(p, mask, W, wpc, nch);
  if (bits_out) *bits_out = bits;
  const uint64_t stored_words = (bits + 31) / 32;
  uint32_t stored;
  if (4 * stored_words >= R) {
    memcpy(out, row, R);
    *is_raw = 1;
    stored = R;
  } else {
    bit_writer bw = {words, 0};
    for (uint32_t k = 0; k < nch; ++k) put_bit(&bw, p[k]);
    for (uint32_t k = 0; k < nch; ++k)
      for (uint32_t w = chunk_first(k, wpc); w < chunk_end(k, wpc, W); ++w) {
        const uint32_t x = load_le32(row + 4 * w);
        for (unsigned b = 0; b < 32; ++b)
          if (!p[k] || !bit_of(mask[w], b)) put_bit(&bw, bit_of(x, b));
      }
    for (uint64_t i = 0; i < stored_words; ++i) store_le32(out + 4 * i, words[i]);
    *is_raw = 0;
    stored = (uint32_t)(4 * stored_words);
  }
  free(p);
  free(words);
  return stored;
}

/* ------------------------------------------------------------------ */
/* Decompression of one row.                                           */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint8_t* bytes;
  uint64_t avail_bits; /* bits available in the stored stream */
  uint64_t pos;
  int overrun;
} bit_reader;

static int get_bit(bit_reader* br) {
  if (br->pos >= br->avail_bits) {
    br->overrun = 1;
    return 0;
  }
  const uint32_t word = load_le32(br->bytes + 4 * (br->pos / 32));
  const int v = bit_of(word, (unsigned)(br->pos % 32));
  br->pos += 1;
  return v;
}

/*
 * Decompress one stored row into `out` (R bytes).  `stored` holds
 * `stored_bytes` bytes (a multiple of 4).  A raw row is copied.  A compressed
 * row whose stream runs past `stored_bytes`, or which claims R bytes or more,
 * is corrupt: `out` is zero-filled and IBP_REF_ECORRUPT returned.
 */
int ibp_ref_decompress_row(const uint8_t* stored, uint32_t stored_bytes, int is_raw, uint32_t R,
                           uint32_t C, const uint32_t* mask, const uint32_t* bitval,
                           uint8_t* out) {
  uint32_t W, wpc, nch;
  if (geometry(R, C, &W, &wpc, &nch) != IBP_REF_OK) return IBP_REF_EINVAL;
  if (is_raw) {
    if (stored_bytes < R) {
      memset(out, 0, R);
      return IBP_REF_ECORRUPT;
    }
    memcpy(out, stored, R);
    return IBP_REF_OK;
  }
  bit_reader br = {stored, 8ull * (stored_bytes & ~3u), 0, 0};
  int* p = (int*)calloc(nch, sizeof(int));
  for (uint32_t k = 0; k < nch; ++k) p[k] = get_bit(&br);
  const uint64_t bits = stream_bits(p, mask, W, wpc, nch);
  int status = IBP_REF_OK;
  if (4 * ((bits + 31) / 32) >= R) status = IBP_REF_ECORRUPT; /* would have been raw */
  for (uint32_t k = 0; k < nch && status == IBP_REF_OK; ++k)
    for (uint32_t w = chunk_first(k, wpc); w < chunk_end(k, wpc, W); ++w) {
      uint32_t x = 0;
      for (unsigned b = 0; b < 32; ++b) {
        int v;
        if (!p[k] || !bit_of(mask[w], b))
          v = get_bit(&br);
        else
          v = bit_of(bitval[w], b);
        if (v) x |= 1u << b;
      }
      store_le32(out + 4 * w, x);
    }
  if (br.overrun) status = IBP_REF_ECORRUPT;
  if (status != IBP_REF_OK) memset(out, 0, R);
  free(p);
  return status;
}

/* ------------------------------------------------------------------ */
/* Batch helpers: loops over the row functions above, nothing more.    */
/* OpenMP only splits the loop over rows; every row is independent.    */
/* ------------------------------------------------------------------ */

/* Stored bytes of row `id`: the raw bitmap decides raw; a compressed row's
 * length is not known up front, so the reader is given the whole slot. */
static int bitmap_get(const uint32_t* bitmap, uint64_t id) {
  return (int)((bitmap[id / 32] >> (id % 32)) & 1u);
}

/*
 * Compress rows src[i] (i < n, stride src_stride) into slots
 * dst + slot_ids[i]*slot_stride (slot_ids NULL = i).  Sets/clears the raw
 * bitmap bit of each slot and writes its stored byte count to stored_bytes[i]
 * (optional).  Returns the number of rows that failed (0 = all good).
 */
uint64_t ibp_ref_compress_batch(const uint8_t* src, uint64_t src_stride, uint64_t n,
                                const int64_t* slot_ids, uint8_t* dst, uint64_t slot_stride,
                                uint32_t R, uint32_t C, const uint32_t* mask,
                                const uint32_t* bitval, uint32_t* bitmap,
                                uint32_t* stored_bytes, int nthreads) {
  uint64_t bad = 0;
  (void)nthreads;
  int* raw = (int*)calloc(n ? n : 1, sizeof(int));
#ifdef _OPENMP
#pragma omp parallel for schedule(static) reduction(+ : bad) num_threads(nthreads > 0 ? nthreads : 1)
#endif
  for (uint64_t i = 0; i < n; ++i) {
    const uint64_t s = slot_ids ? (uint64_t)slot_ids[i] : i;
    const uint32_t st = ibp_ref_compress_row(src + i * src_stride, R, C, mask, bitval,
                                             dst + s * slot_stride, &raw[i], NULL);
    if (st == 0) bad += 1;
    if (stored_bytes) stored_bytes[i] = st;
  }
  for (uint64_t i = 0; i < n; ++i) {
    const uint64_t s = slot_ids ? (uint64_t)slot_ids[i] : i;
    if (raw[i])
      bitmap[s / 32] |= 1u << (s % 32);
    else
      bitmap[s / 32] &= ~(1u << (s % 32));
  }
  free(raw);
  return bad;
}

/*
 * Decompress rows ids[i] (NULL = i) of a store into out + i*out_stride.
 * Row id's stored bytes start at src + offsets[id] (offsets NULL:
 * src + id*slot_stride) and at most `avail` bytes of it may be read
 * (the slot size, or R for a packed cache).  Returns the number of rows
 * that were corrupt (their output is zero).
 */
uint64_t ibp_ref_decompress_batch(const uint8_t* src, const uint64_t* offsets,
                                  uint64_t slot_stride, uint32_t avail, const uint32_t* bitmap,
                                  const int64_t* ids, uint64_t n, uint32_t R, uint32_t C,
                                  const uint32_t* mask, const uint32_t* bitval, uint8_t* out,
                                  uint64_t out_stride, int nthreads) {
  uint64_t bad = 0;
  (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) reduction(+ : bad) num_threads(nthreads > 0 ? nthreads : 1)
#endif
  for (uint64_t i = 0; i < n; ++i) {
    const uint64_t id = ids ? (uint64_t)ids[i] : i;
    const uint8_t* s = src + (offsets ? offsets[id] : id * slot_stride);
    const int st = ibp_ref_decompress_row(s, avail, bitmap_get(bitmap, id), R, C, mask, bitval,
                                          out + i * out_stride);
    if (st != IBP_REF_OK) bad += 1;
  }
  return bad;
}

/* Threads an OpenMP region would use (1 without OpenMP). */
int ibp_ref_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
