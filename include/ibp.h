/*
 * ibp.h -- C ABI of the GB300 Invariant Bit Packing (IBP) library (libibp.so).
 *
 * IBP is the lossless scheme of "Reducing the GPU Memory Bottleneck with
 * Lossless Compression for ML -- Extended" (Kamath, Krishnamurthy, Canini,
 * Peter).  The gist.science explainer, Technical Summary, Methodology > Core
 * Algorithm defines the three operations exposed here (preprocessing into a
 * Mask/Bitval pair, chunked compression with participation bits, warp-parallel
 * decompression); its System Integration section defines the two storage
 * layouts (a compressed GPU cache, and in-place fixed-size host buffers with a
 * GPU bitmask of compressed tensors).
 *
 * Stream format (the pages fix the idea, not the bits; this library's choice):
 *   - a row of R bytes is R/4 little-endian 32-bit words; Mask and Bitval have
 *     one bit per row bit position;
 *   - chunk k covers words [k*C/4, min((k+1)*C/4, R/4)); nch = ceil(R/C);
 *   - chunk k participates (p_k = 1) iff every word w in it satisfies
 *     (x_w & Mask_w) == Bitval_w and the chunk has at least one invariant bit;
 *   - the stream is LSB-first 32-bit words: nch participation bits, then per
 *     chunk the non-Mask bits of each word (p_k = 1) or all its bits (p_k = 0);
 *   - a row whose stream needs 4*ceil(bits/32) >= R bytes is stored raw (its
 *     R bytes unchanged) and its raw-bitmap bit is set.
 *
 * Conventions shared by every call:
 *   - All device work is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  A synchronous return covers argument errors
 *     only.  Data errors found by a kernel (row id out of range, corrupt
 *     stream, misaligned offset) set the store's device status word and the
 *     affected output row is zero-filled; read it with ibp_stream_status.
 *   - Pointers marked "device" may be device memory or pinned, mapped host
 *     memory (cudaHostAlloc / torch pin_memory) -- the kernels read and write
 *     host memory zero-copy over the host link.  The caller owns every buffer
 *     it passes; the store owns its metadata, derived tables, raw bitmap and
 *     status word.
 *   - Limits: R = row_bytes is a multiple of 16 and <= IBP_MAX_ROW_BYTES;
 *     C = chunk_bytes is a multiple of 4; nch <= IBP_MAX_CHUNKS.  Row, slot
 *     and destination base addresses are 16-byte aligned.
 *   - No call traps, asserts or spins without bound on the device.
 */
#ifndef IBP_H_
#define IBP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define IBP_API __attribute__((visibility("default")))
#else
#define IBP_API
#endif

#define IBP_MAX_ROW_BYTES 32768u
#define IBP_MAX_CHUNKS 256u
#define IBP_NOALLOC_MAX_ROW_BYTES 8192u
#define IBP_MAX_TUNE_CANDIDATES 8u
#define IBP_MAX_GROUP_STORES 64u
/* device workspace bytes of the ordered gathers for n ids (or batch*T items) */
#define IBP_ORDER_WORKSPACE_BYTES(n) (20ull * (uint64_t)(n) + 65536ull)
/* device workspace bytes of ibp_project_compress for m rows of R bytes */
#define IBP_PROJECT_WORKSPACE_BYTES(m, R) \
  ((((uint64_t)(m) * ((uint64_t)(R) / 16ull) + 255ull) / 256ull) * 256ull + \
   (uint64_t)(m) * (uint64_t)(R))

typedef enum {
  IBP_OK = 0,
  IBP_EINVAL = 1,   /* bad argument (NULL, size, threshold, geometry) */
  IBP_EALIGN = 2,   /* a pointer, stride or offset is not 16-byte aligned */
  IBP_ERANGE = 3,   /* a row / slot id outside [0, n_rows) */
  IBP_ECORRUPT = 4, /* a stored stream that cannot be a valid IBP stream */
  IBP_ENOMEM = 5,   /* device allocation failed (store creation only) */
  IBP_ECUDA = 6,    /* a CUDA runtime call failed */
  IBP_ETIMEOUT = 7  /* reserved: a bounded device wait gave up */
} ibp_status;

/* Opaque store: geometry, Mask/Bitval, tables derived from them, the raw
 * bitmap of its n_rows slots and a device status word, all in HBM. */
typedef struct ibp_store ibp_store;

/* Opaque group of stores of one geometry, decoded together (see
 * ibp_group_gather_decompress). */
typedef struct ibp_group ibp_group;

/* A cudaStream_t. */
typedef struct CUstream_st* ibp_stream_t;

typedef struct {
  uint32_t row_bytes;   /* R */
  uint32_t chunk_bytes; /* C */
  uint32_t n_chunks;    /* nch = ceil(R / C) */
  uint32_t min_bits;    /* nch + sum of kept bits: shortest possible stream */
  uint64_t n_rows;      /* slots the raw bitmap covers */
  uint64_t slot_bytes;  /* host-store slot stride S (>= R, multiple of 16) */
  uint32_t meta_valid;  /* 1 once a Mask/Bitval has been built or set */
  uint32_t max_runs;    /* most runs of kept bits in one word of ~Mask */
} ibp_store_info;

/* Create a store for rows of `row_bytes` bytes cut into `chunk_bytes`
 * chunks, with a raw bitmap for `n_rows` slots of stride `slot_bytes`
 * (0 = roundup(row_bytes, 128), the 128-byte line the host link moves).
 * Allocates device memory; *out receives the store.  Mask and Bitval start
 * as all-zero (every row would be stored raw).  Synchronous.
 * Errors: IBP_EINVAL (geometry outside the limits), IBP_EALIGN (slot_bytes
 * not a multiple of 16 or < row_bytes), IBP_ENOMEM, IBP_ECUDA. */
IBP_API ibp_status ibp_store_create(ibp_store** out, uint32_t row_bytes, uint32_t chunk_bytes,
                            uint64_t n_rows, uint64_t slot_bytes);

/* Free a store and its device memory (synchronises the device). NULL is a no-op. */
IBP_API ibp_status ibp_store_destroy(ibp_store* store);

/* Fill *info (host struct).  Synchronous: waits for the last derive kernel. */
IBP_API ibp_status ibp_store_get_info(const ibp_store* store, ibp_store_info* info);

/* Preprocessing (Core Algorithm > Preprocessing; the review's sampling
 * experiment: 1/5/10 % samples): count, for every row bit position j, the
 * ones over the analysed rows -- rows[sample_ids[i]] for i < n, or rows[0..n)
 * when sample_ids is NULL -- and mark j invariant when
 * ones*den >= num*n (Bitval bit 1) or (n-ones)*den >= num*n (Bitval bit 0),
 * i.e. threshold T = num/den with 1/2 < T <= 1.  Then derives the store's
 * decode tables.
 *   rows        device/host-mapped, row r at rows + r*row_stride (R bytes)
 *   row_stride  bytes, multiple of 16
 *   sample_ids  device int64[n] or NULL; ids must lie in [0, 2^40)
 *   n           analysed rows, 1 <= n < 2^32
 * Errors: IBP_EINVAL (n, threshold), IBP_EALIGN, IBP_ECUDA. */
IBP_API ibp_status ibp_build_meta(ibp_store* store, const void* rows, uint64_t row_stride,
                          const int64_t* sample_ids, uint64_t n, uint32_t thr_num,
                          uint32_t thr_den, ibp_stream_t stream);

/* Chunk-aware preprocessing.  Core Algorithm > Preprocessing leaves the
 * threshold T a free parameter; this builder picks it from the sample itself:
 * for each candidate T_c = thr_num[c]/thr_den[c] (host arrays, n_thr <=
 * IBP_MAX_TUNE_CANDIDATES, each 1/2 < T_c <= 1) it builds the Mask/Bitval
 * exactly as ibp_build_meta would, then prices it by the bytes the sampled
 * rows would be stored in (participation per chunk, stream bits, raw
 * fallback), and installs the cheapest (the first on ties).  A Mask bit that
 * makes chunks fall back to raw costs more than it saves, so this drops such
 * bits -- e.g. at T = 0.95 a sparse feature matrix keeps its rare non-zero
 * bits in the Mask and most rows go raw, while T = 0.999 packs every row.
 * Everything runs on the device, asynchronously on `stream`.
 *   chosen_out  optional device uint32: index of the installed candidate
 *   sizes_out   optional device uint64[n_thr]: the sample's stored bytes per candidate
 * Other arguments and errors as ibp_build_meta. */
IBP_API ibp_status ibp_build_meta_tuned(ibp_store* store, const void* rows, uint64_t row_stride,
                                        const int64_t* sample_ids, uint64_t n,
                                        const uint32_t* thr_num, const uint32_t* thr_den,
                                        uint32_t n_thr, uint32_t* chosen_out, uint64_t* sizes_out,
                                        ibp_stream_t stream);

/* Allocation-free builder.  The paper has no counterpart: this entry point
 * exists for callers that cannot allocate device memory when they build a
 * Mask/Bitval -- code inside another framework's memory pool, whose allocator
 * must own every device allocation, or a latency-sensitive loop where
 * cudaMalloc's implicit device synchronisation would stall other streams.
 * It computes exactly what ibp_build_meta computes (same arguments and
 * threshold rule) but needs no store and calls no allocating routine: the
 * per-bit ones counters live in a fixed 256 KiB array of device memory that
 * the library holds on every GPU that loads it, until the process exits.
 *   rows, row_stride, sample_ids, n, thr_num, thr_den  as for ibp_build_meta
 *   row_bytes    R, a multiple of 16, at most IBP_NOALLOC_MAX_ROW_BYTES
 *                (larger rows are rejected with IBP_EINVAL)
 *   mask_out, bitval_out  device uint32[R/4] each (4-byte aligned), written
 *                by the call; sample_ids, when given, is 8-byte aligned
 * Each call outside a stream capture looks up the array's device address
 * with the current device (after a cudaDeviceReset, or in another context of
 * that device, the array lives elsewhere); a call being captured uses the
 * address the last uncaptured call on that device saw, so make one call on a
 * device before capturing any (a capture with none before it returns
 * IBP_EINVAL).  Every call clears and reuses the same array, so calls whose
 * work overlaps on the GPU (other streams, other host threads) race and give
 * wrong results: serialise them.  Errors: IBP_EINVAL, IBP_EALIGN (rows,
 * row_stride, the outputs or sample_ids misaligned), IBP_ECUDA. */
IBP_API ibp_status ibp_build_meta_noalloc(const void* rows, uint64_t row_stride,
                                          uint32_t row_bytes, const int64_t* sample_ids,
                                          uint64_t n, uint32_t thr_num, uint32_t thr_den,
                                          uint32_t* mask_out, uint32_t* bitval_out,
                                          ibp_stream_t stream);

/* Compression (Core Algorithm > Compression; System Integration: in-place
 * compression into fixed-size buffers, GPU bitmask of compressed tensors):
 * compress row i (src_rows + i*src_stride, i < n) into slot slot_ids[i]
 * (NULL: slot i) at dst_slots + slot*slot_bytes: the stored bytes go to the
 * slot start (16-byte granules; the slot tail is not defined), and the slot's
 * raw-bitmap bit is set or cleared.  stored_bytes_out (optional, device
 * uint32[n]) receives each row's stored size (R for a raw row).  dst_slots may
 * be pinned host memory (zero-copy writes over the host link).  Rows whose
 * slot ids collide race.  Errors: IBP_EINVAL, IBP_EALIGN, IBP_ECUDA;
 * a slot id out of range sets IBP_ERANGE in the status word. */
IBP_API ibp_status ibp_compress(ibp_store* store, void* dst_slots, const void* src_rows,
                        uint64_t src_stride, const int64_t* slot_ids, uint64_t n,
                        uint32_t* stored_bytes_out, ibp_stream_t stream);

/* Decompression of rows 0..n-1 (Core Algorithm > Decompression):
 * row i's stored bytes start at src + offsets[i] (a packed HBM cache; offsets
 * device uint64[n], multiples of 16) or, with offsets NULL, at
 * src + i*slot_bytes (a slot store).  dst receives n rows of R bytes,
 * contiguous.  A valid stream is read only within its own stored bytes
 * (rounded up to 16); a corrupt one is detected after reading at most R bytes
 * from its start (slot stores: within the slot), so a packed cache that may
 * hold corrupt data should keep R readable bytes after its last row.  With
 * offsets in GPU memory (src 16-byte aligned), where the starts of 32
 * consecutive rows increase and each lies at most R bytes before the next
 * (a cache written by ibp_pack), the bytes from each row's start to the
 * next row's start are read: the tile's bytes in one bulk copy.
 * Errors: IBP_EINVAL, IBP_EALIGN, IBP_ECUDA; corrupt streams and misaligned
 * offsets set the status word.  Calls on one store from several host threads
 * are safe for decompression; building or setting the Mask/Bitval or the
 * bitmap while other calls use the store is not.  The decompression and
 * compression calls may be captured into a CUDA graph once the store's
 * properties have reached the host (after any such call that follows the
 * Mask/Bitval build and a synchronisation of its stream; earlier captures
 * run the slower forms that read them on the device); the builder calls may
 * not be captured.  A captured call keeps the store properties of the
 * Mask/Bitval current at capture time: replayed after the Mask/Bitval was
 * rebuilt or set again, it finds a newer generation of the store on the
 * device, sets IBP_EINVAL in the status word and zero-fills its output rows
 * (decompression) or writes nothing (compression).  Capture again after every
 * Mask/Bitval change. */
IBP_API ibp_status ibp_decompress(const ibp_store* store, void* dst, const void* src,
                          const uint64_t* offsets, uint64_t n, ibp_stream_t stream);

/* Gather-decompression (the hot path): row i of dst (R bytes, contiguous) is
 * the decompressed row ids[i] of the store, read from host_or_dev_src +
 * offsets[id] (offsets may be NULL: + id*slot_bytes).  ids: device int64[n].
 * With a pinned host source every stored byte crosses the host link inside
 * the kernel (GPU-initiated zero-copy reads, 16-byte vectors, 128-byte lines).
 * Errors: as ibp_decompress; an id outside [0, n_rows) sets IBP_ERANGE. */
IBP_API ibp_status ibp_gather_decompress(const ibp_store* store, void* dst, const void* host_or_dev_src,
                                 const uint64_t* offsets, const int64_t* ids, uint64_t n,
                                 ibp_stream_t stream);

/* As ibp_gather_decompress, with row i written to dst + i*dst_stride_bytes
 * (dst_stride_bytes >= R, multiple of 16): e.g. one table's column of a
 * [batch, tables, dim] embedding output. */
IBP_API ibp_status ibp_gather_decompress_strided(const ibp_store* store, void* dst,
                                         uint64_t dst_stride_bytes,
                                         const void* host_or_dev_src, const uint64_t* offsets,
                                         const int64_t* ids, uint64_t n, ibp_stream_t stream);

/* A group of n stores (1 <= n <= IBP_MAX_GROUP_STORES) that share row and
 * chunk size, with the slot storage srcs[t] of each (host-mapped or device,
 * 16-byte aligned), for fused gathers: one launch serves a batch of lookups
 * into every store, e.g. the per-table lookups of a DLRM batch (the review's
 * DLRM embedding-lookup integration).  Rows must be <= 2 KB with chunks a
 * multiple of 16 bytes, slots <= 64 KB.  Waits for the stores' pending
 * Mask/Bitval builds and takes each store's properties and its length table
 * (ibp_store_set_lengths) as they are now: a store whose Mask/Bitval changes
 * later needs a new group (until then its lookups set IBP_EINVAL in its
 * status word and are zero-filled), and so does one whose length table is
 * attached or detached later.  Allocates device memory.  Errors: IBP_EINVAL,
 * IBP_EALIGN, IBP_ENOMEM, IBP_ECUDA. */
IBP_API ibp_status ibp_group_create(ibp_group** out, ibp_store* const* stores,
                                    const void* const* srcs, uint32_t n);

/* Free a group (synchronises the device; the stores are not touched). */
IBP_API ibp_status ibp_group_destroy(ibp_group* group);

/* Fused gather-decompression over a group of T stores: ids is a device int64
 * [batch, T] array; item (b, t) is the decompressed row ids[b*T + t] of store
 * t and lands at dst + b*dst_row_stride + t*R (dst_row_stride >= T*R,
 * multiple of 16), e.g. a dense [batch, T, dim] embedding output.  Data
 * errors set the status word of the store concerned.  Errors: IBP_EINVAL,
 * IBP_EALIGN, IBP_ECUDA. */
IBP_API ibp_status ibp_group_gather_decompress(const ibp_group* group, void* dst,
                                               uint64_t dst_row_stride, const int64_t* ids,
                                               uint64_t batch, ibp_stream_t stream);

/* As ibp_group_gather_decompress, in address order (see
 * ibp_gather_decompress_ordered): the batch*T items are bucketed by store
 * and by region within it, each bucket of up to 2048 items is sorted by row
 * id, and the list is decoded in contiguous shares of equal cost (a lookup
 * that fetches a row counts as four that repeat the row before it), each
 * item to its own place in dst.  Repeated lookups of a row (Zipf batches)
 * next to each other are fetched and decoded once: the repeats are stored
 * from the decoded copy.  For groups whose slots together exceed the GPU's
 * reach into host memory (DLRM tables of 1-2 KB rows: 26-53 GB), and for
 * batches that repeat rows.
 *   workspace  device memory of IBP_ORDER_WORKSPACE_BYTES(batch*T) bytes,
 *              16-byte aligned
 * Errors: as ibp_group_gather_decompress; IBP_EINVAL for a missing or short
 * workspace or batch*T above 2^32 - 1, IBP_EALIGN for a misaligned one. */
IBP_API ibp_status ibp_group_gather_decompress_ordered(const ibp_group* group, void* dst,
                                                       uint64_t dst_row_stride,
                                                       const int64_t* ids, uint64_t batch,
                                                       void* workspace, uint64_t workspace_bytes,
                                                       ibp_stream_t stream);

/* ibp_group_gather_decompress_ordered in two calls, so that a batch's plan
 * (its bucketing, grouping and warp shares: a chain of short latency-bound
 * launches) runs ahead, e.g. on a second stream while the previous batch is
 * gathered (a DLRM loop knows its next batch's ids).  The output equals
 * ibp_group_gather_decompress_ordered's.
 *
 * ibp_group_order_plan writes the plan of ids [batch, T] into workspace
 * (IBP_ORDER_WORKSPACE_BYTES(batch*T) bytes, 16-byte aligned), including a
 * stamp of batch*T and the warp shares.  ibp_group_gather_decompress_planned
 * then gathers ids (the same device array, unchanged since the plan) into dst
 * as the ordered call would, with as many CTAs per SM as leave room for one
 * CTA of the plan's grouping kernel, so that another stream's plan runs
 * beside it.  The caller orders the two calls (same stream,
 * or an event) and keeps one workspace per batch in flight: a plan must not
 * overwrite a workspace a gather still reads.  A planned gather whose
 * workspace holds no plan for batch*T items writes nothing and sets
 * IBP_EINVAL in the status word of the group's first store; a plan made for
 * other ids of the same size still gives the right rows, in a worse order.
 * Like the group's other calls, both may be captured into a CUDA graph once
 * an uncaptured pair has run on the device (it sets the kernels' shared-memory
 * limits and reads their resources).
 * Errors: as ibp_group_gather_decompress_ordered. */
IBP_API ibp_status ibp_group_order_plan(const ibp_group* group, const int64_t* ids,
                                        uint64_t batch, void* workspace,
                                        uint64_t workspace_bytes, ibp_stream_t stream);
IBP_API ibp_status ibp_group_gather_decompress_planned(const ibp_group* group, void* dst,
                                                       uint64_t dst_row_stride,
                                                       const int64_t* ids, uint64_t batch,
                                                       const void* workspace,
                                                       uint64_t workspace_bytes,
                                                       ibp_stream_t stream);

/* Gather-decompression into a layout that splits each row by chunks (the
 * KV-cache fetch of System Integration, decompressed straight into the
 * attention layout): output row i = g*group_rows + r puts its chunk k (C
 * bytes; the last chunk of a row may be shorter) at
 *   dst + g*group_stride + r*row_stride + k*chunk_stride.
 * KV rows of one token (H heads x D fp16, chunk = one head), gathered for B
 * sequences of T tokens each in order, land in a [B, H, T, D] tensor with
 * group_rows = T, group_stride = H*T*D*2, row_stride = D*2,
 * chunk_stride = T*D*2.  The caller keeps the placements disjoint.  Needs
 * C % 16 == 0 and R <= 8192 (IBP_EINVAL otherwise); the three strides are
 * multiples of 16 (IBP_EALIGN); chunk_stride and group_rows are nonzero.
 * Other errors: as ibp_gather_decompress. */
IBP_API ibp_status ibp_gather_decompress_split(const ibp_store* store, void* dst,
                                               uint64_t group_rows, uint64_t group_stride,
                                               uint64_t row_stride, uint64_t chunk_stride,
                                               const void* host_or_dev_src,
                                               const uint64_t* offsets, const int64_t* ids,
                                               uint64_t n, ibp_stream_t stream);

/* Attach (or, with NULL, detach) a table of each slot's stored bytes: device
 * uint32[n_rows], as ibp_compress writes to stored_bytes_out, owned by the
 * caller and kept current by it.  With the table a decompression fetches each
 * row's whole stream at once; without it the first fetch is the shortest
 * stream any compressed row can have and rows whose raw chunks made theirs
 * longer need a second round trip (over the host link, a second wait).  The
 * pages keep only the raw bitmap on the GPU; the table is 4 bytes per row of
 * HBM.  A wrong entry costs time, not bytes: fetches are clamped to
 * [shortest stream, R] and the stream's own header decides what is decoded
 * (a packed cache then needs R readable bytes after each row, as for corrupt
 * streams).  Not for use while other calls run on the store.
 * Errors: IBP_EINVAL (NULL store). */
IBP_API ibp_status ibp_store_set_lengths(ibp_store* store, const uint32_t* lengths);

/* Gather-decompression in address order, for stores larger than the GPU's
 * reach into host memory.  The pages have no counterpart: it is the gather of
 * System Integration (GPU-initiated zero-copy reads of compressed tensors),
 * scheduled for this GPU's address translation.  As
 * ibp_gather_decompress_strided, but the ids are
 * first bucketed by the region of the store they address (1024 regions, a
 * counting sort in the workspace) and the rows decoded region by region, each
 * written to its own output row.  A GPU reads pinned host memory through
 * address translation whose reach is limited: measured on GB300, random
 * 1 KB gathers over 26-52 GB of host slots ran at 22-45 GB/s and the same
 * gathers in address order at 124-210 GB/s.  No difference in the output;
 * the bucketing costs three small kernels.
 *   workspace  device memory of IBP_ORDER_WORKSPACE_BYTES(n) bytes, 16-byte
 *              aligned, used during the call (stream-ordered)
 * Errors: as ibp_gather_decompress_strided; IBP_EINVAL for a missing or
 * short workspace, IBP_EALIGN for a misaligned one. */
IBP_API ibp_status ibp_gather_decompress_ordered(const ibp_store* store, void* dst,
                                                 uint64_t dst_stride_bytes,
                                                 const void* host_or_dev_src,
                                                 const uint64_t* offsets, const int64_t* ids,
                                                 uint64_t n, void* workspace,
                                                 uint64_t workspace_bytes, ibp_stream_t stream);

/* Gather-decompression through a compressed HBM cache in front of the host
 * store (System Integration: cache compression and PCIe-transfer compression
 * together): row i of dst (at dst + i*dst_stride_bytes) is the decompressed
 * row ids[i]; if cache_map[id] >= 0 its stored bytes are read from the HBM
 * cache slot cache_src + cache_map[id]*slot_bytes, otherwise from
 * host_src + id*slot_bytes over the host link -- in one launch.  The cache
 * holds copies of the store's slots (same stride, same raw bitmap).
 *   cache_slots  slots in the cache; a map entry >= cache_slots sets IBP_ERANGE
 *                and zeroes the row instead of reading past the cache
 *   cache_map  device int64[n_rows]: cache slot of each row, -1 if not cached
 * Errors: as ibp_gather_decompress_strided. */
IBP_API ibp_status ibp_gather_decompress_cached(const ibp_store* store, void* dst,
                                                uint64_t dst_stride_bytes, const void* host_src,
                                                const void* cache_src, uint64_t cache_slots,
                                                const int64_t* cache_map,
                                                const int64_t* ids, uint64_t n,
                                                ibp_stream_t stream);

/* Build a packed HBM cache (System Integration: compressed GPU software
 * cache) from compressed slots: row i's stored_bytes[i] bytes at
 * src_slots + i*slot_bytes are copied to dst_packed + offsets_out[i], where
 * offsets_out[i] = sum over i' < i of roundup(stored_bytes[i'], 16) and
 * offsets_out[n] is the total.  With dst_packed NULL only the offsets are
 * written (size query).  offsets_out: device uint64[n+1]; stored_bytes:
 * device uint32[n] as written by ibp_compress.  The raw bitmap of the slots
 * applies unchanged to the packed rows.  Errors: IBP_EINVAL, IBP_EALIGN,
 * IBP_ECUDA. */
IBP_API ibp_status ibp_pack(const ibp_store* store, void* dst_packed, uint64_t* offsets_out,
                            const void* src_slots, const uint32_t* stored_bytes, uint64_t n,
                            ibp_stream_t stream);

/* K/V projection with the compressor in its epilogue (the review's LLM
 * paragraph: the K/V of each decode token are compressed on the GPU with the
 * Mask/Bitval built from the prompt's K/V, and offloaded to host memory).
 * Computes Y = X W^T (+ bias) on the tensor cores, fp32 accumulation, and
 * compresses each row of Y into its slot as ibp_compress would: the GEMM's
 * epilogue tests each tile of a row against the Mask/Bitval and gathers its
 * kept bits; a second kernel, launched behind it on the same stream
 * (programmatic dependent launch), places them in each row's stream.
 *   x          device [m, k_dim] 16-bit values, row-major (the tokens' inputs)
 *   k_dim      contraction length, a multiple of 64
 *   w          device [N, k_dim] 16-bit values, row-major (a K or V projection
 *              weight, one output channel per row), N = R / 2
 *   bias       NULL or device [N] values of the same type (16-byte aligned)
 *   dtype      0: fp16 inputs, weights, bias and output; 1: bf16
 *   y          device [m, N] output (R bytes per row): the projection itself,
 *              rounded to the 16-bit type; the compressed rows are exactly
 *              ibp_compress applied to these rows
 *   dst_slots, slot_ids, stored_bytes_out  as for ibp_compress (row r of Y
 *              goes to slot slot_ids[r], or r when slot_ids is NULL)
 *   workspace  device memory of IBP_PROJECT_WORKSPACE_BYTES(m, R) bytes,
 *              16-byte aligned, used during the call (stream-ordered)
 * The store's chunks must be 256 bytes (one head of 128 16-bit values) and R
 * a multiple of 256.  Reads the store's current Mask/Bitval on the device (no
 * store properties are fixed on the host).  Errors: IBP_EINVAL (geometry,
 * dtype, k_dim, workspace, m above 65535 * 128), IBP_EALIGN, IBP_ERANGE,
 * IBP_ECUDA; a slot id out of range sets IBP_ERANGE in the status word (that
 * row's slot is not written), and a device wait that gave up sets
 * IBP_ETIMEOUT.
 * The call may be captured into a CUDA graph after one uncaptured call of the
 * same shape on the device (it sets the kernels' shared-memory limits once);
 * a replay reads x, w, bias and the store's tables at the addresses given at
 * capture. */
IBP_API ibp_status ibp_project_compress(ibp_store* store, const void* x, uint64_t m,
                                        uint64_t k_dim, const void* w, const void* bias,
                                        uint32_t dtype, void* y, void* dst_slots,
                                        const int64_t* slot_ids, uint32_t* stored_bytes_out,
                                        void* workspace, uint64_t workspace_bytes,
                                        ibp_stream_t stream);

/* Copy the store's Mask and Bitval (R/4 words each) to host arrays.  Synchronous. */
IBP_API ibp_status ibp_meta_get(const ibp_store* store, uint32_t* mask_host, uint32_t* bitval_host);

/* Install a Mask/Bitval from host arrays (R/4 words each; Bitval bits outside
 * the Mask must be zero, else IBP_EINVAL) and derive the decode tables.  Synchronous. */
IBP_API ibp_status ibp_meta_set(ibp_store* store, const uint32_t* mask_host, const uint32_t* bitval_host);

/* Copy the raw bitmap (ceil(n_rows/32) words; bit id%32 of word id/32) to the host.  Synchronous. */
IBP_API ibp_status ibp_bitmap_get(const ibp_store* store, uint32_t* bitmap_host);

/* Install a raw bitmap from the host (e.g. for streams compressed elsewhere).  Synchronous. */
IBP_API ibp_status ibp_bitmap_set(ibp_store* store, const uint32_t* bitmap_host);

/* Synchronise `stream`, then report the store's device status word (IBP_OK
 * or the first data error a kernel recorded) in *out; reset != 0 clears it. */
IBP_API ibp_status ibp_stream_status(const ibp_store* store, ibp_stream_t stream, ibp_status* out,
                             int reset);

/* Aligned zero-copy copy of `bytes` (multiple of 16, 16-byte aligned ends)
 * from src to dst by GPU warps issuing 16-byte loads that cover whole
 * 128-byte lines (the review's "GPU aligned transfer", Figure 5).  Used as the
 * host-link bandwidth probe.  Errors: IBP_EINVAL, IBP_EALIGN, IBP_ECUDA. */
IBP_API ibp_status ibp_link_copy(void* dst, const void* src, uint64_t bytes, ibp_stream_t stream);

/* Uncompressed gather: row i of dst (row_bytes, contiguous) = the row_bytes
 * at src + ids[i]*slot_bytes.  The raw-transfer baseline of the review's
 * Table 1 speedups.  row_bytes and slot_bytes are multiples of 16; a row whose
 * id lies outside [0, n_rows) is zero-filled (no status word: no store). */
IBP_API ibp_status ibp_gather_copy(void* dst, const void* src, uint64_t slot_bytes, uint32_t row_bytes,
                           const int64_t* ids, uint64_t n, uint64_t n_rows,
                           ibp_stream_t stream);

/* CPU-initiated baselines of the review's Figure 5 (transfer methods for
 * small random tensors), for comparison with the GPU-initiated gathers above.
 * Both gather rows ids_host[i] (a HOST int64 array, ids in [0, n_rows)) of
 * row_bytes from src + id*slot_bytes (host memory) into dst (device, row i at
 * dst + i*row_bytes).
 * ibp_gather_copy_dma: "CPU fine-grained" -- one cudaMemcpyAsync per row.
 * ibp_gather_copy_staged: "CPU bulk" -- the host copies the rows into
 * staging_host (pinned, n*row_bytes, 16-byte aligned) and issues one
 * cudaMemcpyAsync; it first synchronises `stream` (the staging buffer may
 * still feed an earlier copy).
 * Errors: IBP_EINVAL, IBP_EALIGN, IBP_ERANGE (checked on the host), IBP_ECUDA. */
IBP_API ibp_status ibp_gather_copy_dma(void* dst, const void* src, uint64_t slot_bytes,
                                       uint32_t row_bytes, const int64_t* ids_host, uint64_t n,
                                       uint64_t n_rows, ibp_stream_t stream);
IBP_API ibp_status ibp_gather_copy_staged(void* dst, const void* src, uint64_t slot_bytes,
                                          uint32_t row_bytes, const int64_t* ids_host, uint64_t n,
                                          uint64_t n_rows, void* staging_host,
                                          ibp_stream_t stream);

/* Static text of a status code. */
IBP_API const char* ibp_status_str(ibp_status s);

#ifdef __cplusplus
}
#endif
#endif /* IBP_H_ */
