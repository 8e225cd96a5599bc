// Internal declarations shared by the IBP kernels and the C-ABI host code.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ibp.h"

namespace ibp {

// Read-only views of a store's metadata and the tables derived from it.
//   mask, bitval  W words each (the Mask / Bitval of the Core Algorithm)
//   nm            ~mask: the positions whose bits are kept in a packed chunk
//   pre           kept bits of the earlier words of the same chunk
//   kr            chunk index (bits 0..15) | word index inside the chunk (16..31)
//   mv            5 x W move masks of the bit-gather network of nm (stage i at i*W)
//   ckeep         nch words: kept bits per chunk
//   scal          [0] min_bits = nch + sum(ckeep), [1] max runs of one word's nm,
//                 [2] meta valid flag, [3] uniform flag (all words share ~Mask
//                 and Bitval, <= 2 runs), [4] run0, [5] run1, [6] s0 | s1 << 8,
//                 [7] Bitval, [8] kept bits per word (of the uniform word),
//                 [9] generation: bumped by every derive (every Mask/Bitval
//                 build or install), so a launch whose store properties were
//                 fixed on the host can tell that they are out of date
struct MetaView {
  const uint32_t* mask;
  const uint32_t* bitval;
  const uint32_t* nm;
  const uint32_t* pre;
  const uint32_t* kr;
  const uint32_t* mv;
  const uint32_t* ckeep;
  const uint32_t* scal;
  uint32_t R, W, wpc, nch;
};

struct DecodeArgs {
  MetaView m;
  const uint4* t2;          // fast-decoder descriptors (two-run form), W entries
  const uint4* t5;          // fast-decoder descriptors (network form), 2W entries
  const uint32_t* gtab;     // fast-decoder group table, W/4 entries
  const uint32_t* bitmap;
  uint32_t* status;
  const uint8_t* src;
  const uint64_t* offsets;  // NULL: slot layout
  uint64_t slot;            // slot stride (slot layout)
  uint64_t avail;           // bytes of a row's storage the decoder may read
  const int64_t* ids;       // NULL: row i
  uint64_t n;
  uint64_t n_rows;
  uint8_t* dst;
  uint64_t dst_stride;
  const int64_t* cache_map;  // NULL, or per row id: its slot in the HBM cache, -1 if none
  const uint8_t* cache_src;  // the HBM cache's slots (stride `slot`)
  uint64_t cache_slots;      // slots in the HBM cache; a map entry beyond it is an error
  // split output (chunk_stride != 0): output row i = g*group_rows + r puts its
  // chunk k at dst + g*group_stride + r*dst_stride + k*chunk_stride
  uint64_t chunk_stride;
  uint64_t group_rows;
  uint64_t group_stride;
  // ordered gather (out_pos != NULL): ids come sorted by address region and
  // row i lands at dst + out_pos[i]*dst_stride; each warp takes a contiguous
  // share of the sorted ids, so each SM reads a narrow address range
  const int64_t* out_pos;
  // NULL, or each row id's stored bytes (in HBM): the first fetch then takes
  // the whole stream, so rows with raw chunks need no second round trip
  const uint32_t* lengths;
  uint32_t host_src;  // src is pinned host memory (sets the launch shape only)
  // test hook of the bounded waits: the tile decoder's producer never
  // releases this tile (~0: none; IBP_DEBUG_WITHHOLD_TILE in the environment)
  uint64_t withhold_tile;
};

struct EncodeArgs {
  MetaView m;
  const uint4* t5;        // per-word network descriptors (k_derive_fast), 2W entries
  const uint32_t* gtab;   // group table: chunk | word in chunk << 16, then chunk starts
  uint32_t* bitmap;
  uint32_t* status;
  const uint8_t* src;
  uint64_t src_stride;
  const int64_t* slot_ids;
  uint64_t n;
  uint64_t n_rows;
  uint8_t* dst;
  uint64_t slot;
  uint32_t* stored_out;
  uint32_t um0, um1, ush, ubv, ukeep;  // uniform store (the k_encode<true> form)
  uint32_t gen;       // store generation the uniform parameters belong to
  uint32_t chunk_lg;  // log2 of the rows a warp takes at a time: 5 (32 rows, one
                      // raw-bitmap word) or 0 (one row; bitmap bits set by atomics)
};

struct CountArgs {
  const uint8_t* rows;
  uint64_t row_stride;
  const int64_t* ids;
  uint64_t n;
  uint32_t W;
  uint32_t* counts;  // 32 * W
};

// Shared-memory layout of one warp in the decode / encode kernels (in words).
struct WarpSmem {
  uint32_t sbuf_words;  // stream (decode) or packed output (encode) buffer
  uint32_t xbuf_words;  // raw row (encode only)
  uint32_t cinfo_words; // per chunk start | p << 31
  uint32_t total_words; // per warp
};

// Store modes of the fast decoder: kModeRuntime reads the store's properties
// from device memory; the others are specialised for a store whose
// properties the host already knows (uniform: every word has the same ~Mask
// and Bitval with <= 2 runs; uniform1: the same with one run; run2: every
// word has <= 2 runs; net5: any Mask).
enum { kModeRuntime = 0, kModeUniform = 1, kModeRun2 = 2, kModeNet5 = 3, kModeUniform1 = 4 };

// Host-side copy of a store's derived properties (valid when `known`).
struct HostProps {
  bool known;
  bool uniform;
  uint32_t gen;  // generation of the derive these properties come from
  uint32_t min_bits, max_runs;
  uint32_t um0, um1, ush, ubv, ukeep;  // uniform word: run masks, s0 | s1 << 8, Bitval, keep
};

// Launch parameters of the fast decoder: shared-memory layout (in words:
// descriptor table and group table per CTA, then per warp a ring of S
// single-row stream buffers and the chunk starts) and the store properties of
// the specialised modes, with the generation they belong to (a launch replayed
// from a CUDA graph after the Mask/Bitval changed sees a newer one on the
// device, reports IBP_EINVAL and zero-fills its rows).
struct FastParams {
  uint32_t table_words;
  uint32_t gtab_words;
  uint32_t sbuf_words;
  uint32_t warp_words;
  uint32_t S;
  uint32_t min_bits;
  uint32_t um0, um1, ush, ubv, ukeep;
  uint32_t gen;
};

// One store of a fused multi-store gather (all stores share R and C).
struct GroupEntry {
  const uint8_t* src;      // the store's slots (host-mapped or HBM)
  const uint32_t* bitmap;  // raw bitmap
  uint32_t* status;        // device status word
  const uint4* tab;        // two-run (t2) or network (t5) descriptors, global memory
  const uint32_t* gtab;    // group table, then the all-packed chunk starts
  const uint32_t* ckeep;   // kept bits per chunk
  uint64_t slot;
  uint64_t n_rows;
  uint32_t mode;           // kModeUniform / kModeUniform1 / kModeRun2 / kModeNet5
  uint32_t min_vec;        // 16-byte vectors of the shortest compressed stream
  uint32_t can_pack;       // some compressed row can exist
  uint32_t um0, um1, ush, ubv, ukeep;  // uniform stores
  const uint32_t* scal;    // the store's scalars: its current generation at scal[9]
  const uint32_t* lengths; // NULL, or each slot's stored bytes (the store's length table)
  uint32_t gen;            // generation the fields above were read at
  uint32_t pad[3];
};
static_assert(sizeof(GroupEntry) % 16 == 0, "group entries are staged as 16-byte vectors");

struct GroupArgs {
  const GroupEntry* entries;
  uint32_t T;               // stores in the group
  uint32_t R, W, wpc, nch;  // shared geometry
  const int64_t* ids;       // [batch, T]: item b*T + t looks up ids[b*T + t] in store t
  uint64_t n_items;         // batch * T
  uint8_t* dst;             // item (b, t) at dst + b*dst_row_stride + t*R
  uint64_t dst_row_stride;
  uint32_t sbuf_words;
  uint32_t warp_words;
  const int64_t* order;     // NULL, or the items in address order (ordered gather)
  const uint32_t* shares;   // NULL, or warp w's items order[shares[w] .. shares[w+1])
  uint32_t host_src;        // some store's slots are pinned host memory (launch shape only)
  // NULL, or the stamp a plan made ahead left in its workspace: {kPlanMagic,
  // n_items, shares}; a gather whose stamp differs writes nothing and sets
  // IBP_EINVAL in store 0's status word
  const uint32_t* plan_stamp;
};
constexpr uint32_t kPlanMagic = 0x49425050u;

// K/V projection with the compressor in its epilogue (ibp_project_compress):
// Y[m, N] = X[m, k_dim] W[N, k_dim]^T (+ bias), 16-bit in and out, in tiles
// of 128 rows x (128 / seg) columns (N = nch * 128: a chunk is 1, 2 or 4
// tiles), then each row of Y compressed into its slot.
struct ProjectArgs {
  const uint32_t* mask;     // the store's Mask, Bitval, ~Mask, move masks, kept bits per chunk
  const uint32_t* bitval;
  const uint32_t* nm;
  const uint32_t* mv;
  const uint32_t* ckeep;
  const uint32_t* pre;      // kept bits of the earlier words of each word's chunk
  uint32_t* bitmap;
  uint32_t* status;
  uint32_t W, nch;          // row words (R / 4) and chunks (R / 256)
  uint32_t bf16;            // 1: bf16 values, 0: fp16
  uint64_t m, k_dim;        // rows (tokens) and the contraction length (multiple of 64)
  const void* bias;         // NULL or [N] values of the output type
  uint8_t* y;               // [m, R bytes]: the projection's output
  uint8_t* dst;             // slots (host-mapped or device)
  uint64_t slot;            // slot stride
  const int64_t* slot_ids;  // NULL: row r -> slot r
  uint64_t n_rows;
  uint32_t* stored_out;     // NULL or [m]
  uint32_t* flags;          // [m, tiles]: every word of the (row, tile) matches the Mask
  uint32_t* staged;         // [m, tiles, 64 / seg] packed kept bits of matching tiles
};

cudaError_t launch_project(const ProjectArgs& a, const void* x, const void* w, int sm_count,
                           cudaStream_t st);

cudaError_t launch_group(const GroupArgs& g, int sm_count, cudaStream_t st);
uint64_t launch_blocks(uint64_t n, uint64_t full, uint64_t warps, uint64_t rpw, bool host,
                       bool ordered);
// Whether p points into pinned host memory (false when unknown).
bool host_pointer(const void* p);
bool fast_geometry(uint32_t R, uint32_t C);

WarpSmem decode_smem(uint32_t W, uint32_t nch);
WarpSmem encode_smem(uint32_t W, uint32_t nch);

// Launchers (return the cudaError_t of the launch).
cudaError_t launch_count_ones(const CountArgs& a, int sm_count, cudaStream_t st);
// Candidate thresholds num[c]/den[c] (host arrays): a Mask per candidate into
// cand, the sample's stored size under each into sizes, the cheapest into
// mask/bitval (counts must already hold the sample's ones counts).
cudaError_t launch_tune(const CountArgs& a, const uint32_t* counts, const uint32_t* num,
                        const uint32_t* den, uint32_t n_c, uint32_t wpc, uint32_t nch,
                        uint32_t* cand, unsigned long long* sizes, uint32_t* mask,
                        uint32_t* bitval, uint32_t* chosen_out, uint64_t* sizes_out,
                        int sm_count, cudaStream_t st);
cudaError_t launch_finish_meta(const uint32_t* counts, uint32_t W, uint64_t n, uint32_t num,
                               uint32_t den, uint32_t* mask, uint32_t* bitval, cudaStream_t st);
cudaError_t launch_derive(uint32_t* mask, uint32_t* bitval, uint32_t* nm, uint32_t* pre,
                          uint32_t* kr, uint32_t* mv, uint32_t* ckeep, uint32_t* scal,
                          uint4* t2, uint4* t5, uint32_t* gtab, uint32_t W, uint32_t wpc,
                          uint32_t nch, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, const HostProps& hp, int sm_count,
                          cudaStream_t st);
// Bucket the ids by address region (a counting sort on id * kOrderBuckets /
// n_rows): ids_out, in bucket order, and pos_out, each id's index in ids.
// hist: kOrderBuckets zeroed counters.
#ifndef IBP_ORDER_BUCKETS
#define IBP_ORDER_BUCKETS 1024u
#endif
constexpr uint32_t kOrderBuckets = IBP_ORDER_BUCKETS;
cudaError_t launch_order_ids(const int64_t* ids, uint64_t n, uint64_t n_rows, int64_t* ids_out,
                             int64_t* pos_out, uint32_t* hist, int sm_count, cudaStream_t st);
// The same for a group's items (b, t): bucket t * (kOrderBuckets / T) plus the
// region of ids[b*T + t] in store t; order_out receives the item indices.
cudaError_t launch_order_items(const GroupEntry* entries, uint32_t T, const int64_t* ids,
                               uint64_t n_items, int64_t* order_out, uint32_t* hist,
                               int sm_count, cudaStream_t st);
// The ordered group gather after launch_order_items: each bucket of g.order
// sorted by row id (repeats of a row side by side), the list cut into warp
// shares of equal cost (an item that fetches a row costs as much as several
// repeats), then the gather.  hist: the bucket ends launch_order_items left;
// wpre: n_items words; cost: kOrderBuckets words; shares: n_items / 32 + 9
// words at least.
cudaError_t launch_group_ordered(GroupArgs g, const uint32_t* hist, uint32_t* wpre,
                                 uint32_t* cost, uint32_t* shares, int sm_count,
                                 cudaStream_t st);
// The two halves of launch_group_ordered, for a plan made ahead of its gather
// (ibp_group_order_plan, ibp_group_gather_decompress_planned):
// group_gather_blocks: the gather's CTAs (at most max_per_sm per SM, 0 = as
// many as fit), 8 warps each, one share per warp; launch_group_plan: the
// grouping and share kernels for nw shares (stamp: NULL, or 3 words where the
// share kernel writes {kPlanMagic, n_items, nw}); launch_group_gather: the
// gather over g.order in g.shares.
uint64_t group_gather_blocks(const GroupArgs& g, int sm_count, uint32_t max_per_sm);
// CTAs per SM of a gather planned ahead: the most that leave room on each SM
// (shared memory, registers, threads) for one CTA of the plan's grouping
// kernel, so that the next batch's plan runs during the gather
uint32_t group_planned_per_sm(const GroupArgs& g);
cudaError_t launch_group_plan(GroupArgs g, const uint32_t* hist, uint32_t* wpre, uint32_t* cost,
                              uint32_t* shares, uint32_t nw, uint32_t* stamp, cudaStream_t st);
cudaError_t launch_group_gather(const GroupArgs& g, uint64_t blocks, cudaStream_t st);
cudaError_t launch_encode(const EncodeArgs& a, const HostProps& hp, int sm_count,
                          cudaStream_t st);
cudaError_t launch_pack(uint8_t* dst, uint64_t* offsets, const uint8_t* src, uint64_t slot,
                        const uint32_t* stored, uint64_t n, int sm_count, cudaStream_t st);
cudaError_t launch_link_copy(uint4* dst, const uint4* src, uint64_t nvec, int sm_count,
                             cudaStream_t st);
cudaError_t launch_gather_copy(uint8_t* dst, const uint8_t* src, uint64_t slot,
                               uint32_t row_bytes, const int64_t* ids, uint64_t n,
                               uint64_t n_rows, int sm_count, cudaStream_t st);

}  // namespace ibp
