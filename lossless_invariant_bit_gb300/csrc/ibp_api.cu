// C-ABI of the IBP library: store objects, argument checks, launches.
// The operations are those of "Reducing the GPU Memory Bottleneck with
// Lossless Compression for ML -- Extended" (gist.science explainer, Technical
// Summary, Methodology > Core Algorithm and System Integration); see ibp.h
// for the contract of each entry point.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <new>

#include "ibp_internal.cuh"

struct ibp_store {
  uint32_t R, C, W, wpc, nch;
  uint64_t n_rows, slot;
  int device;
  int sm_count;
  void* base;  // one device allocation, carved below
  uint32_t *mask, *bitval, *nm, *pre, *kr, *mv, *ckeep, *scal, *counts, *bitmap, *status;
  uint32_t* cand;             // tuned builder: a Mask/Bitval per candidate threshold
  unsigned long long* sizes;  // tuned builder: the sample's stored size per candidate
  uint4 *t2, *t5;  // fast-decoder descriptors
  uint32_t* gtab;
  uint32_t* h_scal;       // pinned host mirror of scal, filled after each derive
  cudaEvent_t props_ev;   // completes when h_scal is current
  std::atomic<int> props_ready{0};  // 1 once props_ev was seen complete (reset by derive)
  const uint32_t* lengths = nullptr;  // caller's stored bytes per slot (device), or NULL
  uint64_t bitmap_words;
  // the last source pointer a decode saw, with bit 0 set when it was pinned
  // host memory (a pointer query costs more host time than a small launch)
  std::atomic<uintptr_t> src_kind{0};
};

struct ibp_group {
  uint32_t T, R, C, W, wpc, nch;
  int device, sm_count;
  uint32_t host_src;  // some store's slots are pinned host memory
  ibp::GroupEntry* entries;  // device copy, one per store
};

namespace ibp {

bool host_pointer(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

}  // namespace ibp

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether `src` is pinned host memory, remembered per store for the last
// source seen.  Only the launch shape depends on it.  A stream being captured
// makes no pointer query: an unseen source counts as device memory there.
bool source_is_host(const ibp_store* s, const void* src, cudaStream_t st) {
  const uintptr_t v = s->src_kind.load(std::memory_order_relaxed);
  if ((v & ~(uintptr_t)1) == reinterpret_cast<uintptr_t>(src)) return (v & 1u) != 0;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return false;
  }
  const bool host = ibp::host_pointer(src);
  const_cast<ibp_store*>(s)->src_kind.store(reinterpret_cast<uintptr_t>(src) | (host ? 1u : 0u),
                                            std::memory_order_relaxed);
  return host;
}

inline ibp_status cu(cudaError_t e) { return e == cudaSuccess ? IBP_OK : IBP_ECUDA; }

// Test hook of the bounded waits (read once): IBP_DEBUG_WITHHOLD_TILE=k makes
// the tile decoder's producer withhold tile k, so the warps waiting for it give
// up after ~2 s and the call reports IBP_ETIMEOUT.  Unset: no tile withheld.
uint64_t withheld_tile() {
  static const uint64_t tile = [] {
    const char* v = std::getenv("IBP_DEBUG_WITHHOLD_TILE");
    if (!v || !*v) return ~0ull;
    char* end = nullptr;
    const unsigned long long t = std::strtoull(v, &end, 10);
    return (end && *end == '\0') ? (uint64_t)t : ~0ull;
  }();
  return tile;
}

// Calls on a store run on the device it was created on.
ibp_status on_device(const ibp_store* s) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return IBP_ECUDA;
  return d == s->device ? IBP_OK : IBP_EINVAL;
}

ibp::MetaView view(const ibp_store* s) {
  ibp::MetaView m;
  m.mask = s->mask;
  m.bitval = s->bitval;
  m.nm = s->nm;
  m.pre = s->pre;
  m.kr = s->kr;
  m.mv = s->mv;
  m.ckeep = s->ckeep;
  m.scal = s->scal;
  m.R = s->R;
  m.W = s->W;
  m.wpc = s->wpc;
  m.nch = s->nch;
  return m;
}

// Derive the decode tables, then mirror the store's properties to the host
// (asynchronously: a decode launched before the copy lands uses the kernel
// that reads them on the device).
ibp_status derive(ibp_store* s, cudaStream_t st) {
  ibp_status e = cu(ibp::launch_derive(s->mask, s->bitval, s->nm, s->pre, s->kr, s->mv,
                                       s->ckeep, s->scal, s->t2, s->t5, s->gtab, s->W, s->wpc,
                                       s->nch, st));
  if (e != IBP_OK) return e;
  s->props_ready.store(0);
  e = cu(cudaMemcpyAsync(s->h_scal, s->scal, 16 * sizeof(uint32_t), cudaMemcpyDeviceToHost, st));
  if (e != IBP_OK) return e;
  return cu(cudaEventRecord(s->props_ev, st));
}

// The store's properties as the host knows them.  Once the mirror has been
// seen current no query is made, so calls captured into a CUDA graph (where
// querying an event is not allowed) use it; a capture before that runs the
// decoders' runtime forms.
ibp::HostProps host_props(const ibp_store* s, cudaStream_t st) {
  ibp::HostProps hp = {};
  if (s->props_ready.load() != 1) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return hp;
    }
    if (cudaEventQuery(s->props_ev) != cudaSuccess) {
      cudaGetLastError();  // cudaErrorNotReady: not known yet
      return hp;
    }
    const_cast<ibp_store*>(s)->props_ready.store(1);
  }
  const volatile uint32_t* h = s->h_scal;
  hp.known = true;
  hp.gen = h[9];
  hp.min_bits = h[0];
  hp.max_runs = h[1];
  hp.uniform = h[3] != 0;
  hp.um0 = h[4];
  hp.um1 = h[5];
  hp.ush = h[6];
  hp.ubv = h[7];
  hp.ukeep = h[8];
  return hp;
}

// Where output rows go when each row is split by chunks (chunk_stride != 0).
struct SplitOut {
  uint64_t chunk_stride = 0, group_rows = 1, group_stride = 0;
};

ibp_status decode(const ibp_store* s, void* dst, uint64_t dst_stride, const void* src,
                  const uint64_t* offsets, const int64_t* ids, uint64_t n, cudaStream_t st,
                  const int64_t* cache_map = nullptr, const void* cache_src = nullptr,
                  uint64_t cache_slots = 0,
                  SplitOut split = SplitOut(), const int64_t* out_pos = nullptr) {
  if (!s) return IBP_EINVAL;
  if (n == 0) return IBP_OK;
  if (!dst || !src) return IBP_EINVAL;
  if (!aligned16(dst) || !aligned16(src) || (dst_stride & 15u) ||
      (split.chunk_stride == 0 && dst_stride < s->R))
    return IBP_EALIGN;
  if (!ids && n > s->n_rows) return IBP_ERANGE;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  ibp::DecodeArgs a;
  a.m = view(s);
  a.t2 = s->t2;
  a.t5 = s->t5;
  a.gtab = s->gtab;
  a.bitmap = s->bitmap;
  a.status = s->status;
  a.src = static_cast<const uint8_t*>(src);
  a.offsets = offsets;
  a.slot = s->slot;
  a.avail = offsets ? s->R : s->slot;
  a.ids = ids;
  a.n = n;
  a.n_rows = s->n_rows;
  a.dst = static_cast<uint8_t*>(dst);
  a.dst_stride = dst_stride;
  a.cache_map = cache_map;
  a.cache_src = static_cast<const uint8_t*>(cache_src);
  a.cache_slots = cache_slots;
  a.chunk_stride = split.chunk_stride;
  a.group_rows = split.group_rows;
  a.group_stride = split.group_stride;
  a.out_pos = out_pos;
  a.lengths = s->lengths;
  a.host_src = source_is_host(s, src, st) ? 1u : 0u;
  a.withhold_tile = withheld_tile();
  return cu(ibp::launch_decode(a, host_props(s, st), s->sm_count, st));
}


// The gather arguments of a group call (no order, shares or plan stamp).
ibp::GroupArgs group_args(const ibp_group* g, const int64_t* ids, uint64_t batch, void* dst,
                          uint64_t dst_row_stride) {
  ibp::GroupArgs a;
  a.entries = g->entries;
  a.T = g->T;
  a.R = g->R;
  a.W = g->W;
  a.wpc = g->wpc;
  a.nch = g->nch;
  a.ids = ids;
  a.n_items = batch * g->T;
  a.dst = static_cast<uint8_t*>(dst);
  a.dst_row_stride = dst_row_stride;
  a.sbuf_words = ((g->W + 8u) + 3u) & ~3u;
  a.warp_words = 4u * a.sbuf_words + 256u + ((g->nch + 3u) & ~3u) + g->W;
  a.order = nullptr;
  a.shares = nullptr;
  a.host_src = g->host_src;
  a.plan_stamp = nullptr;
  return a;
}

// The ordered gathers' workspace: the item order (8 bytes per item), each
// item's cost prefix within its bucket (4 per item), the warp shares (at most
// n/32 + 9 words), then in the 64 KB tail a plan's stamp (4 words) and the
// bucket counters and the bucket costs (4 bytes per bucket each) at its end.
struct OrderWorkspace {
  int64_t* order;
  uint32_t* wpre;
  uint32_t* shares;
  uint32_t* stamp;
  uint32_t* hist;
  uint32_t* cost;
};

OrderWorkspace order_workspace(void* workspace, uint64_t n_items) {
  static_assert(8ull * ibp::kOrderBuckets + 16ull <= 32768ull,
                "bucket arrays and stamp in the workspace's tail");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  OrderWorkspace w;
  w.order = reinterpret_cast<int64_t*>(ws);
  w.wpre = reinterpret_cast<uint32_t*>(ws + 8ull * n_items);
  w.shares = reinterpret_cast<uint32_t*>(ws + 12ull * n_items);
  w.hist = reinterpret_cast<uint32_t*>(ws + IBP_ORDER_WORKSPACE_BYTES(n_items) -
                                       8ull * ibp::kOrderBuckets);
  w.cost = w.hist + ibp::kOrderBuckets;
  w.stamp = w.hist - 4;
  return w;
}

// Arguments of the ordered group calls, checked on the host.
ibp_status check_ordered(const ibp_group* g, const int64_t* ids, uint64_t n_items,
                         const void* workspace, uint64_t workspace_bytes) {
  if (!ids) return IBP_EINVAL;
  if (n_items > 0xFFFFFFFFull) return IBP_EINVAL;
  if (!workspace || workspace_bytes < IBP_ORDER_WORKSPACE_BYTES(n_items)) return IBP_EINVAL;
  if (!aligned16(workspace)) return IBP_EALIGN;
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return IBP_ECUDA;
  if (d != g->device) return IBP_EINVAL;
  return IBP_OK;
}

}  // namespace

extern "C" {

const char* ibp_status_str(ibp_status s) {
  switch (s) {
    case IBP_OK: return "IBP_OK";
    case IBP_EINVAL: return "IBP_EINVAL: invalid argument";
    case IBP_EALIGN: return "IBP_EALIGN: pointer, stride or offset not 16-byte aligned";
    case IBP_ERANGE: return "IBP_ERANGE: row or slot id out of range";
    case IBP_ECORRUPT: return "IBP_ECORRUPT: stored stream is not a valid IBP stream";
    case IBP_ENOMEM: return "IBP_ENOMEM: device allocation failed";
    case IBP_ECUDA: return "IBP_ECUDA: CUDA runtime error";
    case IBP_ETIMEOUT: return "IBP_ETIMEOUT: bounded device wait gave up";
  }
  return "IBP: unknown status";
}

ibp_status ibp_store_create(ibp_store** out, uint32_t row_bytes, uint32_t chunk_bytes,
                            uint64_t n_rows, uint64_t slot_bytes) {
  if (!out) return IBP_EINVAL;
  *out = nullptr;
  if (row_bytes == 0 || row_bytes > IBP_MAX_ROW_BYTES || (row_bytes & 15u)) return IBP_EINVAL;
  if (chunk_bytes == 0 || (chunk_bytes & 3u) || n_rows == 0) return IBP_EINVAL;
  const uint32_t W = row_bytes / 4, wpc = chunk_bytes / 4;
  const uint32_t nch = (W + wpc - 1) / wpc;
  if (nch > IBP_MAX_CHUNKS) return IBP_EINVAL;
  if (slot_bytes == 0) slot_bytes = ((uint64_t)row_bytes + 127u) & ~(uint64_t)127u;
  if ((slot_bytes & 15u) || slot_bytes < row_bytes) return IBP_EALIGN;
  if (n_rows > (1ull << 40)) return IBP_EINVAL;

  ibp_store* s = new (std::nothrow) ibp_store();
  if (!s) return IBP_ENOMEM;
  s->R = row_bytes;
  s->C = chunk_bytes;
  s->W = W;
  s->wpc = wpc;
  s->nch = nch;
  s->n_rows = n_rows;
  s->slot = slot_bytes;
  s->bitmap_words = (n_rows + 31) / 32;
  if (cudaGetDevice(&s->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&s->sm_count, cudaDevAttrMultiProcessorCount, s->device) !=
          cudaSuccess) {
    delete s;
    return IBP_ECUDA;
  }
  // words: mask, bitval, nm, pre, kr (5W) + mv (5W) + ckeep (nch) + scal (4)
  //        + counts (32W) + status (4) + t2 (4W) + t5 (8W) + gtab (W/4) + bitmap,
  //        each piece 16-byte aligned
  auto r4 = [](uint64_t x) { return (x + 3u) & ~(uint64_t)3u; };
  const uint64_t words = 10ull * r4(W) + r4(nch) + 16 + 32ull * W + 4 + 12ull * W +
                         r4(W / 4) + r4(nch) + 2ull * IBP_MAX_TUNE_CANDIDATES * r4(W) +
                         2ull * IBP_MAX_TUNE_CANDIDATES + r4(s->bitmap_words);
  if (cudaMalloc(&s->base, words * 4) != cudaSuccess) {
    cudaGetLastError();
    delete s;
    return IBP_ENOMEM;
  }
  if (cudaHostAlloc(reinterpret_cast<void**>(&s->h_scal), 16 * sizeof(uint32_t),
                    cudaHostAllocDefault) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->props_ev, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    if (s->h_scal) cudaFreeHost(s->h_scal);
    cudaFree(s->base);
    delete s;
    return IBP_ENOMEM;
  }
  uint32_t* p = static_cast<uint32_t*>(s->base);
  auto take = [&](uint64_t n) {
    uint32_t* q = p;
    p += r4(n);
    return q;
  };
  s->mask = take(W);
  s->bitval = take(W);
  s->nm = take(W);
  s->pre = take(W);
  s->kr = take(W);
  s->mv = take(5ull * W);
  s->ckeep = take(nch);
  s->scal = take(16);
  s->counts = take(32ull * W);
  s->status = take(4);
  s->t2 = reinterpret_cast<uint4*>(take(4ull * W));
  s->t5 = reinterpret_cast<uint4*>(take(8ull * W));
  s->gtab = take(r4(W / 4) + r4(nch));
  s->cand = take(2ull * IBP_MAX_TUNE_CANDIDATES * r4(W));
  s->sizes = reinterpret_cast<unsigned long long*>(take(2ull * IBP_MAX_TUNE_CANDIDATES));
  s->bitmap = take(s->bitmap_words);
  ibp_status e = cu(cudaMemset(s->base, 0, words * 4));
  if (e == IBP_OK) e = derive(s, 0);  // all-zero Mask: tables for "everything raw"
  if (e == IBP_OK) e = cu(cudaDeviceSynchronize());
  // derive() sets the valid flag; a fresh store has no built Mask yet
  uint32_t zero = 0;
  if (e == IBP_OK) e = cu(cudaMemcpy(s->scal + 2, &zero, 4, cudaMemcpyHostToDevice));
  if (e == IBP_OK) s->h_scal[2] = 0;
  if (e != IBP_OK) {
    cudaEventDestroy(s->props_ev);
    cudaFreeHost(s->h_scal);
    cudaFree(s->base);
    delete s;
    return e;
  }
  *out = s;
  return IBP_OK;
}

ibp_status ibp_store_destroy(ibp_store* s) {
  if (!s) return IBP_OK;
  cudaDeviceSynchronize();
  cudaEventDestroy(s->props_ev);
  cudaFreeHost(s->h_scal);
  const cudaError_t e = cudaFree(s->base);
  delete s;
  return cu(e);
}

ibp_status ibp_store_get_info(const ibp_store* s, ibp_store_info* info) {
  if (!s || !info) return IBP_EINVAL;
  uint32_t sc[4];
  if (cudaDeviceSynchronize() != cudaSuccess) return IBP_ECUDA;
  if (cudaMemcpy(sc, s->scal, sizeof sc, cudaMemcpyDeviceToHost) != cudaSuccess) return IBP_ECUDA;
  info->row_bytes = s->R;
  info->chunk_bytes = s->C;
  info->n_chunks = s->nch;
  info->min_bits = sc[0];
  info->max_runs = sc[1];
  info->meta_valid = sc[2];
  info->n_rows = s->n_rows;
  info->slot_bytes = s->slot;
  return IBP_OK;
}

ibp_status ibp_build_meta(ibp_store* s, const void* rows, uint64_t row_stride,
                          const int64_t* sample_ids, uint64_t n, uint32_t thr_num,
                          uint32_t thr_den, ibp_stream_t stream) {
  if (!s || !rows) return IBP_EINVAL;
  if (n == 0 || n >= (1ull << 32)) return IBP_EINVAL;
  if (thr_den == 0 || thr_num > thr_den || 2ull * thr_num <= thr_den) return IBP_EINVAL;
  if (!aligned16(rows) || (row_stride & 15u) || row_stride < s->R) return IBP_EALIGN;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  e = cu(cudaMemsetAsync(s->counts, 0, 32ull * s->W * 4, st));
  if (e != IBP_OK) return e;
  ibp::CountArgs a;
  a.rows = static_cast<const uint8_t*>(rows);
  a.row_stride = row_stride;
  a.ids = sample_ids;
  a.n = n;
  a.W = s->W;
  a.counts = s->counts;
  e = cu(ibp::launch_count_ones(a, s->sm_count, st));
  if (e != IBP_OK) return e;
  e = cu(ibp::launch_finish_meta(s->counts, s->W, n, thr_num, thr_den, s->mask, s->bitval, st));
  if (e != IBP_OK) return e;
  return derive(s, st);
}

ibp_status ibp_build_meta_tuned(ibp_store* s, const void* rows, uint64_t row_stride,
                                const int64_t* sample_ids, uint64_t n, const uint32_t* thr_num,
                                const uint32_t* thr_den, uint32_t n_thr, uint32_t* chosen_out,
                                uint64_t* sizes_out, ibp_stream_t stream) {
  if (!s || !rows || !thr_num || !thr_den) return IBP_EINVAL;
  if (n_thr == 0 || n_thr > IBP_MAX_TUNE_CANDIDATES) return IBP_EINVAL;
  for (uint32_t c = 0; c < n_thr; ++c)
    if (thr_den[c] == 0 || thr_num[c] > thr_den[c] || 2ull * thr_num[c] <= thr_den[c])
      return IBP_EINVAL;
  if (n == 0 || n >= (1ull << 32)) return IBP_EINVAL;
  if (!aligned16(rows) || (row_stride & 15u) || row_stride < s->R) return IBP_EALIGN;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  e = cu(cudaMemsetAsync(s->counts, 0, 32ull * s->W * 4, st));
  if (e != IBP_OK) return e;
  ibp::CountArgs a;
  a.rows = static_cast<const uint8_t*>(rows);
  a.row_stride = row_stride;
  a.ids = sample_ids;
  a.n = n;
  a.W = s->W;
  a.counts = s->counts;
  e = cu(ibp::launch_count_ones(a, s->sm_count, st));
  if (e != IBP_OK) return e;
  e = cu(ibp::launch_tune(a, s->counts, thr_num, thr_den, n_thr, s->wpc, s->nch, s->cand,
                          s->sizes, s->mask, s->bitval, chosen_out, sizes_out, s->sm_count, st));
  if (e != IBP_OK) return e;
  return derive(s, st);
}

ibp_status ibp_compress(ibp_store* s, void* dst_slots, const void* src_rows, uint64_t src_stride,
                        const int64_t* slot_ids, uint64_t n, uint32_t* stored_bytes_out,
                        ibp_stream_t stream) {
  if (!s) return IBP_EINVAL;
  if (n == 0) return IBP_OK;
  if (!dst_slots || !src_rows) return IBP_EINVAL;
  if (!aligned16(dst_slots) || !aligned16(src_rows) || (src_stride & 15u) || src_stride < s->R)
    return IBP_EALIGN;
  if (!slot_ids && n > s->n_rows) return IBP_ERANGE;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  ibp::EncodeArgs a;
  a.m = view(s);
  a.t5 = s->t5;
  a.gtab = s->gtab;
  a.bitmap = s->bitmap;
  a.status = s->status;
  a.src = static_cast<const uint8_t*>(src_rows);
  a.src_stride = src_stride;
  a.slot_ids = slot_ids;
  a.n = n;
  a.n_rows = s->n_rows;
  a.dst = static_cast<uint8_t*>(dst_slots);
  a.slot = s->slot;
  a.stored_out = stored_bytes_out;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return cu(ibp::launch_encode(a, host_props(s, st), s->sm_count, st));
}

ibp_status ibp_decompress(const ibp_store* s, void* dst, const void* src, const uint64_t* offsets,
                          uint64_t n, ibp_stream_t stream) {
  return decode(s, dst, s ? s->R : 0, src, offsets, nullptr, n,
                reinterpret_cast<cudaStream_t>(stream));
}

ibp_status ibp_gather_decompress(const ibp_store* s, void* dst, const void* src,
                                 const uint64_t* offsets, const int64_t* ids, uint64_t n,
                                 ibp_stream_t stream) {
  if (!ids && n) return IBP_EINVAL;
  return decode(s, dst, s ? s->R : 0, src, offsets, ids, n,
                reinterpret_cast<cudaStream_t>(stream));
}

ibp_status ibp_gather_decompress_strided(const ibp_store* s, void* dst, uint64_t dst_stride,
                                         const void* src, const uint64_t* offsets,
                                         const int64_t* ids, uint64_t n, ibp_stream_t stream) {
  if (!ids && n) return IBP_EINVAL;
  return decode(s, dst, dst_stride, src, offsets, ids, n, reinterpret_cast<cudaStream_t>(stream));
}

ibp_status ibp_gather_decompress_split(const ibp_store* s, void* dst, uint64_t group_rows,
                                       uint64_t group_stride, uint64_t row_stride,
                                       uint64_t chunk_stride, const void* src,
                                       const uint64_t* offsets, const int64_t* ids, uint64_t n,
                                       ibp_stream_t stream) {
  if (!s || group_rows == 0 || chunk_stride == 0) return IBP_EINVAL;
  if (!ids && n) return IBP_EINVAL;
  // the fast decoder's geometries: chunks of whole 16-byte groups, rows <= 8 KB
  if (s->C % 16u != 0u || s->R > 8192u) return IBP_EINVAL;
  if ((group_stride | row_stride | chunk_stride) & 15u) return IBP_EALIGN;
  SplitOut sp;
  sp.chunk_stride = chunk_stride;
  sp.group_rows = group_rows;
  sp.group_stride = group_stride;
  return decode(s, dst, row_stride, src, offsets, ids, n, reinterpret_cast<cudaStream_t>(stream),
                nullptr, nullptr, 0, sp);
}

ibp_status ibp_store_set_lengths(ibp_store* s, const uint32_t* lengths) {
  if (!s) return IBP_EINVAL;
  s->lengths = lengths;
  return IBP_OK;
}

ibp_status ibp_gather_decompress_ordered(const ibp_store* s, void* dst, uint64_t dst_stride,
                                         const void* src, const uint64_t* offsets,
                                         const int64_t* ids, uint64_t n, void* workspace,
                                         uint64_t workspace_bytes, ibp_stream_t stream) {
  if (!s) return IBP_EINVAL;
  if (n == 0) return IBP_OK;
  if (!ids || !workspace || workspace_bytes < IBP_ORDER_WORKSPACE_BYTES(n)) return IBP_EINVAL;
  if (!aligned16(workspace)) return IBP_EALIGN;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int64_t* ids_out = static_cast<int64_t*>(workspace);
  int64_t* pos_out = ids_out + n;
  uint32_t* hist = reinterpret_cast<uint32_t*>(pos_out + n);
  e = cu(cudaMemsetAsync(hist, 0, 4ull * ibp::kOrderBuckets, st));
  if (e != IBP_OK) return e;
  e = cu(ibp::launch_order_ids(ids, n, s->n_rows, ids_out, pos_out, hist, s->sm_count, st));
  if (e != IBP_OK) return e;
  return decode(s, dst, dst_stride, src, offsets, ids_out, n, st, nullptr, nullptr, 0, SplitOut(),
                pos_out);
}

ibp_status ibp_gather_decompress_cached(const ibp_store* s, void* dst, uint64_t dst_stride,
                                        const void* host_src, const void* cache_src,
                                        uint64_t cache_slots, const int64_t* cache_map,
                                        const int64_t* ids, uint64_t n, ibp_stream_t stream) {
  if (!ids && n) return IBP_EINVAL;
  if (n && (!cache_map || !cache_src)) return IBP_EINVAL;
  if (cache_src && !aligned16(cache_src)) return IBP_EALIGN;
  return decode(s, dst, dst_stride, host_src, nullptr, ids, n,
                reinterpret_cast<cudaStream_t>(stream), cache_map, cache_src, cache_slots);
}

ibp_status ibp_pack(const ibp_store* s, void* dst_packed, uint64_t* offsets_out,
                    const void* src_slots, const uint32_t* stored_bytes, uint64_t n,
                    ibp_stream_t stream) {
  if (!s || !offsets_out) return IBP_EINVAL;
  if (n && (!src_slots || !stored_bytes)) return IBP_EINVAL;
  if ((dst_packed && !aligned16(dst_packed)) || (src_slots && !aligned16(src_slots)))
    return IBP_EALIGN;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  return cu(ibp::launch_pack(static_cast<uint8_t*>(dst_packed), offsets_out,
                             static_cast<const uint8_t*>(src_slots), s->slot, stored_bytes, n,
                             s->sm_count, reinterpret_cast<cudaStream_t>(stream)));
}

ibp_status ibp_group_create(ibp_group** out, ibp_store* const* stores, const void* const* srcs,
                            uint32_t n) {
  if (!out || !stores || !srcs || n == 0 || n > IBP_MAX_GROUP_STORES) return IBP_EINVAL;
  *out = nullptr;
  const ibp_store* s0 = stores[0];
  if (!s0) return IBP_EINVAL;
  if (!ibp::fast_geometry(s0->R, s0->C)) return IBP_EINVAL;
  ibp::GroupEntry* h = new (std::nothrow) ibp::GroupEntry[n];
  if (!h) return IBP_ENOMEM;
  ibp_status e = on_device(s0);
  for (uint32_t t = 0; t < n && e == IBP_OK; ++t) {
    const ibp_store* s = stores[t];
    if (!s || !srcs[t] || s->R != s0->R || s->C != s0->C || s->device != s0->device) {
      e = IBP_EINVAL;
      break;
    }
    if (!aligned16(srcs[t])) {
      e = IBP_EALIGN;
      break;
    }
    if (s->n_rows > (1ull << 40) || s->slot > (1ull << 16)) {  // item offsets fit 56 bits
      e = IBP_EINVAL;
      break;
    }
    if (cudaEventSynchronize(s->props_ev) != cudaSuccess) {
      e = IBP_ECUDA;
      break;
    }
    const ibp::HostProps hp = host_props(s, 0);
    ibp::GroupEntry& g = h[t];
    g.src = static_cast<const uint8_t*>(srcs[t]);
    g.bitmap = s->bitmap;
    g.status = s->status;
    g.gtab = s->gtab;
    g.ckeep = s->ckeep;
    g.slot = s->slot;
    g.n_rows = s->n_rows;
    g.mode = hp.uniform ? (hp.um1 == 0 ? ibp::kModeUniform1 : ibp::kModeUniform)
                        : (hp.max_runs <= 2 ? ibp::kModeRun2 : ibp::kModeNet5);
    g.tab = g.mode == ibp::kModeNet5 ? s->t5 : s->t2;
    const uint32_t min_words = (hp.min_bits + 31u) / 32u;
    const uint32_t nvec = s->R / 16u;
    const uint32_t mv = (4u * min_words + 15u) / 16u;
    g.min_vec = mv < nvec ? mv : nvec;
    g.can_pack = 4u * min_words < s->R ? 1u : 0u;
    g.um0 = hp.um0;
    g.um1 = hp.um1;
    g.ush = hp.ush;
    g.ubv = hp.ubv;
    g.ukeep = hp.ukeep;
    g.scal = s->scal;
    g.lengths = s->lengths;
    g.gen = hp.gen;
    g.pad[0] = g.pad[1] = g.pad[2] = 0;
  }
  ibp_group* grp = nullptr;
  if (e == IBP_OK) {
    grp = new (std::nothrow) ibp_group();
    if (!grp) e = IBP_ENOMEM;
  }
  if (e == IBP_OK) {
    grp->T = n;
    grp->R = s0->R;
    grp->C = s0->C;
    grp->W = s0->W;
    grp->wpc = s0->wpc;
    grp->nch = s0->nch;
    grp->device = s0->device;
    grp->sm_count = s0->sm_count;
    grp->host_src = 0;
    for (uint32_t t = 0; t < n; ++t)
      if (ibp::host_pointer(srcs[t])) grp->host_src = 1;
    if (cudaMalloc(&grp->entries, sizeof(ibp::GroupEntry) * n) != cudaSuccess) {
      cudaGetLastError();
      e = IBP_ENOMEM;
    } else if (cudaMemcpy(grp->entries, h, sizeof(ibp::GroupEntry) * n, cudaMemcpyHostToDevice) !=
               cudaSuccess) {
      cudaFree(grp->entries);
      e = IBP_ECUDA;
    }
    if (e != IBP_OK) {
      delete grp;
      grp = nullptr;
    }
  }
  delete[] h;
  if (e == IBP_OK) *out = grp;
  return e;
}

ibp_status ibp_group_destroy(ibp_group* g) {
  if (!g) return IBP_OK;
  cudaDeviceSynchronize();
  const cudaError_t e = cudaFree(g->entries);
  delete g;
  return cu(e);
}

ibp_status ibp_group_gather_decompress(const ibp_group* g, void* dst, uint64_t dst_row_stride,
                                       const int64_t* ids, uint64_t batch, ibp_stream_t stream) {
  if (!g) return IBP_EINVAL;
  if (batch == 0) return IBP_OK;
  if (!dst || !ids) return IBP_EINVAL;
  if (!aligned16(dst) || (dst_row_stride & 15u) || dst_row_stride < (uint64_t)g->T * g->R)
    return IBP_EALIGN;
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return IBP_ECUDA;
  if (d != g->device) return IBP_EINVAL;
  const ibp::GroupArgs a = group_args(g, ids, batch, dst, dst_row_stride);
  return cu(ibp::launch_group(a, g->sm_count, reinterpret_cast<cudaStream_t>(stream)));
}

ibp_status ibp_group_gather_decompress_ordered(const ibp_group* g, void* dst,
                                               uint64_t dst_row_stride, const int64_t* ids,
                                               uint64_t batch, void* workspace,
                                               uint64_t workspace_bytes, ibp_stream_t stream) {
  if (!g) return IBP_EINVAL;
  if (batch == 0) return IBP_OK;
  if (!dst || !ids) return IBP_EINVAL;
  if (!aligned16(dst) || (dst_row_stride & 15u) || dst_row_stride < (uint64_t)g->T * g->R)
    return IBP_EALIGN;
  const uint64_t n_items = batch * g->T;
  ibp_status e = check_ordered(g, ids, n_items, workspace, workspace_bytes);
  if (e != IBP_OK) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const OrderWorkspace w = order_workspace(workspace, n_items);
  e = cu(cudaMemsetAsync(w.hist, 0, 4ull * ibp::kOrderBuckets, st));
  if (e != IBP_OK) return e;
  e = cu(ibp::launch_order_items(g->entries, g->T, ids, n_items, w.order, w.hist, g->sm_count,
                                 st));
  if (e != IBP_OK) return e;
  ibp::GroupArgs a = group_args(g, ids, batch, dst, dst_row_stride);
  a.order = w.order;
  return cu(ibp::launch_group_ordered(a, w.hist, w.wpre, w.cost, w.shares, g->sm_count, st));
}

ibp_status ibp_group_order_plan(const ibp_group* g, const int64_t* ids, uint64_t batch,
                                void* workspace, uint64_t workspace_bytes, ibp_stream_t stream) {
  if (!g) return IBP_EINVAL;
  if (batch == 0) return IBP_OK;
  const uint64_t n_items = batch * g->T;
  ibp_status e = check_ordered(g, ids, n_items, workspace, workspace_bytes);
  if (e != IBP_OK) return e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const OrderWorkspace w = order_workspace(workspace, n_items);
  e = cu(cudaMemsetAsync(w.hist, 0, 4ull * ibp::kOrderBuckets, st));
  if (e != IBP_OK) return e;
  e = cu(ibp::launch_order_items(g->entries, g->T, ids, n_items, w.order, w.hist, g->sm_count,
                                 st));
  if (e != IBP_OK) return e;
  ibp::GroupArgs a = group_args(g, ids, batch, nullptr, 0);
  a.order = w.order;
  const uint64_t blocks = ibp::group_gather_blocks(a, g->sm_count, ibp::group_planned_per_sm(a));
  return cu(ibp::launch_group_plan(a, w.hist, w.wpre, w.cost, w.shares, (uint32_t)(8u * blocks),
                                   w.stamp, st));
}

ibp_status ibp_group_gather_decompress_planned(const ibp_group* g, void* dst,
                                               uint64_t dst_row_stride, const int64_t* ids,
                                               uint64_t batch, const void* workspace,
                                               uint64_t workspace_bytes, ibp_stream_t stream) {
  if (!g) return IBP_EINVAL;
  if (batch == 0) return IBP_OK;
  if (!dst || !ids) return IBP_EINVAL;
  if (!aligned16(dst) || (dst_row_stride & 15u) || dst_row_stride < (uint64_t)g->T * g->R)
    return IBP_EALIGN;
  const uint64_t n_items = batch * g->T;
  ibp_status e = check_ordered(g, ids, n_items, workspace, workspace_bytes);
  if (e != IBP_OK) return e;
  const OrderWorkspace w = order_workspace(const_cast<void*>(workspace), n_items);
  ibp::GroupArgs a = group_args(g, ids, batch, dst, dst_row_stride);
  a.order = w.order;
  a.shares = w.shares;
  a.plan_stamp = w.stamp;
  const uint64_t blocks = ibp::group_gather_blocks(a, g->sm_count, ibp::group_planned_per_sm(a));
  return cu(ibp::launch_group_gather(a, blocks, reinterpret_cast<cudaStream_t>(stream)));
}

ibp_status ibp_project_compress(ibp_store* s, const void* x, uint64_t m, uint64_t k_dim,
                                const void* w, const void* bias, uint32_t dtype, void* y,
                                void* dst_slots, const int64_t* slot_ids,
                                uint32_t* stored_bytes_out, void* workspace,
                                uint64_t workspace_bytes, ibp_stream_t stream) {
  if (!s) return IBP_EINVAL;
  if (m == 0) return IBP_OK;
  if (!x || !w || !y || !dst_slots || !workspace) return IBP_EINVAL;
  if (dtype > 1u || k_dim == 0 || (k_dim % 64u) != 0 || k_dim > (1ull << 31)) return IBP_EINVAL;
  // one chunk = one 128-column tile of 16-bit values
  if (s->C != 256u || (s->R % 256u) != 0) return IBP_EINVAL;
  if (!slot_ids && m > s->n_rows) return IBP_ERANGE;
  if (m > 65535ull * 128ull) return IBP_EINVAL;  // row tiles in one grid dimension
  if (workspace_bytes < IBP_PROJECT_WORKSPACE_BYTES(m, s->R)) return IBP_EINVAL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(dst_slots) ||
      !aligned16(workspace) || (bias && !aligned16(bias)) ||
      (reinterpret_cast<uintptr_t>(slot_ids) & 7u) ||
      (reinterpret_cast<uintptr_t>(stored_bytes_out) & 3u))
    return IBP_EALIGN;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  ibp::ProjectArgs a;
  a.mask = s->mask;
  a.bitval = s->bitval;
  a.nm = s->nm;
  a.mv = s->mv;
  a.ckeep = s->ckeep;
  a.pre = s->pre;
  a.bitmap = s->bitmap;
  a.status = s->status;
  a.W = s->W;
  a.nch = s->nch;
  a.bf16 = dtype;
  a.m = m;
  a.k_dim = k_dim;
  a.bias = bias;
  a.y = static_cast<uint8_t*>(y);
  a.dst = static_cast<uint8_t*>(dst_slots);
  a.slot = s->slot;
  a.slot_ids = slot_ids;
  a.n_rows = s->n_rows;
  a.stored_out = stored_bytes_out;
  // workspace: a participation flag per (row, tile), up to 4 tiles per chunk,
  // then the staged kept bits (R bytes per row)
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.flags = reinterpret_cast<uint32_t*>(ws);
  a.staged = reinterpret_cast<uint32_t*>(ws + ((m * (s->R / 16u) + 255u) / 256u) * 256u);
  return cu(ibp::launch_project(a, x, w, s->sm_count, reinterpret_cast<cudaStream_t>(stream)));
}

ibp_status ibp_meta_get(const ibp_store* s, uint32_t* mask_host, uint32_t* bitval_host) {
  if (!s || !mask_host || !bitval_host) return IBP_EINVAL;
  if (cudaDeviceSynchronize() != cudaSuccess) return IBP_ECUDA;
  if (cudaMemcpy(mask_host, s->mask, 4ull * s->W, cudaMemcpyDeviceToHost) != cudaSuccess)
    return IBP_ECUDA;
  return cu(cudaMemcpy(bitval_host, s->bitval, 4ull * s->W, cudaMemcpyDeviceToHost));
}

ibp_status ibp_meta_set(ibp_store* s, const uint32_t* mask_host, const uint32_t* bitval_host) {
  if (!s || !mask_host || !bitval_host) return IBP_EINVAL;
  for (uint32_t w = 0; w < s->W; ++w)
    if (bitval_host[w] & ~mask_host[w]) return IBP_EINVAL;
  ibp_status e = on_device(s);
  if (e != IBP_OK) return e;
  if (cudaDeviceSynchronize() != cudaSuccess) return IBP_ECUDA;
  if (cudaMemcpy(s->mask, mask_host, 4ull * s->W, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(s->bitval, bitval_host, 4ull * s->W, cudaMemcpyHostToDevice) != cudaSuccess)
    return IBP_ECUDA;
  e = derive(s, 0);
  if (e != IBP_OK) return e;
  return cu(cudaDeviceSynchronize());
}

ibp_status ibp_bitmap_get(const ibp_store* s, uint32_t* host) {
  if (!s || !host) return IBP_EINVAL;
  if (cudaDeviceSynchronize() != cudaSuccess) return IBP_ECUDA;
  return cu(cudaMemcpy(host, s->bitmap, 4ull * s->bitmap_words, cudaMemcpyDeviceToHost));
}

ibp_status ibp_bitmap_set(ibp_store* s, const uint32_t* host) {
  if (!s || !host) return IBP_EINVAL;
  if (cudaDeviceSynchronize() != cudaSuccess) return IBP_ECUDA;
  return cu(cudaMemcpy(s->bitmap, host, 4ull * s->bitmap_words, cudaMemcpyHostToDevice));
}

ibp_status ibp_stream_status(const ibp_store* s, ibp_stream_t stream, ibp_status* out,
                             int reset) {
  if (!s || !out) return IBP_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return IBP_ECUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, s->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return IBP_ECUDA;
  *out = static_cast<ibp_status>(v);
  if (reset && v) {
    if (cudaMemset(s->status, 0, 4) != cudaSuccess) return IBP_ECUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return IBP_ECUDA;
  }
  return IBP_OK;
}

ibp_status ibp_link_copy(void* dst, const void* src, uint64_t bytes, ibp_stream_t stream) {
  if (bytes == 0) return IBP_OK;
  if (!dst || !src) return IBP_EINVAL;
  if (!aligned16(dst) || !aligned16(src) || (bytes & 15u)) return IBP_EALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return IBP_ECUDA;
  return cu(ibp::launch_link_copy(static_cast<uint4*>(dst), static_cast<const uint4*>(src),
                                  bytes / 16, sms, reinterpret_cast<cudaStream_t>(stream)));
}

ibp_status ibp_gather_copy(void* dst, const void* src, uint64_t slot_bytes, uint32_t row_bytes,
                           const int64_t* ids, uint64_t n, uint64_t n_rows,
                           ibp_stream_t stream) {
  if (n == 0) return IBP_OK;
  if (!dst || !src || !ids || row_bytes == 0) return IBP_EINVAL;
  if (!aligned16(dst) || !aligned16(src) || (row_bytes & 15u) || (slot_bytes & 15u))
    return IBP_EALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return IBP_ECUDA;
  return cu(ibp::launch_gather_copy(static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src),
                                    slot_bytes, row_bytes, ids, n, n_rows, sms,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
