// Allocation-free Mask/Bitval builder.
//
// Some callers cannot allocate device memory at the point where they need a
// Mask/Bitval: code that runs inside another framework's memory pool (whose
// allocator owns the device memory and must see every allocation), or a
// latency-sensitive loop where cudaMalloc's implicit device synchronisation
// would stall work on other streams.  ibp_build_meta needs a store, and a
// store owns device memory.  This entry point runs the same two builder
// kernels with their per-bit ones counters in a fixed array of device memory
// that belongs to this library, so the call itself allocates nothing: the
// caller passes the rows and the two output arrays.
#include <mutex>

#include "ibp_internal.cuh"

// One 32-bit ones counter per row bit position, for rows of up to
// IBP_NOALLOC_MAX_ROW_BYTES bytes: 256 KiB, held by every GPU that loads the
// library until the process exits.
static __device__ __align__(256) uint32_t g_noalloc_counts[8u * IBP_NOALLOC_MAX_ROW_BYTES];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_setup_mu;
uint32_t* g_counts_addr[kMaxDevices] = {};  // last looked-up device address, per device

// The array's name in host code is only a host-side stand-in; the kernels
// need its device address, looked up with the device current.  Outside a
// stream capture the lookup runs on every call (it is cheap once the module
// is loaded, and after a cudaDeviceReset, or in another context of the same
// device, the array lives at another address); a call being captured cannot
// make the lookup and takes the address the last uncaptured call on this
// device saw.
ibp_status counts_on(int dev, cudaStream_t st, uint32_t** out) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return IBP_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_counts) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return IBP_ECUDA;
    }
    g_counts_addr[dev] = static_cast<uint32_t*>(p);
  } else if (g_counts_addr[dev] == nullptr) {
    return IBP_EINVAL;  // no uncaptured call on this device yet
  }
  *out = g_counts_addr[dev];
  return IBP_OK;
}

}  // namespace

extern "C" ibp_status ibp_build_meta_noalloc(const void* rows, uint64_t row_stride,
                                             uint32_t row_bytes, const int64_t* sample_ids,
                                             uint64_t n, uint32_t thr_num, uint32_t thr_den,
                                             uint32_t* mask_out, uint32_t* bitval_out,
                                             ibp_stream_t stream) {
  if (!rows || !mask_out || !bitval_out) return IBP_EINVAL;
  if (row_bytes == 0 || (row_bytes & 15u)) return IBP_EINVAL;
  if (row_bytes > IBP_NOALLOC_MAX_ROW_BYTES) return IBP_EINVAL;
  if (n == 0 || n >= (1ull << 32)) return IBP_EINVAL;
  if (thr_den == 0 || thr_num > thr_den || 2ull * thr_num <= thr_den) return IBP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(rows) & 15u) || (row_stride & 15u) || row_stride < row_bytes)
    return IBP_EALIGN;
  // the kernels store whole 32-bit words to the outputs and read 64-bit ids
  if (((reinterpret_cast<uintptr_t>(mask_out) | reinterpret_cast<uintptr_t>(bitval_out)) & 3u) ||
      (reinterpret_cast<uintptr_t>(sample_ids) & 7u))
    return IBP_EALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IBP_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return IBP_EINVAL;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return IBP_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* counts = nullptr;
  ibp_status e = counts_on(dev, st, &counts);
  if (e != IBP_OK) return e;
  const uint32_t W = row_bytes / 4;
  // the array keeps the previous call's counts: clear the part this call uses
  if (cudaMemsetAsync(counts, 0, 32ull * W * sizeof(uint32_t), st) != cudaSuccess)
    return IBP_ECUDA;
  ibp::CountArgs a;
  a.rows = static_cast<const uint8_t*>(rows);
  a.row_stride = row_stride;
  a.ids = sample_ids;
  a.n = n;
  a.W = W;
  a.counts = counts;
  if (ibp::launch_count_ones(a, sms, st) != cudaSuccess) return IBP_ECUDA;
  if (ibp::launch_finish_meta(counts, W, n, thr_num, thr_den, mask_out, bitval_out, st) !=
      cudaSuccess)
    return IBP_ECUDA;
  return IBP_OK;
}
