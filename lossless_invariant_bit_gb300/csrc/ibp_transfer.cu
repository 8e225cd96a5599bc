// CPU-initiated transfer baselines for the host -> GPU gather of rows.
//
// The juhe.plus review of "Reducing the GPU Memory Bottleneck with Lossless
// Compression for ML -- Extended" compares four ways of moving small random
// tensors from CPU memory to the GPU (Figure 5): CPU fine-grained copies (one
// DMA per tensor), CPU bulk copies (gather on the CPU, then one DMA), GPU
// zero-copy and GPU aligned zero-copy.  The two GPU-initiated ways are
// ibp_gather_copy (on 128-byte aligned slots, or on a source shifted off the
// line boundaries); these are the two CPU-initiated ones, as host code.
#include <cstring>

#include "ibp_internal.cuh"

namespace {
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

extern "C" ibp_status ibp_gather_copy_dma(void* dst, const void* src, uint64_t slot_bytes,
                                          uint32_t row_bytes, const int64_t* ids_host,
                                          uint64_t n, uint64_t n_rows, ibp_stream_t stream) {
  if (n == 0) return IBP_OK;
  if (!dst || !src || !ids_host || row_bytes == 0) return IBP_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint8_t* d = static_cast<uint8_t*>(dst);
  for (uint64_t i = 0; i < n; ++i) {
    const int64_t id = ids_host[i];
    if (id < 0 || (uint64_t)id >= n_rows) return IBP_ERANGE;
    if (cudaMemcpyAsync(d + i * row_bytes, s + (uint64_t)id * slot_bytes, row_bytes,
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
      return IBP_ECUDA;
  }
  return IBP_OK;
}

extern "C" ibp_status ibp_gather_copy_staged(void* dst, const void* src, uint64_t slot_bytes,
                                             uint32_t row_bytes, const int64_t* ids_host,
                                             uint64_t n, uint64_t n_rows, void* staging_host,
                                             ibp_stream_t stream) {
  if (n == 0) return IBP_OK;
  if (!dst || !src || !ids_host || !staging_host || row_bytes == 0) return IBP_EINVAL;
  if (!aligned16(dst) || !aligned16(staging_host)) return IBP_EALIGN;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the staging buffer may still feed the previous call's copy
  if (cudaStreamSynchronize(st) != cudaSuccess) return IBP_ECUDA;
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint8_t* g = static_cast<uint8_t*>(staging_host);
  for (uint64_t i = 0; i < n; ++i) {
    const int64_t id = ids_host[i];
    if (id < 0 || (uint64_t)id >= n_rows) return IBP_ERANGE;
    std::memcpy(g + i * row_bytes, s + (uint64_t)id * slot_bytes, row_bytes);
  }
  if (cudaMemcpyAsync(dst, staging_host, n * row_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return IBP_ECUDA;
  return IBP_OK;
}
