// IBP kernels for sm_103a: Mask/Bitval builder, table derivation, compressor,
// decompressor (dense and gather, HBM or zero-copy host source) and the
// aligned zero-copy copy used as the host-link probe.
//
// Method: "Reducing the GPU Memory Bottleneck with Lossless Compression for
// ML -- Extended", gist.science explainer, Technical Summary, Methodology >
// Core Algorithm (Preprocessing, Compression, Decompression) and System
// Integration; juhe.plus review (one warp per tensor with only warp-local
// communication, 128-byte aligned GPU-initiated transfers).
//
// Nothing here is a dense contraction, so there are no tensor-core paths: the
// decoder is bound by the host link (zero-copy source) or by HBM (cache
// source), the builder by the bandwidth of the rows it reads, and the bit
// work runs on the integer pipes.
#include <cooperative_groups.h>
#include <mutex>
#include <vector>

#include "ibp_internal.cuh"

namespace ibp {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t code) {
  atomicCAS(st, 0u, code);
}

__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v, uint32_t lane) {
#pragma unroll
  for (uint32_t d = 1; d < 32; d <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, v, d);
    if (lane >= d) v += t;
  }
  return v;
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) { return __ldg(p); }


__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_n() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Scatter network of a kept-bit mask: the low popcount(nm) bits of v move to
// the set positions of nm, in order (5 stages of shifts by 16, 8, 4, 2, 1,
// the inverse of the gather below).  Bits of v above popcount(nm) may be
// anything; the caller masks the result with nm.
__device__ __forceinline__ uint32_t scatter_bits(uint32_t v, const uint32_t* mv, uint32_t W,
                                                 uint32_t w) {
#pragma unroll
  for (int i = 4; i >= 0; --i) {
    const uint32_t m = __ldg(mv + (uint32_t)i * W + w);
    v = (v & ~m) | ((v << (1u << i)) & m);
  }
  return v;
}

// Gather network: the bits of x at the set positions of nm, packed to the
// low end in order (x must already be masked with nm).
__device__ __forceinline__ uint32_t gather_bits(uint32_t x, const uint32_t* mv, uint32_t W,
                                                uint32_t w) {
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const uint32_t t = x & __ldg(mv + (uint32_t)i * W + w);
    x = (x ^ t) | (t >> (1u << i));
  }
  return x;
}

// ------------------------------------------------------------------------
// Builder (Core Algorithm > Preprocessing): ones count per row bit position.
// Thread = one word position; block.x tiles words, grid.x splits the rows.
// Eight rows at a time go through a carry-save adder tree (the Harley-Seal
// positional popcount: W. Muła, N. Kurz, D. Lemire, "Faster Population
// Counts Using AVX2 Instructions", 2018): running bit vectors of weight 1, 2
// and 4 absorb the rows, and the weight-8 carries feed 8 bit-plane counters
// (a vertical ripple-carry adder).  A carry-save step is two 3-input logic
// ops, so eight rows cost ~30 logic ops instead of 8 x 16.  The planes spill
// into 32 per-bit counts every 255 blocks of 8 rows; the per-thread totals go
// to the global counts with one atomic per bit.
// ------------------------------------------------------------------------
__device__ __forceinline__ void vadd(uint32_t (&c)[8], uint32_t x) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t t = c[p] & x;
    c[p] ^= x;
    x = t;
  }
}

__device__ __forceinline__ void vspill(uint32_t (&c)[8], uint32_t (&ones)[32]) {
#pragma unroll
  for (int b = 0; b < 32; ++b) {
    uint32_t s = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) s += ((c[p] >> b) & 1u) << p;
    ones[b] += s;
  }
#pragma unroll
  for (int p = 0; p < 8; ++p) c[p] = 0;
}

// carry-save add of three bit vectors: sum bits (weight 1), carry bits (weight 2)
__device__ __forceinline__ void csa(uint32_t& hi, uint32_t& lo, uint32_t a, uint32_t b,
                                    uint32_t c) {
  const uint32_t u = a ^ b;
  hi = (a & b) | (u & c);
  lo = u ^ c;
}

// Rows reach the counting threads through shared memory: a CTA copies the
// slice of 16 rows it counts next with 16-byte cp.async copies (lane v of
// warp q copies vector v of rows q, q+4, q+8, q+12) into a ring of 4 stages,
// 3 of them in flight while one is counted, so many bytes are in flight
// without costing registers; each thread then reads its word position of the
// 16 rows from shared memory.
constexpr uint32_t kCountRows = 16;   // rows per stage: two carry-save blocks
constexpr uint32_t kCountStages = 4;  // ring stages
constexpr uint32_t kCountTile = 128;  // word positions per CTA, one per thread (4 warps)
constexpr uint32_t kCountCluster = 8; // CTAs (same word tile, other rows) that pool their totals

__device__ __forceinline__ void count8(const uint32_t* sg, uint32_t& o1, uint32_t& o2,
                                       uint32_t& o4, uint32_t (&c)[8]) {
  uint32_t x[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) x[u] = sg[u * kCountTile];
  uint32_t t2a, t2b, t4a, t4b, t8;
  csa(t2a, o1, o1, x[0], x[1]);
  csa(t2b, o1, o1, x[2], x[3]);
  csa(t4a, o2, o2, t2a, t2b);
  csa(t2a, o1, o1, x[4], x[5]);
  csa(t2b, o1, o1, x[6], x[7]);
  csa(t4b, o2, o2, t2a, t2b);
  csa(t8, o4, o4, t4a, t4b);
  vadd(c, t8);
}

// The CTAs of a cluster cover the same word positions: at the end they add
// their totals through distributed shared memory (CTA r of the cluster sums
// bits 4r..4r+3 of all eight), so the global counters take one atomic per
// cluster instead of one per CTA.
__global__ void __cluster_dims__(kCountCluster, 1, 1) __launch_bounds__(128)
    k_count_ones(CountArgs a) {
  extern __shared__ __align__(16) uint32_t cring[];  // [stage][row][word of the tile]
  const uint32_t t = threadIdx.x;
  const uint32_t w0 = blockIdx.y * kCountTile;
  const uint32_t tw = min(kCountTile, a.W - w0);  // a multiple of 4 (rows are 16-byte multiples)
  const uint32_t nvr = tw >> 2;                   // 16-byte vectors of a row's slice, <= 32
  const uint32_t w = w0 + t;
  const bool active = t < tw;
  // this CTA's rows: a contiguous share [r0, r1) of [0, n)
  const uint64_t r0 = a.n * blockIdx.x / gridDim.x;
  const uint64_t r1 = a.n * (blockIdx.x + 1) / gridDim.x;
  const uint64_t ngrp = (r1 - r0 + kCountRows - 1) / kCountRows;
  const uint32_t cv = t & 31u, cq = t >> 5;  // the vector and first row this thread copies
  const uint32_t ring_sa =
      static_cast<uint32_t>(__cvta_generic_to_shared(cring)) + 16u * cv + 4u * cq * kCountTile;
  const uint8_t* src_v = a.rows + 4ull * w0 + 16u * cv;
  auto issue = [&](uint64_t j) {  // rows of group j into stage j % kCountStages
    if (j < ngrp && cv < nvr) {
      const uint32_t sb = ring_sa + 4u * (uint32_t)(j % kCountStages) * kCountRows * kCountTile;
      const uint64_t ib = r0 + kCountRows * j + cq;
#pragma unroll
      for (uint32_t k = 0; k < kCountRows / 4u; ++k) {
        const uint64_t i = ib + 4u * k;
        if (i < r1) {
          const uint64_t row = a.ids ? (uint64_t)__ldg(a.ids + i) : i;
          asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(
                           sb + 16u * k * kCountTile),
                       "l"(src_v + row * a.row_stride));
        }
      }
    }
    cp_async_commit();
  };

  uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // planes counting weight-8 carries
  uint32_t n8[32];                            // spilled plane counts (units of 8 rows)
#pragma unroll
  for (int b = 0; b < 32; ++b) n8[b] = 0;
  uint32_t o1 = 0, o2 = 0, o4 = 0;  // running bit vectors of weight 1, 2, 4
  uint32_t blocks = 0;
  for (uint32_t j = 0; j + 1 < kCountStages; ++j) issue(j);
  for (uint64_t j = 0; j < ngrp; ++j) {
    issue(j + kCountStages - 1);
    cp_async_wait_n<kCountStages - 1>();  // this thread's copies of group j have landed
    __syncthreads();                       // and everyone else's
    const uint32_t* sg = cring + (uint32_t)(j % kCountStages) * kCountRows * kCountTile + t;
    const uint64_t left = r1 - r0 - kCountRows * j;
    if (active) {
      if (left >= kCountRows) {
        count8(sg, o1, o2, o4, c);
        count8(sg + 8u * kCountTile, o1, o2, o4, c);
        blocks += 2;
        if (blocks >= 254u) {  // the 8-bit planes hold at most 255 carries
          vspill(c, n8);
          blocks = 0;
        }
      } else {  // the last < 16 rows
        uint32_t u = 0;
        if (left >= 8u) {
          count8(sg, o1, o2, o4, c);
          u = 8;
        }
        vspill(c, n8);  // room for the tail's carries in the 8-bit planes
        for (; u < (uint32_t)left; ++u) {  // half adders down the chain
          const uint32_t x = sg[u * kCountTile];
          const uint32_t k1 = o1 & x;
          o1 ^= x;
          const uint32_t k2 = o2 & k1;
          o2 ^= k1;
          const uint32_t k4 = o4 & k2;
          o4 ^= k2;
          vadd(c, k4);
        }
      }
    }
    __syncthreads();  // stage j % kCountStages is refilled by the next issue
  }
  cp_async_wait_n<0>();
  __syncthreads();  // the ring is free: it takes this CTA's totals, [bit][word of the tile]
  vspill(c, n8);
#pragma unroll
  for (int b = 0; b < 32; ++b)
    cring[(uint32_t)b * kCountTile + t] = 8u * n8[b] + 4u * ((o4 >> b) & 1u) +
                                          2u * ((o2 >> b) & 1u) + ((o1 >> b) & 1u);
  cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
  cl.sync();
  constexpr uint32_t kBitsPer = 32u / kCountCluster;
  const uint32_t b0 = cl.block_rank() * kBitsPer;
#pragma unroll
  for (uint32_t bb = 0; bb < kBitsPer; ++bb) {
    uint32_t sum = 0;
#pragma unroll
    for (uint32_t r = 0; r < kCountCluster; ++r)
      sum += cl.map_shared_rank(cring, r)[(b0 + bb) * kCountTile + t];
    if (active && sum) atomicAdd(a.counts + 32u * w + b0 + bb, sum);
  }
  cl.sync();  // no CTA leaves while the others read its totals
}

// Threshold: bit j is invariant when ones*den >= num*n (value 1) or
// (n-ones)*den >= num*n (value 0); 64-bit integer arithmetic.
__global__ void k_finish_meta(const uint32_t* counts, uint32_t W, uint64_t n, uint32_t num,
                              uint32_t den, uint32_t* mask, uint32_t* bitval) {
  const uint32_t w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= W) return;
  const uint64_t lim = (uint64_t)num * n;
  uint32_t m = 0, bv = 0;
  for (uint32_t b = 0; b < 32; ++b) {
    const uint64_t o = counts[32u * w + b];
    const bool inv1 = o * den >= lim;
    const bool inv0 = (n - o) * den >= lim;
    m |= (uint32_t)(inv1 || inv0) << b;
    bv |= (uint32_t)inv1 << b;
  }
  mask[w] = m;
  bitval[w] = bv;
}

// Chunk-aware choice among candidate thresholds (the review's sampling
// experiment uses the sample for the Mask; here the same sample also prices
// each candidate Mask): for candidate c (blockIdx.y), the stored size every
// sampled row would take -- participation per chunk, stream bits, raw
// fallback -- summed into sizes[c].  cand holds, per candidate, W Mask words
// then W Bitval words.
__global__ void __launch_bounds__(256) k_size_estimate(const uint8_t* rows, uint64_t row_stride,
                                                       const int64_t* ids, uint64_t n,
                                                       const uint32_t* cand, uint32_t W,
                                                       uint32_t wpc, uint32_t nch,
                                                       unsigned long long* sizes) {
  extern __shared__ uint32_t sm[];
  const uint32_t c = blockIdx.y;
  const uint32_t* M = cand + 2ull * W * c;
  const uint32_t* B = M + W;
  const uint32_t nr = (nch + 3u) & ~3u;
  uint32_t* ck = sm;  // kept bits per chunk under this candidate
  const uint32_t lane = threadIdx.x & 31u, wid = threadIdx.x >> 5;
  uint32_t* mism = sm + nr * (1u + wid);
  for (uint32_t k = threadIdx.x; k < nch; k += blockDim.x) ck[k] = 0;
  __syncthreads();
  for (uint32_t w = threadIdx.x; w < W; w += blockDim.x) atomicAdd(&ck[w / wpc], (uint32_t)__popc(~M[w]));
  __syncthreads();
  const uint32_t R = 4u * W;
  unsigned long long local = 0;
  const uint64_t wstride = (uint64_t)gridDim.x * (blockDim.x >> 5);
  for (uint64_t i = (uint64_t)blockIdx.x * (blockDim.x >> 5) + wid; i < n; i += wstride) {
    const uint64_t row = ids ? (uint64_t)__ldg(ids + i) : i;
    const uint32_t* x = reinterpret_cast<const uint32_t*>(rows + row * row_stride);
    for (uint32_t k = lane; k < nch; k += 32) mism[k] = 0;
    __syncwarp();
    for (uint32_t w = lane; w < W; w += 32)
      if ((__ldg(x + w) & __ldg(M + w)) != __ldg(B + w)) mism[w / wpc] = 1u;
    __syncwarp();
    uint32_t part = 0;
    for (uint32_t k = lane; k < nch; k += 32) {
      const uint32_t full = 32u * min(wpc, W - k * wpc);
      part += (mism[k] == 0u && ck[k] < full) ? ck[k] : full;
    }
    const uint32_t bits = nch + __reduce_add_sync(0xFFFFFFFFu, part);
    const uint32_t stored = 4u * ((bits + 31u) >> 5);
    local += stored >= R ? R : stored;
    __syncwarp();
  }
  if (lane == 0 && local) atomicAdd(sizes + c, local);
}

// The cheapest candidate (the first on ties) becomes the store's Mask/Bitval.
__global__ void __launch_bounds__(256) k_pick_meta(const uint32_t* cand,
                                                   const unsigned long long* sizes, uint32_t n_c,
                                                   uint32_t W, uint32_t* mask, uint32_t* bitval,
                                                   uint32_t* chosen_out, uint64_t* sizes_out) {
  __shared__ uint32_t best;
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (uint32_t c = 1; c < n_c; ++c)
      if (sizes[c] < sizes[b]) b = c;
    best = b;
    if (chosen_out) *chosen_out = b;
  }
  if (sizes_out)
    for (uint32_t c = threadIdx.x; c < n_c; c += blockDim.x) sizes_out[c] = sizes[c];
  __syncthreads();
  const uint32_t* M = cand + 2ull * W * best;
  for (uint32_t w = threadIdx.x; w < W; w += blockDim.x) {
    mask[w] = M[w];
    bitval[w] = M[W + w];
  }
}

// Decode tables from the Mask (one block).  The move masks are those of the
// classic 5-stage bit gather (H. S. Warren, Hacker's Delight, sec. 7-4 and
// 7-5): at stage i, the bits of the current mask with an odd number of
// not-yet-consumed zeros below them (parallel suffix parity) move right by
// 2^i.
__device__ void move_masks(uint32_t m, uint32_t (&mv)[5]) {
  uint32_t zeros_below = ~m << 1;
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    uint32_t par = zeros_below ^ (zeros_below << 1);
    par ^= par << 2;
    par ^= par << 4;
    par ^= par << 8;
    par ^= par << 16;
    const uint32_t mov = par & m;
    mv[i] = mov;
    m = (m ^ mov) | (mov >> (1u << i));
    zeros_below &= ~par;
  }
}

__global__ void __launch_bounds__(1024) k_derive(uint32_t* mask, uint32_t* bitval, uint32_t* nm,
                                                 uint32_t* pre, uint32_t* kr, uint32_t* mv,
                                                 uint32_t* ckeep, uint32_t* scal, uint32_t W,
                                                 uint32_t wpc, uint32_t nch) {
  __shared__ uint32_t s_sum, s_runs;
  if (threadIdx.x == 0) {
    s_sum = 0;
    s_runs = 0;
  }
  __syncthreads();
  for (uint32_t w = threadIdx.x; w < W; w += blockDim.x) {
    const uint32_t keepm = ~mask[w];
    bitval[w] &= mask[w];
    nm[w] = keepm;
    uint32_t m5[5];
    move_masks(keepm, m5);
#pragma unroll
    for (int i = 0; i < 5; ++i) mv[(uint32_t)i * W + w] = m5[i];
    kr[w] = (w / wpc) | ((w % wpc) << 16);
    atomicMax(&s_runs, (uint32_t)__popc(keepm & ~(keepm << 1)));
  }
  for (uint32_t k = threadIdx.x; k < nch; k += blockDim.x) {
    const uint32_t e = min((k + 1) * wpc, W);
    uint32_t acc = 0;
    for (uint32_t w = k * wpc; w < e; ++w) {
      pre[w] = acc;
      acc += __popc(~mask[w]);
    }
    ckeep[k] = acc;
    atomicAdd(&s_sum, acc);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    scal[0] = nch + s_sum;
    scal[1] = s_runs;
    scal[2] = 1;
    scal[9] += 1u;  // a new generation of the store's tables
  }
}

// Shared-memory decode descriptors for the fast decoder (one block; runs
// after k_derive, whose nm/pre/mv/ckeep it reads).  soff[w] is word w's bit
// offset in a stream whose chunks all participate: nch + the kept bits of
// every earlier word.
//   t2 = {run0, run1, Bitval, soff | s0 << 20 | s1 << 25} -- ~Mask as at most
//        two runs of kept bits: run r takes the next len_r stream bits, shifted
//        left by s_r (its start minus the kept bits before it); valid when
//        every word has <= 2 runs
//   t5 = {mv0, mv1, mv2, mv3}, {mv4, ~Mask, Bitval, soff} -- scatter network
//   gtab[g] = chunk of words 4g..4g+3 | (4g - first word of that chunk) << 16,
//   then (from word roundup(W/4, 4)) the all-packed start of each chunk
// Word w = 4g + e sits at t2[e*G + g] and t5[(2e + h)*G + g] (G = W/4): the
// lanes of a warp read consecutive 16-byte entries, free of bank conflicts.
__global__ void __launch_bounds__(1024) k_derive_fast(const uint32_t* nm, const uint32_t* bitval,
                                                      const uint32_t* pre, const uint32_t* mv,
                                                      const uint32_t* ckeep, uint4* t2, uint4* t5,
                                                      uint32_t* gtab, uint32_t* scal, uint32_t W,
                                                      uint32_t wpc, uint32_t nch) {
  __shared__ uint32_t s_start[IBP_MAX_CHUNKS];
  __shared__ uint32_t s_same;
  if (threadIdx.x == 0) {
    s_same = 1;
    uint32_t run = nch;
    for (uint32_t k = 0; k < nch; ++k) {
      s_start[k] = run;
      run += ckeep[k];
    }
  }
  __syncthreads();
  const uint32_t G = W >> 2;
  const uint32_t G4 = (G + 3u) & ~3u;
  for (uint32_t w = threadIdx.x; w < W; w += blockDim.x) {
    const uint32_t keepm = nm[w];
    const uint32_t r0 = keepm & ~(keepm + (keepm & (0u - keepm)));
    const uint32_t rest = keepm & ~r0;
    const uint32_t r1 = rest & ~(rest + (rest & (0u - rest)));
    const uint32_t s0 = r0 ? (uint32_t)(__ffs(r0) - 1) : 0u;
    const uint32_t s1 = r1 ? (uint32_t)(__ffs(r1) - 1) - (uint32_t)__popc(r0) : 0u;
    const uint32_t soff = s_start[w / wpc] + pre[w];
    const uint32_t g = w >> 2, e = w & 3u;
    if (g < G) {
      t2[e * G + g] = make_uint4(r0, r1, bitval[w], soff | (s0 << 20) | (s1 << 25));
      t5[2 * e * G + g] = make_uint4(mv[w], mv[W + w], mv[2 * W + w], mv[3 * W + w]);
      t5[(2 * e + 1) * G + g] = make_uint4(mv[4 * W + w], keepm, bitval[w], soff);
    }
  }
  for (uint32_t g = threadIdx.x; g < G; g += blockDim.x) {
    const uint32_t k = (4 * g) / wpc;
    gtab[g] = k | ((4 * g - k * wpc) << 16);
  }
  for (uint32_t k = threadIdx.x; k < nch; k += blockDim.x) gtab[G4 + k] = s_start[k];
  // uniform store: every word has the same ~Mask and Bitval, with <= 2 runs
  for (uint32_t w = threadIdx.x; w < W; w += blockDim.x)
    if (nm[w] != nm[0] || bitval[w] != bitval[0]) atomicAnd(&s_same, 0u);
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t keepm = nm[0];
    const uint32_t r0 = keepm & ~(keepm + (keepm & (0u - keepm)));
    const uint32_t rest = keepm & ~r0;
    const uint32_t r1 = rest & ~(rest + (rest & (0u - rest)));
    const uint32_t s0 = r0 ? (uint32_t)(__ffs(r0) - 1) : 0u;
    const uint32_t s1 = r1 ? (uint32_t)(__ffs(r1) - 1) - (uint32_t)__popc(r0) : 0u;
    const bool two = (rest & ~r1) == 0u;
    scal[3] = (s_same && two) ? 1u : 0u;
    scal[4] = r0;
    scal[5] = r1;
    scal[6] = s0 | (s1 << 8);
    scal[7] = bitval[0];
    scal[8] = (uint32_t)__popc(keepm);
  }
}

// ------------------------------------------------------------------------
// Decompression.  One warp per row (the pages' "one warp per tensor"), but
// the lanes split the row's output words rather than its chunks, so a row
// with fewer than 32 chunks still keeps all lanes busy.  Per row:
//   resolve   id, raw bit, source address;
//   fetch     the shortest stream any compressed row can have (min_bits) in
//             16-byte cp.async copies, staged in the warp's shared memory;
//   scan      participation bits -> chunk sizes -> exclusive warp scan;
//   fetch     the rest of the stream when raw chunks made it longer;
//   re-insert each lane builds 4 output words at a time: a funnel shift
//             pulls the word's bits out of the staged stream, the scatter
//             network spreads them over ~Mask, Bitval fills the rest; one
//             coalesced 16-byte store.
// A raw row is a straight 16-byte vector copy.
// ------------------------------------------------------------------------
// Where row `id`'s stored bytes start, relative to a.src: packed offsets,
// a slot, or -- with a cache map -- the row's slot in the HBM cache when it
// has one (the unsigned difference of the two bases wraps, so a.src + result
// addresses the cache).
constexpr uint64_t kBadSource = ~0ull;  // a cache map entry past the cache's slots

__device__ __forceinline__ uint64_t source_offset(const DecodeArgs& a, int64_t id) {
  if (a.cache_map) {
    const int64_t cs = __ldg(a.cache_map + id);
    if (cs >= 0) {
      if ((uint64_t)cs >= a.cache_slots) return kBadSource;
      return (uint64_t)((uintptr_t)a.cache_src - (uintptr_t)a.src) + (uint64_t)cs * a.slot;
    }
  }
  return a.offsets ? __ldg(a.offsets + id) : (uint64_t)id * a.slot;
}

// 16-byte vectors [v0, v1) of a stored stream into the warp's buffer at
// shared address `sa`, all issued before any is waited for: one round trip
// to host memory per fetch instead of one per 512 bytes.
__device__ __forceinline__ void fetch_vectors(uint32_t sa, const uint4* src, uint32_t v0,
                                              uint32_t v1, uint32_t lane) {
  for (uint32_t v = v0 + lane; v < v1; v += 32)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(sa + 16u * v),
                 "l"(src + v));
  cp_async_commit();
  cp_async_wait_n<0>();
  __syncwarp();
}

__device__ __forceinline__ void zero_row(uint4* drow, uint32_t nvec, uint32_t lane) {
  for (uint32_t v = lane; v < nvec; v += 32) drow[v] = make_uint4(0, 0, 0, 0);
}

template <bool kIds>
__global__ void __launch_bounds__(256) k_decode(DecodeArgs a, WarpSmem L) {
  extern __shared__ __align__(16) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t wid = threadIdx.x >> 5;
  uint32_t* sbuf = smem + wid * L.total_words;
  uint32_t* cinfo = sbuf + L.sbuf_words;
  const uint32_t sbuf_sa = static_cast<uint32_t>(__cvta_generic_to_shared(sbuf));
  const uint32_t R = a.m.R, W = a.m.W, wpc = a.m.wpc, nch = a.m.nch;
  const uint32_t nvec = R >> 4;
  const uint32_t min_words = (__ldg(a.m.scal) + 31u) >> 5;
  const uint32_t min_vec = (4u * min_words + 15u) >> 4;
  const uint64_t wpb = blockDim.x >> 5;
  const uint64_t stride = (uint64_t)gridDim.x * wpb;

  for (uint64_t i = (uint64_t)blockIdx.x * wpb + wid; i < a.n; i += stride) {
    const uint64_t orow = (kIds && a.out_pos) ? (uint64_t)__ldg(a.out_pos + i) : i;
    uint4* drow = reinterpret_cast<uint4*>(a.dst + orow * a.dst_stride);
    const int64_t id = kIds ? __ldg(a.ids + i) : (int64_t)i;
    if (id < 0 || (uint64_t)id >= a.n_rows) {
      if (lane == 0) set_status(a.status, IBP_ERANGE);
      zero_row(drow, nvec, lane);
      continue;
    }
    const uint64_t off = source_offset(a, id);
    if (off == kBadSource) {
      if (lane == 0) set_status(a.status, IBP_ERANGE);
      zero_row(drow, nvec, lane);
      continue;
    }
    if (off & 15u) {
      if (lane == 0) set_status(a.status, IBP_EALIGN);
      zero_row(drow, nvec, lane);
      continue;
    }
    const uint4* srow = reinterpret_cast<const uint4*>(a.src + off);
    const bool raw = (__ldg(a.bitmap + (id >> 5)) >> (id & 31)) & 1u;
    if (raw) {
      for (uint32_t v = lane; v < nvec; v += 32) drow[v] = ld_nc_v4(srow + v);
      continue;
    }
    if (4u * min_words >= R) {  // no compressed row can exist for this Mask
      if (lane == 0) set_status(a.status, IBP_ECORRUPT);
      zero_row(drow, nvec, lane);
      continue;
    }
    // the first fetch: the whole stream when its length is known, else the shortest one
    const uint32_t first =
        a.lengths ? min(max((__ldg(a.lengths + id) + 15u) >> 4, min_vec), nvec) : min_vec;
    fetch_vectors(sbuf_sa, srow, 0u, first, lane);
    // chunk starts: exclusive scan of the chunk sizes, 32 chunks per pass
    uint32_t run = nch;
    for (uint32_t k0 = 0; k0 < nch; k0 += 32) {
      const uint32_t k = k0 + lane;
      uint32_t size = 0, p = 0;
      if (k < nch) {
        p = (sbuf[k >> 5] >> (k & 31u)) & 1u;
        size = p ? __ldg(a.m.ckeep + k) : 32u * min(wpc, W - k * wpc);
      }
      const uint32_t incl = warp_inclusive_scan(size, lane);
      if (k < nch) cinfo[k] = (run + incl - size) | (p << 31);
      run += __shfl_sync(kFull, incl, 31);
    }
    const uint32_t words = (run + 31u) >> 5;
    if (4u * words >= R || 4ull * words > a.avail) {
      if (lane == 0) set_status(a.status, IBP_ECORRUPT);
      __syncwarp();
      zero_row(drow, nvec, lane);
      continue;
    }
    const uint32_t need_vec = (4u * words + 15u) >> 4;
    if (need_vec > first) fetch_vectors(sbuf_sa, srow, first, need_vec, lane);
    for (uint32_t v = lane; v < nvec; v += 32) {
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t w = 4u * v + (uint32_t)e;
        const uint32_t krw = __ldg(a.m.kr + w);
        const uint32_t ci = cinfo[krw & 0xFFFFu];
        const bool packed = (ci >> 31) != 0u;
        const uint32_t bit = (ci & 0x7FFFFFFFu) + (packed ? __ldg(a.m.pre + w) : ((krw >> 16) << 5));
        const uint32_t q = bit >> 5;
        uint32_t x = __funnelshift_r(sbuf[q], sbuf[q + 1], bit & 31u);
        if (packed)
          x = (scatter_bits(x, a.m.mv, W, w) & __ldg(a.m.nm + w)) | __ldg(a.m.bitval + w);
        o[e] = x;
      }
      drow[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------------
// Fast decompression for rows of at most 8 KB whose chunks hold whole groups
// of 4 words (C % 16 == 0): the common geometries (512 B - 8 KB rows, chunks
// of 256 B / 1 KB / 4 KB).  Differences from k_decode:
//   - a warp resolves 32 rows at a time, one per lane (id -> offset -> raw
//     bit, coalesced), the next 32 one chunk ahead, and then walks them one
//     by one; each row's (offset, flags) sit in a shared-memory ring;
//   - the stored bytes travel by cp.async (.ca) into a ring of S single-row
//     stages in shared memory, S-1 rows ahead of the row being decoded, so the
//     bytes in flight cost no registers; this holds for HBM sources and for
//     pinned host memory read over the link (rows above 2 KB: the kBig
//     instances, with a 3-row ring and up to 16 copies per lane);
//   - a row whose chunks all participate (the usual case) needs no scan: word
//     w's kept bits sit at a static offset (for a uniform store, one whose
//     words all share the same ~Mask and Bitval, nch + w*keep);
//   - the per-word decode descriptors sit in shared memory, staged once per
//     persistent CTA; where no word of ~Mask has more than two runs of kept
//     bits (fp32 sign/exponent masks), the scatter is two shift-and-mask
//     steps instead of the 5-stage network.
// ------------------------------------------------------------------------



// Four output words 4g..4g+3 of a row whose chunk participates: their kept
// bits start at the static offsets plus `delta` (the extra bits of raw chunks
// earlier in the row).
__device__ __forceinline__ uint4 decode_group(const uint4* tab, const uint32_t* sb, uint32_t g,
                                              uint32_t G, uint32_t delta, bool net5) {
  uint32_t o[4];
  if (!net5) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint4 t = tab[(uint32_t)e * G + g];
      const uint32_t bit = (t.w & 0xFFFFFu) + delta;
      const uint32_t q = bit >> 5;
      const uint32_t x = __funnelshift_r(sb[q], sb[q + 1], bit);
      o[e] = ((x << ((t.w >> 20) & 31u)) & t.x) | ((x << (t.w >> 25)) & t.y) | t.z;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint4 t0 = tab[2u * (uint32_t)e * G + g];
      const uint4 t1 = tab[(2u * (uint32_t)e + 1u) * G + g];
      const uint32_t bit = t1.w + delta;
      const uint32_t q = bit >> 5;
      uint32_t x = __funnelshift_r(sb[q], sb[q + 1], bit);
      x = (x & ~t1.x) | ((x << 16) & t1.x);
      x = (x & ~t0.w) | ((x << 8) & t0.w);
      x = (x & ~t0.z) | ((x << 4) & t0.z);
      x = (x & ~t0.y) | ((x << 2) & t0.y);
      x = (x & ~t0.x) | ((x << 1) & t0.x);
      o[e] = (x & t1.y) | t1.z;
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8-warp CTAs per SM the register budget is cut for: the uniform mode fits 64
// registers without spilling (4 CTAs, 32 warps per SM), the others 80 (3 CTAs)
#define IBP_FAST_MIN_BLOCKS(mode) ((mode) == kModeUniform || (mode) == kModeUniform1 ? 4 : 3)

// Decode of a word group under each store mode (FastMode): the uniform form
// takes its run masks and shifts from the launch parameters.
template <int kMode>
__device__ __forceinline__ uint4 decode_packed_group(const uint4* tab, const uint32_t* sb,
                                                     uint32_t g, uint32_t G, uint32_t nch,
                                                     uint32_t delta, bool net5, bool uni,
                                                     const FastParams& F, const uint32_t* up) {
  if (kMode == kModeUniform1) {  // one run: a funnel shift and a mask per word
    // The window starts ush bits before the word's kept bits, so they land at
    // the run's place [ush, ush + ukeep) without a second shift.  For a
    // stream's first word (bit < ush) the window takes its low word from the
    // shared-memory word before the stream: every stream buffer has other
    // shared memory in front of it, and those bits fall below ush, outside
    // the mask.
    int bit = (int)(nch + 4u * g * F.ukeep + delta) - (int)(F.ush & 31u);
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int q = bit >> 5;  // -1 at the least
      const uint32_t x = __funnelshift_r(sb[q], sb[q + 1], (uint32_t)bit);
      o[e] = (x & F.um0) | F.ubv;
      bit += (int)F.ukeep;
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (kMode == kModeUniform || (kMode == kModeRuntime && uni)) {
    uint32_t m0, m1, sh, bv, keep;
    if (kMode == kModeUniform) {
      m0 = F.um0; m1 = F.um1; sh = F.ush; bv = F.ubv; keep = F.ukeep;
    } else {
      m0 = up[0]; m1 = up[1]; sh = up[2]; bv = up[3]; keep = up[4];
    }
    uint32_t bit = nch + 4u * g * keep + delta;  // word w's kept bits at nch + w*keep
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t q = bit >> 5;
      const uint32_t x = __funnelshift_r(sb[q], sb[q + 1], bit);
      o[e] = ((x << (sh & 31u)) & m0) | ((x << (sh >> 8)) & m1) | bv;
      bit += keep;
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
  return decode_group(tab, sb, g, G, delta, kMode == kModeNet5 || (kMode == kModeRuntime && net5));
}

constexpr uint32_t kRingStages = 4;     // rows per warp ring: 3 in flight while one decodes
constexpr uint32_t kRingStagesBig = 3;  // rows above 2 KB: 2 in flight, more warps per SM

// Split output: where the 16-byte group g of a row lands, from the group
// table entry (chunk k | word offset in the chunk << 16).
__device__ __forceinline__ uint4* split_group(uint4* drow, const uint32_t* gtab, uint32_t g,
                                              uint64_t chunk_stride) {
  const uint32_t gd = gtab[g];
  return reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(drow) +
                                  (uint64_t)(gd & 0xFFFFu) * chunk_stride + 4u * (gd >> 16));
}

template <bool kIds, int kMode, bool kBig, bool kSplit>
__global__ void __launch_bounds__(256, IBP_FAST_MIN_BLOCKS(kMode)) k_decode_fast(DecodeArgs a, FastParams F) {
  extern __shared__ __align__(16) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t wid = threadIdx.x >> 5;
  const uint32_t R = a.m.R, W = a.m.W, wpc = a.m.wpc, nch = a.m.nch;
  constexpr uint32_t S = kBig ? kRingStagesBig : kRingStages;
  const uint32_t nvec = R >> 4;
  const uint32_t G = W >> 2;
  const uint32_t min_bits = kMode == kModeRuntime ? __ldg(a.m.scal) : F.min_bits;
  const bool net5 = kMode == kModeNet5 || (kMode == kModeRuntime && __ldg(a.m.scal + 1) > 2u);
  const bool uni = kMode == kModeUniform || kMode == kModeUniform1 ||
                   (kMode == kModeRuntime && __ldg(a.m.scal + 3) != 0u);
  const uint32_t min_words = (min_bits + 31u) >> 5;
  const bool can_pack = 4u * min_words < R;
  const uint32_t min_vec = min((4u * min_words + 15u) >> 4, nvec);
  // the specialised modes carry store properties fixed on the host; a launch
  // replayed (from a CUDA graph) after the Mask/Bitval changed must not use them
  const bool stale = kMode != kModeRuntime && __ldg(a.m.scal + 9) != F.gen;

  uint4* tab = reinterpret_cast<uint4*>(smem);
  uint32_t* gtab = smem + F.table_words;
  uint32_t* uparm = gtab + F.gtab_words;  // uniform-store parameters (runtime mode)
  uint32_t* ring = uparm + 8 + wid * F.warp_words;
  // row info ring, two 32-row chunks: {offset | flags (lo, hi), output offset (lo, hi)}
  // flags (low 4 bits, offsets are 16-byte aligned): 1 present, 2 raw, 4 bad id,
  // 8 misaligned, 4|8 store properties out of date
  uint4* rinfo = reinterpret_cast<uint4*>(ring + S * F.sbuf_words);
  uint32_t* cinfo = ring + S * F.sbuf_words + 256;
  {
    if (F.table_words && !uni) {
      const uint4* t = net5 ? a.t5 : a.t2;
      const uint32_t nv = net5 ? 2u * W : W;
      for (uint32_t v = threadIdx.x; v < nv; v += blockDim.x) tab[v] = __ldg(t + v);
    }
    for (uint32_t g = threadIdx.x; g < F.gtab_words; g += blockDim.x) gtab[g] = __ldg(a.gtab + g);
    if (kMode == kModeRuntime && threadIdx.x < 8) uparm[threadIdx.x] = __ldg(a.m.scal + 4 + threadIdx.x);
  }
  __syncthreads();
  const uint32_t* cstat = gtab + ((G + 3u) & ~3u);  // all-packed start of each chunk
  const uint32_t nhw = (nch + 31u) >> 5;             // header words
  const uint32_t hexp = (lane + 1u < nhw || (nch & 31u) == 0u) ? 0xFFFFFFFFu
                                                                 : ((1u << (nch & 31u)) - 1u);

  // this warp's rows: a contiguous, balanced share [r0, r0 + cnt) of [0, n);
  // for an ordered gather, of the address-sorted list, so that each SM reads
  // within a narrow range of the store's addresses (measured on 26 tables of
  // 2 KB rows, 53 GB: 281 GB/s, against 240 for 32-row chunks taken in turn
  // by all warps and 131 for rows dealt out one by one across the warps)
  const uint64_t nw = (uint64_t)gridDim.x * (blockDim.x >> 5);
  const uint64_t gw = (uint64_t)blockIdx.x * (blockDim.x >> 5) + wid;
  const bool ordered = kIds && a.out_pos != nullptr;
  const uint64_t r0 = a.n * gw / nw;
  const uint32_t cnt = (uint32_t)(a.n * (gw + 1) / nw - r0);
  if (cnt == 0) return;
  auto row_index = [&](uint32_t t) -> uint64_t { return r0 + t; };  // the warp's t-th row

  // Resolving chunk q (rows r0 + 32q + lane) is a chain of dependent loads
  // (id -> offset, raw bit); it runs in three steps spread over the chunk two
  // ahead, so the loads complete while other rows are decoded.
  int64_t pid = 0, ppos = 0;
  uint64_t poff = 0;
  uint32_t pbm = 0, plen = 0;
  bool pin = false;
  auto step_ids = [&](uint32_t q) {
    const uint32_t t = 32u * q + lane;
    const uint64_t ri = row_index(t);
    pin = q < (cnt + 31u) / 32u && t < cnt && ri < a.n;
    if (pin) {
      pid = kIds ? __ldg(a.ids + ri) : (int64_t)ri;
      if (ordered) ppos = __ldg(a.out_pos + ri);
    }
  };
  auto step_loads = [&]() {
    if (pin && pid >= 0 && (uint64_t)pid < a.n_rows) {
      poff = source_offset(a, pid);
      pbm = __ldg(a.bitmap + (pid >> 5));
      if (a.lengths) plen = __ldg(a.lengths + pid);
    }
  };
  auto step_store = [&](uint32_t q) {
    uint32_t fl = 0;
    uint64_t off = 0;
    if (pin) {
      if (stale) {
        fl = 1u | 12u;
      } else if (pid < 0 || (uint64_t)pid >= a.n_rows || poff == kBadSource) {
        fl = 1u | 4u;
      } else if (poff & 15u) {
        fl = 1u | 8u;
      } else {
        fl = 1u | (((pbm >> (pid & 31)) & 1u) << 1);
        off = poff;
      }
    }
    const uint64_t ri = row_index(32u * q + lane);
    const uint64_t dsto = ordered ? (uint64_t)ppos * a.dst_stride
                          : !kSplit ? ri * a.dst_stride
                                    : (ri / a.group_rows) * a.group_stride +
                                          (ri % a.group_rows) * a.dst_stride;
    // vectors of the first fetch: the raw row, the whole stream when its length
    // is known, else the shortest stream; they ride in the top 12 bits of the
    // output offset's high word (output offsets stay below 2^52)
    const uint32_t nv = (fl & 2u) ? nvec
                        : a.lengths ? min(max((plen + 15u) >> 4, min_vec), nvec) : min_vec;
    rinfo[((q & 1u) << 5) + lane] =
        make_uint4((uint32_t)off | fl, (uint32_t)(off >> 32), (uint32_t)dsto,
                   ((uint32_t)(dsto >> 32) & 0xFFFFFu) | (nv << 20));
  };
  // copy row tt into ring stage tt % S (one commit group, empty past the end);
  // rows of at most 2 KB: four predicated 16-byte copies per lane; larger
  // rows (kBig, up to 8 KB): up to sixteen
  const uint32_t ring_sa = static_cast<uint32_t>(__cvta_generic_to_shared(ring)) + 16u * lane;
  const uint8_t* src_lane = a.src + 16u * lane;
  auto issue = [&](uint32_t tt) {
    if (tt < cnt) {
      const uint4 e = rinfo[tt & 63u];
      const uint32_t fl = e.x & 15u;
      if ((fl & 13u) == 1u) {
        const uint32_t nv = e.w >> 20;
        const uint8_t* src = src_lane + ((((uint64_t)e.y) << 32) | (uint64_t)(e.x & ~15u));
        const uint32_t sa = ring_sa + 4u * (tt % S) * F.sbuf_words;
        // one copy per lane covers a stream of up to 512 bytes (measured: the
        // HBM cache path, 324-byte streams, 3 % faster than four predicated
        // copies per lane; a 64-bit window read of 3 stream words per 4 output
        // words measured 3 % slower than the per-word reads, and 5 CTAs per SM
        // instead of 4 4 % slower)
        if (lane < nv)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(src));
        if (nv > 32u) {  // streams above 512 bytes (and raw rows above 512 bytes)
#pragma unroll
          for (uint32_t j = 1; j < (kBig ? 16u : 4u); ++j)
            if (lane + 32u * j < nv)
              asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(sa + 512u * j),
                           "l"(src + 512u * j));
        }
      }
    }
    cp_async_commit();
  };

  for (uint32_t q = 0; q < 2u; ++q) {
    step_ids(q);
    step_loads();
    step_store(q);
  }
  __syncwarp();
  for (uint32_t t = 0; t + 1u < S; ++t) issue(t);
#pragma unroll 1
  for (uint32_t t = 0; t < cnt; ++t) {
    const uint32_t l = t & 31u;
    if (l == 0u) step_ids((t >> 5) + 2u);
    if (l == 16u) step_loads();
    issue(t + S - 1u);           // S-1 rows stay in flight
    cp_async_wait_n<S - 1>();    // row t has landed
    __syncwarp();
    do {
      const uint4 e = rinfo[t & 63u];
      const uint32_t fl = e.x & 15u;
      if (!(fl & 1u)) break;  // no row here (past the end of the warp's rows)
      uint4* drow = reinterpret_cast<uint4*>(
          a.dst + ((((uint64_t)(e.w & 0xFFFFFu)) << 32) | (uint64_t)e.z));
      uint32_t* sb = ring + (t % S) * F.sbuf_words;
      constexpr bool split = kSplit;
      if (fl & 12u) {
        if (lane == 0)
          set_status(a.status, (fl & 12u) == 12u ? IBP_EINVAL
                               : (fl & 4u)       ? IBP_ERANGE
                                                 : IBP_EALIGN);
        if (split)
          for (uint32_t v = lane; v < nvec; v += 32)
            *split_group(drow, gtab, v, a.chunk_stride) = make_uint4(0, 0, 0, 0);
        else
          zero_row(drow, nvec, lane);
        break;
      }
      if (fl & 2u) {  // raw row
        if (split) {
          for (uint32_t v = lane; v < nvec; v += 32)
            *split_group(drow, gtab, v, a.chunk_stride) = *reinterpret_cast<const uint4*>(sb + 4u * v);
          break;
        }
        uint4* dp = drow + lane;
        for (uint32_t v = lane; v < nvec; v += 32, dp += 32)
          *dp = *reinterpret_cast<const uint4*>(sb + 4u * v);
        break;
      }
      if (!can_pack) {
        if (lane == 0) set_status(a.status, IBP_ECORRUPT);
        if (split)
          for (uint32_t v = lane; v < nvec; v += 32)
            *split_group(drow, gtab, v, a.chunk_stride) = make_uint4(0, 0, 0, 0);
        else
          zero_row(drow, nvec, lane);
        break;
      }
      const bool all_packed = nhw == 1u ? (sb[0] & hexp) == hexp
                                        : __all_sync(kFull, lane >= nhw || (sb[lane] & hexp) == hexp);
      if (all_packed) {
        // every chunk participates: static offsets, no scan
        if (split) {
          for (uint32_t g = lane; g < G; g += 32)
            *split_group(drow, gtab, g, a.chunk_stride) =
                decode_packed_group<kMode>(tab, sb, g, G, nch, 0u, net5, uni, F, uparm);
          break;
        }
        uint4* dp = drow + lane;
        for (uint32_t g = lane; g < G; g += 32, dp += 32)
          *dp = decode_packed_group<kMode>(tab, sb, g, G, nch, 0u, net5, uni, F, uparm);
        break;
      }
      // some chunks are raw: scan the chunk sizes
      uint32_t run = nch;
      for (uint32_t k0 = 0; k0 < nch; k0 += 32) {
        const uint32_t k = k0 + lane;
        uint32_t size = 0, pk = 0;
        if (k < nch) {
          pk = (sb[k >> 5] >> (k & 31u)) & 1u;
          size = pk ? __ldg(a.m.ckeep + k) : 32u * min(wpc, W - k * wpc);
        }
        const uint32_t incl = warp_inclusive_scan(size, lane);
        if (k < nch) cinfo[k] = (run + incl - size) | (pk << 31);
        run += __shfl_sync(kFull, incl, 31);
      }
      const uint32_t words = (run + 31u) >> 5;
      if (4u * words >= R || 4ull * words > a.avail) {
        if (lane == 0) set_status(a.status, IBP_ECORRUPT);
        __syncwarp();
        if (split)
          for (uint32_t v = lane; v < nvec; v += 32)
            *split_group(drow, gtab, v, a.chunk_stride) = make_uint4(0, 0, 0, 0);
        else
          zero_row(drow, nvec, lane);
        break;
      }
      const uint32_t need_vec = (4u * words + 15u) >> 4;
      const uint32_t fetched = e.w >> 20;
      if (need_vec > fetched) {  // the raw chunks made the stream longer: second fetch
        // (every copy issued before any is awaited: one round trip, not one per 512 bytes)
        const uint4* src = reinterpret_cast<const uint4*>(
            a.src + ((((uint64_t)e.y) << 32) | (uint64_t)(e.x & ~15u)));
        fetch_vectors(static_cast<uint32_t>(__cvta_generic_to_shared(sb)), src, fetched,
                      need_vec, lane);
      }
      __syncwarp();
      for (uint32_t g = lane; g < G; g += 32) {
        const uint32_t gd = gtab[g];
        const uint32_t k = gd & 0xFFFFu;
        const uint32_t ci = cinfo[k];
        const uint32_t start = ci & 0x7FFFFFFFu;
        uint4* dp = split ? reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(drow) +
                                                     (uint64_t)k * a.chunk_stride + 4u * (gd >> 16))
                          : drow + g;
        if (ci >> 31) {
          *dp = decode_packed_group<kMode>(tab, sb, g, G, nch, start - cstat[k], net5, uni, F,
                                           uparm);
        } else {
          const uint32_t bit = start + ((gd >> 16) << 5);
          const uint32_t q = bit >> 5;
          *dp = make_uint4(__funnelshift_r(sb[q], sb[q + 1], bit),
                           __funnelshift_r(sb[q + 1], sb[q + 2], bit),
                           __funnelshift_r(sb[q + 2], sb[q + 3], bit),
                           __funnelshift_r(sb[q + 3], sb[q + 4], bit));
        }
      }
    } while (false);
    __syncwarp();  // stage t % S and row info slot t % 64 are refilled later
    if (l == 31u) {
      step_store((t >> 5) + 2u);  // chunk t/32 + 2 takes the slots of chunk t/32
      __syncwarp();
    }
  }
  cp_async_wait_n<0>();
}

// ------------------------------------------------------------------------
// Decompression of a packed cache in row order (ibp_decompress with offsets,
// the source in GPU memory).  The stored bytes of rows r0 .. r0+31 lie back
// to back when their offsets increase (a cache written by ibp_pack), so one
// bulk copy (cp.async.bulk, completing on an mbarrier) brings a tile's bytes
// into a shared-memory stage, and the warps decode its rows from there: no
// per-row copies, commits or waits.  A producer warp fills kTileStages stages
// ahead of kTileWarps decoding warps.  A row whose bytes are not all in the
// stage -- the call's last row (its end is not known), a stream longer than
// the bytes up to the next row's start, every row of a tile whose offsets are
// out of order, not 16-byte aligned, more than R bytes apart, or span more
// than a stage's 16 KB -- is read by its warp from global memory, within its
// own stream as the other decoders read it; the output and status codes are
// those of k_decode_fast.
// ------------------------------------------------------------------------
constexpr uint32_t kTileRows = 32;
constexpr uint32_t kTileStages = 3;  // measured: 2 or 4 stages slower
constexpr uint32_t kTileWarps = 8;  // decoding warps (one more produces); 12 or 16 measured slower

struct TileInfo {
  uint64_t off[kTileRows + 1];  // the rows' starts, then the end of the stage's bytes
  uint32_t nr;                  // rows in the tile
  uint32_t ok;                  // 1: the stage holds [off[0], off[nr])
};

__device__ __forceinline__ bool tile_bar_try(uint32_t a, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(a), "r"(parity)
      : "memory");
  return done != 0u;
}

// Wait for the phase of `parity`, for at most ~2 s.
__device__ __forceinline__ bool tile_bar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  if (tile_bar_try(a, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (true) {
    if (tile_bar_try(a, parity)) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 2000000000ull) return false;
  }
}

// One row from its stream at sb (shared memory, 16-byte aligned), of which
// `have` bytes are valid.  Returns 0 once the row is written (decoded, or
// zero-filled with a status), else the bytes of stream it needs (> have).
template <int kMode>
__device__ __forceinline__ uint32_t tile_row(const DecodeArgs& a, const FastParams& F,
                                             const uint4* tab, const uint32_t* gtab,
                                             const uint32_t* uparm, uint32_t* cinfo,
                                             const uint32_t* sb, uint32_t have, bool raw,
                                             uint4* drow, uint32_t lane, bool can_pack,
                                             bool net5, bool uni) {
  const uint32_t R = a.m.R, W = a.m.W, wpc = a.m.wpc, nch = a.m.nch;
  const uint32_t nvec = R >> 4, G = W >> 2;
  if (raw) {
    if (have < R) return R;
    uint4* dp = drow + lane;
    for (uint32_t v = lane; v < nvec; v += 32, dp += 32)
      *dp = *reinterpret_cast<const uint4*>(sb + 4u * v);
    return 0u;
  }
  if (!can_pack) {
    if (lane == 0) set_status(a.status, IBP_ECORRUPT);
    zero_row(drow, nvec, lane);
    return 0u;
  }
  const uint32_t nhw = (nch + 31u) >> 5;
  if (have < 4u * nhw) return 4u * nhw;
  const uint32_t hexp = (lane + 1u < nhw || (nch & 31u) == 0u) ? 0xFFFFFFFFu
                                                                 : ((1u << (nch & 31u)) - 1u);
  const bool all_packed = nhw == 1u ? (sb[0] & hexp) == hexp
                                    : __all_sync(kFull, lane >= nhw || (sb[lane] & hexp) == hexp);
  if (all_packed) {
    const uint32_t need = 4u * ((F.min_bits + 31u) >> 5);
    if (have < need) return need;
    uint4* dp = drow + lane;
    for (uint32_t g = lane; g < G; g += 32, dp += 32)
      *dp = decode_packed_group<kMode>(tab, sb, g, G, nch, 0u, net5, uni, F, uparm);
    return 0u;
  }
  uint32_t run = nch;
  for (uint32_t k0 = 0; k0 < nch; k0 += 32) {
    const uint32_t k = k0 + lane;
    uint32_t size = 0, pk = 0;
    if (k < nch) {
      pk = (sb[k >> 5] >> (k & 31u)) & 1u;
      size = pk ? __ldg(a.m.ckeep + k) : 32u * min(wpc, W - k * wpc);
    }
    const uint32_t incl = warp_inclusive_scan(size, lane);
    if (k < nch) cinfo[k] = (run + incl - size) | (pk << 31);
    run += __shfl_sync(kFull, incl, 31);
  }
  const uint32_t words = (run + 31u) >> 5;
  if (4u * words >= R || 4ull * words > a.avail) {
    if (lane == 0) set_status(a.status, IBP_ECORRUPT);
    __syncwarp();
    zero_row(drow, nvec, lane);
    return 0u;
  }
  if (have < 4u * words) return 4u * words;
  __syncwarp();
  const uint32_t* cstat = gtab + ((G + 3u) & ~3u);
  for (uint32_t g = lane; g < G; g += 32) {
    const uint32_t gd = gtab[g];
    const uint32_t k = gd & 0xFFFFu;
    const uint32_t ci = cinfo[k];
    const uint32_t start = ci & 0x7FFFFFFFu;
    uint4* dp = drow + g;
    if (ci >> 31) {
      *dp = decode_packed_group<kMode>(tab, sb, g, G, nch, start - cstat[k], net5, uni, F, uparm);
    } else {
      const uint32_t bit = start + ((gd >> 16) << 5);
      const uint32_t q = bit >> 5;
      *dp = make_uint4(__funnelshift_r(sb[q], sb[q + 1], bit),
                       __funnelshift_r(sb[q + 1], sb[q + 2], bit),
                       __funnelshift_r(sb[q + 2], sb[q + 3], bit),
                       __funnelshift_r(sb[q + 3], sb[q + 4], bit));
    }
  }
  return 0u;
}

template <int kMode>
__global__ void __launch_bounds__(32 * (kTileWarps + 1), 3) k_decode_tiles(DecodeArgs a,
                                                                           FastParams F,
                                                                           uint32_t stage_bytes) {
  extern __shared__ __align__(16) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u, wid = threadIdx.x >> 5;
  const uint32_t R = a.m.R, W = a.m.W, nch = a.m.nch;
  const uint32_t nvec = R >> 4, G = W >> 2;
  const uint32_t min_bits = kMode == kModeRuntime ? __ldg(a.m.scal) : F.min_bits;
  const bool net5 = kMode == kModeNet5 || (kMode == kModeRuntime && __ldg(a.m.scal + 1) > 2u);
  const bool uni = kMode == kModeUniform || kMode == kModeUniform1 ||
                   (kMode == kModeRuntime && __ldg(a.m.scal + 3) != 0u);
  const uint32_t min_words = (min_bits + 31u) >> 5;
  const bool can_pack = 4u * min_words < R;
  const uint32_t min_vec = min((4u * min_words + 15u) >> 4, nvec);
  const bool stale = kMode != kModeRuntime && __ldg(a.m.scal + 9) != F.gen;
  FastParams P = F;
  P.min_bits = min_bits;  // the runtime mode reads it on the device
  (void)G;

  uint4* tab = reinterpret_cast<uint4*>(smem);
  uint32_t* gtab = smem + F.table_words;
  uint32_t* uparm = gtab + F.gtab_words;
  TileInfo* info = reinterpret_cast<TileInfo*>(uparm + 8);
  uint64_t* full = reinterpret_cast<uint64_t*>(info + kTileStages);
  uint64_t* empty = full + kTileStages;
  uint32_t* s_fail = reinterpret_cast<uint32_t*>(empty + kTileStages);
  const uint32_t scr_words = W + 16u;
  uint32_t* scratch = s_fail + 4;                         // kTileWarps x scr_words
  uint32_t* cinfo_all = scratch + kTileWarps * scr_words;  // kTileWarps x nch (rounded)
  const uint32_t nch4 = (nch + 3u) & ~3u;
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(cinfo_all + kTileWarps * nch4) + 127u) & ~uintptr_t(127));
  {
    if (F.table_words && !uni) {
      const uint4* t = net5 ? a.t5 : a.t2;
      const uint32_t nv = net5 ? 2u * W : W;
      for (uint32_t v = threadIdx.x; v < nv; v += blockDim.x) tab[v] = __ldg(t + v);
    }
    for (uint32_t g = threadIdx.x; g < F.gtab_words; g += blockDim.x) gtab[g] = __ldg(a.gtab + g);
    if (kMode == kModeRuntime && threadIdx.x < 8) uparm[threadIdx.x] = __ldg(a.m.scal + 4 + threadIdx.x);
    if (threadIdx.x == 0) {
      for (uint32_t st = 0; st < kTileStages; ++st) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(full + st))),
                     "r"(1u)
                     : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(empty + st))),
                     "r"(kTileWarps)
                     : "memory");
      }
      s_fail[0] = 0u;  // a wait gave up
      s_fail[1] = 0u;  // tiles the producer issued
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  __syncthreads();

  const uint64_t ntiles = (a.n + kTileRows - 1) / kTileRows;
  const uint64_t t0 = ntiles * blockIdx.x / gridDim.x;
  const uint32_t cnt = (uint32_t)(ntiles * (blockIdx.x + 1) / gridDim.x - t0);
  const uint64_t cap = (uint64_t)stage_bytes - 64u;  // bytes a stage takes (64 bytes of slack)

  if (wid == kTileWarps) {  // producer
    for (uint32_t k = 0; k < cnt; ++k) {
      const uint32_t s = k % kTileStages, round = k / kTileStages;
      if (round > 0 && !tile_bar_wait(empty + s, (round - 1u) & 1u)) {
        if (lane == 0) atomicExch(s_fail, 1u);
        break;
      }
      if (*reinterpret_cast<volatile uint32_t*>(s_fail)) break;
      const uint64_t r0 = (t0 + k) * kTileRows;
      const uint32_t nr = (uint32_t)min((uint64_t)kTileRows, a.n - r0);
      const bool has_next = r0 + nr < a.n;
      uint64_t o = 0, oe = 0;
      if (lane < nr) o = __ldg(a.offsets + r0 + lane);
      if (lane == 0 && has_next) oe = __ldg(a.offsets + r0 + nr);
      oe = __shfl_sync(kFull, oe, 0);
      const uint64_t base = __shfl_sync(kFull, o, 0);
      const uint64_t last = __shfl_sync(kFull, o, nr - 1u);
      const uint64_t end = has_next ? oe : last;  // the call's last row: its end is unknown
      const uint64_t nxt = __shfl_down_sync(kFull, o, 1);
      // each start 16-byte aligned and at most R bytes before the next: the
      // copy then reads only bytes the decoders may read (R from a row's start)
      const uint64_t to = lane + 1u == nr ? end : nxt;
      const bool in_order = lane >= nr || ((o & 15u) == 0u && o <= to && to - o <= R);
      const bool ok = __all_sync(kFull, in_order) && (end & 15u) == 0u && end - base <= cap;
      TileInfo& ti = info[s];
      if (lane < nr) ti.off[lane] = o;
      if (lane == 0) {
        ti.off[nr] = end;
        ti.nr = nr;
        ti.ok = ok ? 1u : 0u;
      }
      __syncwarp();
      if (t0 + k == a.withhold_tile) continue;  // test hook: this tile is never released
      if (lane == 0) {
        const uint32_t fb = static_cast<uint32_t>(__cvta_generic_to_shared(full + s));
        const uint32_t bytes = ok ? (uint32_t)(end - base) : 0u;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                     "r"(bytes)
                     : "memory");
        if (bytes)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
              "%2, [%3];" ::"r"(static_cast<uint32_t>(
                                  __cvta_generic_to_shared(stages + (size_t)s * stage_bytes))),
              "l"(a.src + base), "r"(bytes), "r"(fb)
              : "memory");
        s_fail[1] = k + 1u;  // tiles issued
      }
    }
  } else {  // decoding warps
    uint32_t* scr = scratch + wid * scr_words;
    uint32_t* cinfo = cinfo_all + wid * nch4;
    static_assert(kTileRows == 32u, "a tile's raw bits are one bitmap word");
    // the raw bits of the tile (rows 32k .. 32k+31: one bitmap word), loaded
    // a tile ahead
    uint32_t bm_next = cnt ? __ldg(a.bitmap + t0) : 0u;
    for (uint32_t k = 0; k < cnt; ++k) {
      const uint32_t s = k % kTileStages;
      const uint32_t bm = bm_next;
      if (k + 1u < cnt) bm_next = __ldg(a.bitmap + t0 + k + 1u);
      if (!tile_bar_wait(full + s, (k / kTileStages) & 1u)) {
        if (lane == 0) atomicExch(s_fail, 1u);
        break;
      }
      if (*reinterpret_cast<volatile uint32_t*>(s_fail)) break;
      const TileInfo& ti = info[s];
      const uint32_t nr = ti.nr;
      const bool ok = ti.ok != 0u;
      const uint64_t base = ti.off[0], end = ti.off[nr];
      const uint32_t* stage = reinterpret_cast<const uint32_t*>(stages + (size_t)s * stage_bytes);
      const uint64_t r0 = (t0 + k) * kTileRows;
      for (uint32_t j = wid; j < nr; j += kTileWarps) {
        const uint64_t i = r0 + j;
        uint4* drow = reinterpret_cast<uint4*>(a.dst + i * a.dst_stride);
        const uint64_t o = ti.off[j];
        if (stale) {
          if (lane == 0) set_status(a.status, IBP_EINVAL);
          zero_row(drow, nvec, lane);
          continue;
        }
        if (o & 15u) {
          if (lane == 0) set_status(a.status, IBP_EALIGN);
          zero_row(drow, nvec, lane);
          continue;
        }
        const bool raw = (bm >> j) & 1u;
        uint32_t need = 0xFFFFFFFFu;
        if (ok) {
          const uint64_t h = end - o;
          need = tile_row<kMode>(a, P, tab, gtab, uparm, cinfo, stage + ((o - base) >> 2),
                                 h > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)h, raw, drow, lane,
                                 can_pack, net5, uni);
        }
        if (need == 0u) continue;
        // from global memory: the first fetch as the other decoders take it
        // (the raw row, the stream's length when a length table is attached,
        // else the shortest stream), then the rest of the stream if it needs it
        const uint4* src = reinterpret_cast<const uint4*>(a.src + o);
        uint4* sv = reinterpret_cast<uint4*>(scr);
        uint32_t nv = raw ? nvec
                          : a.lengths ? min(max((__ldg(a.lengths + i) + 15u) >> 4, min_vec), nvec)
                                      : min_vec;
        __syncwarp();
        for (uint32_t v = lane; v < nv; v += 32) sv[v] = src[v];
        __syncwarp();
        need = tile_row<kMode>(a, P, tab, gtab, uparm, cinfo, scr, 16u * nv, raw, drow, lane,
                               can_pack, net5, uni);
        if (need == 0u) continue;
        const uint32_t nv2 = min((need + 15u) >> 4, nvec);
        for (uint32_t v = nv + lane; v < nv2; v += 32) sv[v] = src[v];
        __syncwarp();
        tile_row<kMode>(a, P, tab, gtab, uparm, cinfo, scr, 16u * nv2, raw, drow, lane, can_pack,
                        net5, uni);
      }
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(empty + s)))
                     : "memory");
    }
  }
  __syncthreads();
  if (*reinterpret_cast<volatile uint32_t*>(s_fail)) {
    // a wait gave up: report it and let the copies in flight land before the
    // CTA's shared memory goes away (each with its own bounded wait)
    if (threadIdx.x == 0) {
      set_status(a.status, IBP_ETIMEOUT);
      // a stage is refilled only after its tile was decoded: the last
      // kTileStages tiles issued are the only copies that can be in flight
      const uint32_t issued = s_fail[1];
      for (uint32_t k = issued > kTileStages ? issued - kTileStages : 0u; k < issued; ++k)
        tile_bar_wait(full + (k % kTileStages), (k / kTileStages) & 1u);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------
// Fused multi-store gather (a batch of lookups into several stores of one
// geometry -- the 26 embedding tables of a DLRM batch -- in one launch, so
// small per-table batches still fill the GPU).  Item i = b*T + t looks up
// ids[i] in store t and lands at dst + b*dst_row_stride + t*R.  The pipeline
// is k_decode_fast's; each row takes its store's parameters from a per-store
// entry staged in shared memory, and stores that are not uniform read their
// decode descriptors from global memory (L1/L2 resident: a few KB each).
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 3) k_gather_group(GroupArgs g) {
  extern __shared__ __align__(16) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t wid = threadIdx.x >> 5;
  const uint32_t R = g.R, W = g.W, wpc = g.wpc, nch = g.nch, T = g.T;
  const uint32_t nvec = R >> 4;
  const uint32_t G = W >> 2;
  const uint32_t G4 = (G + 3u) & ~3u;
  constexpr uint32_t S = kRingStages;
  GroupEntry* ent = reinterpret_cast<GroupEntry*>(smem);
  const uint32_t ent_words = T * (uint32_t)(sizeof(GroupEntry) / 4);
  // stores whose Mask/Bitval changed since the group read their properties
  // (a launch replayed from a CUDA graph): their items report IBP_EINVAL
  __shared__ uint32_t s_stale[IBP_MAX_GROUP_STORES / 32];
  {
    const uint4* src = reinterpret_cast<const uint4*>(g.entries);
    uint4* dstv = reinterpret_cast<uint4*>(smem);
    for (uint32_t v = threadIdx.x; v < ent_words / 4u; v += blockDim.x) dstv[v] = __ldg(src + v);
    if (threadIdx.x < IBP_MAX_GROUP_STORES / 32) s_stale[threadIdx.x] = 0u;
  }
  __syncthreads();
  if (g.plan_stamp) {  // a plan made ahead: for this many items and shares?
    const uint64_t nwarps = (uint64_t)gridDim.x * (blockDim.x >> 5);
    if (__ldg(g.plan_stamp) != kPlanMagic || __ldg(g.plan_stamp + 1) != (uint32_t)g.n_items ||
        __ldg(g.plan_stamp + 2) != (uint32_t)nwarps) {
      if (blockIdx.x == 0 && threadIdx.x == 0) set_status(ent[0].status, IBP_EINVAL);
      return;
    }
  }
  for (uint32_t t = threadIdx.x; t < T; t += blockDim.x)
    if (__ldg(ent[t].scal + 9) != ent[t].gen) atomicOr(&s_stale[t >> 5], 1u << (t & 31u));

  uint32_t* ring = smem + ent_words + wid * g.warp_words;
  uint4* rinfo = reinterpret_cast<uint4*>(ring + S * g.sbuf_words);
  uint32_t* cinfo = ring + S * g.sbuf_words + 256;
  // the warp's last decoded row, kept while the next items repeat it
  uint4* lastrow = reinterpret_cast<uint4*>(cinfo + ((nch + 3u) & ~3u));
  __syncthreads();
  const uint32_t nhw = (nch + 31u) >> 5;
  const uint32_t hexp = (lane + 1u < nhw || (nch & 31u) == 0u) ? 0xFFFFFFFFu
                                                                 : ((1u << (nch & 31u)) - 1u);
  // contiguous item shares: of the sorted list, as cut for an ordered gather
  // (equal numbers of distinct rows), else equal numbers of items
  const uint64_t nw = (uint64_t)gridDim.x * (blockDim.x >> 5);
  const uint64_t gw = (uint64_t)blockIdx.x * (blockDim.x >> 5) + wid;
  const bool ordered = g.order != nullptr;
  // (shares read from a workspace are clamped to the list)
  const uint64_t r0 = g.shares ? min((uint64_t)__ldg(g.shares + gw), g.n_items)
                               : g.n_items * gw / nw;
  const uint64_t r1 = g.shares ? min((uint64_t)__ldg(g.shares + gw + 1), g.n_items)
                               : g.n_items * (gw + 1) / nw;
  const uint32_t cnt = (uint32_t)(r1 > r0 ? r1 - r0 : 0u);
  if (cnt == 0) return;
  auto row_index = [&](uint32_t t) -> uint64_t { return r0 + t; };  // the warp's t-th item

  int64_t pid = 0;
  uint64_t poff = 0, pitem = 0;
  uint32_t pbm = 0, pt = 0, plen = 0;
  bool pin = false, pdup = false;
  // an ordered gather's list has the lookups of one row next to each other
  // (Zipf batches repeat rows): an item that repeats the warp's previous item
  // is not fetched; its row is stored from the warp's copy of the last one
  int64_t carry_id = -1;
  uint32_t carry_t = 0xFFFFFFFFu;
  auto step_ids = [&](uint32_t q) {
    const uint32_t t = 32u * q + lane;
    const uint64_t ri = row_index(t);
    pin = q < (cnt + 31u) / 32u && t < cnt && ri < g.n_items;
    if (pin) {
      pitem = ordered ? (uint64_t)__ldg(g.order + ri) : ri;
      pin = pitem < g.n_items;  // an item of the list, as every plan makes it
    }
    if (pin) {
      pid = __ldg(g.ids + pitem);
      pt = (uint32_t)(pitem % T);
    }
    if (ordered) {
      const int64_t key_id = pin ? pid : -1;
      const uint32_t key_t = pin ? pt : 0xFFFFFFFFu;
      int64_t prev_id = __shfl_up_sync(kFull, key_id, 1);
      uint32_t prev_t = __shfl_up_sync(kFull, key_t, 1);
      if (lane == 0) {
        prev_id = carry_id;
        prev_t = carry_t;
      }
      pdup = pin && key_id >= 0 && prev_t == key_t && prev_id == key_id;
      carry_id = __shfl_sync(kFull, key_id, 31);
      carry_t = __shfl_sync(kFull, key_t, 31);
    }
  };
  auto step_loads = [&]() {
    if (pin && pid >= 0 && (uint64_t)pid < ent[pt].n_rows) {
      poff = (uint64_t)pid * ent[pt].slot;
      pbm = __ldg(ent[pt].bitmap + (pid >> 5));
      if (ent[pt].lengths) plen = __ldg(ent[pt].lengths + pid);
    }
  };
  auto step_store = [&](uint32_t q) {
    uint32_t fl = 0;
    uint64_t off = 0;
    if (pin) {
      if ((s_stale[pt >> 5] >> (pt & 31u)) & 1u) {
        fl = 1u | 12u;
      } else if (pid < 0 || (uint64_t)pid >= ent[pt].n_rows) {
        fl = 1u | 4u;
      } else if (pdup) {
        fl = 7u;  // 1 | 2 | 4: a repeat of the previous item (never a fetch)
      } else {
        fl = 1u | (((pbm >> (pid & 31)) & 1u) << 1);
        off = poff;
      }
    }
    const uint64_t dsto = (pitem / T) * g.dst_row_stride + (uint64_t)pt * R;
    // vectors of the first fetch (the raw row; the whole stream when the store
    // has a length table; else the shortest stream) ride in the top 12 bits of
    // the output offset's high word (output offsets stay below 2^52)
    const GroupEntry& en = ent[pt];
    const uint32_t nv = (fl & 2u) ? nvec
                        : en.lengths ? min(max((plen + 15u) >> 4, en.min_vec), nvec) : en.min_vec;
    rinfo[((q & 1u) << 5) + lane] =
        make_uint4((uint32_t)off | fl, (uint32_t)(off >> 32) | (pt << 24), (uint32_t)dsto,
                   ((uint32_t)(dsto >> 32) & 0xFFFFFu) | (nv << 20));
  };
  const uint32_t ring_sa = static_cast<uint32_t>(__cvta_generic_to_shared(ring)) + 16u * lane;
  auto issue = [&](uint32_t tt) {
    if (tt < cnt) {
      const uint4 e = rinfo[tt & 63u];
      const uint32_t fl = e.x & 15u;
      if ((fl & 13u) == 1u) {
        const GroupEntry& en = ent[e.y >> 24];
        const uint32_t nv = e.w >> 20;
        const uint8_t* src = en.src + 16u * lane +
                             ((((uint64_t)(e.y & 0xFFFFFFu)) << 32) | (uint64_t)(e.x & ~15u));
        const uint32_t sa = ring_sa + 4u * (tt & (S - 1u)) * g.sbuf_words;
#pragma unroll
        for (uint32_t j = 0; j < 4u; ++j)
          if (lane + 32u * j < nv)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(sa + 512u * j),
                         "l"(src + 512u * j));
      }
    }
    cp_async_commit();
  };

  for (uint32_t q = 0; q < 2u; ++q) {
    step_ids(q);
    step_loads();
    step_store(q);
  }
  __syncwarp();
  for (uint32_t t = 0; t + 1u < S; ++t) issue(t);
#pragma unroll 1
  for (uint32_t t = 0; t < cnt; ++t) {
    const uint32_t l = t & 31u;
    if (l == 0u) step_ids((t >> 5) + 2u);
    if (l == 16u) step_loads();
    issue(t + S - 1u);
    cp_async_wait_n<S - 1>();
    __syncwarp();
    do {
      const uint4 e = rinfo[t & 63u];
      const uint32_t fl = e.x & 15u;
      if (!(fl & 1u)) break;  // no row here (past the end of the warp's rows)
      const GroupEntry& en = ent[e.y >> 24];
      uint4* drow = reinterpret_cast<uint4*>(
          g.dst + ((((uint64_t)(e.w & 0xFFFFFu)) << 32) | (uint64_t)e.z));
      uint32_t* sb = ring + (t & (S - 1u)) * g.sbuf_words;
      if (fl == 7u) {  // a repeat: the row this warp decoded last (each lane its own groups)
        for (uint32_t v = lane; v < nvec; v += 32) drow[v] = lastrow[v];
        break;
      }
      // the next item repeats this one: keep the row (set only in an ordered
      // gather, where the item after a repeat's first lookup is flagged)
      const bool keep = t + 1u < cnt && (rinfo[(t + 1u) & 63u].x & 15u) == 7u;
      if (fl & 12u) {
        if (lane == 0) set_status(en.status, (fl & 12u) == 12u ? IBP_EINVAL : IBP_ERANGE);
        zero_row(drow, nvec, lane);
        if (keep) zero_row(lastrow, nvec, lane);
        break;
      }
      if (fl & 2u) {
        uint4* dp = drow + lane;
        for (uint32_t v = lane; v < nvec; v += 32, dp += 32) {
          const uint4 x = *reinterpret_cast<const uint4*>(sb + 4u * v);
          *dp = x;
          if (keep) lastrow[v] = x;
        }
        break;
      }
      if (!en.can_pack) {
        if (lane == 0) set_status(en.status, IBP_ECORRUPT);
        zero_row(drow, nvec, lane);
        if (keep) zero_row(lastrow, nvec, lane);
        break;
      }
      const uint32_t mode = en.mode;
      const bool uni = mode == (uint32_t)kModeUniform || mode == (uint32_t)kModeUniform1;
      const bool net5 = mode == (uint32_t)kModeNet5;
      const bool all_packed = nhw == 1u ? (sb[0] & hexp) == hexp
                                        : __all_sync(kFull, lane >= nhw || (sb[lane] & hexp) == hexp);
      uint32_t words = 0;
      if (!all_packed) {
        uint32_t run = nch;
        for (uint32_t k0 = 0; k0 < nch; k0 += 32) {
          const uint32_t k = k0 + lane;
          uint32_t size = 0, pk = 0;
          if (k < nch) {
            pk = (sb[k >> 5] >> (k & 31u)) & 1u;
            size = pk ? __ldg(en.ckeep + k) : 32u * min(wpc, W - k * wpc);
          }
          const uint32_t incl = warp_inclusive_scan(size, lane);
          if (k < nch) cinfo[k] = (run + incl - size) | (pk << 31);
          run += __shfl_sync(kFull, incl, 31);
        }
        words = (run + 31u) >> 5;
        if (4u * words >= R || 4ull * words > en.slot) {
          if (lane == 0) set_status(en.status, IBP_ECORRUPT);
          __syncwarp();
          zero_row(drow, nvec, lane);
          if (keep) zero_row(lastrow, nvec, lane);
          break;
        }
        const uint32_t need_vec = (4u * words + 15u) >> 4;
        const uint32_t fetched = e.w >> 20;
        if (need_vec > fetched) {  // the raw chunks made the stream longer: second fetch
          const uint4* src = reinterpret_cast<const uint4*>(
              en.src + ((((uint64_t)(e.y & 0xFFFFFFu)) << 32) | (uint64_t)(e.x & ~15u)));
          fetch_vectors(static_cast<uint32_t>(__cvta_generic_to_shared(sb)), src, fetched,
                        need_vec, lane);
        }
        __syncwarp();
      }
      const uint32_t* cstat = en.gtab + G4;
      uint4* dp = drow + lane;
      for (uint32_t gi = lane; gi < G; gi += 32, dp += 32) {
        uint32_t delta = 0;
        bool packed = true;
        uint32_t start = 0, gd = 0;
        if (!all_packed) {
          gd = __ldg(en.gtab + gi);
          const uint32_t k = gd & 0xFFFFu;
          const uint32_t ci = cinfo[k];
          start = ci & 0x7FFFFFFFu;
          packed = (ci >> 31) != 0u;
          delta = start - __ldg(cstat + k);
        }
        uint4 val;
        if (!packed) {
          const uint32_t bit = start + ((gd >> 16) << 5);
          const uint32_t q = bit >> 5;
          val = make_uint4(__funnelshift_r(sb[q], sb[q + 1], bit), __funnelshift_r(sb[q + 1], sb[q + 2], bit),
                           __funnelshift_r(sb[q + 2], sb[q + 3], bit), __funnelshift_r(sb[q + 3], sb[q + 4], bit));
        } else if (uni) {
          uint32_t bit = nch + 4u * gi * en.ukeep + delta;
          uint32_t o[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const uint32_t q = bit >> 5;
            const uint32_t v = __funnelshift_r(sb[q], sb[q + 1], bit);
            o[x] = ((v << (en.ush & 31u)) & en.um0) | ((v << (en.ush >> 8)) & en.um1) | en.ubv;
            bit += en.ukeep;
          }
          val = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          val = decode_group(en.tab, sb, gi, G, delta, net5);
        }
        *dp = val;
        if (keep) lastrow[gi] = val;
      }
    } while (false);
    __syncwarp();
    if (l == 31u) {
      step_store((t >> 5) + 2u);
      __syncwarp();
    }
  }
  cp_async_wait_n<0>();
}

// ------------------------------------------------------------------------
// Compression (Core Algorithm > Compression).  One warp per row (a warp
// takes 32 consecutive rows at a time): stage the row in shared memory, flag
// chunks with a Mask mismatch, decide the participation bits, scan the chunk
// sizes, then every lane gathers the kept bits of its words (or takes the
// whole word of a raw chunk) and ORs them into the packed buffer at their
// stream offset with shared-memory atomics.  A row that would not shrink is
// written raw and flagged in the bitmap.
// ------------------------------------------------------------------------
// kUni: a uniform store (every word has the same ~Mask, at most two runs,
// and the same Bitval, known on the host): the match test and the bit gather
// take their masks and shifts from the launch parameters.
constexpr uint32_t kEncodeStages = 4;  // rows per warp ring (rows up to 2 KB)

// kVpl: 16-byte vectors per lane of a row staged in the ring (1, 2 or 4:
// rows up to 512 B, 1 KB, 2 KB); 0: larger rows, loaded when their turn comes.
template <bool kUni, int kVpl>
__global__ void __launch_bounds__(256, 3) k_encode(EncodeArgs a, WarpSmem L) {
  extern __shared__ __align__(16) uint32_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t wid = threadIdx.x >> 5;
  uint32_t* obuf = smem + wid * L.total_words;
  uint32_t* cinfo = obuf + L.sbuf_words;
  uint32_t* rows = cinfo + L.cinfo_words;  // kEncodeStages rows (ring), or one row
  const uint32_t R = a.m.R, W = a.m.W, wpc = a.m.wpc, nch = a.m.nch;
  const uint32_t nvec = R >> 4;
  const uint64_t wpb = blockDim.x >> 5;
  const uint64_t stride = (uint64_t)gridDim.x * wpb;
  // the uniform parameters were fixed on the host for one generation of the
  // store's tables; a launch replayed (from a CUDA graph) after the Mask/Bitval
  // changed writes nothing and reports IBP_EINVAL
  if (kUni && __ldg(a.m.scal + 9) != a.gen) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(a.status, IBP_EINVAL);
    return;
  }

  // A warp takes rpc consecutive rows at a time: 32 for large batches with
  // identity slots (the warp owns one raw-bitmap word and writes it once,
  // instead of 32 warps contending on it with atomics), else 1 (small batches
  // spread over many warps).  Rows up to 2 KB travel by cp.async into a ring
  // of 4 single-row stages, 3 rows ahead of the row being packed; larger rows
  // are fetched when their turn comes, every copy issued before any is awaited.
  constexpr bool use_ring = kVpl > 0;
  constexpr uint32_t S = kEncodeStages;
  const uint32_t lg = a.chunk_lg, rpc = 1u << lg;
  const bool word_owner = lg == 5u && a.slot_ids == nullptr;
  const uint64_t nchunk = (a.n + rpc - 1) >> lg;
  const uint64_t c0 = (uint64_t)blockIdx.x * wpb + wid;
  const uint32_t ring_sa = static_cast<uint32_t>(__cvta_generic_to_shared(rows)) + 16u * lane;
  auto issue = [&](uint64_t r, uint32_t stage) {  // row r into ring stage `stage`
    if (use_ring && r < a.n) {
      const uint8_t* src = a.src + r * a.src_stride + 16u * lane;
      const uint32_t sa = ring_sa + 4u * stage * W;
#pragma unroll
      for (int q = 0; q < kVpl; ++q)
        if (lane + 32u * q < nvec)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(sa + 512u * q),
                       "l"(src + 512u * q));
    }
    cp_async_commit();
  };
  // the warp's rows in order: chunk c0, c0 + stride, ... of rpc rows each
  auto row_at = [&](uint64_t c, uint32_t p) {  // p rows after the start of chunk c
    return ((c + (uint64_t)(p >> lg) * stride) << lg) + (p & (rpc - 1u));
  };
  for (uint32_t t = 0; t + 1 < S; ++t) issue(row_at(c0, t), t);

  uint64_t t = 0;  // the warp's row counter
  for (uint64_t c = c0; c < nchunk; c += stride) {
    uint32_t rawmask = 0, donemask = 0;
#pragma unroll 1
    for (uint32_t j = 0; j < rpc; ++j, ++t) {
      const uint64_t i = (c << lg) + j;
      if (i >= a.n) break;
      // the row S-1 ahead: later in this chunk or in one of the warp's next ones
      issue(j + S - 1u < rpc ? i + S - 1u : row_at(c, j + S - 1u), (uint32_t)((t + S - 1u) % S));
      cp_async_wait_n<S - 1>();  // row t has landed
      __syncwarp();
      uint32_t* xbuf = use_ring ? rows + (uint32_t)(t % S) * W : rows;
      const int64_t slot = a.slot_ids ? __ldg(a.slot_ids + i) : (int64_t)i;
      if (slot < 0 || (uint64_t)slot >= a.n_rows) {
        if (lane == 0) set_status(a.status, IBP_ERANGE);
        if (a.stored_out && lane == 0) a.stored_out[i] = 0;
        __syncwarp();
        continue;
      }
      uint4* dslot = reinterpret_cast<uint4*>(a.dst + (uint64_t)slot * a.slot);
      bool raw = false, done = false;
      uint32_t words = 0;
      if (kUni && use_ring) {
        // Uniform store: when no word misses the Mask every chunk participates
        // and word w's kept bits go to nch + w*keep; when the row is one chunk
        // and some word misses, the row is raw.  Other rows take the general
        // path below.
        uint4 cur[kVpl > 0 ? kVpl : 1];
        const uint32_t msk = ~(a.um0 | a.um1);
        uint32_t diff = 0;
#pragma unroll
        for (int q = 0; q < kVpl; ++q) {
          if (lane + 32u * q < nvec) {
            cur[q] = *reinterpret_cast<const uint4*>(xbuf + 4u * (lane + 32u * q));
            diff |= ((cur[q].x & msk) ^ a.ubv) | ((cur[q].y & msk) ^ a.ubv) |
                    ((cur[q].z & msk) ^ a.ubv) | ((cur[q].w & msk) ^ a.ubv);
          }
        }
        const bool mis = __any_sync(kFull, diff != 0u);
        if (a.ukeep >= 32u || (mis && nch == 1u)) {
          raw = done = true;
        } else if (!mis) {
          words = (nch + W * a.ukeep + 31u) >> 5;
          raw = 4u * words >= R;
          done = true;
        }
        if (done && raw) {
#pragma unroll
          for (int q = 0; q < kVpl; ++q)
            if (lane + 32u * q < nvec) dslot[lane + 32u * q] = cur[q];
        } else if (done) {
          const uint32_t padded = (words + 3u) & ~3u;
          const uint32_t hw = nch >> 5;  // header: nch one bits from bit 0
          for (uint32_t z = lane; z < padded; z += 32)
            obuf[z] = z < hw ? 0xFFFFFFFFu : (z == hw ? (1u << (nch & 31u)) - 1u : 0u);
          __syncwarp();
          if (a.ukeep) {
#pragma unroll
            for (int q = 0; q < kVpl; ++q) {
              if (lane + 32u * q < nvec) {
                const uint32_t xs[4] = {cur[q].x, cur[q].y, cur[q].z, cur[q].w};
                uint32_t bit = nch + 4u * (lane + 32u * q) * a.ukeep;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const uint32_t v = ((xs[e] & a.um0) >> (a.ush & 31u)) |
                                     ((xs[e] & a.um1) >> (a.ush >> 8));
                  const uint32_t qw = bit >> 5, sh = bit & 31u;
                  atomicOr(obuf + qw, v << sh);
                  if (sh != 0u && sh + a.ukeep > 32u) atomicOr(obuf + qw + 1, v >> (32u - sh));
                  bit += a.ukeep;
                }
              }
            }
          }
          __syncwarp();
          for (uint32_t v = lane; 4u * v < padded; v += 32)
            dslot[v] = *reinterpret_cast<const uint4*>(obuf + 4u * v);
        }
      }
      if (!done) {
        if (!use_ring)
          fetch_vectors(static_cast<uint32_t>(__cvta_generic_to_shared(xbuf)),
                        reinterpret_cast<const uint4*>(a.src + i * a.src_stride), 0u, nvec, lane);
        for (uint32_t k = lane; k < nch; k += 32) cinfo[k] = 0;
        __syncwarp();
        // chunks of whole 4-word groups: the work goes by 16-byte groups (one
        // table entry per group, 4 words' loads in flight together)
        const bool by_group = (wpc & 3u) == 0u;
        const uint32_t G = W >> 2;
        if (by_group) {
          const uint32_t msk = ~(a.um0 | a.um1);
          for (uint32_t g = lane; g < G; g += 32) {
            const uint4 x4 = *reinterpret_cast<const uint4*>(xbuf + 4u * g);
            uint32_t d;
            if (kUni) {
              d = ((x4.x & msk) ^ a.ubv) | ((x4.y & msk) ^ a.ubv) | ((x4.z & msk) ^ a.ubv) |
                  ((x4.w & msk) ^ a.ubv);
            } else {
              const uint4 m4 = __ldg(reinterpret_cast<const uint4*>(a.m.mask) + g);
              const uint4 b4 = __ldg(reinterpret_cast<const uint4*>(a.m.bitval) + g);
              d = ((x4.x & m4.x) ^ b4.x) | ((x4.y & m4.y) ^ b4.y) | ((x4.z & m4.z) ^ b4.z) |
                  ((x4.w & m4.w) ^ b4.w);
            }
            if (d) cinfo[__ldg(a.gtab + g) & 0xFFFFu] = 1u;  // mismatch flag
          }
        } else if (kUni) {
          const uint32_t msk = ~(a.um0 | a.um1);
          for (uint32_t w = lane; w < W; w += 32)
            if ((xbuf[w] & msk) != a.ubv) cinfo[__ldg(a.m.kr + w) & 0xFFFFu] = 1u;  // mismatch flag
        } else {
          for (uint32_t w = lane; w < W; w += 32)
            if ((xbuf[w] & __ldg(a.m.mask + w)) != __ldg(a.m.bitval + w))
              cinfo[__ldg(a.m.kr + w) & 0xFFFFu] = 1u;  // mismatch flag
        }
        __syncwarp();
        uint32_t run = nch;
        for (uint32_t k0 = 0; k0 < nch; k0 += 32) {
          const uint32_t k = k0 + lane;
          uint32_t size = 0, p = 0;
          if (k < nch) {
            const uint32_t full = 32u * min(wpc, W - k * wpc);
            const uint32_t keep = __ldg(a.m.ckeep + k);
            p = (cinfo[k] == 0u && keep < full) ? 1u : 0u;
            size = p ? keep : full;
          }
          const uint32_t incl = warp_inclusive_scan(size, lane);
          __syncwarp();
          if (k < nch) cinfo[k] = (run + incl - size) | (p << 31);
          run += __shfl_sync(kFull, incl, 31);
        }
        words = (run + 31u) >> 5;
        raw = 4u * words >= R;
        if (raw) {
          for (uint32_t v = lane; v < nvec; v += 32)
            dslot[v] = *reinterpret_cast<const uint4*>(xbuf + 4u * v);
        } else {
          const uint32_t padded = (words + 3u) & ~3u;
          for (uint32_t z = lane; z < padded + 4u; z += 32) obuf[z] = 0;
          __syncwarp();
          for (uint32_t k = lane; k < nch; k += 32)
            if (cinfo[k] >> 31) atomicOr(obuf + (k >> 5), 1u << (k & 31u));
          auto put = [&](uint32_t v, uint32_t bit, uint32_t nbits) {
            const uint32_t q = bit >> 5, sh = bit & 31u;
            atomicOr(obuf + q, v << sh);
            if (sh != 0u && sh + nbits > 32u) atomicOr(obuf + q + 1, v >> (32u - sh));
          };
          const uint32_t G4 = (G + 3u) & ~3u;
          for (uint32_t g = lane; by_group && g < G; g += 32) {
            const uint32_t gd = __ldg(a.gtab + g);
            const uint32_t k = gd & 0xFFFFu;
            const uint32_t ci = cinfo[k];
            const uint32_t start = ci & 0x7FFFFFFFu;
            const uint4 x4 = *reinterpret_cast<const uint4*>(xbuf + 4u * g);
            const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w};
            if (ci >> 31) {  // packed chunk: word w's kept bits at its all-packed offset + delta
              const uint32_t delta = start - __ldg(a.gtab + G4 + k);
              if (kUni) {
                uint32_t bit = start + (gd >> 16) * a.ukeep;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const uint32_t v = ((xs[e] & a.um0) >> (a.ush & 31u)) |
                                     ((xs[e] & a.um1) >> (a.ush >> 8));
                  if (a.ukeep) put(v, bit, a.ukeep);
                  bit += a.ukeep;
                }
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const uint4 t0 = __ldg(a.t5 + (2u * (uint32_t)e) * G + g);
                  const uint4 t1 = __ldg(a.t5 + (2u * (uint32_t)e + 1u) * G + g);
                  uint32_t x = xs[e] & t1.y;  // the kept bits, gathered to the low end
                  uint32_t t = x & t0.x;
                  x = (x ^ t) | (t >> 1);
                  t = x & t0.y;
                  x = (x ^ t) | (t >> 2);
                  t = x & t0.z;
                  x = (x ^ t) | (t >> 4);
                  t = x & t0.w;
                  x = (x ^ t) | (t >> 8);
                  t = x & t1.x;
                  x = (x ^ t) | (t >> 16);
                  const uint32_t nb = __popc(t1.y);
                  if (nb) put(x, t1.w + delta, nb);
                }
              }
            } else {  // raw chunk: the 4 words verbatim
              uint32_t bit = start + ((gd >> 16) << 5);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                put(xs[e], bit, 32u);
                bit += 32u;
              }
            }
          }
          for (uint32_t w = lane; !by_group && w < W; w += 32) {
            const uint32_t krw = __ldg(a.m.kr + w);  // chunk | word in chunk << 16
            const uint32_t ci = cinfo[krw & 0xFFFFu];
            const bool packed = (ci >> 31) != 0u;
            uint32_t v = xbuf[w];
            uint32_t nbits = 32;
            uint32_t bit;
            if (kUni) {
              bit = (ci & 0x7FFFFFFFu) + (krw >> 16) * (packed ? a.ukeep : 32u);
              if (packed) {
                v = ((v & a.um0) >> (a.ush & 31u)) | ((v & a.um1) >> (a.ush >> 8));
                nbits = a.ukeep;
              }
            } else {
              bit = (ci & 0x7FFFFFFFu) + (packed ? __ldg(a.m.pre + w) : ((krw >> 16) << 5));
              if (packed) {
                const uint32_t keepm = __ldg(a.m.nm + w);
                v = gather_bits(v & keepm, a.m.mv, W, w);
                nbits = __popc(keepm);
              }
            }
            if (nbits) {
              const uint32_t q = bit >> 5, sh = bit & 31u;
              atomicOr(obuf + q, v << sh);
              if (sh != 0u && sh + nbits > 32u) atomicOr(obuf + q + 1, v >> (32u - sh));
            }
          }
          __syncwarp();
          for (uint32_t v = lane; 4u * v < padded; v += 32)
            dslot[v] = *reinterpret_cast<const uint4*>(obuf + 4u * v);
        }
      }
      if (!word_owner) {
        if (lane == 0) {
          const uint32_t bitm = 1u << ((uint64_t)slot & 31u);
          if (raw)
            atomicOr(a.bitmap + ((uint64_t)slot >> 5), bitm);
          else
            atomicAnd(a.bitmap + ((uint64_t)slot >> 5), ~bitm);
        }
      } else {
        rawmask |= (uint32_t)raw << j;
        donemask |= 1u << j;
      }
      if (lane == 0 && a.stored_out) a.stored_out[i] = raw ? R : 4u * words;
      __syncwarp();
    }
    if (word_owner && lane == 0 && donemask) {
      if (donemask == 0xFFFFFFFFu) {
        a.bitmap[c] = rawmask;  // this warp wrote every row of the word
      } else {
        atomicOr(a.bitmap + c, rawmask);
        atomicAnd(a.bitmap + c, rawmask | ~donemask);
      }
    }
  }
  cp_async_wait_n<0>();
}

// ------------------------------------------------------------------------
// Compression of rows above 2 KB, one CTA per row: the CTA's threads stage
// the row in shared memory together and split its 16-byte groups between
// them for the mismatch test and the packing, so a row costs a few memory
// round trips instead of one warp walking 4-32 KB alone (a decode step's
// handful of 8 KB K/V rows took ~25 us per call that way).  Same steps and
// output as k_encode.
// ------------------------------------------------------------------------
template <bool kUni>
__global__ void __launch_bounds__(256) k_encode_rows(EncodeArgs a) {
  extern __shared__ __align__(16) uint32_t smem[];
  __shared__ uint32_t s_words;
  const uint32_t R = a.m.R, W = a.m.W, wpc = a.m.wpc, nch = a.m.nch;
  const uint32_t nvec = R >> 4, G = W >> 2;
  const uint32_t tid = threadIdx.x, T = blockDim.x, lane = tid & 31u, wid = tid >> 5;
  uint32_t* xbuf = smem;           // the row: W words
  uint32_t* obuf = xbuf + W;       // the packed stream: W + 8 words
  uint32_t* cinfo = obuf + W + 8;  // per chunk: mismatch flag, then start | p << 31
  // uniform parameters fixed on the host for an older Mask/Bitval (a launch
  // replayed from a CUDA graph): write nothing, report IBP_EINVAL
  if (kUni && __ldg(a.m.scal + 9) != a.gen) {
    if (tid == 0 && blockIdx.x == 0) set_status(a.status, IBP_EINVAL);
    return;
  }
  const bool by_group = (wpc & 3u) == 0u;
  const uint32_t msk = ~(a.um0 | a.um1);
  const uint32_t G4 = (G + 3u) & ~3u;
  const uint32_t xs_sa = static_cast<uint32_t>(__cvta_generic_to_shared(xbuf));
  auto put = [&](uint32_t v, uint32_t bit, uint32_t nbits) {
    const uint32_t q = bit >> 5, sh = bit & 31u;
    atomicOr(obuf + q, v << sh);
    if (sh != 0u && sh + nbits > 32u) atomicOr(obuf + q + 1, v >> (32u - sh));
  };
  for (uint64_t i = blockIdx.x; i < a.n; i += gridDim.x) {
    const int64_t slot = a.slot_ids ? __ldg(a.slot_ids + i) : (int64_t)i;
    if (slot < 0 || (uint64_t)slot >= a.n_rows) {  // the same for every thread
      if (tid == 0) {
        set_status(a.status, IBP_ERANGE);
        if (a.stored_out) a.stored_out[i] = 0;
      }
      continue;
    }
    const uint8_t* src = a.src + i * a.src_stride;
    for (uint32_t v = tid; v < nvec; v += T)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(xs_sa + 16u * v),
                   "l"(src + 16u * v));
    cp_async_commit();
    for (uint32_t k = tid; k < nch; k += T) cinfo[k] = 0;
    cp_async_wait_n<0>();
    __syncthreads();
    // chunks with a Mask mismatch
    if (by_group) {
      for (uint32_t g = tid; g < G; g += T) {
        const uint4 x4 = *reinterpret_cast<const uint4*>(xbuf + 4u * g);
        uint32_t d;
        if (kUni) {
          d = ((x4.x & msk) ^ a.ubv) | ((x4.y & msk) ^ a.ubv) | ((x4.z & msk) ^ a.ubv) |
              ((x4.w & msk) ^ a.ubv);
        } else {
          const uint4 m4 = __ldg(reinterpret_cast<const uint4*>(a.m.mask) + g);
          const uint4 b4 = __ldg(reinterpret_cast<const uint4*>(a.m.bitval) + g);
          d = ((x4.x & m4.x) ^ b4.x) | ((x4.y & m4.y) ^ b4.y) | ((x4.z & m4.z) ^ b4.z) |
              ((x4.w & m4.w) ^ b4.w);
        }
        if (d) cinfo[__ldg(a.gtab + g) & 0xFFFFu] = 1u;
      }
    } else {
      for (uint32_t w = tid; w < W; w += T) {
        const uint32_t m = kUni ? msk : __ldg(a.m.mask + w);
        const uint32_t b = kUni ? a.ubv : __ldg(a.m.bitval + w);
        if ((xbuf[w] & m) != b) cinfo[__ldg(a.m.kr + w) & 0xFFFFu] = 1u;
      }
    }
    __syncthreads();
    if (wid == 0) {  // participation, chunk sizes -> starts, stream words
      uint32_t run = nch;
      for (uint32_t k0 = 0; k0 < nch; k0 += 32) {
        const uint32_t k = k0 + lane;
        uint32_t size = 0, p = 0;
        if (k < nch) {
          const uint32_t full = 32u * min(wpc, W - k * wpc);
          const uint32_t keep = __ldg(a.m.ckeep + k);
          p = (cinfo[k] == 0u && keep < full) ? 1u : 0u;
          size = p ? keep : full;
        }
        const uint32_t incl = warp_inclusive_scan(size, lane);
        if (k < nch) cinfo[k] = (run + incl - size) | (p << 31);
        run += __shfl_sync(kFull, incl, 31);
      }
      if (lane == 0) s_words = (run + 31u) >> 5;
    }
    __syncthreads();
    const uint32_t words = s_words;
    const bool raw = 4u * words >= R;
    uint4* dslot = reinterpret_cast<uint4*>(a.dst + (uint64_t)slot * a.slot);
    if (raw) {
      for (uint32_t v = tid; v < nvec; v += T)
        dslot[v] = *reinterpret_cast<const uint4*>(xbuf + 4u * v);
    } else {
      const uint32_t padded = (words + 3u) & ~3u;
      for (uint32_t z = tid; z < padded + 4u; z += T) obuf[z] = 0;
      __syncthreads();
      for (uint32_t k = tid; k < nch; k += T)
        if (cinfo[k] >> 31) atomicOr(obuf + (k >> 5), 1u << (k & 31u));
      for (uint32_t g = tid; by_group && g < G; g += T) {
        const uint32_t gd = __ldg(a.gtab + g);
        const uint32_t k = gd & 0xFFFFu;
        const uint32_t ci = cinfo[k];
        const uint32_t start = ci & 0x7FFFFFFFu;
        const uint4 x4 = *reinterpret_cast<const uint4*>(xbuf + 4u * g);
        const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w};
        if (ci >> 31) {  // packed chunk: word w's kept bits at its all-packed offset + delta
          if (kUni) {
            uint32_t bit = start + (gd >> 16) * a.ukeep;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t v = ((xs[e] & a.um0) >> (a.ush & 31u)) |
                                 ((xs[e] & a.um1) >> (a.ush >> 8));
              if (a.ukeep) put(v, bit, a.ukeep);
              bit += a.ukeep;
            }
          } else {
            const uint32_t delta = start - __ldg(a.gtab + G4 + k);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint4 t0 = __ldg(a.t5 + (2u * (uint32_t)e) * G + g);
              const uint4 t1 = __ldg(a.t5 + (2u * (uint32_t)e + 1u) * G + g);
              uint32_t x = xs[e] & t1.y;  // the kept bits, gathered to the low end
              uint32_t t = x & t0.x;
              x = (x ^ t) | (t >> 1);
              t = x & t0.y;
              x = (x ^ t) | (t >> 2);
              t = x & t0.z;
              x = (x ^ t) | (t >> 4);
              t = x & t0.w;
              x = (x ^ t) | (t >> 8);
              t = x & t1.x;
              x = (x ^ t) | (t >> 16);
              const uint32_t nb = __popc(t1.y);
              if (nb) put(x, t1.w + delta, nb);
            }
          }
        } else {  // raw chunk: the 4 words verbatim
          uint32_t bit = start + ((gd >> 16) << 5);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            put(xs[e], bit, 32u);
            bit += 32u;
          }
        }
      }
      for (uint32_t w = tid; !by_group && w < W; w += T) {
        const uint32_t krw = __ldg(a.m.kr + w);  // chunk | word in chunk << 16
        const uint32_t ci = cinfo[krw & 0xFFFFu];
        const bool packed = (ci >> 31) != 0u;
        uint32_t v = xbuf[w];
        uint32_t nbits = 32;
        uint32_t bit;
        if (kUni) {
          bit = (ci & 0x7FFFFFFFu) + (krw >> 16) * (packed ? a.ukeep : 32u);
          if (packed) {
            v = ((v & a.um0) >> (a.ush & 31u)) | ((v & a.um1) >> (a.ush >> 8));
            nbits = a.ukeep;
          }
        } else {
          bit = (ci & 0x7FFFFFFFu) + (packed ? __ldg(a.m.pre + w) : ((krw >> 16) << 5));
          if (packed) {
            const uint32_t keepm = __ldg(a.m.nm + w);
            v = gather_bits(v & keepm, a.m.mv, W, w);
            nbits = __popc(keepm);
          }
        }
        if (nbits) put(v, bit, nbits);
      }
      __syncthreads();
      for (uint32_t v = tid; 4u * v < padded; v += T)
        dslot[v] = *reinterpret_cast<const uint4*>(obuf + 4u * v);
    }
    if (tid == 0) {
      const uint32_t bitm = 1u << ((uint64_t)slot & 31u);
      if (raw)
        atomicOr(a.bitmap + ((uint64_t)slot >> 5), bitm);
      else
        atomicAnd(a.bitmap + ((uint64_t)slot >> 5), ~bitm);
      if (a.stored_out) a.stored_out[i] = raw ? R : 4u * words;
    }
    __syncthreads();  // the buffers are refilled for the next row
  }
}

// ------------------------------------------------------------------------
// Aligned zero-copy copy (the review's GPU aligned transfer): consecutive
// lanes take consecutive 16-byte vectors, so every warp load covers four
// whole 128-byte lines; eight loads per thread are in flight before the
// first store.
// ------------------------------------------------------------------------
__global__ void __launch_bounds__(512) k_link_copy(uint4* __restrict__ dst,
                                                   const uint4* __restrict__ src,
                                                   uint64_t nvec) {
  const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t T = (uint64_t)gridDim.x * blockDim.x;
  uint64_t v = t;
  for (; v + 7 * T < nvec; v += 8 * T) {
    uint4 r[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) r[u] = ld_nc_v4(src + v + (uint64_t)u * T);
#pragma unroll
    for (int u = 0; u < 8; ++u) dst[v + (uint64_t)u * T] = r[u];
  }
  for (; v < nvec; v += T) dst[v] = ld_nc_v4(src + v);
}

__global__ void __launch_bounds__(256) k_gather_copy(uint8_t* dst, const uint8_t* src,
                                                     uint64_t slot, uint32_t row_bytes,
                                                     const int64_t* ids, uint64_t n,
                                                     uint64_t n_rows) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t wpb = blockDim.x >> 5;
  const uint32_t nvec = row_bytes >> 4;
  for (uint64_t i = (uint64_t)blockIdx.x * wpb + (threadIdx.x >> 5); i < n;
       i += (uint64_t)gridDim.x * wpb) {
    const int64_t id = __ldg(ids + i);
    uint4* d = reinterpret_cast<uint4*>(dst + i * row_bytes);
    if (id < 0 || (uint64_t)id >= n_rows) {
      zero_row(d, nvec, lane);
      continue;
    }
    const uint4* s = reinterpret_cast<const uint4*>(src + (uint64_t)id * slot);
    for (uint32_t v = lane; v < nvec; v += 32) d[v] = ld_nc_v4(s + v);
  }
}

// Packed-cache offsets: exclusive scan of roundup(stored, 16), in tiles of
// 8192 rows.  (1) each tile's sum is parked in offsets[first row of the next
// tile] (offsets[n] for the last tile); (2) one block turns those sums into
// tile bases in place and writes the total to offsets[n]; (3) each tile scans
// its rows from its base, one warp per 1024 rows, 32 at a time with a
// shuffle scan (coalesced reads and writes).  The slots that (1) and (2) use
// are rewritten by (3) with the same value, so the tiles never race.
constexpr uint32_t kPackTile = 8192;

__device__ __forceinline__ uint64_t pack_len(const uint32_t* stored, uint64_t i) {
  return (__ldg(stored + i) + 15u) & ~15u;
}

__global__ void __launch_bounds__(256) k_pack_tile_sums(const uint32_t* stored, uint64_t n,
                                                        uint64_t* offsets) {
  __shared__ uint64_t wsum[8];
  const uint64_t t0 = (uint64_t)blockIdx.x * kPackTile;
  const uint64_t t1 = min(t0 + kPackTile, n);
  uint64_t sum = 0;
  for (uint64_t i = t0 + threadIdx.x; i < t1; i += blockDim.x) sum += pack_len(stored, i);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) sum += __shfl_down_sync(0xFFFFFFFFu, sum, d);
  if ((threadIdx.x & 31u) == 0) wsum[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t tot = 0;
    for (uint32_t w = 0; w < (blockDim.x >> 5); ++w) tot += wsum[w];
    offsets[t1] = tot;  // the next tile's first slot, or offsets[n]
  }
}

__global__ void __launch_bounds__(1024) k_pack_tile_bases(uint64_t n, uint64_t* offsets) {
  __shared__ uint64_t part[1024];
  const uint64_t T = (n + kPackTile - 1) / kPackTile;
  uint64_t carry = 0;
  for (uint64_t b0 = 0; b0 < T; b0 += blockDim.x) {
    const uint64_t t = b0 + threadIdx.x;
    const uint64_t v = t < T ? offsets[min((t + 1) * kPackTile, n)] : 0;
    part[threadIdx.x] = v;
    __syncthreads();
    for (uint32_t d = 1; d < blockDim.x; d <<= 1) {
      const uint64_t x = threadIdx.x >= d ? part[threadIdx.x - d] : 0;
      __syncthreads();
      part[threadIdx.x] += x;
      __syncthreads();
    }
    // tile t + 1 starts where tiles 0..t end; the last one's end is the total
    if (t < T) offsets[min((t + 1) * kPackTile, n)] = carry + part[threadIdx.x];
    carry += part[blockDim.x - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[0] = 0;
}

__global__ void __launch_bounds__(256) k_pack_tile_scan(const uint32_t* stored, uint64_t n,
                                                        uint64_t* offsets) {
  __shared__ uint64_t wsum[8];
  const uint32_t lane = threadIdx.x & 31u, wid = threadIdx.x >> 5;
  const uint64_t t0 = (uint64_t)blockIdx.x * kPackTile;
  const uint64_t w0 = t0 + (uint64_t)wid * (kPackTile / 8u);
  const uint64_t w1 = min(w0 + kPackTile / 8u, n);
  const uint64_t base = offsets[t0];  // written by k_pack_tile_bases
  uint64_t sum = 0;
  for (uint64_t i = w0 + lane; i < w1; i += 32) sum += pack_len(stored, i);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, d);
  if (lane == 0) wsum[wid] = sum;
  __syncthreads();
  uint64_t run = base;
  for (uint32_t w = 0; w < wid; ++w) run += wsum[w];
  for (uint64_t i0 = w0; i0 < w1; i0 += 32) {
    const uint64_t i = i0 + lane;
    const uint64_t v = i < w1 ? pack_len(stored, i) : 0;
    uint64_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t x = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= (uint32_t)d) incl += x;
    }
    if (i < w1) offsets[i] = run + incl - v;
    run += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
}

__global__ void __launch_bounds__(256) k_pack_copy(uint8_t* dst, const uint64_t* offsets,
                                                   const uint8_t* src, uint64_t slot,
                                                   const uint32_t* stored, uint64_t n) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t wpb = blockDim.x >> 5;
  for (uint64_t i = (uint64_t)blockIdx.x * wpb + (threadIdx.x >> 5); i < n;
       i += (uint64_t)gridDim.x * wpb) {
    const uint32_t nv = (__ldg(stored + i) + 15u) >> 4;
    const uint4* s = reinterpret_cast<const uint4*>(src + i * slot);
    uint4* d = reinterpret_cast<uint4*>(dst + __ldg(offsets + i));
    for (uint32_t v = lane; v < nv; v += 32) d[v] = ld_nc_v4(s + v);
  }
}

// Resident blocks per SM of a kernel at a launch shape, with its dynamic
// shared-memory limit raised as needed.  Both runtime queries cost more host
// time than a small launch takes on the GPU, so the answers are kept per
// (device, kernel, threads, shared memory).
struct LaunchCfg {
  int dev;
  const void* fn;
  int threads;
  size_t smem;
  int bps;
};
std::mutex g_cfg_mu;
std::vector<LaunchCfg> g_cfg;

template <typename K>
int blocks_per_sm(K kernel, int threads, size_t smem) {
  const void* fn = reinterpret_cast<const void*>(kernel);
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_cfg_mu);
  size_t max_smem = 0;
  for (const LaunchCfg& c : g_cfg) {
    if (c.dev != dev || c.fn != fn) continue;
    if (c.threads == threads && c.smem == smem) return c.bps;
    if (c.smem > max_smem) max_smem = c.smem;
  }
  if (smem > max_smem && smem > 48u * 1024u)
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    b = 1;
  }
  if (b < 1) b = 1;
  g_cfg.push_back({dev, fn, threads, smem, b});
  return b;
}

// Clusters of a kernel with compile-time cluster dimensions that fit on the
// GPU at once (0 if the runtime cannot tell).
template <typename K>
int max_active_clusters(K kernel, int threads, size_t smem) {
  const void* fn = reinterpret_cast<const void*>(kernel);
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_cfg_mu);
  for (const LaunchCfg& c : g_cfg)
    if (c.dev == dev && c.fn == fn && c.threads == -threads && c.smem == smem) return c.bps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCountCluster * 1024u, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  g_cfg.push_back({dev, fn, -threads, smem, n});  // cached under a negative thread count
  return n;
}

uint32_t warps_for(uint32_t per_warp_bytes) {
  uint32_t w = (96u * 1024u) / per_warp_bytes;
  if (w > 8u) w = 8u;
  if (w < 1u) w = 1u;
  return w;
}

}  // namespace

WarpSmem decode_smem(uint32_t W, uint32_t nch) {
  WarpSmem L;
  L.sbuf_words = ((W + 8u) + 3u) & ~3u;
  L.xbuf_words = 0;
  L.cinfo_words = (nch + 3u) & ~3u;
  L.total_words = L.sbuf_words + L.cinfo_words;
  return L;
}

WarpSmem encode_smem(uint32_t W, uint32_t nch) {
  WarpSmem L;
  L.sbuf_words = ((W + 8u) + 3u) & ~3u;
  L.cinfo_words = (nch + 3u) & ~3u;
  // rows up to 2 KB: a ring of kEncodeStages rows; larger rows: one
  L.xbuf_words = (W <= 512u ? kEncodeStages : 1u) * ((W + 3u) & ~3u);
  L.total_words = L.sbuf_words + L.xbuf_words + L.cinfo_words;
  return L;
}

// ------------------------------------------------------------------------
// Ordered gathers.  A GPU reads pinned host memory through address
// translation whose reach is limited: random gathers over a store larger than
// that reach (measured on GB300: beyond ~20 GB of host slots) fall to a
// fraction of the link, while the same gathers in address order keep it
// busy.  The ids are bucketed by region (a counting sort on
// id * kOrderBuckets / n_rows, order within a bucket arbitrary) and the
// decoder's warps sweep the bucketed list together, each row written back to
// its original output position.
// ------------------------------------------------------------------------
namespace {

__device__ __forceinline__ uint32_t order_bucket(int64_t id, uint64_t n_rows) {
  if (id < 0 || (uint64_t)id >= n_rows) return 0;  // flagged by the decoder later
  return (uint32_t)((uint64_t)id * kOrderBuckets / n_rows);
}

__global__ void __launch_bounds__(256) k_order_count(const int64_t* ids, uint64_t n,
                                                     uint64_t n_rows, uint32_t* hist) {
  __shared__ uint32_t h[kOrderBuckets];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) h[b] = 0;
  __syncthreads();
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    atomicAdd(&h[order_bucket(__ldg(ids + i), n_rows)], 1u);
  __syncthreads();
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x)
    if (h[b]) atomicAdd(hist + b, h[b]);
}

// counts -> exclusive starts, in place: one block of 1024 threads,
// ceil(kOrderBuckets / 1024) consecutive counters each
__global__ void __launch_bounds__(1024) k_order_scan(uint32_t* hist) {
  constexpr uint32_t kPer = (kOrderBuckets + 1023u) / 1024u;
  __shared__ uint32_t part[1024];
  // behind the count (programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t t = threadIdx.x;
  uint32_t c[kPer], v = 0;
#pragma unroll
  for (uint32_t q = 0; q < kPer; ++q) {
    c[q] = kPer * t + q < kOrderBuckets ? hist[kPer * t + q] : 0u;
    v += c[q];
  }
  part[t] = v;
  __syncthreads();
  for (uint32_t d = 1; d < 1024u; d <<= 1) {
    const uint32_t x = t >= d ? part[t - d] : 0u;
    __syncthreads();
    part[t] += x;
    __syncthreads();
  }
  uint32_t run = part[t] - v;
#pragma unroll
  for (uint32_t q = 0; q < kPer; ++q) {
    if (kPer * t + q < kOrderBuckets) hist[kPer * t + q] = run;
    run += c[q];
  }
}

// One id per thread (the grid covers the n ids): a rank among the CTA's ids
// of the same bucket (shared memory), one global atomic per bucket the CTA
// touched for its base (a bucket of hot rows takes one per CTA, not one per
// lookup), the id and its position at base + rank.
__global__ void __launch_bounds__(256) k_order_scatter(const int64_t* ids, uint64_t n,
                                                       uint64_t n_rows, uint32_t* cursor,
                                                       int64_t* ids_out, int64_t* pos_out) {
  __shared__ uint32_t lc[kOrderBuckets];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) lc[b] = 0;
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool has = i < n;
  int64_t id = 0;
  uint32_t bk = 0, rank = 0;
  __syncthreads();
  if (has) {
    id = __ldg(ids + i);
    bk = order_bucket(id, n_rows);
    rank = atomicAdd(&lc[bk], 1u);
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the scanned cursors
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x)
    if (lc[b]) lc[b] = atomicAdd(cursor + b, lc[b]);
  __syncthreads();
  if (has) {
    const uint32_t p = lc[bk] + rank;
    ids_out[p] = id;
    pos_out[p] = (int64_t)i;
  }
}

}  // namespace

// A launch that may start while the stream's previous kernel finishes
// (programmatic dependent launch): the kernel waits for that kernel's results
// with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_behind(void (*kern)(KArgs...), uint32_t grid, uint32_t block, size_t smem,
                          cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_order_ids(const int64_t* ids, uint64_t n, uint64_t n_rows, int64_t* ids_out,
                             int64_t* pos_out, uint32_t* hist, int sm_count, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const uint64_t need = (n + 255) / 256;  // the scatter: one id per thread
  if (need > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  uint64_t blocks = (uint64_t)sm_count * 4;
  if (blocks > need) blocks = need;
  k_order_count<<<(uint32_t)blocks, 256, 0, st>>>(ids, n, n_rows, hist);
  cudaError_t e = launch_behind(k_order_scan, 1u, 1024u, 0, st, hist);
  if (e != cudaSuccess) return e;
  return launch_behind(k_order_scatter, (uint32_t)need, 256u, 0, st, ids, n, n_rows, hist,
                       ids_out, pos_out);
}

namespace {

__device__ __forceinline__ uint32_t item_bucket(const GroupEntry* ent, uint32_t T, uint32_t bpt,
                                                const int64_t* ids, uint64_t i) {
  const uint32_t t = (uint32_t)(i % T);
  const int64_t id = __ldg(ids + i);
  const uint64_t nr = ent[t].n_rows;
  const uint32_t r = (id < 0 || (uint64_t)id >= nr) ? 0u : (uint32_t)((uint64_t)id * bpt / nr);
  return t * bpt + r;
}

// The items are visited table by table (x = t * batch + b is item b*T + t),
// so that the 256 items of a CTA come from one or two tables and touch a few
// dozen buckets: the CTA adds up its counts in shared memory and sends one
// global atomic per bucket it touched.  (Visited in item order, the bucket
// of a table's hottest rows took a returning global atomic per lookup, more
// than a thousand in a row on one address.)
__device__ __forceinline__ uint64_t table_major_item(uint64_t x, uint32_t T, uint64_t batch) {
  return (x % batch) * T + x / batch;
}

__global__ void __launch_bounds__(256) k_order_items_count(const GroupEntry* ent, uint32_t T,
                                                           const int64_t* ids, uint64_t n,
                                                           uint32_t* hist) {
  __shared__ uint32_t h[kOrderBuckets];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t bpt = kOrderBuckets / T;
  const uint64_t batch = n / T;
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) h[b] = 0;
  __syncthreads();
  for (uint64_t x = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n;
       x += (uint64_t)gridDim.x * blockDim.x)
    atomicAdd(&h[item_bucket(ent, T, bpt, ids, table_major_item(x, T, batch))], 1u);
  __syncthreads();
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x)
    if (h[b]) atomicAdd(hist + b, h[b]);
}

// One item per thread (the grid covers the n items), in table-major order:
// a rank within the CTA's items of the same bucket (shared memory), one
// global atomic per bucket the CTA touched for its base, the item at base +
// rank.  cursor: each bucket's next free position (the scanned counts).
__global__ void __launch_bounds__(256) k_order_items_scatter(const GroupEntry* ent, uint32_t T,
                                                             const int64_t* ids, uint64_t n,
                                                             uint32_t* cursor, int64_t* order) {
  __shared__ uint32_t lc[kOrderBuckets];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t bpt = kOrderBuckets / T;
  const uint64_t batch = n / T;
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) lc[b] = 0;
  const uint64_t x = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool has = x < n;
  uint64_t item = 0;
  uint32_t bk = 0, rank = 0;
  __syncthreads();
  if (has) {
    item = table_major_item(x, T, batch);
    bk = item_bucket(ent, T, bpt, ids, item);
    rank = atomicAdd(&lc[bk], 1u);
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the scanned cursors
  for (uint32_t b = threadIdx.x; b < kOrderBuckets; b += blockDim.x)
    if (lc[b]) lc[b] = atomicAdd(cursor + b, lc[b]);
  __syncthreads();
  if (has) order[lc[bk] + rank] = (int64_t)item;
}

// Largest bucket grouped in shared memory (larger ones keep the scatter's order).
constexpr uint32_t kGroupCap = 2048;
constexpr uint32_t kGroupHash = 2 * kGroupCap;  // hash slots (load at most 1/2)
// Cost of an item that fetches a row, in units of an item that repeats the
// row before it (stored from the warp's copy: no fetch, no decode), for
// cutting the list into warp shares of equal cost.  Measured on 26 Zipf DLRM
// tables: 4 best at 512 B rows (2-4 within 1 %, 8 5 % slower, 15 20 %), 4-6
// best at 2 KB rows.
constexpr uint32_t kFetchWeight = 4;
// dynamic shared memory of k_order_items_group: hash keys, slot counters,
// and each position's slot after grouping (4 CTAs per SM)
constexpr size_t kGroupSmem = 8ull * kGroupHash + 4ull * kGroupHash + 2ull * kGroupCap;

// One CTA per bucket of the ordered group list: the bucket's lookups of each
// row brought next to each other (each item's row id inserted into a hash
// table in shared memory, then the items counting-sorted by their row's hash
// slot: the rows in hash order, their lookups side by side).  Each item's
// cost (a row's first item kFetchWeight, its repeats 1), the cost of the
// bucket's earlier items in wpre, the bucket's total in cost.  ends: bucket
// ends in order (the scatter's cursors).  A bucket above kGroupCap items
// keeps its order, every item costing kFetchWeight (cost = its item count;
// wpre unused).  Launched behind the scatter (programmatic dependent launch).
__global__ void __launch_bounds__(256) k_order_items_group(const int64_t* ids,
                                                           const uint32_t* ends,
                                                           int64_t* order, uint32_t* wpre,
                                                           uint32_t* cost) {
  extern __shared__ __align__(16) unsigned long long gsm[];
  unsigned long long* hkey = gsm;                                    // kGroupHash
  uint32_t* hcnt = reinterpret_cast<uint32_t*>(hkey + kGroupHash);  // kGroupHash
  uint16_t* slot2 = reinterpret_cast<uint16_t*>(hcnt + kGroupHash);  // kGroupCap
  __shared__ uint32_t wsum[8];
  constexpr unsigned long long kEmpty = 0x8000000000000000ull;
  constexpr uint32_t kPer = kGroupCap / 256u;  // items per thread at most
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t b = blockIdx.x, tid = threadIdx.x, lane = tid & 31u, wid = tid >> 5;
  const uint32_t start = b ? ends[b - 1] : 0u, nb = ends[b] - start;
  if (nb == 0u || nb > kGroupCap) {
    if (tid == 0) cost[b] = nb;
    return;
  }
  uint32_t hs = 4u;  // hash slots: a power of two at least twice the items
  while (hs < 2u * nb) hs <<= 1;
  uint32_t lg = 0;
  while ((1u << lg) < hs) ++lg;
  for (uint32_t i = tid; i < hs; i += 256u) {
    hkey[i] = kEmpty;
    hcnt[i] = 0u;
  }
  __syncthreads();
  // each item's row into the table (linear probing; a row's lookups share a
  // slot); item j = tid + 256 q is held in registers
  uint32_t it[kPer], sl[kPer];
#pragma unroll
  for (uint32_t q = 0; q < kPer; ++q) {
    const uint32_t j = tid + 256u * q;
    it[q] = 0u;
    sl[q] = 0u;
    if (j < nb) {
      const int64_t item = order[start + j];
      const int64_t id = __ldg(ids + item);
      const unsigned long long k =
          (unsigned long long)id == kEmpty ? kEmpty + 1ull : (unsigned long long)id;
      uint32_t h = (uint32_t)((k * 0x9E3779B97F4A7C15ull) >> (64u - lg));
      for (uint32_t probe = 0; probe < hs; ++probe) {
        const unsigned long long prev = atomicCAS(hkey + h, kEmpty, k);
        if (prev == kEmpty || prev == k) break;
        h = (h + 1u) & (hs - 1u);
      }
      it[q] = (uint32_t)item;
      sl[q] = h;
      atomicAdd(hcnt + h, 1u);
    }
  }
  __syncthreads();
  // slot starts: an exclusive scan of the counts (hs / 256 slots per thread)
  const uint32_t per = (hs + 255u) / 256u, s0 = tid * per;
  uint32_t sum = 0;
  for (uint32_t q = 0; q < per; ++q)
    if (s0 + q < hs) sum += hcnt[s0 + q];
  uint32_t incl = sum;
#pragma unroll
  for (uint32_t d = 1; d < 32u; d <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31u) wsum[wid] = incl;
  __syncthreads();
  uint32_t base = 0;
  for (uint32_t w = 0; w < wid; ++w) base += wsum[w];
  uint32_t run = base + incl - sum;
  for (uint32_t q = 0; q < per; ++q) {
    if (s0 + q < hs) {
      const uint32_t c = hcnt[s0 + q];
      hcnt[s0 + q] = run;
      run += c;
    }
  }
  __syncthreads();
  // every read of the bucket's old order happened before the first barrier
#pragma unroll
  for (uint32_t q = 0; q < kPer; ++q) {
    if (tid + 256u * q < nb) {
      const uint32_t p = atomicAdd(hcnt + sl[q], 1u);
      order[start + p] = (int64_t)it[q];
      slot2[p] = (uint16_t)sl[q];
    }
  }
  __syncthreads();
  // costs in the new order: a position starts a row when its slot differs
  // from the one before; 8 consecutive positions per thread
  const uint32_t j0 = tid * 8u;
  uint32_t wts = 0, csum = 0;
#pragma unroll
  for (uint32_t q = 0; q < 8u; ++q) {
    const uint32_t j = j0 + q;
    if (j < nb) {
      const uint32_t w = (j == 0u || slot2[j] != slot2[j - 1u]) ? kFetchWeight : 1u;
      wts |= w << (4u * q);
      csum += w;
    }
  }
  __syncthreads();  // wsum is reused
  incl = csum;
#pragma unroll
  for (uint32_t d = 1; d < 32u; d <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31u) wsum[wid] = incl;
  __syncthreads();
  uint32_t cbase = 0, total = 0;
  for (uint32_t w = 0; w < 8u; ++w) {
    if (w < wid) cbase += wsum[w];
    total += wsum[w];
  }
  uint32_t r = cbase + incl - csum;
#pragma unroll
  for (uint32_t q = 0; q < 8u; ++q) {
    const uint32_t j = j0 + q;
    if (j < nb) {
      wpre[start + j] = r;
      r += (wts >> (4u * q)) & 15u;
    }
  }
  if (tid == 0) cost[b] = total;
}

constexpr uint32_t kSharePer = kOrderBuckets / 256u;  // bucket costs per thread
static_assert(kSharePer * 256u == kOrderBuckets, "k_order_shares: whole buckets per thread");

// Warp shares of the grouped list with equal costs: share w starts at the
// item whose cost interval holds floor(w * total / nw); shares[nw] = n.  A
// share may start on a repeat (its first item then fetches the row again).
// One warp per share (nw + 1 warps); each CTA first scans the bucket costs.
__global__ void __launch_bounds__(256) k_order_shares(const uint32_t* ends, const uint32_t* cost,
                                                      const uint32_t* wpre, uint32_t nw,
                                                      uint32_t n, uint32_t* shares,
                                                      uint32_t* stamp) {
  __shared__ unsigned long long pre[kOrderBuckets];
  __shared__ unsigned long long wsum[8];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // behind the grouping kernel
  const uint32_t tid = threadIdx.x, lane = tid & 31u, wid = tid >> 5;
  // bucket costs, kSharePer per thread, and their exclusive scan
  unsigned long long c[kSharePer], sum = 0;
#pragma unroll
  for (uint32_t q = 0; q < kSharePer; ++q) {
    const uint32_t bk = kSharePer * tid + q;
    const uint32_t nb = ends[bk] - (bk ? ends[bk - 1u] : 0u);
    c[q] = nb > kGroupCap ? (unsigned long long)kFetchWeight * nb : (unsigned long long)cost[bk];
    sum += c[q];
  }
  unsigned long long incl = sum;
#pragma unroll
  for (uint32_t d = 1; d < 32u; d <<= 1) {
    const unsigned long long v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31u) wsum[wid] = incl;
  __syncthreads();
  unsigned long long run = 0, total = 0;
  for (uint32_t w = 0; w < 8u; ++w) {
    if (w < wid) run += wsum[w];
    total += wsum[w];
  }
  run += incl - sum;
#pragma unroll
  for (uint32_t q = 0; q < kSharePer; ++q) {
    pre[kSharePer * tid + q] = run;
    run += c[q];
  }
  __syncthreads();
  const uint32_t w = blockIdx.x * 8u + wid;
  if (w > nw) return;
  if (w == nw) {
    if (lane == 0) {
      shares[w] = n;
      if (stamp) {  // the plan is complete once this kernel is
        stamp[0] = kPlanMagic;
        stamp[1] = n;
        stamp[2] = nw;
      }
    }
    return;
  }
  const unsigned long long k = (unsigned long long)w * total / nw;
  // the last bucket whose cost starts at or before k (it holds k)
  uint32_t lo = 0, hi = kOrderBuckets - 1u;
  while (lo < hi) {
    const uint32_t mid = (lo + hi + 1u) >> 1;
    if (pre[mid] <= k) lo = mid; else hi = mid - 1u;
  }
  const uint32_t start = lo ? ends[lo - 1u] : 0u, nbl = ends[lo] - start;
  const unsigned long long off = k - pre[lo];
  uint32_t j;
  if (nbl > kGroupCap) {
    j = (uint32_t)(off / kFetchWeight);
  } else {  // the last item whose cost starts at or before off: a 32-way search
    uint32_t a = 0, span = nbl;  // the answer lies in [a, a + span)
    while (span > 1u) {
      const uint32_t step = (span + 31u) >> 5;
      const uint32_t cand = a + lane * step;
      const bool le = cand < a + span && __ldg(wpre + start + cand) <= off;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, le);  // lane 0 always true
      const uint32_t last = 31u - __clz(m);
      a += last * step;
      span = min(step, span - last * step);
    }
    j = a;
  }
  if (lane == 0) shares[w] = start + j;
}

}  // namespace

cudaError_t launch_order_items(const GroupEntry* entries, uint32_t T, const int64_t* ids,
                               uint64_t n_items, int64_t* order_out, uint32_t* hist,
                               int sm_count, cudaStream_t st) {
  if (n_items == 0) return cudaSuccess;
  if (T == 0 || T > kOrderBuckets) return cudaErrorInvalidValue;
  const uint64_t need = (n_items + 255) / 256;  // the scatter: one item per thread
  if (need > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  uint64_t blocks = (uint64_t)sm_count * 4;
  if (blocks > need) blocks = need;
  k_order_items_count<<<(uint32_t)blocks, 256, 0, st>>>(entries, T, ids, n_items, hist);
  cudaError_t e = launch_behind(k_order_scan, 1u, 1024u, 0, st, hist);
  if (e != cudaSuccess) return e;
  const uint64_t sblocks = need;
  return launch_behind(k_order_items_scatter, (uint32_t)sblocks, 256u, 0, st, entries, T, ids,
                       n_items, hist, order_out);
}

cudaError_t launch_count_ones(const CountArgs& a, int sm_count, cudaStream_t st) {
  const uint32_t tpb = kCountTile;
  const uint32_t gy = (a.W + tpb - 1) / tpb;
  const size_t smem = 4ull * kCountStages * kCountRows * kCountTile;  // 32 KB
  // one wave: as many CTAs as fit on the GPU at once, split over the word
  // tiles; each CTA covers n/gx rows
  const int clusters = max_active_clusters(k_count_ones, (int)tpb, smem);
  uint64_t gx = clusters > 0
                    ? ((uint64_t)clusters / gy) * kCountCluster
                    : ((uint64_t)sm_count * blocks_per_sm(k_count_ones, (int)tpb, smem) / 2) / gy;
  if (gx < kCountCluster) gx = kCountCluster;
  const uint64_t max_gx = (a.n + 63) / 64;  // at least 64 rows per CTA
  if (gx > max_gx) gx = max_gx;
  if (gx > 65528) gx = 65528;
  gx = (gx + kCountCluster - 1) / kCountCluster * kCountCluster;  // whole clusters
  k_count_ones<<<dim3((uint32_t)gx, gy), tpb, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_finish_meta(const uint32_t* counts, uint32_t W, uint64_t n, uint32_t num,
                               uint32_t den, uint32_t* mask, uint32_t* bitval, cudaStream_t st) {
  k_finish_meta<<<(W + 127) / 128, 128, 0, st>>>(counts, W, n, num, den, mask, bitval);
  return cudaGetLastError();
}

cudaError_t launch_tune(const CountArgs& a, const uint32_t* counts, const uint32_t* num,
                        const uint32_t* den, uint32_t n_c, uint32_t wpc, uint32_t nch,
                        uint32_t* cand, unsigned long long* sizes, uint32_t* mask,
                        uint32_t* bitval, uint32_t* chosen_out, uint64_t* sizes_out,
                        int sm_count, cudaStream_t st) {
  const uint32_t W = a.W;
  for (uint32_t c = 0; c < n_c; ++c) {
    k_finish_meta<<<(W + 127) / 128, 128, 0, st>>>(counts, W, a.n, num[c], den[c],
                                                    cand + 2ull * W * c, cand + 2ull * W * c + W);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(sizes, 0, sizeof(unsigned long long) * n_c, st);
  if (e != cudaSuccess) return e;
  const uint32_t nr = (nch + 3u) & ~3u;
  const size_t smem = 4ull * nr * 9u;
  uint64_t gx = ((uint64_t)sm_count * 4 + n_c - 1) / n_c;
  const uint64_t need = (a.n + 7) / 8;
  if (gx > need) gx = need;
  if (gx < 1) gx = 1;
  k_size_estimate<<<dim3((uint32_t)gx, n_c), 256, smem, st>>>(a.rows, a.row_stride, a.ids, a.n,
                                                              cand, W, wpc, nch, sizes);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_pick_meta<<<1, 256, 0, st>>>(cand, sizes, n_c, W, mask, bitval, chosen_out, sizes_out);
  return cudaGetLastError();
}

cudaError_t launch_derive(uint32_t* mask, uint32_t* bitval, uint32_t* nm, uint32_t* pre,
                          uint32_t* kr, uint32_t* mv, uint32_t* ckeep, uint32_t* scal,
                          uint4* t2, uint4* t5, uint32_t* gtab, uint32_t W, uint32_t wpc,
                          uint32_t nch, cudaStream_t st) {
  k_derive<<<1, 1024, 0, st>>>(mask, bitval, nm, pre, kr, mv, ckeep, scal, W, wpc, nch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_derive_fast<<<1, 1024, 0, st>>>(nm, bitval, pre, mv, ckeep, t2, t5, gtab, scal, W, wpc, nch);
  return cudaGetLastError();
}

bool fast_geometry(uint32_t R, uint32_t C) { return R <= 2048u && (C % 16u) == 0u; }

namespace {
int max_smem_optin() {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    v = 48 * 1024;
  }
  return v;
}
}  // namespace

// CTAs for a gather of n rows (or items) by persistent warps, `full` CTAs
// filling the GPU:
//   - ordered gathers: as many CTAs as fit, each warp a contiguous share of
//     the sorted list (a grid cut so that fewer warps sweep the list in more
//     rounds measured slower: 192 against 243 GB/s on 26 tables of 2 KB rows,
//     53 GB of host slots, with 32-row chunks taken in turn);
//   - other gathers from pinned host memory spread the rows over every SM (a
//     few rows per warp: the link's latency wants many rows in flight, and
//     a few thousand rows would otherwise sit on a few SMs);
//   - from HBM, at least `rpw` rows per warp (one resolve chunk: measured best
//     for batches of a few thousand rows), else as many CTAs as fit.
uint64_t launch_blocks(uint64_t n, uint64_t full, uint64_t warps, uint64_t rpw, bool host,
                       bool ordered) {
  if (ordered) return (n + 32ull * warps - 1) / (32ull * warps);
  if (host) {
    uint64_t r = (n + full * warps - 1) / (full * warps);
    if (r > 32) r = 32;
    if (r < 1) r = 1;
    return (n + r * warps - 1) / (r * warps);
  }
  return (n + rpw * warps - 1) / (rpw * warps);
}

template <bool kIds, int kMode, bool kBig, bool kSplit>
cudaError_t launch_fast(const DecodeArgs& a, const HostProps& hp, int sm_count, cudaStream_t st) {
  FastParams F;
  const uint32_t W = a.m.W, nch = a.m.nch;
  F.S = kBig ? kRingStagesBig : kRingStages;
  F.table_words = (kMode == kModeUniform || kMode == kModeUniform1) ? 0u : 8u * W;
  F.gtab_words = (((W >> 2) + 3u) & ~3u) + ((nch + 3u) & ~3u);
  F.sbuf_words = ((W + 8u) + 3u) & ~3u;
  F.warp_words = F.S * F.sbuf_words + 256u + ((nch + 3u) & ~3u);
  F.min_bits = hp.min_bits;
  F.um0 = hp.um0;
  F.um1 = hp.um1;
  F.ush = hp.ush;
  F.ubv = hp.ubv;
  F.ukeep = hp.ukeep;
  F.gen = hp.gen;
  // 8 warps per CTA; rows above 2 KB take as many as their rings leave room for
  int warps = 8;
  size_t smem = 4ull * (F.table_words + F.gtab_words + 8 + (uint64_t)warps * F.warp_words);
  if (kBig) {
    const size_t cap = (size_t)max_smem_optin();
    while (warps > 1 && smem > cap) {
      --warps;
      smem = 4ull * (F.table_words + F.gtab_words + 8 + (uint64_t)warps * F.warp_words);
    }
    if (smem > cap) return cudaErrorInvalidConfiguration;
  }
  auto kern = k_decode_fast<kIds, kMode, kBig, kSplit>;
  const int bps = blocks_per_sm(kern, 32 * warps, smem);
  uint64_t blocks = (uint64_t)sm_count * bps;
  const uint64_t need = launch_blocks(a.n, blocks, (uint64_t)warps, kBig ? 8ull : 32ull,
                                      a.host_src != 0u, kIds && a.out_pos != nullptr);
  if (blocks > need) blocks = need;
  kern<<<(uint32_t)blocks, 32 * warps, smem, st>>>(a, F);
  return cudaGetLastError();
}

// The tile decoder for a packed cache read in row order; cudaErrorNotSupported
// when its stages do not fit (the caller then takes k_decode_fast).
template <int kMode>
cudaError_t launch_tiles(const DecodeArgs& a, const HostProps& hp, int sm_count,
                         cudaStream_t st) {
  FastParams F = {};
  const uint32_t W = a.m.W, nch = a.m.nch;
  F.table_words = (kMode == kModeUniform || kMode == kModeUniform1) ? 0u : 8u * W;
  F.gtab_words = (((W >> 2) + 3u) & ~3u) + ((nch + 3u) & ~3u);
  F.min_bits = hp.min_bits;
  F.um0 = hp.um0;
  F.um1 = hp.um1;
  F.ush = hp.ush;
  F.ubv = hp.ubv;
  F.ukeep = hp.ukeep;
  F.gen = hp.gen;
  // a stage takes up to 16 KB of stream bytes (a tile above that is read
  // row by row): three stages and three CTAs per SM for rows of 1 KB
  const uint32_t stage_bytes = ((min(kTileRows * a.m.R, 16384u) + 64u) + 127u) & ~127u;
  const size_t fixed = 4ull * (F.table_words + F.gtab_words + 8) + sizeof(TileInfo) * kTileStages +
                       16ull * kTileStages + 16ull +
                       4ull * kTileWarps * ((W + 16u) + ((nch + 3u) & ~3u)) + 128ull;
  const size_t smem = fixed + (size_t)kTileStages * stage_bytes;
  if (smem > (size_t)max_smem_optin()) return cudaErrorNotSupported;
  auto kern = k_decode_tiles<kMode>;
  const int threads = 32 * (int)(kTileWarps + 1);
  const int bps = blocks_per_sm(kern, threads, smem);
  if (bps < 1) return cudaErrorNotSupported;
  const uint64_t ntiles = (a.n + kTileRows - 1) / kTileRows;
  uint64_t blocks = (uint64_t)sm_count * bps;
  if (blocks > ntiles) blocks = ntiles;
  kern<<<(uint32_t)blocks, threads, smem, st>>>(a, F, stage_bytes);
  return cudaGetLastError();
}

cudaError_t launch_tiles_mode(const DecodeArgs& a, const HostProps& hp, int sm_count,
                              cudaStream_t st) {
  if (!hp.known) return launch_tiles<kModeRuntime>(a, hp, sm_count, st);
  if (hp.uniform && hp.um1 == 0u) return launch_tiles<kModeUniform1>(a, hp, sm_count, st);
  if (hp.uniform) return launch_tiles<kModeUniform>(a, hp, sm_count, st);
  if (hp.max_runs <= 2u) return launch_tiles<kModeRun2>(a, hp, sm_count, st);
  return launch_tiles<kModeNet5>(a, hp, sm_count, st);
}

template <bool kIds, bool kBig, bool kSplit = false>
cudaError_t launch_fast_mode(const DecodeArgs& a, const HostProps& hp, int sm_count,
                             cudaStream_t st) {
  if (!hp.known) return launch_fast<kIds, kModeRuntime, kBig, kSplit>(a, hp, sm_count, st);
  if (hp.uniform && hp.um1 == 0u)
    return launch_fast<kIds, kModeUniform1, kBig, kSplit>(a, hp, sm_count, st);
  if (hp.uniform) return launch_fast<kIds, kModeUniform, kBig, kSplit>(a, hp, sm_count, st);
  if (hp.max_runs <= 2u) return launch_fast<kIds, kModeRun2, kBig, kSplit>(a, hp, sm_count, st);
  return launch_fast<kIds, kModeNet5, kBig, kSplit>(a, hp, sm_count, st);
}

cudaError_t launch_decode(const DecodeArgs& a, const HostProps& hp, int sm_count,
                          cudaStream_t st) {
  if (a.n == 0) return cudaSuccess;
  if (a.chunk_stride) {  // split output: gathers on the fast decoder's geometries only
    if (!a.ids || !a.t2 || a.m.R > 8192u || (a.m.wpc & 3u) != 0u || a.group_rows == 0)
      return cudaErrorInvalidValue;
    return a.m.R <= 2048u ? launch_fast_mode<true, false, true>(a, hp, sm_count, st)
                          : launch_fast_mode<true, true, true>(a, hp, sm_count, st);
  }
  // rows up to 2 KB take the fast decoder from HBM and from host memory alike
  // (its cp.async copies use the .ca form: measured, the L2-only .cg form
  // reads host memory over the link at 60 % of the rate)
  if (a.t2 && fast_geometry(a.m.R, a.m.wpc * 4u)) {
    // a packed cache in GPU memory read in row order: whole tiles of rows by
    // bulk copies (the source 16-byte aligned, as the copies need)
    if (!a.ids && a.offsets && !a.host_src && !a.cache_map &&
        (reinterpret_cast<uintptr_t>(a.src) & 15u) == 0u) {
      const cudaError_t e = launch_tiles_mode(a, hp, sm_count, st);
      if (e != cudaErrorNotSupported) return e;
      cudaGetLastError();
    }
    return a.ids ? launch_fast_mode<true, false>(a, hp, sm_count, st)
                 : launch_fast_mode<false, false>(a, hp, sm_count, st);
  }
  // rows of 2-8 KB: the same pipeline with longer copies and, where the rings
  // need it, fewer warps per CTA
  if (a.t2 && a.m.R <= 8192u && (a.m.wpc & 3u) == 0u)
    return a.ids ? launch_fast_mode<true, true>(a, hp, sm_count, st)
                 : launch_fast_mode<false, true>(a, hp, sm_count, st);
  const WarpSmem L = decode_smem(a.m.W, a.m.nch);
  const uint32_t warps = warps_for(4u * L.total_words);
  const int threads = (int)(32u * warps);
  const size_t smem = (size_t)4u * L.total_words * warps;
  int bps;
  if (a.ids)
    bps = blocks_per_sm(k_decode<true>, threads, smem);
  else
    bps = blocks_per_sm(k_decode<false>, threads, smem);
  uint64_t blocks = (uint64_t)sm_count * bps;
  const uint64_t need = (a.n + warps - 1) / warps;
  if (blocks > need) blocks = need;
  if (a.ids)
    k_decode<true><<<(uint32_t)blocks, threads, smem, st>>>(a, L);
  else
    k_decode<false><<<(uint32_t)blocks, threads, smem, st>>>(a, L);
  return cudaGetLastError();
}

template <bool kUni, int kVpl>
cudaError_t launch_encode_v(const EncodeArgs& a, int sm_count, cudaStream_t st) {
  const WarpSmem L = encode_smem(a.m.W, a.m.nch);
  const uint32_t warps = warps_for(4u * L.total_words);
  const int threads = (int)(32u * warps);
  const size_t smem = (size_t)4u * L.total_words * warps;
  const int bps = blocks_per_sm(k_encode<kUni, kVpl>, threads, smem);
  uint64_t blocks = (uint64_t)sm_count * bps;
  // 32-row chunks only when there are enough of them to fill every warp
  EncodeArgs b = a;
  b.chunk_lg = (a.slot_ids == nullptr && a.n >= 32ull * warps * blocks) ? 5u : 0u;
  const uint64_t need = (((a.n + (1ull << b.chunk_lg) - 1) >> b.chunk_lg) + warps - 1) / warps;
  if (blocks > need) blocks = need;
  k_encode<kUni, kVpl><<<(uint32_t)blocks, threads, smem, st>>>(b, L);
  return cudaGetLastError();
}

template <bool kUni>
cudaError_t launch_encode_rows(const EncodeArgs& a, int sm_count, cudaStream_t st) {
  const uint32_t W = a.m.W;
  const size_t smem = 4ull * (2ull * W + 8ull + ((a.m.nch + 3u) & ~3u));
  const int threads = 256;
  const int bps = blocks_per_sm(k_encode_rows<kUni>, threads, smem);
  uint64_t blocks = (uint64_t)sm_count * bps;
  if (blocks > a.n) blocks = a.n;
  k_encode_rows<kUni><<<(uint32_t)blocks, threads, smem, st>>>(a);
  return cudaGetLastError();
}

template <bool kUni>
cudaError_t launch_encode_t(const EncodeArgs& a, int sm_count, cudaStream_t st) {
  const uint32_t nvec = a.m.R >> 4;
  if (nvec <= 32u) return launch_encode_v<kUni, 1>(a, sm_count, st);
  if (nvec <= 64u) return launch_encode_v<kUni, 2>(a, sm_count, st);
  if (nvec <= 128u) return launch_encode_v<kUni, 4>(a, sm_count, st);
  return launch_encode_rows<kUni>(a, sm_count, st);  // rows above 2 KB: a CTA per row
}

cudaError_t launch_encode(const EncodeArgs& a, const HostProps& hp, int sm_count,
                          cudaStream_t st) {
  if (a.n == 0) return cudaSuccess;
  if (hp.known && hp.uniform) {
    EncodeArgs u = a;
    u.um0 = hp.um0;
    u.um1 = hp.um1;
    u.ush = hp.ush;
    u.ubv = hp.ubv;
    u.ukeep = hp.ukeep;
    u.gen = hp.gen;
    return launch_encode_t<true>(u, sm_count, st);
  }
  return launch_encode_t<false>(a, sm_count, st);
}

cudaError_t launch_pack(uint8_t* dst, uint64_t* offsets, const uint8_t* src, uint64_t slot,
                        const uint32_t* stored, uint64_t n, int sm_count, cudaStream_t st) {
  const uint64_t T = (n + kPackTile - 1) / kPackTile;
  if (n == 0) {
    k_pack_tile_bases<<<1, 1024, 0, st>>>(0, offsets);  // offsets[0] = 0
    return cudaGetLastError();
  }
  if (T > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  k_pack_tile_sums<<<(uint32_t)T, 256, 0, st>>>(stored, n, offsets);
  k_pack_tile_bases<<<1, 1024, 0, st>>>(n, offsets);
  k_pack_tile_scan<<<(uint32_t)T, 256, 0, st>>>(stored, n, offsets);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || dst == nullptr) return e;
  uint64_t blocks = (uint64_t)sm_count * blocks_per_sm(k_pack_copy, 256, 0);
  const uint64_t need = (n + 7) / 8;
  if (blocks > need) blocks = need;
  k_pack_copy<<<(uint32_t)blocks, 256, 0, st>>>(dst, offsets, src, slot, stored, n);
  return cudaGetLastError();
}

static size_t group_smem(const GroupArgs& g, int warps) {
  return 4ull * (g.T * (sizeof(GroupEntry) / 4) + (uint64_t)warps * g.warp_words);
}

static uint64_t group_blocks(const GroupArgs& g, int sm_count, int warps) {
  const int bps = blocks_per_sm(k_gather_group, 32 * warps, group_smem(g, warps));
  uint64_t blocks = (uint64_t)sm_count * bps;
  const uint64_t need = launch_blocks(g.n_items, blocks, (uint64_t)warps, 8ull, g.host_src != 0u,
                                      g.order != nullptr);
  return blocks > need ? need : blocks;
}

static cudaError_t launch_group_blocks(const GroupArgs& g, uint64_t blocks, int warps,
                                       cudaStream_t st) {
  k_gather_group<<<(uint32_t)blocks, 32 * warps, group_smem(g, warps), st>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_group(const GroupArgs& g, int sm_count, cudaStream_t st) {
  if (g.n_items == 0) return cudaSuccess;
  const int warps = 8;
  return launch_group_blocks(g, group_blocks(g, sm_count, warps), warps, st);
}

uint32_t group_planned_per_sm(const GroupArgs& g) {
  struct Sm {
    int dev = -1, smem = 0, regs = 0, reserved = 0, threads = 0;
    int gather_regs = 0, group_regs = 0;
    size_t gather_static = 0, group_static = 0;
  };
  static Sm c;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_cfg_mu);
    if (c.dev != dev) {
      Sm n;
      n.dev = dev;
      cudaDeviceGetAttribute(&n.smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
      cudaDeviceGetAttribute(&n.regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
      cudaDeviceGetAttribute(&n.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
      cudaDeviceGetAttribute(&n.threads, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
      cudaFuncAttributes fa = {}, fg = {};
      cudaFuncGetAttributes(&fa, k_gather_group);
      cudaFuncGetAttributes(&fg, k_order_items_group);
      cudaGetLastError();
      n.gather_regs = fa.numRegs;
      n.group_regs = fg.numRegs;
      n.gather_static = fa.sharedSizeBytes;
      n.group_static = fg.sharedSizeBytes;
      c = n;
    }
  }
  // registers are given out in units of 8 per thread
  auto regs = [](int per_thread) { return (uint64_t)((per_thread + 7) / 8) * 8u * 256u; };
  const size_t gsm = group_smem(g, 8);
  const int kmax = blocks_per_sm(k_gather_group, 256, gsm);
  const uint64_t gather_smem = gsm + c.gather_static + (uint64_t)c.reserved;
  const uint64_t group_smem_b = kGroupSmem + c.group_static + (uint64_t)c.reserved;
  for (int k = kmax; k > 1; --k)
    if ((uint64_t)k * gather_smem + group_smem_b <= (uint64_t)c.smem &&
        (uint64_t)k * regs(c.gather_regs) + regs(c.group_regs) <= (uint64_t)c.regs &&
        (k + 1) * 256 <= c.threads)
      return (uint32_t)k;
  return 1u;
}

uint64_t group_gather_blocks(const GroupArgs& g, int sm_count, uint32_t max_per_sm) {
  const uint64_t blocks = group_blocks(g, sm_count, 8);
  const uint64_t cap = (uint64_t)sm_count * max_per_sm;
  return max_per_sm && blocks > cap ? cap : blocks;
}

cudaError_t launch_group_plan(GroupArgs g, const uint32_t* hist, uint32_t* wpre, uint32_t* cost,
                              uint32_t* shares, uint32_t nw, uint32_t* stamp, cudaStream_t st) {
  if (g.n_items == 0) return cudaSuccess;
  if (g.n_items > 0xFFFFFFFFull || nw == 0) return cudaErrorInvalidValue;
  // sets the kernel's shared-memory limit once (cached), so the call stays
  // capturable in a CUDA graph
  blocks_per_sm(k_order_items_group, 256, kGroupSmem);
  cudaError_t e = launch_behind(k_order_items_group, kOrderBuckets, 256u, kGroupSmem, st, g.ids, hist,
                    const_cast<int64_t*>(g.order), wpre, cost);
  if (e != cudaSuccess) return e;
  return launch_behind(k_order_shares, (nw + 1u + 7u) / 8u, 256u, 0, st, (const uint32_t*)hist,
                       (const uint32_t*)cost, (const uint32_t*)wpre, nw, (uint32_t)g.n_items,
                       shares, stamp);
}

cudaError_t launch_group_gather(const GroupArgs& g, uint64_t blocks, cudaStream_t st) {
  if (g.n_items == 0) return cudaSuccess;
  // a plain launch: started early (behind the share kernel) its CTAs, sized
  // to fill the SMs, measured 3x slower on 2 KB rows
  return launch_group_blocks(g, blocks, 8, st);
}

cudaError_t launch_group_ordered(GroupArgs g, const uint32_t* hist, uint32_t* wpre,
                                 uint32_t* cost, uint32_t* shares, int sm_count,
                                 cudaStream_t st) {
  if (g.n_items == 0) return cudaSuccess;
  const uint64_t blocks = group_gather_blocks(g, sm_count, 0);
  cudaError_t e =
      launch_group_plan(g, hist, wpre, cost, shares, (uint32_t)(blocks * 8u), nullptr, st);
  if (e != cudaSuccess) return e;
  g.shares = shares;
  return launch_group_gather(g, blocks, st);
}

cudaError_t launch_link_copy(uint4* dst, const uint4* src, uint64_t nvec, int sm_count,
                             cudaStream_t st) {
  if (nvec == 0) return cudaSuccess;
  const int threads = 512;
  uint64_t blocks = (uint64_t)sm_count * blocks_per_sm(k_link_copy, threads, 0);
  const uint64_t need = (nvec + threads - 1) / threads;
  if (blocks > need) blocks = need;
  k_link_copy<<<(uint32_t)blocks, threads, 0, st>>>(dst, src, nvec);
  return cudaGetLastError();
}

cudaError_t launch_gather_copy(uint8_t* dst, const uint8_t* src, uint64_t slot,
                               uint32_t row_bytes, const int64_t* ids, uint64_t n,
                               uint64_t n_rows, int sm_count, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  uint64_t blocks = (uint64_t)sm_count * blocks_per_sm(k_gather_copy, threads, 0);
  const uint64_t need = (n + 7) / 8;
  if (blocks > need) blocks = need;
  k_gather_copy<<<(uint32_t)blocks, threads, 0, st>>>(dst, src, slot, row_bytes, ids, n, n_rows);
  return cudaGetLastError();
}

}  // namespace ibp
