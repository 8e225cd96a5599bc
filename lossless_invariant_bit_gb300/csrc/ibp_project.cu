// K/V projection with the IBP compressor in its epilogue.
//
// The juhe.plus review's LLM paragraph and the gist.science explainer
// (Technical Summary, Results: KV movement) have the K/V of each decode
// token compressed on the GPU, with the Mask/Bitval built from the prompt's
// K/V, and offloaded to host memory.  The K/V come out of a projection
// Y = X W^T (+ bias): here the compressor's work happens where Y is produced.
//
// k_project_compress: one CTA computes a 128-row x BN-column tile of Y,
// BN = 128 / kSeg: a 256-byte chunk (one attention head of 16-bit values)
// when kSeg = 1, half or a quarter of one when few rows leave most SMs idle
// (a decode step has 20 rows: 32 chunk-wide tiles would stream the 32 MB
// weight through 32 SMs).
//   - warp 0, one thread: TMA loads of X and W tiles (64 K-elements, 128-byte
//     swizzle) into a ring of shared-memory stages, each with a full and an
//     empty mbarrier (for at most 32 rows only 32 rows of X are loaded: the
//     MMA's other rows read whatever the shared memory holds, and their
//     results, rows past m, are never used);
//   - warp 1, one thread: tcgen05.mma (kind::f16, M = 128, N = BN, K = 16)
//     into a BN-column fp32 accumulator in tensor memory; tcgen05.commit
//     frees each stage and, at the end, signals the epilogue;
//   - all four warps (thread = tensor-memory lane = row): the row's BN
//     accumulators plus bias, rounded to 16 bits, written to Y; the tile
//     tested against Mask/Bitval (does every word match?) and its kept bits
//     gathered (5-stage network of the store's move masks) into a staging
//     area, with a flag per (row, tile).
// k_project_assemble (one CTA per row, launched behind the first with
// programmatic dependent launch, so its launch overlaps the GEMM's tail): a
// row's stream needs every chunk's participation before any chunk's place is
// known, and the chunks of a row come from different CTAs of the first
// kernel.  Per row: participation of each chunk (all its tiles matched and it
// has an invariant bit), chunk starts by a warp scan, the raw fallback; the
// staged kept bits (or Y's words, for a raw chunk) copied into shared
// memory, OR'd into the stream at their bit offsets, and the stored bytes,
// raw bit and stored size written -- as ibp_compress would write them.
//
// Every wait on an mbarrier gives up after about two seconds, records
// IBP_ETIMEOUT and lets the CTA free its tensor memory and exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "ibp_internal.cuh"

namespace ibp {
namespace {

// Most tiles a chunk is cut into for small batches (1, 2 or 4).
#ifndef IBP_PROJECT_MAX_SEG
#define IBP_PROJECT_MAX_SEG 4u
#endif
// Most stages in the ring (fewer when the stages are larger).
#ifndef IBP_PROJECT_MAX_STAGES
#define IBP_PROJECT_MAX_STAGES 16u
#endif
// Accumulators in tensor memory, taken by the k-blocks in turn (1, 2 or 4).
#ifndef IBP_PROJECT_ACCUMULATORS
#define IBP_PROJECT_ACCUMULATORS 4u
#endif

constexpr uint32_t kPjBM = 128;           // rows per tile (the MMA's M)
constexpr uint32_t kPjBK = 64;            // K elements per stage: one 128-byte row
constexpr uint32_t kPjRing = 200u * 1024u;  // shared-memory bytes of the stage ring
// shared memory: 1 KB alignment slack, the ring, the tile's metadata (8 x 64
// words at most: mask, bitval, ~mask, 5 move masks), barriers
constexpr uint32_t kPjMetaWords = 8u * 64u;

// Shape of one instance: kSeg tiles per chunk, kAR rows of X loaded per stage.
template <int kSeg, int kAR>
struct PjShape {
  static constexpr uint32_t BN = 128u / kSeg;             // columns per tile
  static constexpr uint32_t WPT = 64u / kSeg;             // row words per tile
  static constexpr uint32_t A = (uint32_t)kAR * 128u;     // bytes of X per k-block
  static constexpr uint32_t B = BN * 128u;                // bytes of W per k-block
  // k-blocks per stage: one TMA copy of each operand fetches them all (a
  // copy has a cost of its own besides its bytes: with one k-block per
  // stage, narrow tiles streamed W at the same k-blocks per second whatever
  // their width)
  static constexpr uint32_t KB = (A + B) <= 12288u ? 4u : (A + B) <= 24576u ? 2u : 1u;
  static constexpr uint32_t SA = KB * A, SB = KB * B;     // bytes per stage
  static constexpr uint32_t S0 = kPjRing / (SA + SB);
  static constexpr uint32_t S = S0 > IBP_PROJECT_MAX_STAGES ? IBP_PROJECT_MAX_STAGES : S0;
  static constexpr uint32_t RING = S * (SA + SB);         // bytes of the ring
  // dynamic shared memory: 1 KB alignment slack, the ring, the tile's
  // metadata, the barriers (only what this shape uses: a smaller carve-out
  // of shared memory)
  static constexpr uint32_t SMEM = 1024u + RING + 4u * kPjMetaWords + 512u;
  // independent accumulators the k-blocks take in turn: consecutive MMAs into
  // one accumulator wait for each other, and a narrow tile's MMAs are short
  static constexpr uint32_t ACC = IBP_PROJECT_ACCUMULATORS;
  static constexpr uint32_t TMEM = ACC * BN;             // accumulator columns (<= 512)
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(a), "r"(parity), "r"(1000000u)
      : "memory");
  return done != 0u;
}

// Wait for the phase of `parity` to complete, for at most ~2 s (the clock is
// read only once the first test has failed).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try(a, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try(a, parity)) return true;
    if (global_ns() - t0 > 2000000000ull) return false;
  }
}

// One TMA copy of a 3-D box {64 elements, rows, k-blocks} into shared memory
// (coordinates: element 0, first row, first k-block), completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t row, int32_t kblock) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(0), "r"(row), "r"(kblock)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1u << 16;                           // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset: one 8-row atom
  d |= (uint64_t)1u << 46;                           // descriptor version
  d |= (uint64_t)2u << 61;                           // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, fp32 accumulator, A and B of one 16-bit
// type (fp16 or bf16), both K-major, M = 128, N = bn.
__device__ __forceinline__ uint32_t mma_idesc(uint32_t bf16, uint32_t bn) {
  return (1u << 4) | (bf16 << 7) | (bf16 << 10) | ((bn >> 3) << 17) | ((kPjBM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, uint32_t bf16) {
  if (bf16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float to_float(uint16_t v, uint32_t bf16) {
  if (bf16) return __uint_as_float((uint32_t)v << 16);
  return __half2float(__ushort_as_half(v));
}

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t code) {
  atomicCAS(st, 0u, code);
}

template <int kSeg, int kAR>
__global__ void __launch_bounds__(128, 1)
    k_project_compress(const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_w, ProjectArgs a) {
  using P = PjShape<kSeg, kAR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  uint8_t* s_x = smem;                 // P::S stages of X: KB tiles of kAR rows each
  uint8_t* s_w = smem + P::S * P::SA;  // P::S stages of W: KB tiles of BN rows each
  uint32_t* s_meta = reinterpret_cast<uint32_t*>(smem + P::RING);
  uint64_t* full = reinterpret_cast<uint64_t*>(s_meta + kPjMetaWords);
  uint64_t* empty = full + P::S;
  uint64_t* done = empty + P::S;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  uint32_t* s_fail = s_tmem + 1;

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t t = blockIdx.x;               // column tile
  const uint32_t ntiles = gridDim.x;           // nch * kSeg
  const uint32_t n0 = t * P::BN, m0 = blockIdx.y * kPjBM;
  const uint32_t w0 = t * P::WPT;              // the tile's first row word
  const uint32_t W = a.W;
  const uint32_t kb_n = (uint32_t)(a.k_dim / kPjBK);

  // the tile's Mask, Bitval, ~Mask and move masks (WPT words each)
  for (uint32_t i = threadIdx.x; i < P::WPT; i += blockDim.x) {
    const uint32_t w = w0 + i;
    s_meta[i] = __ldg(a.mask + w);
    s_meta[P::WPT + i] = __ldg(a.bitval + w);
    s_meta[2u * P::WPT + i] = __ldg(a.nm + w);
#pragma unroll
    for (uint32_t st = 0; st < 5u; ++st)
      s_meta[(3u + st) * P::WPT + i] = __ldg(a.mv + st * W + w);
  }
  if (threadIdx.x == 0) {
    // the tensor maps' descriptors, fetched while the CTA sets up
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
    for (uint32_t s = 0; s < P::S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(done, 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // tensor memory for the accumulator (one warp allocates)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(s_tmem)),
                 "r"(P::TMEM)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *s_tmem;

  const uint32_t st_n = (kb_n + P::KB - 1) / P::KB;  // stages to fill
  if (warp == 0 && lane == 0) {  // producer
    for (uint32_t ks = 0; ks < st_n; ++ks) {
      const uint32_t s = ks % P::S, round = ks / P::S;
      if (round > 0 && !mbar_wait(empty + s, (round - 1u) & 1u)) {
        atomicExch(s_fail, 1u);
        break;
      }
      if (*reinterpret_cast<volatile uint32_t*>(s_fail)) break;
      // k-blocks past the end of K read as zero (and are not multiplied)
      mbar_expect_tx(full + s, P::SA + P::SB);
      tma_load_3d(s_x + s * P::SA, &tmap_x, full + s, (int32_t)m0, (int32_t)(ks * P::KB));
      tma_load_3d(s_w + s * P::SB, &tmap_w, full + s, (int32_t)n0, (int32_t)(ks * P::KB));
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    const uint32_t idesc = mma_idesc(a.bf16, P::BN);
    for (uint32_t ks = 0; ks < st_n; ++ks) {
      const uint32_t s = ks % P::S, round = ks / P::S;
      if (!mbar_wait(full + s, round & 1u)) {
        atomicExch(s_fail, 1u);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
      for (uint32_t j = 0; j < P::KB; ++j) {
        const uint32_t kb = ks * P::KB + j;
        if (kb >= kb_n) break;
        const uint32_t xa = smem_addr(s_x + s * P::SA + j * P::A);
        const uint32_t wa = smem_addr(s_w + s * P::SB + j * P::B);
        const uint32_t acc = kb % P::ACC;  // this k-block's accumulator
#pragma unroll
        for (uint32_t kk = 0; kk < kPjBK / 16u; ++kk)
          mma_f16(tmem + acc * P::BN, sw128_desc(xa + 32u * kk), sw128_desc(wa + 32u * kk),
                  idesc, (kb >= P::ACC || kk != 0u) ? 1u : 0u);
      }
      mma_commit(empty + s);  // the stage is free once these MMAs have read it
    }
    mma_commit(done);  // every MMA issued so far has completed
  }
  __syncwarp();

  // ---- epilogue: thread = tensor-memory lane = row m0 + 32*warp + lane
  const bool waited = mbar_wait(done, 0);
  const bool ok =
      __syncthreads_and(waited && *reinterpret_cast<volatile uint32_t*>(s_fail) == 0u) != 0;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint64_t row = (uint64_t)m0 + 32u * warp + lane;
  const bool valid = ok && row < a.m;
  uint32_t x[P::WPT];  // the row's tile: BN 16-bit values, two per word
  const uint32_t used = kb_n < P::ACC ? kb_n : P::ACC;  // accumulators written
#pragma unroll
  for (uint32_t j = 0; j < P::BN / 32u; ++j) {
    float f[32];
#pragma unroll
    for (uint32_t i = 0; i < 32u; ++i) f[i] = 0.f;
    for (uint32_t q = 0; ok && q < used; ++q) {  // the accumulators' sum
      uint32_t r[32];
      tmem_ld32(tmem + ((32u * warp) << 16) + q * P::BN + 32u * j, r);
#pragma unroll
      for (uint32_t i = 0; i < 32u; ++i) f[i] += __uint_as_float(r[i]);
    }
#pragma unroll
    for (uint32_t i = 0; i < 16u; ++i) {
      float lo = f[2u * i], hi = f[2u * i + 1u];
      if (a.bias) {
        const uint32_t bw = __ldg(reinterpret_cast<const uint32_t*>(a.bias) + w0 + 16u * j + i);
        lo += to_float((uint16_t)(bw & 0xFFFFu), a.bf16);
        hi += to_float((uint16_t)(bw >> 16), a.bf16);
      }
      x[16u * j + i] = pack2(lo, hi, a.bf16);
    }
  }
  // the accumulator has been read: free the tensor memory (after a timeout,
  // first give the MMAs already issued their own bounded wait)
  if (!ok && threadIdx.x == 32u) mbar_wait(done, 0);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(P::TMEM)
                 : "memory");
  if (!ok) {
    if (threadIdx.x == 0) set_status(a.status, IBP_ETIMEOUT);
    return;
  }
  if (valid) {
    uint4* yrow = reinterpret_cast<uint4*>(a.y + row * (uint64_t)(4u * W) + 4u * w0);
#pragma unroll
    for (uint32_t v = 0; v < P::WPT / 4u; ++v)
      yrow[v] = make_uint4(x[4u * v], x[4u * v + 1u], x[4u * v + 2u], x[4u * v + 3u]);
    // does every word of the tile agree with the Bitval on the Mask?
    uint32_t diff = 0;
#pragma unroll
    for (uint32_t i = 0; i < P::WPT; ++i) diff |= (x[i] & s_meta[i]) ^ s_meta[P::WPT + i];
    a.flags[row * ntiles + t] = diff == 0u ? 1u : 0u;
    if (diff == 0u) {  // the kept bits, LSB-first, word after word
      uint32_t* out = a.staged + (row * ntiles + t) * P::WPT;
      uint64_t acc = 0;
      uint32_t nacc = 0, wo = 0;
#pragma unroll
      for (uint32_t i = 0; i < P::WPT; ++i) {
        const uint32_t keepm = s_meta[2u * P::WPT + i];
        uint32_t v = x[i] & keepm;
#pragma unroll
        for (uint32_t st = 0; st < 5u; ++st) {
          const uint32_t tt = v & s_meta[(3u + st) * P::WPT + i];
          v = (v ^ tt) | (tt >> (1u << st));
        }
        acc |= (uint64_t)v << nacc;
        nacc += __popc(keepm);
        if (nacc >= 32u) {
          out[wo++] = (uint32_t)acc;
          acc >>= 32;
          nacc -= 32u;
        }
      }
      if (nacc) out[wo] = (uint32_t)acc;
    }
  }
  // this CTA's part is staged: the assembling grid may launch
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One row per CTA: its stream from the staged tiles (see the file comment).
__global__ void __launch_bounds__(128) k_project_assemble(ProjectArgs a, uint32_t seg) {
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ uint32_t s_words;
  __shared__ int64_t s_slot;
  // wait for the projection grid: its staged bits, flags and Y are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t W = a.W, nch = a.nch, R = 4u * W, ntiles = nch * seg, wpt = 64u / seg;
  const uint32_t tid = threadIdx.x, T = blockDim.x, lane = tid & 31u;
  const uint64_t r = blockIdx.x;
  uint32_t* src = sm;                       // W words: each chunk's source
  uint32_t* out = src + W;                  // W + 8 words: the stream
  uint32_t* seg_keep = out + W + 8u;        // kept bits of each tile (ntiles)
  uint32_t* seg_start = seg_keep + ntiles;  // each tile's flag, then its stream offset
  uint32_t* cst = seg_start + ntiles;       // per chunk: start | p << 31
  // every tile's flag and kept bits (from the chunk-relative prefix of kept
  // bits), and the slot: one round of independent loads
  for (uint32_t ti = tid; ti < ntiles; ti += T) {
    const uint32_t c = ti / seg, h = ti % seg, w = 64u * c + h * wpt;
    const uint32_t hi = h + 1u < seg ? __ldg(a.pre + w + wpt) : __ldg(a.ckeep + c);
    seg_keep[ti] = hi - __ldg(a.pre + w);
    seg_start[ti] = __ldcg(a.flags + r * ntiles + ti);
  }
  if (tid == 0) s_slot = a.slot_ids ? __ldg(a.slot_ids + r) : (int64_t)r;
  __syncthreads();
  if (tid < 32u) {  // participation, chunk sizes -> starts (a warp scan)
    uint32_t run = nch;
    for (uint32_t k0 = 0; k0 < nch; k0 += 32u) {
      const uint32_t c = k0 + lane;
      uint32_t p = 0, size = 0;
      if (c < nch) {
        const uint32_t keep = __ldg(a.ckeep + c);
        p = keep < 2048u ? 1u : 0u;
        for (uint32_t h = 0; h < seg; ++h) p &= seg_start[c * seg + h];
        size = p ? keep : 2048u;
      }
      uint32_t incl = size;
#pragma unroll
      for (uint32_t d = 1; d < 32u; d <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += v;
      }
      if (c < nch) {
        uint32_t st = run + incl - size;
        cst[c] = st | (p << 31);
        for (uint32_t h = 0; h < seg; ++h) {
          seg_start[c * seg + h] = st;
          st += seg_keep[c * seg + h];
        }
      }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) s_words = (run + 31u) >> 5;
  }
  __syncthreads();
  const uint32_t words = s_words;
  const bool raw = 4u * words >= R;
  const int64_t slot = s_slot;
  if (slot < 0 || (uint64_t)slot >= a.n_rows) {
    if (tid == 0) {
      set_status(a.status, IBP_ERANGE);
      if (a.stored_out) a.stored_out[r] = 0;
    }
    return;
  }
  uint4* dslot = reinterpret_cast<uint4*>(a.dst + (uint64_t)slot * a.slot);
  const uint4* yrow = reinterpret_cast<const uint4*>(a.y + r * (uint64_t)R);
  if (raw) {
    for (uint32_t v = tid; v < R / 16u; v += T) dslot[v] = __ldcg(yrow + v);
  } else {
    const uint32_t padded = (words + 3u) & ~3u;
    for (uint32_t z = tid; z < padded + 4u; z += T) out[z] = 0;
    // each chunk's source, 16 bytes at a time, all copies in flight together:
    // a packed chunk's tiles (their kept bits) or a raw chunk's words of Y
    for (uint32_t v = tid; v < W / 4u; v += T) {
      const uint32_t w = 4u * v, c = w >> 6, i = w & 63u;  // word i of chunk c
      const uint32_t* from;
      if (cst[c] >> 31) {
        const uint32_t h = i / wpt, o = i % wpt;  // word o of tile h's kept bits
        if (32u * o >= seg_keep[c * seg + h]) continue;
        from = a.staged + (r * ntiles + c * seg + h) * wpt + o;
      } else {
        from = reinterpret_cast<const uint32_t*>(yrow) + w;
      }
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                       static_cast<uint32_t>(__cvta_generic_to_shared(src + w))),
                   "l"(from));
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();
    for (uint32_t c = tid; c < nch; c += T)
      if (cst[c] >> 31) atomicOr(out + (c >> 5), 1u << (c & 31u));
    for (uint32_t w = tid; w < W; w += T) {
      const uint32_t c = w >> 6, i = w & 63u;
      uint32_t bit, nbits;
      if (cst[c] >> 31) {
        const uint32_t h = i / wpt, o = i % wpt;
        const uint32_t kh = seg_keep[c * seg + h];
        if (32u * o >= kh) continue;
        bit = seg_start[c * seg + h] + 32u * o;
        nbits = min(32u, kh - 32u * o);
      } else {
        bit = (cst[c] & 0x7FFFFFFFu) + 32u * i;
        nbits = 32u;
      }
      const uint32_t v = src[w], q = bit >> 5, sh = bit & 31u;
      atomicOr(out + q, v << sh);
      if (sh != 0u && sh + nbits > 32u) atomicOr(out + q + 1u, v >> (32u - sh));
    }
    __syncthreads();
    for (uint32_t v = tid; 4u * v < padded; v += T)
      dslot[v] = *reinterpret_cast<const uint4*>(out + 4u * v);
  }
  if (tid == 0) {
    const uint32_t bitm = 1u << ((uint64_t)slot & 31u);
    if (raw)
      atomicOr(a.bitmap + ((uint64_t)slot >> 5), bitm);
    else
      atomicAnd(a.bitmap + ((uint64_t)slot >> 5), ~bitm);
    if (a.stored_out) a.stored_out[r] = raw ? R : 4u * words;
  }
}

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// links no driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_enc_mu;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lock(g_enc_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// A 3-D map of a row-major [rows, k] matrix of 16-bit values seen as
// {64 elements, rows, k / 64 k-blocks} (the k-blocks 128 bytes apart), boxes
// of {64, box_rows, box_kb} with the 128-byte swizzle: box_kb K-major tiles
// of box_rows x 64 one after another.  Rows and k-blocks past the end read as
// zero.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t k, uint32_t box_rows,
              uint32_t box_kb, uint32_t bf16) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t dims[3] = {kPjBK, rows, k / kPjBK};
  const cuuint64_t strides[2] = {k * 2u, kPjBK * 2u};
  const cuuint32_t box[3] = {kPjBK, box_rows, box_kb};
  const cuuint32_t estr[3] = {1, 1, 1};
  return f(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
           const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared-memory limit to `smem` once per device (a
// call being captured into a CUDA graph then sets nothing).
cudaError_t smem_limit(const void* fn, size_t smem) {
  struct Seen {
    const void* fn;
    int dev;
    size_t smem;
  };
  static std::mutex mu;
  static Seen seen[64];
  static int n_seen = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_seen; ++i)
    if (seen[i].fn == fn && seen[i].dev == dev && seen[i].smem >= smem) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n_seen; ++i)
    if (seen[i].fn == fn && seen[i].dev == dev) {
      seen[i].smem = smem;
      return cudaSuccess;
    }
  if (n_seen < 64) seen[n_seen++] = Seen{fn, dev, smem};
  return cudaSuccess;
}

template <int kSeg, int kAR>
cudaError_t launch_shape(const ProjectArgs& a, const void* x, const void* w, cudaStream_t st) {
  using P = PjShape<kSeg, kAR>;
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, a.m, a.k_dim, (uint32_t)kAR, P::KB, a.bf16) ||
      !make_map(&mw, w, (uint64_t)a.nch * 128u, a.k_dim, P::BN, P::KB, a.bf16))
    return cudaErrorInvalidValue;
  auto kern = k_project_compress<kSeg, kAR>;
  cudaError_t e = smem_limit(reinterpret_cast<const void*>(kern), P::SMEM);
  if (e != cudaSuccess) return e;
  const uint64_t mtiles = (a.m + kPjBM - 1) / kPjBM;
  kern<<<dim3(a.nch * kSeg, (uint32_t)mtiles), 128, P::SMEM, st>>>(mx, mw, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the row assembly, launched behind the projection (programmatic dependent
  // launch: it starts while the projection's last CTAs finish and waits for
  // them on the device)
  const uint32_t ntiles = a.nch * kSeg;
  const size_t smem = 4ull * (2ull * a.W + 8ull + 2ull * ntiles + ((a.nch + 3u) & ~3u));
  auto asmk = k_project_assemble;
  if (smem > 48u * 1024u) {
    e = smem_limit(reinterpret_cast<const void*>(asmk), smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.m, 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, asmk, a, (uint32_t)kSeg);
}

}  // namespace

cudaError_t launch_project(const ProjectArgs& a, const void* x, const void* w, int sm_count,
                           cudaStream_t st) {
  if (a.m == 0) return cudaSuccess;
  const uint64_t mtiles = (a.m + kPjBM - 1) / kPjBM;
  if (mtiles > 65535u || a.m > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  // narrower tiles while the grid would leave a quarter of the SMs idle
  // (measured: 20 rows x 32 chunks best at 4 tiles per chunk, 128 CTAs; 160
  // rows at 2, 128 CTAs: 41.6 against 58.0 us at 4)
  uint32_t seg = 1;
  while (seg < IBP_PROJECT_MAX_SEG && 4ull * a.nch * seg * mtiles < 3ull * (uint64_t)sm_count)
    seg *= 2u;
  const bool few = a.m <= 32u;  // one row tile, at most 32 rows of X to load
  if (seg == 1u) return few ? launch_shape<1, 32>(a, x, w, st) : launch_shape<1, 128>(a, x, w, st);
  if (seg == 2u) return few ? launch_shape<2, 32>(a, x, w, st) : launch_shape<2, 128>(a, x, w, st);
  return few ? launch_shape<4, 32>(a, x, w, st) : launch_shape<4, 128>(a, x, w, st);
}

}  // namespace ibp
