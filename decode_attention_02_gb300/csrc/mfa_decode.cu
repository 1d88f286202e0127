// MFA decode attention for GB300 (sm_103a): split-KV decode kernel, log-sum-exp
// combine kernel, and the C ABI declared in include/mfa.h.
//
// The step (Step-3, paperlayer.ai/abs/2507.19427v1, sections 2 and 5): 64 query
// heads of width 256 attend over ONE shared K head and ONE shared V head in a
// paged cache, so every KV page is a dense [64 x 256] . [256 x tokens] contraction
// shared by all heads.  Section 4 states the cost model: the larger of compute and
// KV-memory access.  At 64 FLOP/B (bf16 KV) the step is HBM-bound on GB300, so the
// design streams each KV byte exactly once per step:
//
//  * One CTA per SM (persistent).  CTA g owns tiles [floor(gW/G), floor((g+1)W/G))
//    of the batch's W 128-token tiles laid end to end, so the load is even for any
//    length mix; a sequence cut by a CTA boundary yields partial results that the
//    combine kernel merges (split-KV with a log-sum-exp merge).
//  * Each CTA holds all 64 heads of its sequence, so K and V are read once.
//  * Warp 0 streams K/V pages with TMA (3-D tensor maps over the page pool; the
//    block table supplies the page coordinate) into a 10-slot, 16 KB/slot ring.
//  * Warp 1 issues tcgen05 MMAs in the transposed form, which fills the M=128
//    datapath: S^T[128 tokens x 64 heads] = K_tile . Q^T and
//    O^T[256 d x 64 heads] += V^T . P^T (two M=128 halves), fp32 accumulators in
//    tensor memory (S double-buffered, O double-buffered across sequences).
//  * Warps 2-5 (one thread per tensor-memory lane = token) run the online softmax
//    in fp32.  The running max is lazy: a head's reference max moves only when a
//    score exceeds it by 2^8, so the common tile needs no cross-thread reduction;
//    row sums accumulate per thread and are reduced once per sequence.
//  * The ragged last page is loaded with its valid rows shifted to the end of the
//    box (negative row start; TMA fills the rest with zeros), so NaN or stale data
//    in unused page slots never enters an MMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "mfa.h"
#include "ptx.cuh"

namespace mfa {

constexpr int kH = 64;             // query heads
constexpr int kD = 256;            // head width
constexpr int kPage = 64;          // tokens per KV page
constexpr int kTile = 128;         // tokens per pipeline tile (MMA M)
constexpr int kThreads = 320;      // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr int kSoftmaxThreads = 256;  // two warps per TMEM lane quarter, 32 heads each
constexpr int kMaxTilesPerCta = 128;
constexpr int kMaxSeg = kMaxTilesPerCta;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 domain: p <= 2^8 between rescales
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per pipeline wait
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 0.1 s for drains after an abort

// Shared-memory map (offsets from a 1024-byte aligned base).  Both KV formats put the
// barriers at the same offset; they differ below it:
//   bf16 : Q 32 KB | P 16 KB | ring 10 x 16 KB (K/V operand tiles as TMA writes them)
//   e4m3 : Q 32 KB | P 16 KB | V f16 64 KB (dequantised PV operand) | ring 12 x 8 KB (raw
//          e4m3 boxes) and, after the common area, a 4-tile ring of per-token scales
constexpr int kOffQ = 0;                                     // 4 x [64 heads x 128 B]
constexpr int kOffP = 32768;                                 // [128 tokens x 128 B]
constexpr int kOffBar = 212992;                              // mbarriers
template <bool kFp8>
struct KvLayout;
template <>
struct KvLayout<false> {
  static constexpr int kOffRing = 49152;
  static constexpr int kNumSlots = 10;
  static constexpr int kSlotBytes = 16384;
  static constexpr int kOffStageFinal = kOffRing;   // 128 KB free after the last MMA
  static constexpr int kExtraSmem = 0;
};
template <>
struct KvLayout<true> {
  static constexpr int kOffVh = 49152;              // 4 x 16 KB: (page, d-half) f16 tiles
  static constexpr int kOffRing = 114688;
  static constexpr int kNumSlots = 12;
  static constexpr int kSlotBytes = 8192;
  static constexpr int kOffStageFinal = kOffVh;     // V f16 + ring: 160 KB free after the last MMA
  // scale ring, per tile: K scales of the 2 pages, then V scales of the 2 pages once per
  // d-half (each half's box brings its own copy, so its consumers wait on their own box)
  static constexpr int kScaleTiles = 4;
  static constexpr int kScaleTileBytes = 6 * 256;
  static constexpr int kExtraSmem = kScaleTiles * kScaleTileBytes;
};
static_assert(KvLayout<false>::kOffRing + KvLayout<false>::kNumSlots * KvLayout<false>::kSlotBytes == kOffBar, "");
static_assert(KvLayout<true>::kOffRing + KvLayout<true>::kNumSlots * KvLayout<true>::kSlotBytes == kOffBar, "");
constexpr int kOffMisc = kOffBar + 512;  // int: [0] tmem base [1] abort [2] nseg [3] ntiles [4..15] scan
constexpr int kOffMref = kOffMisc + 128;      // float[64]  reference max per head (log2 domain)
constexpr int kOffAlpha = kOffMref + 256;     // float[64]  rescale factor per head
constexpr int kOffRed = kOffAlpha + 256;      // float[2][4][64] cross-warp reduction scratch
constexpr int kOffLinv = kOffRed + 2048;      // float[2][64]  1 / row sum per O buffer
constexpr int kOffSeg = kOffLinv + 512;       // int4[kMaxSeg] {b, first tile, end tile, L}
constexpr int kOffSegN0 = kOffSeg + 16 * kMaxSeg;       // int[kMaxSeg] CTA-local index of first tile
constexpr int kOffTileBlk = kOffSegN0 + 4 * kMaxSeg;    // int2[kMaxTilesPerCta] page ids
constexpr int kSmemUsed = kOffTileBlk + 8 * kMaxTilesPerCta;
constexpr int kOffScale = kSmemUsed;                    // e4m3 only
template <bool kFp8>
constexpr int smem_bytes() { return kSmemUsed + KvLayout<kFp8>::kExtraSmem + 1024; }
static_assert(smem_bytes<true>() <= 232448, "shared memory budget");

enum Bar : int {
  kBarFull = 0,
  kBarEmpty = kBarFull + 12,   // room for the larger ring
  kBarQFull = kBarEmpty + 12,
  kBarQEmpty,
  kBarSFull,   // 2
  kBarSEmpty = kBarSFull + 2,
  kBarPFull = kBarSEmpty + 2,
  kBarPvDone,
  kBarOFull,   // 2
  kBarOEmpty = kBarOFull + 2,
  kBarDrain = kBarOEmpty + 2,
  kBarQReady,   // e4m3: q converted to f16 in place
  kBarKReady,   // e4m3: K tile dequantised into tensor memory
  kBarKFree,    // e4m3: the QK MMAs have read that K tile
  kBarCount
};
static_assert(kBarCount * 8 <= 512, "barrier area");

// Tensor-memory columns.
constexpr uint32_t kTmemS = 0;     // S^T buffers: [0,64) and [64,128)
constexpr uint32_t kTmemO = 128;   // O^T buffer k, half hh: 128 + 128k + 64hh
constexpr uint32_t kTmemL = 384;   // bf16: per-lane row sums of the bf16-rounded weights (normalise O)
constexpr uint32_t kTmemLx = 448;  // bf16: per-lane row sums of the fp32 weights (lse)
constexpr uint32_t kTmemK = 384;   // e4m3: K tile in f16, lane = token, 2 d per column (A operand)

struct DecodeParams {
  CUtensorMap tm_q;   // 2-D [B*64 rows, 256] bf16, box 64x64, 128B swizzle
  CUtensorMap tm_k;   // 3-D [num_blocks, 64, 256]: bf16 box {64, 64, 1}, e4m3 box {128, 64, 1}; 128B swizzle
  CUtensorMap tm_v;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;          // bf16 or fp32 [B, 64, 256]
  float* lse;
  float* part_o;
  float* part_lse;
  unsigned int* status;
  int batch;
  int max_pages;
  int num_blocks;
  int out_f32;        // 1: fp32 output, 0: bf16 output
  int early_metadata; // 1: seq_lens/block_table may be read before the preceding grid completes
  float scale_log2;   // softmax_scale * log2(e)
};

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  const int32_t* seq_lens;
  void* out;
  float* lse;
  int batch;
  int max_pages;
  int num_ctas;
  int out_f32;
  int heads_per_cta;  // 1, 4 or 16
};

// ------------------------------------------------------------------ helpers

// tcgen05 shared-memory matrix descriptor: start, leading/stride byte offsets,
// descriptor version 1 (bits 46..47), 128-byte swizzle (bits 61..63 = 2).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// tcgen05 instruction descriptor for kind::f16: fp32 D, bf16 or f16 A/B,
// K-major (0) or MN-major (1) operands, N>>3 at bit 17, M>>4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool a_mn, bool b_mn, int m, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ int clamp_len(int L, int cap, bool& bad) {
  if (L < 0) { bad = true; return 0; }
  if (L > cap) { bad = true; return cap; }
  return L;
}

__device__ __forceinline__ int tiles_of(int L) { return (L + kTile - 1) / kTile; }

// Bounded wait on an mbarrier phase.  Returns false after kWaitLimitNs, or at
// once when another role has raised the CTA's abort flag.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const bool ok = wait_slow(bar, parity, abort_flag, kWaitLimitNs);
  if (!ok && abort_flag != nullptr) *abort_flag = 1;
  return ok;
}

// Block-wide (kThreads) inclusive scan of one int per thread; also returns the total.
__device__ __forceinline__ int block_incl_scan(int v, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int x = scratch[w];
    before += (w < warp) ? x : 0;
    tot += x;
  }
  __syncthreads();
  total = tot;
  return v + before;
}

// Reduce 64 per-thread values across the 32 lanes of a warp by halving exchanges;
// lane l ends with the results for heads 2l and 2l+1.
template <bool kMax>
__device__ __forceinline__ void warp_reduce_scatter64(float (&v)[64], float& r0, float& r1) {
  const int lane = threadIdx.x & 31;
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const bool hi = lane & 16;
    const float keep = hi ? v[i + 32] : v[i], send = hi ? v[i] : v[i + 32];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool hi = lane & 8;
    const float keep = hi ? v[i + 16] : v[i], send = hi ? v[i] : v[i + 16];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 4;
    const float keep = hi ? v[i + 8] : v[i], send = hi ? v[i] : v[i + 8];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 2;
    const float keep = hi ? v[i + 4] : v[i], send = hi ? v[i] : v[i + 4];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 1;
    const float keep = hi ? v[i + 2] : v[i], send = hi ? v[i] : v[i + 2];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
  }
  r0 = v[0];
  r1 = v[1];
}

// Reduce 32 per-thread values across the 32 lanes of a warp by halving exchanges;
// lane l ends with the result for value index l.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool hi = lane & 16;
    const float keep = hi ? v[i + 16] : v[i], send = hi ? v[i] : v[i + 16];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 8;
    const float keep = hi ? v[i + 8] : v[i], send = hi ? v[i] : v[i + 8];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 4;
    const float keep = hi ? v[i + 4] : v[i], send = hi ? v[i] : v[i + 4];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 2;
    const float keep = hi ? v[i + 2] : v[i], send = hi ? v[i] : v[i + 2];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  {
    const bool hi = lane & 1;
    const float keep = hi ? v[1] : v[0], send = hi ? v[0] : v[1];
    v[0] = op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
  }
  return v[0];
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 64 consecutive TMEM columns of this thread's lane, as two 32-register halves.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&a)[32], uint32_t (&b)[32]) {
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_ld_wait(a);
  tmem_ld_wait(b);
}
#define SV(h) ((h) < 32 ? sa[(h)] : sb[(h) - 32])

// Warp-uniform bounded wait (all lanes poll; the warp agrees on the outcome).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = wait_bar(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ decode kernel

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Ring use index of the K (is_v = false) or V part (page pg, d-half dh) of tile t of a
// CTA with `ntiles` tiles.  The producer issues K(0), then K(t) and V(t-1) for t = 1..N-1,
// then V(N-1), four uses each: K(0) = 0..3, K(t) = 8t-4.., V(t) = 8t+8.. except the last
// tile's V, which directly follows its K: V(N-1) = 8N-4...
__device__ __forceinline__ uint32_t ring_use(int t, int ntiles, bool is_v, int pg, int dh) {
  const uint32_t base = is_v ? (t + 1 < ntiles ? 8u * t + 8u : 8u * t + 4u) : (t == 0 ? 0u : 8u * t - 4u);
  return base + 2u * pg + dh;
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) mfa_decode_kernel(const __grid_constant__ DecodeParams p) {
  using Lay = KvLayout<kFp8>;
  constexpr int kNumSlots = Lay::kNumSlots;
  constexpr int kSlotBytes = Lay::kSlotBytes;
  constexpr int kOffRing = Lay::kOffRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  int* misc = reinterpret_cast<int*>(smem + kOffMisc);
  volatile int* abort_flag = misc + 1;
  int4* seg = reinterpret_cast<int4*>(smem + kOffSeg);
  int* seg_n0 = reinterpret_cast<int*>(smem + kOffSegN0);
  int2* tile_blk = reinterpret_cast<int2*>(smem + kOffTileBlk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };

  // ---------------- set-up: barriers, tensor memory
  if (tid == 0) {
    for (int i = 0; i < kNumSlots; ++i) {
      mbar_init(bar(kBarFull + i), 1);
      // bf16: released by the MMA commit; e4m3: by the 64 threads that dequantise the box
      mbar_init(bar(kBarEmpty + i), kFp8 ? 64 : 1);
    }
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSEmpty + i), kSoftmaxThreads);
      mbar_init(bar(kBarOFull + i), 1);
      mbar_init(bar(kBarOEmpty + i), kSoftmaxThreads);
    }
    mbar_init(bar(kBarPFull), kSoftmaxThreads);
    mbar_init(bar(kBarPvDone), 1);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarQReady), kSoftmaxThreads);
    mbar_init(bar(kBarKReady), kSoftmaxThreads);
    mbar_init(bar(kBarKFree), 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32 * 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }

  // Launched as a programmatic dependent of the preceding kernel on the stream: nothing
  // that kernel may write is touched before griddepcontrol.wait.  With early metadata
  // the lengths and the block table are read first (the caller guarantees the preceding
  // kernel does not write them); q, K, V and every output wait.
  if (!p.early_metadata) grid_dep_wait();

  // ---------------- schedule: this CTA's tile range and its per-sequence segments
  const int cap = p.max_pages * kPage;
  {
    int* scratch = misc + 4;
    bool bad = false;
    int loc = 0;
    const int L_first = (tid < p.batch) ? p.seq_lens[tid] : 0;   // reused by the segment scan below
    loc += tiles_of(clamp_len(L_first, cap, bad));
    for (int b = tid + kThreads; b < p.batch; b += kThreads) loc += tiles_of(clamp_len(p.seq_lens[b], cap, bad));
    if (bad) atomicOr(p.status, MFA_DEV_BAD_LENGTH);
    int W = 0;
    block_incl_scan(loc, scratch, W);
    const int G = gridDim.x, g = blockIdx.x;
    const int t0 = static_cast<int>((static_cast<long long>(g) * W) / G);
    const int t1 = static_cast<int>((static_cast<long long>(g + 1) * W) / G);
    int nseg = 0;
    if (t1 - t0 > kMaxTilesPerCta) {
      if (tid == 0) atomicOr(p.status, MFA_DEV_SCHEDULE);
    } else {
      int carry = 0;
      for (int c0 = 0; c0 < p.batch && carry < t1; c0 += kThreads) {
        const int b = c0 + tid;
        bool dummy = false;
        const int L = (b < p.batch) ? clamp_len(c0 == 0 ? L_first : p.seq_lens[b], cap, dummy) : 0;
        const int T = tiles_of(L);
        int tot = 0, ftot = 0;
        const int incl = block_incl_scan(T, scratch, tot) + carry;
        const int excl = incl - T;
        const int f = (max(t0, excl) < min(t1, incl)) ? 1 : 0;   // non-empty overlap
        const int fidx = nseg + block_incl_scan(f, scratch, ftot) - f;
        if (f) {
          const int lo = max(t0, excl), hi = min(t1, incl);
          seg[fidx] = make_int4(b, lo - excl, hi - excl, L);
          seg_n0[fidx] = lo - t0;
        }
        carry += tot;
        nseg += ftot;
      }
    }
    if (tid == 0) {
      misc[2] = nseg;
      misc[3] = (nseg > 0) ? (t1 - t0) : 0;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  const int nseg = misc[2];
  const int ntiles = misc[3];

  if (warp == 0) {
    // ---------------- producer: page ids, then TMA loads of Q, K, V (and e4m3 scales)
    bool bad_blk = false;
    // all of this CTA's page ids in one round of independent loads (lane = tile)
    for (int n = lane; n < ntiles; n += 32) {
      int s = 0;
      while (s + 1 < nseg && seg_n0[s + 1] <= n) ++s;
      const int4 sg = seg[s];
      const int32_t* row = p.block_table + static_cast<size_t>(sg.x) * p.max_pages;
      {
        const int j = sg.y + (n - seg_n0[s]);
        int b0 = row[2 * j];
        const bool has1 = kPage * (2 * j + 1) < sg.w;
        int b1 = has1 ? row[2 * j + 1] : -1;
        // an id outside the pool is reported and replaced by page 0, so every TMA
        // coordinate stays inside the pool (the output of that sequence is then wrong)
        if (b0 < 0 || b0 >= p.num_blocks) { bad_blk = true; b0 = 0; }
        if (has1 && (b1 < 0 || b1 >= p.num_blocks)) { bad_blk = true; b1 = 0; }
        tile_blk[n] = make_int2(b0, b1);
      }
    }
    if (bad_blk) atomicOr(p.status, MFA_DEV_BAD_BLOCK);
    __syncwarp();
    if (lane == 0 && ntiles > 0) {
      if (p.early_metadata) grid_dep_wait();
      const uint64_t pol = l2_policy_evict_first();
      uint32_t u = 0;       // ring uses issued
      int nq = 0;           // Q loads issued
      int sk = 0, jk = seg[0].y, sv = 0, jv = seg[0].y;
      bool ok = true;
      // one ring use: wait for the slot, then load a K or V part (bf16: chunk of 64 d over
      // both pages, or page x d-half; e4m3: page x d-half box, plus the page's scales)
      auto issue = [&](bool is_v, int t, int a, int b2, int r0, int r1, const int2 bk) -> bool {
        const uint32_t slot = u % kNumSlots;
        if (!wait_bar(bar(kBarEmpty + slot), ((u / kNumSlots) & 1) ^ 1, abort_flag)) return false;
        const uint32_t dst = sbase + kOffRing + slot * kSlotBytes;
        const uint32_t fb = bar(kBarFull + slot);
        const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
        if constexpr (!kFp8) {
          if (!is_v) {   // a = 64-d chunk, both pages
            mbar_arrive_expect_tx(fb, r1 > 0 ? 16384 : 8192);
            tma_load_3d_hint(dst, map, fb, 64 * a, r0 - kPage, bk.x, pol);
            if (r1 > 0) tma_load_3d_hint(dst + 8192, map, fb, 64 * a, r1 - kPage, bk.y, pol);
          } else {       // a = page, b2 = d-half
            const int r = a ? r1 : r0;
            const int blk = a ? bk.y : bk.x;
            if (r > 0) {
              mbar_arrive_expect_tx(fb, 16384);
              tma_load_3d_hint(dst, map, fb, 128 * b2, r - kPage, blk, pol);
              tma_load_3d_hint(dst + 8192, map, fb, 128 * b2 + 64, r - kPage, blk, pol);
            } else {
              mbar_arrive(fb);
            }
          }
        } else {         // a = page, b2 = d-half
          const int r = a ? r1 : r0;
          const int blk = a ? bk.y : bk.x;
          if (r > 0) {
            // K: the page's scales with its d-half-0 box (read only once QK has run, which
            // needs both halves); V: a copy with each half's box, read by that half's threads
            const bool with_scale = is_v || (b2 == 0);
            mbar_arrive_expect_tx(fb, 8192 + (with_scale ? 256 : 0));
            tma_load_3d_hint(dst, map, fb, 128 * b2, r - kPage, blk, pol);
            if (with_scale) {
              const float* src = (is_v ? p.v_scale : p.k_scale) + static_cast<size_t>(blk) * kPage;
              const int idx = is_v ? 2 + 2 * a + b2 : a;
              const uint32_t sdst = sbase + kOffScale + (t % KvLayout<true>::kScaleTiles) * KvLayout<true>::kScaleTileBytes +
                                    idx * 256;
              bulk_load_g2s(sdst, src, 256, fb);
            }
          } else {
            mbar_arrive(fb);
          }
        }
        ++u;
        return true;
      };
      for (int n = 0; n <= ntiles && ok; ++n) {
        if (n < ntiles) {
          const int4 sg = seg[sk];
          if (jk == sg.y) {
            if (sk > 0) ok = wait_bar(bar(kBarQEmpty), (sk - 1) & 1, abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(kBarQFull), kH * kD * 2);
            for (int c = 0; c < 4; ++c)
              tma_load_2d(sbase + kOffQ + c * 8192, &p.tm_q, bar(kBarQFull), 64 * c, kH * sg.x);
            ++nq;
          }
          const int2 bk = tile_blk[n];
          const int r0 = min(kPage, sg.w - kTile * jk);
          const int r1 = min(kPage, sg.w - kTile * jk - kPage);
          for (int c = 0; c < 4 && ok; ++c) ok = issue(false, n, kFp8 ? (c >> 1) : c, c & 1, r0, r1, bk);
          if (!ok) break;
          if (++jk == sg.z && ++sk < nseg) jk = seg[sk].y;
        }
        if (n >= 1) {
          const int4 sg = seg[sv];
          const int2 bk = tile_blk[n - 1];
          const int rr0 = min(kPage, sg.w - kTile * jv);
          const int rr1 = min(kPage, sg.w - kTile * jv - kPage);
          for (int c = 0; c < 4 && ok; ++c) ok = issue(true, n - 1, c >> 1, c & 1, rr0, rr1, bk);
          if (!ok) break;
          if (++jv == sg.z && ++sv < nseg) jv = seg[sv].y;
        }
      }
      if (!ok) {
        atomicOr(p.status, MFA_DEV_TIMEOUT);
        // let every copy already issued land before the CTA can exit
        const uint32_t first = (u > static_cast<uint32_t>(kNumSlots)) ? u - kNumSlots : 0;
        for (uint32_t v = first; v < u; ++v)
          wait_slow(bar(kBarFull + v % kNumSlots), (v / kNumSlots) & 1, nullptr, kDrainLimitNs);
        if (nq > 0) wait_slow(bar(kBarQFull), (nq - 1) & 1, nullptr, kDrainLimitNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdescQK = idesc_f16(!kFp8, false, false, 128, 64);
      constexpr uint32_t kIdescPV = idesc_f16(!kFp8, true, true, 128, 64);
      uint32_t u = 0;
      int sk = 0, jk = seg[0].y, sv = 0, jv = seg[0].y;
      bool ok = true;
      for (int n = 0; n <= ntiles && ok; ++n) {
        if (n < ntiles) {
          const int4 sg = seg[sk];
          const bool first = (jk == sg.y), last = (jk == sg.z - 1);
          if (first) ok = wait_bar(bar(kFp8 ? kBarQReady : kBarQFull), sk & 1, abort_flag);
          if (ok && n >= 2) ok = wait_bar(bar(kBarSEmpty + (n & 1)), ((n >> 1) - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + kTmemS + 64u * (n & 1);
          if constexpr (!kFp8) {
            for (int c = 0; c < 4; ++c, ++u) {
              const uint32_t slot = u % kNumSlots;
              ok = wait_bar(bar(kBarFull + slot), (u / kNumSlots) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint32_t a0 = sbase + kOffRing + slot * kSlotBytes;
              const uint32_t b0 = sbase + kOffQ + c * 8192;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f16_ss(d_tmem, smem_desc(a0 + 32 * kk, 16, 1024), smem_desc(b0 + 32 * kk, 16, 1024),
                            kIdescQK, (c | kk) != 0);
              umma_commit(bar(kBarEmpty + slot));
            }
            if (!ok) break;
          } else {
            // K(n) in tensor memory: lane = token, column kTmemK + d/2
            ok = wait_bar(bar(kBarKReady), n & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              umma_f16_ts(d_tmem, tmem + kTmemK + 8u * kk,
                          smem_desc(sbase + kOffQ + (kk >> 2) * 8192 + 32 * (kk & 3), 16, 1024), kIdescQK, kk != 0);
            umma_commit(bar(kBarKFree));
          }
          umma_commit(bar(kBarSFull + (n & 1)));
          if (last) umma_commit(bar(kBarQEmpty));
          if (++jk == sg.z && ++sk < nseg) jk = seg[sk].y;
        }
        if (n >= 1) {
          const int m = n - 1;
          const int4 sg = seg[sv];
          const bool first = (jv == sg.y), last = (jv == sg.z - 1);
          const int kb = sv & 1;
          ok = wait_bar(bar(kBarPFull), m & 1, abort_flag);
          if (ok && first && sv >= 2) ok = wait_bar(bar(kBarOEmpty + kb), ((sv >> 1) - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const int rr0 = min(kPage, sg.w - kTile * jv);
          const int rr1 = min(kPage, sg.w - kTile * jv - kPage);
          for (int pg = 0; pg < 2 && ok; ++pg) {
            const int r = pg ? rr1 : rr0;
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t a0;
              if constexpr (!kFp8) {
                const uint32_t slot = u % kNumSlots;
                ok = wait_bar(bar(kBarFull + slot), (u / kNumSlots) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                a0 = sbase + kOffRing + slot * kSlotBytes;
              } else {
                a0 = sbase + KvLayout<true>::kOffVh + (2 * pg + hh) * 16384;   // filled by the softmax warps
              }
              if (r > 0) {
                const uint32_t b0 = sbase + kOffP + pg * 8192;
                const uint32_t d_tmem = tmem + kTmemO + 128u * kb + 64u * hh;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  umma_f16_ss(d_tmem, smem_desc(a0 + 2048 * kk, 8192, 1024),
                              smem_desc(b0 + 2048 * kk, 1024, 1024), kIdescPV,
                              !(first && pg == 0 && kk == 0));
              }
              if constexpr (!kFp8) {
                umma_commit(bar(kBarEmpty + u % kNumSlots));
                ++u;
              }
            }
          }
          if (!ok) break;
          umma_commit(bar(kBarPvDone));
          if (last) umma_commit(bar(kBarOFull + kb));
          if (++jv == sg.z && ++sv < nseg) jv = seg[sv].y;
        }
      }
      if (!ok) atomicOr(p.status, MFA_DEV_TIMEOUT);
      // every MMA must be complete before tensor memory is released
      umma_commit(bar(kBarDrain));
      wait_slow(bar(kBarDrain), 0, nullptr, kDrainLimitNs);
    }
  } else {
    // ---------------- softmax + epilogue (256 threads: two warps per TMEM lane quarter)
    const int ts = tid - 64;                       // 0..255
    const int sw = warp - 2;                       // 0..7
    const int grp = sw >> 2;                       // head half [32*grp, +32); e4m3 dequant: d-half
    const int h0 = 32 * grp;
    const int wq = warp & 3;                       // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;                // token row of a tile / d within an O half
    const int rpg = row >> 6, ri = row & 63;       // page of the tile and row within the page
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    float* m_ref = reinterpret_cast<float*>(smem + kOffMref);
    float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    float* linv = reinterpret_cast<float*>(smem + kOffLinv);
    const float c = p.scale_log2;
    const bool issuer = (lane == 0) && ((sw & 3) == 0);   // one bulk-store thread per head half
    bool range_bad = false;                        // e4m3: a value left the f16 range

    if (p.early_metadata) grid_dep_wait();
    // sequences with no tokens: out = 0, lse = -inf (one CTA each, round robin)
    for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
      bool dummy = false;
      if (clamp_len(p.seq_lens[b], cap, dummy) != 0) continue;
      const int esz = p.out_f32 ? 4 : 2;
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + static_cast<size_t>(b) * kH * kD * esz);
      for (int i = ts; i < kH * kD * esz / 16; i += kSoftmaxThreads) o[i] = make_uint4(0, 0, 0, 0);
      if (p.lse != nullptr && ts < kH) p.lse[b * kH + ts] = -INFINITY;
    }

    bool aborted = false;
    int n = 0;
    const uint32_t l_tmem = tmem + kTmemL + h0 + lane_base;    // bf16: this thread's 32 row-sum partials
    const uint32_t lx_tmem = tmem + kTmemLx + h0 + lane_base;  // bf16: and their fp32-weight twins
    float lreg[32];                                            // e4m3: row-sum partials in registers
    int defer_b[2] = {0, 0}, defer_slot[2] = {0, 0};
    bool defer_whole[2] = {false, false};

    // valid rows of a tile's page pg: the last page's rows sit at the end of the box
    auto page_rows = [&](int L, int j, int pg) { return min(kPage, L - kTile * j - kPage * pg); };

    // e4m3: per-token scale of this thread's row in tile t (0 for rows past the length)
    auto row_scale = [&](int t, bool is_v, int rp) -> float {
      if (rp <= 0 || ri < kPage - rp) return 0.f;
      const int idx = is_v ? 2 + 2 * rpg + grp : rpg;
      const float* sc = reinterpret_cast<const float*>(
          smem + kOffScale + (t % KvLayout<true>::kScaleTiles) * KvLayout<true>::kScaleTileBytes + idx * 256);
      return sc[ri - (kPage - rp)];
    };

    // e4m3: wait until ring use `use` is filled (every consumer waits, even when its page
    // is past the sequence end and nothing is read, so that the slot's full and empty
    // phases advance in step with the producer's)
    auto wait_filled = [&](uint32_t use) -> bool {
      return wait_warp(bar(kBarFull + use % kNumSlots), (use / kNumSlots) & 1, abort_flag);
    };
    // e4m3: this thread's 128 raw codes (its token row, its d-half) of a filled ring box
    auto read_raw = [&](uint32_t use, uint4 (&rw)[8]) {
      const uint8_t* box = smem + kOffRing + (use % kNumSlots) * kSlotBytes + ri * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q) rw[q] = *reinterpret_cast<const uint4*>(box + ((q ^ (ri & 7)) << 4));
    };
    // e4m3: dequantise tile t's K part of this thread into tensor memory (lane = token)
    auto dequant_k = [&](int t, int L, int j) -> bool {
      if (t >= 1 && !wait_warp(bar(kBarKFree), (t - 1) & 1, abort_flag)) return false;
      const uint32_t use = ring_use(t, ntiles, false, rpg, grp);
      if (!wait_filled(use)) return false;
      if (page_rows(L, j, rpg) > 0) {
        uint4 rw[8];
        read_raw(use, rw);
        tc_fence_after();
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          uint32_t kv[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 w = rw[4 * hq + q];
            kv[8 * q + 0] = e4m3x2_to_f16x2(w.x);
            kv[8 * q + 1] = e4m3x2_to_f16x2(w.x >> 16);
            kv[8 * q + 2] = e4m3x2_to_f16x2(w.y);
            kv[8 * q + 3] = e4m3x2_to_f16x2(w.y >> 16);
            kv[8 * q + 4] = e4m3x2_to_f16x2(w.z);
            kv[8 * q + 5] = e4m3x2_to_f16x2(w.z >> 16);
            kv[8 * q + 6] = e4m3x2_to_f16x2(w.w);
            kv[8 * q + 7] = e4m3x2_to_f16x2(w.w >> 16);
          }
          tmem_st32(tmem + kTmemK + 64u * grp + 32u * hq + lane_base, kv);
        }
        tmem_st_wait();
      }
      mbar_arrive(bar(kBarEmpty + use % kNumSlots));
      tc_fence_before();
      mbar_arrive(bar(kBarKReady));
      return true;
    };
    // e4m3: dequantise tile t's V part of this thread into the f16 PV operand tile; the
    // token's V scale (it arrives with the box) multiplies the row here, so that P keeps
    // plain weights.  Scales above 146 would let 448 * scale leave the f16 range: they
    // are clamped and reported.
    auto dequant_v = [&](int t, int L, int j) -> bool {
      const uint32_t use = ring_use(t, ntiles, true, rpg, grp);
      if (!wait_filled(use)) return false;
      const int rp = page_rows(L, j, rpg);
      if (rp > 0) {
        uint4 rw[8];
        read_raw(use, rw);
        float sv = row_scale(t, true, rp);             // 0 for rows past the length
        range_bad |= !(sv <= 146.f);
        sv = fminf(sv, 146.f);
        const uint32_t sv2 = pack_f16_sat(sv, sv);
        auto cv = [&](uint32_t two) { return hmul2(e4m3x2_to_f16x2(two), sv2); };
        // [64 tokens x 64 d] f16 boxes, 128 B rows, 128B swizzle (as TMA would lay them out)
        uint8_t* vh = smem + KvLayout<true>::kOffVh + (2 * rpg + grp) * 16384 + ri * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w = rw[q];
          const uint4 lo = make_uint4(cv(w.x), cv(w.x >> 16), cv(w.y), cv(w.y >> 16));
          const uint4 hi = make_uint4(cv(w.z), cv(w.z >> 16), cv(w.w), cv(w.w >> 16));
          const int j0 = 2 * q, j1 = 2 * q + 1;   // 16-byte f16 chunks 0..15 of the 128-d row
          *reinterpret_cast<uint4*>(vh + (j0 >> 3) * 8192 + (((j0 & 7) ^ (ri & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(vh + (j1 >> 3) * 8192 + (((j1 & 7) ^ (ri & 7)) << 4)) = hi;
        }
      }
      mbar_arrive(bar(kBarEmpty + use % kNumSlots));
      return true;
    };
    // Write the finished accumulator of this CTA's segment `sidx` (O buffer sidx & 1),
    // normalised by 1/l from linv: [head][d] rows are staged in shared memory and sent
    // with bulk async copies.  With `from_ring` the rows go through the idle operand
    // buffers at 64 KB offset `ring_k`; otherwise through this half's 8 KB of the P
    // buffer in double-buffered 4 KB rounds.  Returns false if the CTA is aborting.
    auto write_segment = [&](int sidx, int b, int slot_p, bool whole, bool from_ring, int ring_k) -> bool {
      const int kb = sidx & 1;
      const bool okO = wait_warp(bar(kBarOFull + kb), (sidx >> 1) & 1, abort_flag);
      aborted = aborted || !okO;
      if (named_bar_or(1, kSoftmaxThreads, aborted || *abort_flag)) return false;
      tc_fence_after();
      const uint32_t o_tmem = tmem + kTmemO + 128u * kb + h0 + lane_base;
      uint32_t oa[32], ob[32];
      tmem_ld32(o_tmem, oa);
      tmem_ld32(o_tmem + 64, ob);
      tmem_ld_wait(oa);
      tmem_ld_wait(ob);
      tc_fence_before();
      mbar_arrive(bar(kBarOEmpty + kb));   // the accumulator is free; the stores below use registers
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const float li = linv[kb * kH + h0 + h];
        oa[h] = __float_as_uint(__uint_as_float(oa[h]) * li);
        ob[h] = __float_as_uint(__uint_as_float(ob[h]) * li);
      }
      const bool bf16_out = whole && !p.out_f32;
      const int esz = bf16_out ? 2 : 4;
      uint8_t* gdst = whole ? static_cast<uint8_t*>(p.out) + (static_cast<size_t>(b) * kH + h0) * kD * esz
                            : reinterpret_cast<uint8_t*>(p.part_o) + (static_cast<size_t>(slot_p) * kH + h0) * kD * 4;
      auto put = [&](uint8_t* stg, int hl, float v0, float v1) {
        if (bf16_out) {
          reinterpret_cast<__nv_bfloat16*>(stg)[hl * kD + row] = __float2bfloat16_rn(v0);
          reinterpret_cast<__nv_bfloat16*>(stg)[hl * kD + 128 + row] = __float2bfloat16_rn(v1);
        } else {
          reinterpret_cast<float*>(stg)[hl * kD + row] = v0;
          reinterpret_cast<float*>(stg)[hl * kD + 128 + row] = v1;
        }
      };
      if (from_ring) {
        const uint32_t off = Lay::kOffStageFinal + ring_k * 65536 + grp * 32768;
        uint8_t* stg = smem + off;
#pragma unroll
        for (int h = 0; h < 32; ++h) put(stg, h, __uint_as_float(oa[h]), __uint_as_float(ob[h]));
        fence_proxy_async_smem();
        named_bar_sync(2 + grp, kSoftmaxThreads / 2);
        if (issuer) {
          bulk_store_s2g(gdst, sbase + off, 32 * kD * esz);
          bulk_commit();
        }
        return true;
      }
      // 4 KB per round: 4 heads (fp32) or 8 heads (bf16); round sizes are compile-time so
      // the register arrays are indexed by constants
      constexpr int kRoundBytes = 4096;
      auto rounds = [&](auto hpr_tag) {
        constexpr int hpr = decltype(hpr_tag)::value;
#pragma unroll
        for (int r = 0; r < 32 / hpr; ++r) {
          const int buf = r & 1;
          if (r >= 2) {
            if (issuer) bulk_wait_read1();
            named_bar_sync(2 + grp, kSoftmaxThreads / 2);
          }
          uint8_t* stg = smem + kOffP + grp * 8192 + buf * kRoundBytes;
#pragma unroll
          for (int hl = 0; hl < hpr; ++hl)
            put(stg, hl, __uint_as_float(oa[r * hpr + hl]), __uint_as_float(ob[r * hpr + hl]));
          fence_proxy_async_smem();
          named_bar_sync(2 + grp, kSoftmaxThreads / 2);
          if (issuer) {
            bulk_store_s2g(gdst + static_cast<size_t>(r * hpr) * kD * esz,
                           sbase + kOffP + grp * 8192 + buf * kRoundBytes, kRoundBytes);
            bulk_commit();
          }
        }
      };
      if (bf16_out)
        rounds(std::integral_constant<int, 8>());
      else
        rounds(std::integral_constant<int, 4>());
      // the P buffer must be read out before the next segment's first tile writes it
      if (issuer) bulk_wait_read0();
      named_bar_sync(2 + grp, kSoftmaxThreads / 2);
      return true;
    };

    // e4m3: q of segment sidx arrives in bf16; the e4m3 path multiplies in f16, so convert
    // it in place.  Done as soon as the segment's first K tile is in tensor memory (for a
    // later segment: before the previous segment's epilogue, whose wait for its last PV
    // must not depend on this segment's first QK).
    auto convert_q = [&](int sidx) {
      if (wait_warp(bar(kBarQFull), sidx & 1, abort_flag)) {
        uint4* qv = reinterpret_cast<uint4*>(smem + kOffQ) + ts * 8;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 w = qv[q];
          uint32_t* e = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float x0 = __uint_as_float(e[k] << 16), x1 = __uint_as_float(e[k] & 0xFFFF0000u);
            range_bad |= !(fabsf(x0) <= 65504.f) | !(fabsf(x1) <= 65504.f);
            e[k] = pack_f16_sat(x0, x1);
          }
          qv[q] = w;
        }
        fence_proxy_async_smem();
      } else {
        aborted = true;
      }
      mbar_arrive(bar(kBarQReady));
    };

    if constexpr (kFp8) {
      // the first tile's K goes into tensor memory before the loop; each iteration then
      // dequantises the next tile's K after its own softmax
      if (ntiles > 0) {
        if (!dequant_k(0, seg[0].w, seg[0].y)) aborted = true;
        convert_q(0);
      }
    }

    for (int s = 0; s < nseg && !aborted; ++s) {
      const int4 sg = seg[s];
      const int b = sg.x, L = sg.w, kb = s & 1;
      const bool whole = (sg.y == 0) && (sg.z == tiles_of(L));
      const int slot_p = b + static_cast<int>(blockIdx.x);
      const uint32_t o_tmem = tmem + kTmemO + 128u * kb + h0 + lane_base;   // + 64 for d in [128, 256)
      if (ts < kH) m_ref[ts] = -INFINITY;
      if constexpr (kFp8) {
#pragma unroll
        for (int h = 0; h < 32; ++h) lreg[h] = 0.f;
      }
      named_bar_sync(1, kSoftmaxThreads);
      bool stop = false;
      for (int j = sg.y; j < sg.z; ++j, ++n) {
        const bool first = (j == sg.y);
        const uint32_t s_tmem = tmem + kTmemS + 64u * (n & 1) + h0 + lane_base;
        const bool okS = wait_warp(bar(kBarSFull + (n & 1)), (n >> 1) & 1, abort_flag);
        aborted = aborted || !okS;
        bool pv_waited = (n == 0);   // PV of the previous tile must be done before P or O are touched
        const int rp = page_rows(L, j, rpg);
        const bool valid = okS && rp > 0 && ri >= kPage - rp;
        // score multiplier of this row: scale*log2(e), times the token's K scale for e4m3
        // (the K box and its scales were waited for when K was dequantised)
        float ck = c;
        if constexpr (kFp8) ck = c * row_scale(n, false, rp);
        // --- does any score of this row exceed its head's reference max by > 2^8?
        bool need = false;
        if (okS) {
          tc_fence_after();
          uint32_t sv[32];
          tmem_ld32(s_tmem, sv);
          tmem_ld_wait(sv);
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(m_ref + h0 + h);
            need |= (fmaf(__uint_as_float(sv[h + 0]), ck, -m4.x) > kRescaleThreshold) |
                    (fmaf(__uint_as_float(sv[h + 1]), ck, -m4.y) > kRescaleThreshold) |
                    (fmaf(__uint_as_float(sv[h + 2]), ck, -m4.z) > kRescaleThreshold) |
                    (fmaf(__uint_as_float(sv[h + 3]), ck, -m4.w) > kRescaleThreshold);
          }
          need = need && valid;
        }
        if (named_bar_or(1, kSoftmaxThreads, need || aborted || *abort_flag)) {
          if (named_bar_or(1, kSoftmaxThreads, aborted || *abort_flag)) { stop = true; break; }
          // --- rare path: new reference max for heads whose scores jumped by > 2^8
          {
            uint32_t sv[32];
            tmem_ld32(s_tmem, sv);
            tmem_ld_wait(sv);
            float mv[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) mv[h] = valid ? __uint_as_float(sv[h]) * ck : -INFINITY;
            red[wq * 64 + h0 + lane] = warp_reduce_scatter32<true>(mv);
          }
          named_bar_sync(1, kSoftmaxThreads);
          if (ts < kH) {
            const float mt = fmaxf(fmaxf(red[ts], red[64 + ts]), fmaxf(red[128 + ts], red[192 + ts]));
            const float mo = m_ref[ts];
            float a = 1.f;
            if (mt > mo + kRescaleThreshold) {
              a = exp2f(mo - mt);
              m_ref[ts] = mt;
            }
            alpha_s[ts] = a;
          }
          named_bar_sync(1, kSoftmaxThreads);
          if (!pv_waited) {
            const bool okPV = wait_warp(bar(kBarPvDone), (n - 1) & 1, abort_flag);
            pv_waited = true;
            if (named_bar_or(1, kSoftmaxThreads, !okPV || *abort_flag)) { aborted = true; stop = true; break; }
          }
          if (!first) {
            // row sums and O^T rows (d = row, 128 + row) times alpha per head column
            if constexpr (kFp8) {
#pragma unroll
              for (int h = 0; h < 32; ++h) lreg[h] *= alpha_s[h0 + h];
            }
#pragma unroll 1
            for (int k3 = 0; k3 < (kFp8 ? 2 : 4); ++k3) {
              uint32_t ov[32];
              const uint32_t ta = (k3 == 2) ? l_tmem : (k3 == 3) ? lx_tmem : o_tmem + 64u * k3;
              tmem_ld32(ta, ov);
              tmem_ld_wait(ov);
#pragma unroll
              for (int h = 0; h < 32; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha_s[h0 + h]);
              tmem_st32(ta, ov);
            }
            tmem_st_wait();
          }
        }
        // --- probabilities and row sums; the P^T row piece stays in registers until the
        //     previous tile's PV has released the P buffer
        uint32_t pk[16];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sv[16], lv[16], lx[16];
          tmem_ld16(s_tmem + 16 * half, sv);
          if (!kFp8 && !first) {
            tmem_ld16(l_tmem + 16 * half, lv);
            tmem_ld16(lx_tmem + 16 * half, lx);
          }
          tmem_ld_wait(sv);
          if (!kFp8 && !first) {
            tmem_ld_wait(lv);
            tmem_ld_wait(lx);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) lv[e] = lx[e] = 0u;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int hl = 2 * e, h = 16 * half + hl;
            const float2 m2 = *reinterpret_cast<const float2*>(m_ref + h0 + h);
            const float p0 = valid ? ex2_approx(fmaf(__uint_as_float(sv[hl]), ck, -m2.x)) : 0.f;
            const float p1 = valid ? ex2_approx(fmaf(__uint_as_float(sv[hl + 1]), ck, -m2.y)) : 0.f;
            if constexpr (kFp8) {
              pk[8 * half + e] = pack_f16_sat(p0, p1);   // p <= 2^8: inside the f16 range
              lreg[h] += p0;
              lreg[h + 1] += p1;
            } else {
              const uint32_t w = pack_bf16(p0, p1);
              pk[8 * half + e] = w;
              // the row sum adds the same bf16-rounded weights the PV MMA uses, so the
              // output is an exact convex combination of V rows under those weights
              lv[hl] = __float_as_uint(__uint_as_float(lv[hl]) + __uint_as_float(w << 16));
              lv[hl + 1] = __float_as_uint(__uint_as_float(lv[hl + 1]) + __uint_as_float(w & 0xFFFF0000u));
              lx[hl] = __float_as_uint(__uint_as_float(lx[hl]) + p0);
              lx[hl + 1] = __float_as_uint(__uint_as_float(lx[hl + 1]) + p1);
            }
          }
          if constexpr (!kFp8) {
            tmem_st16(l_tmem + 16 * half, lv);
            tmem_st16(lx_tmem + 16 * half, lx);
          }
        }
        if constexpr (!kFp8) tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarSEmpty + (n & 1)));
        if constexpr (kFp8) {
          // next tile's K into tensor memory (the MMA warp can start its QK right away)
          if (n + 1 < ntiles) {
            const int s1 = (j + 1 < sg.z) ? s : s + 1;
            const int j1 = (j + 1 < sg.z) ? j + 1 : seg[s1].y;
            if (!dequant_k(n + 1, seg[s1].w, j1)) aborted = true;
            if (s1 != s) convert_q(s1);
          }
        }
        if (!pv_waited && !wait_warp(bar(kBarPvDone), (n - 1) & 1, abort_flag)) aborted = true;
        if constexpr (kFp8) {
          // this tile's V into the f16 operand tile (free: the previous PV is done)
          if (!dequant_v(n, L, j)) aborted = true;
        }
        // this thread's 32 heads are 16-byte chunks 4*grp .. 4*grp+3 of the 128-byte P^T row
        uint8_t* prow = smem + kOffP + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(prow + (((4 * grp + q) ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarPFull));
      }
      if (stop) break;

      // ---------------- epilogue of sequence b's segment
#pragma unroll 1
      for (int which = 0; which < (kFp8 ? 1 : 2); ++which) {
        float lsum[32];
        if constexpr (kFp8) {
#pragma unroll
          for (int h = 0; h < 32; ++h) lsum[h] = lreg[h];
        } else {
          uint32_t lv[32];
          tmem_ld32(which ? lx_tmem : l_tmem, lv);
          tmem_ld_wait(lv);
#pragma unroll
          for (int h = 0; h < 32; ++h) lsum[h] = __uint_as_float(lv[h]);
        }
        red[which * 256 + wq * 64 + h0 + lane] = warp_reduce_scatter32<false>(lsum);
      }
      named_bar_sync(1, kSoftmaxThreads);
      if (ts < kH) {
        const float l = (red[ts] + red[64 + ts]) + (red[128 + ts] + red[192 + ts]);
        linv[kb * kH + ts] = 1.f / l;
        const float lx = kFp8 ? l : (red[256 + ts] + red[320 + ts]) + (red[384 + ts] + red[448 + ts]);
        const float lse_v = (m_ref[ts] + log2f(lx)) * 0.69314718055994531f;
        if (whole) {
          if (p.lse != nullptr) p.lse[b * kH + ts] = lse_v;
        } else {
          p.part_lse[static_cast<size_t>(slot_p) * kH + ts] = lse_v;
        }
      }
      named_bar_sync(1, kSoftmaxThreads);
      if (s + 2 < nseg) {
        // the accumulator is needed again by segment s + 2: write it out now
        if (!write_segment(s, b, slot_p, whole, false, 0)) break;
      } else {
        // one of the CTA's last two segments: its accumulator stays in tensor memory
        // and is written after the last tile, when the operand buffers are idle
        defer_b[kb] = b;
        defer_slot[kb] = slot_p;
        defer_whole[kb] = whole;
      }
    }
    if (!aborted && !*abort_flag) {
      // deferred accumulators, newest first: the wait for the last segment's accumulator
      // also means every MMA has finished reading the operand buffers, which then stage
      // the rows (uniform: every thread reads the same values)
      const int first_def = nseg >= 2 ? nseg - 2 : 0;
      for (int s = nseg - 1; s >= first_def; --s) {
        const int kb = s & 1;
        if (!write_segment(s, defer_b[kb], defer_slot[kb], defer_whole[kb], true, s - first_def)) break;
      }
    }
    if (issuer) bulk_wait_read0();
    if (range_bad) atomicOr(p.status, MFA_DEV_RANGE);
    if (aborted && ts == 0) atomicOr(p.status, MFA_DEV_TIMEOUT);
  }

  // ---------------- teardown
  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ combine kernel

__device__ __forceinline__ int cta_of_tile(long long t, long long W, long long G) {
  // largest g with floor(g*W/G) <= t
  return static_cast<int>(((t + 1) * G + W - 1) / W - 1);
}

constexpr int kCombineThreads = 256;
constexpr int kCombineMaxParts = 256;        // partials staged per pass

// One CTA per (sequence, group of `heads_per_cta` heads).  The 256 threads form
// four quads of 64 (each thread owns 4 consecutive d, a float4).  With one head
// per CTA the quads split the partials four ways; with four or more heads each
// quad owns a head and the CTA walks its heads in rounds of four.  Partial lse
// values are staged in shared memory; partial O rows stream in with batched
// independent float4 loads.
__global__ void __launch_bounds__(kCombineThreads) mfa_combine_kernel(const __grid_constant__ CombineParams p) {
  grid_dep_wait();
  grid_dep_launch();   // the next kernel may start its own set-up
  __shared__ int red_b[kCombineThreads / 32], red_t[kCombineThreads / 32];
  __shared__ int slots[kCombineMaxParts];
  __shared__ float wts[4][kCombineMaxParts];
  __shared__ float4 part_acc[3][64];
  __shared__ float pass_max[4], pass_sum[4];
  __shared__ int nparts_s;
  const int b = blockIdx.x;
  const int hpc = p.heads_per_cta;
  const int hpr = hpc < 4 ? hpc : 4;          // heads per round
  const int groups = 4 / hpr;                 // quads sharing one head
  const int rounds = hpc / hpr;
  const int cap = p.max_pages * kPage;
  int before = 0, total = 0;
  for (int i = threadIdx.x; i < p.batch; i += kCombineThreads) {
    bool dummy = false;
    const int T = tiles_of(clamp_len(p.seq_lens[i], cap, dummy));
    total += T;
    before += (i < b) ? T : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red_b[threadIdx.x >> 5] = before;
    red_t[threadIdx.x >> 5] = total;
  }
  __syncthreads();
  before = 0;
  total = 0;
  for (int w = 0; w < kCombineThreads / 32; ++w) {
    before += red_b[w];
    total += red_t[w];
  }
  bool dummy = false;
  const int Tb = tiles_of(clamp_len(p.seq_lens[b], cap, dummy));
  if (Tb == 0) return;
  const int g0 = cta_of_tile(before, total, p.num_ctas);
  const int g1 = cta_of_tile(before + Tb - 1, total, p.num_ctas);
  if (g0 == g1) return;  // written whole by the decode kernel

  const int quad = threadIdx.x >> 6;
  const int hr = quad / groups;               // head of the round owned by this quad
  const int grp = quad % groups;              // partial group within that head
  const int d4 = threadIdx.x & 63;            // float4 column: d = 4*d4 .. 4*d4+3
  for (int r = 0; r < rounds; ++r) {
    const int h = blockIdx.y * hpc + r * hpr + hr;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float run_max = -INFINITY, run_sum = 0.f;
    // partials come from CTAs g0..g1 (CTAs with an empty tile range hold none)
    for (int gs = g0; gs <= g1; gs += kCombineMaxParts) {
      const int ge = min(g1 + 1, gs + kCombineMaxParts);
      __syncthreads();
      if (threadIdx.x < 32) {
        int n = 0;
        for (int g = gs + threadIdx.x; g - static_cast<int>(threadIdx.x) < ge; g += 32) {
          const bool live = g < ge && (static_cast<long long>(g) * total) / p.num_ctas !=
                                          (static_cast<long long>(g + 1) * total) / p.num_ctas;
          const unsigned m = __ballot_sync(0xffffffffu, live);
          if (live) slots[n + __popc(m & ((1u << threadIdx.x) - 1))] = b + g;
          n += __popc(m);
        }
        if (threadIdx.x == 0) nparts_s = n;
      }
      __syncthreads();
      const int n = nparts_s;
      for (int k = threadIdx.x; k < n * hpr; k += kCombineThreads) {
        const int kk = k / hpr, hh = k % hpr;
        wts[hh][kk] = p.part_lse[static_cast<size_t>(slots[kk]) * kH + blockIdx.y * hpc + r * hpr + hh];
      }
      __syncthreads();
      {
        // warp w < hpr turns head w's lse values into weights relative to their max
        const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
        if (w < hpr) {
          float m = -INFINITY;
          for (int k = l; k < n; k += 32) m = fmaxf(m, wts[w][k]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          float sum = 0.f;
          for (int k = l; k < n; k += 32) {
            const float e = expf(wts[w][k] - m);
            wts[w][k] = e;
            sum += e;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          if (l == 0) {
            pass_max[w] = m;
            pass_sum[w] = sum;
          }
        }
      }
      __syncthreads();
      // rescale what earlier passes accumulated to this pass's reference
      const float m_new = fmaxf(run_max, pass_max[hr]);
      const float a_old = (run_max == -INFINITY) ? 0.f : expf(run_max - m_new);
      const float a_new = expf(pass_max[hr] - m_new);
      acc.x *= a_old; acc.y *= a_old; acc.z *= a_old; acc.w *= a_old;
      run_sum = run_sum * a_old + pass_sum[hr] * a_new;
      run_max = m_new;
      const float* wrow = wts[hr];
      int k = grp;
      for (; k + 3 * groups < n; k += 4 * groups) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v[u] = reinterpret_cast<const float4*>(
              p.part_o + (static_cast<size_t>(slots[k + u * groups]) * kH + h) * kD)[d4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = wrow[k + u * groups] * a_new;
          acc.x = fmaf(w, v[u].x, acc.x); acc.y = fmaf(w, v[u].y, acc.y);
          acc.z = fmaf(w, v[u].z, acc.z); acc.w = fmaf(w, v[u].w, acc.w);
        }
      }
      for (; k < n; k += groups) {
        const float4 v = reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(slots[k]) * kH + h) * kD)[d4];
        const float w = wrow[k] * a_new;
        acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
      }
    }
    if (groups > 1) {
      __syncthreads();
      if (grp > 0) part_acc[grp - 1][d4] = acc;
      __syncthreads();
      if (grp != 0) continue;
      for (int k = 0; k < groups - 1; ++k) {
        const float4 o = part_acc[k][d4];
        acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
      }
    }
    const float inv = 1.f / run_sum;
    const size_t oi = (static_cast<size_t>(b) * kH + h) * kD + 4 * d4;
    if (p.out_f32) {
      reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi)[0] =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + oi)[0] = pk;
    }
    if (d4 == 0 && p.lse != nullptr) p.lse[b * kH + h] = run_max + logf(run_sum);
  }
}

// ------------------------------------------------------------------ host side

constexpr uint64_t kWsHeader = 256;

// Text of the last CUDA failure seen by this host thread (static strings only).
static thread_local const char* g_last_error = "no error";

static mfa_status cuda_fail(cudaError_t e, const char* where) {
  (void)where;
  g_last_error = cudaGetErrorString(e);
  return MFA_ERR_CUDA;
}
static mfa_status cuda_fail_msg(const char* msg) {
  g_last_error = msg;
  return MFA_ERR_CUDA;
}

static uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

static uint64_t partial_o_offset() { return kWsHeader; }
static uint64_t partial_lse_offset(int num_partials) {
  return align_up(kWsHeader + static_cast<uint64_t>(num_partials) * kH * kD * 4, 256);
}
static uint64_t workspace_bytes_for(int num_partials) {
  return align_up(partial_lse_offset(num_partials) + static_cast<uint64_t>(num_partials) * kH * 4, 256);
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static mfa_status check_problem(const mfa_problem* pr) {
  if (pr == nullptr) return MFA_ERR_INVALID_ARG;
  if (pr->batch < 0 || pr->max_pages_per_seq < 1 || pr->num_blocks < 1) return MFA_ERR_INVALID_ARG;
  if (pr->kv_dtype != MFA_KV_BF16 && pr->kv_dtype != MFA_KV_FP8_E4M3) return MFA_ERR_INVALID_ARG;
  if (pr->out_dtype != MFA_OUT_BF16 && pr->out_dtype != MFA_OUT_FP32) return MFA_ERR_INVALID_ARG;
  if (!(std::isfinite(pr->softmax_scale) && pr->softmax_scale > 0.f)) return MFA_ERR_INVALID_ARG;
  if (pr->num_q_heads != kH || pr->head_dim != kD || pr->page_size != kPage) return MFA_ERR_UNSUPPORTED;
  if (static_cast<long long>(pr->max_pages_per_seq) * kPage > INT_MAX / 2) return MFA_ERR_INVALID_ARG;
  if (static_cast<long long>(pr->batch) * kH > INT_MAX) return MFA_ERR_INVALID_ARG;
  return MFA_OK;
}

static mfa_status check_plan(const mfa_plan* pl, const mfa_problem* pr) {
  if (pl == nullptr) return MFA_ERR_INVALID_ARG;
  if (pl->batch != pr->batch || pl->kv_dtype != pr->kv_dtype) return MFA_ERR_INVALID_ARG;
  if (pl->num_ctas < 1 || pl->num_partials != pr->batch + pl->num_ctas - 1) return MFA_ERR_INVALID_ARG;
  if (pl->workspace_bytes != workspace_bytes_for(pl->num_partials)) return MFA_ERR_INVALID_ARG;
  return MFA_OK;
}

static mfa_status encode_maps(DecodeParams& prm, const mfa_problem* pr, const void* q, const void* k,
                              const void* v) {
  auto enc = encode_fn();
  if (enc == nullptr) return cuda_fail_msg("cuTensorMapEncodeTiled is not available from the driver");
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(pr->batch) * kH};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    if (enc(&prm.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail_msg("cuTensorMapEncodeTiled rejected a tensor map");
  }
  const void* pools[2] = {k, v};
  CUtensorMap* maps[2] = {&prm.tm_k, &prm.tm_v};
  const bool fp8 = pr->kv_dtype == MFA_KV_FP8_E4M3;
  const cuuint64_t esz = fp8 ? 1 : 2;
  for (int i = 0; i < 2; ++i) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(kPage),
                          static_cast<cuuint64_t>(pr->num_blocks)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * esz, static_cast<cuuint64_t>(kD) * esz * kPage};
    // one 128-byte swizzle row per box row: 64 bf16 or 128 e4m3 codes
    cuuint32_t box[3] = {fp8 ? 128u : 64u, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(maps[i], fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(pools[i]), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail_msg("cuTensorMapEncodeTiled rejected a tensor map");
  }
  return MFA_OK;
}

static mfa_status launch_combine(const mfa_plan* pl, const mfa_problem* pr, const void* workspace,
                                 const int32_t* seq_lens, void* out, float* lse, cudaStream_t stream,
                                 bool dependent) {
  CombineParams cp;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  cp.part_o = reinterpret_cast<const float*>(ws + partial_o_offset());
  cp.part_lse = reinterpret_cast<const float*>(ws + partial_lse_offset(pl->num_partials));
  cp.seq_lens = seq_lens;
  cp.out = out;
  cp.out_f32 = pr->out_dtype == MFA_OUT_FP32 ? 1 : 0;
  cp.lse = lse;
  cp.batch = pr->batch;
  cp.max_pages = pr->max_pages_per_seq;
  cp.num_ctas = pl->num_ctas;
  cudaLaunchConfig_t cfg = {};
  // about two CTAs per SM: many sequences -> more heads per CTA
  const long long want = 2LL * (pl->num_sms > 0 ? pl->num_sms : 148);
  cp.heads_per_cta = (static_cast<long long>(pr->batch) * kH >= 16 * want) ? 16
                     : (static_cast<long long>(pr->batch) * kH >= 4 * want) ? 4 : 1;
  cfg.gridDim = dim3(static_cast<unsigned>(pr->batch), kH / cp.heads_per_cta, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mfa_combine_kernel, cp);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return MFA_OK;
}

}  // namespace mfa

using namespace mfa;

extern "C" {

int32_t mfa_abi_version(void) { return MFA_ABI_VERSION; }

const char* mfa_last_cuda_error(void) { return g_last_error; }

const char* mfa_status_string(mfa_status s) {
  switch (s) {
    case MFA_OK: return "ok";
    case MFA_ERR_INVALID_ARG: return "invalid argument";
    case MFA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MFA_ERR_WORKSPACE: return "workspace too small";
    case MFA_ERR_CUDA: return "CUDA error";
    case MFA_ERR_DEVICE_CHECK: return "device status word is nonzero";
  }
  return "unknown status";
}

mfa_status mfa_decode_plan(const mfa_problem* pr, const int32_t* host_seq_lens, int32_t max_seq_len,
                           int32_t num_sms, int32_t force_ctas, uint32_t flags, mfa_plan* plan) {
  const mfa_status st = check_problem(pr);
  if (st != MFA_OK) return st;
  if (plan == nullptr || force_ctas < 0) return MFA_ERR_INVALID_ARG;
  const long long cap = static_cast<long long>(pr->max_pages_per_seq) * kPage;
  long long W = 0;
  if (host_seq_lens != nullptr) {
    for (int b = 0; b < pr->batch; ++b) {
      if (host_seq_lens[b] < 0 || host_seq_lens[b] > cap) return MFA_ERR_INVALID_ARG;
      W += (host_seq_lens[b] + kTile - 1) / kTile;
    }
  } else {
    if (max_seq_len < 0 || max_seq_len > cap) return MFA_ERR_INVALID_ARG;
    W = static_cast<long long>(pr->batch) * ((max_seq_len + kTile - 1) / kTile);
  }
  if (num_sms <= 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  }
  long long G;
  if (force_ctas > 0) {
    G = force_ctas;
  } else {
    G = W < num_sms ? W : num_sms;
    if (G < 1) G = 1;
  }
  const long long min_ctas = (W + kMaxTilesPerCta - 1) / kMaxTilesPerCta;
  if (G < min_ctas) {
    if (force_ctas > 0) return MFA_ERR_INVALID_ARG;
    G = min_ctas;
  }
  if (G > INT_MAX / 2 || static_cast<long long>(pr->batch) + G - 1 > INT_MAX / 2) return MFA_ERR_INVALID_ARG;
  std::memset(plan, 0, sizeof(*plan));
  plan->num_ctas = static_cast<int32_t>(G);
  plan->tile_tokens = kTile;
  plan->max_tiles_per_cta = static_cast<int32_t>((W + G - 1) / G);
  plan->num_partials = static_cast<int32_t>(pr->batch + G - 1);
  plan->batch = pr->batch;
  plan->kv_dtype = pr->kv_dtype;
  plan->flags = flags;
  plan->num_sms = num_sms;
  plan->total_tiles = static_cast<uint64_t>(W);
  plan->workspace_bytes = workspace_bytes_for(plan->num_partials);
  return MFA_OK;
}

mfa_status mfa_decode_run(const mfa_plan* plan, const mfa_problem* pr, const void* q, const void* k_cache,
                          const void* v_cache, const float* k_scale, const float* v_scale,
                          const int32_t* block_table, const int32_t* seq_lens, void* out, float* lse,
                          void* workspace, uint64_t workspace_bytes, void* stream_ptr) {
  mfa_status st = check_problem(pr);
  if (st != MFA_OK) return st;
  st = check_plan(plan, pr);
  if (st != MFA_OK) return st;
  if (pr->batch == 0) return MFA_OK;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      seq_lens == nullptr || out == nullptr || workspace == nullptr)
    return MFA_ERR_INVALID_ARG;
  if (pr->kv_dtype == MFA_KV_FP8_E4M3 &&
      (k_scale == nullptr || v_scale == nullptr || !aligned(k_scale, 16) || !aligned(v_scale, 16)))
    return MFA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (lse != nullptr && !aligned(lse, 4)))
    return MFA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return MFA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  DecodeParams prm;
  std::memset(&prm, 0, sizeof(prm));
  st = encode_maps(prm, pr, q, k_cache, v_cache);
  if (st != MFA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.out = out;
  prm.out_f32 = pr->out_dtype == MFA_OUT_FP32 ? 1 : 0;
  prm.lse = lse;
  prm.part_o = reinterpret_cast<float*>(ws + partial_o_offset());
  prm.part_lse = reinterpret_cast<float*>(ws + partial_lse_offset(plan->num_partials));
  prm.status = reinterpret_cast<unsigned int*>(ws);
  prm.batch = pr->batch;
  prm.max_pages = pr->max_pages_per_seq;
  prm.num_blocks = pr->num_blocks;
  prm.scale_log2 = static_cast<float>(static_cast<double>(pr->softmax_scale) * 1.4426950408889634);
  prm.early_metadata = (plan->flags & MFA_PLAN_EARLY_METADATA) ? 1 : 0;

  const bool check = (plan->flags & MFA_PLAN_CHECK) != 0;
  cudaError_t e = cudaSuccess;
  if (check && (e = cudaMemsetAsync(ws, 0, 4, stream)) != cudaSuccess) return cuda_fail(e, "memset");
  const bool fp8 = pr->kv_dtype == MFA_KV_FP8_E4M3;
  auto kernel = fp8 ? mfa_decode_kernel<true> : mfa_decode_kernel<false>;
  const int smem = fp8 ? smem_bytes<true>() : smem_bytes<false>();
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan->num_ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, prm);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (plan->num_ctas > 1 && (plan->flags & MFA_PLAN_NO_COMBINE) == 0) {
    st = launch_combine(plan, pr, workspace, seq_lens, out, lse, stream, true);
    if (st != MFA_OK) return st;
  }
  if (check) {
    uint32_t word = 0;
    if ((e = cudaMemcpyAsync(&word, ws, 4, cudaMemcpyDeviceToHost, stream)) != cudaSuccess) return cuda_fail(e, "copy");
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "sync");
    if (word != 0) return MFA_ERR_DEVICE_CHECK;
  }
  return MFA_OK;
}

mfa_status mfa_combine(const mfa_plan* plan, const mfa_problem* pr, const void* workspace,
                       uint64_t workspace_bytes, const int32_t* seq_lens, void* out, float* lse,
                       void* stream_ptr) {
  mfa_status st = check_problem(pr);
  if (st != MFA_OK) return st;
  st = check_plan(plan, pr);
  if (st != MFA_OK) return st;
  if (pr->batch == 0) return MFA_OK;
  if (workspace == nullptr || seq_lens == nullptr || out == nullptr) return MFA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || !aligned(out, 16) || !aligned(seq_lens, 4) || (lse != nullptr && !aligned(lse, 4)))
    return MFA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return MFA_ERR_WORKSPACE;
  return launch_combine(plan, pr, workspace, seq_lens, out, lse, static_cast<cudaStream_t>(stream_ptr), false);
}

mfa_status mfa_read_device_status(void* workspace, uint32_t* status_bits, int32_t clear, void* stream_ptr) {
  if (workspace == nullptr || status_bits == nullptr || !aligned(workspace, 256)) return MFA_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, 4, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copy");
  if (clear && (e = cudaMemsetAsync(workspace, 0, 4, stream)) != cudaSuccess) return cuda_fail(e, "memset");
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_fail(e, "sync");
  *status_bits = word;
  return MFA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ workspace-free entry point
//
// Scratch for mfa_decode_run_static_workspace(): one fixed array per device that
// loads this library, held until the process exits.  In host code the symbol is
// only a stand-in; its device address comes from cudaGetSymbolAddress, looked up
// once per device with that device current.
static __device__ __align__(256) unsigned char g_static_workspace[MFA_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};
}  // namespace

extern "C" mfa_status mfa_decode_run_static_workspace(
    const mfa_plan* plan, const mfa_problem* pr, const void* q, const void* k_cache, const void* v_cache,
    const float* k_scale, const float* v_scale, const int32_t* block_table, const int32_t* seq_lens, void* out,
    float* lse, void* stream_ptr) {
  mfa_status st = check_problem(pr);
  if (st != MFA_OK) return st;
  st = check_plan(plan, pr);
  if (st != MFA_OK) return st;
  if (plan->workspace_bytes > MFA_STATIC_WORKSPACE_BYTES) return MFA_ERR_WORKSPACE;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return MFA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_static_workspace);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
      g_static_ptr[dev] = ptr;
    }
    ws = g_static_ptr[dev];
  }
  // the status word is the only part that must start at zero; partial results are
  // always written before they are read
  e = cudaMemsetAsync(ws, 0, 4, static_cast<cudaStream_t>(stream_ptr));
  if (e != cudaSuccess) return cuda_fail(e, "memset");
  return mfa_decode_run(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse, ws,
                        MFA_STATIC_WORKSPACE_BYTES, stream_ptr);
}
