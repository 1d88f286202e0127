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
//  * One CTA per SM (persistent).  The batch's 128-token tiles are laid end to end
//    and CTA g owns an equal share of their cost, a sequence boundary counting as 3/4
//    of a tile (bf16) or 2.5 tiles (e4m3), so the load is even for any length mix; a
//    sequence cut by a CTA
//    boundary yields partial results that the combine kernel merges (split-KV with a
//    log-sum-exp merge).
//  * Each CTA holds all 64 heads of its sequence, so K and V are read once.
//  * Warp 0 streams K/V pages with TMA (3-D tensor maps over the page pool; the
//    block table supplies the page coordinate) into a ring of shared-memory slots,
//    four ring uses at a time from four lanes.
//  * tcgen05 MMAs in the transposed form fill the M=128 datapath:
//    S^T[128 tokens x 64 heads] = K_tile . Q^T, issued by warp 1, and
//    O^T[256 d x 64 heads] += V^T . P^T (two M=128 halves), issued by another warp so
//    that a PV whose operands are ready never waits behind the issue of the next
//    tile's QK^T; fp32 accumulators in tensor memory (S double-buffered, O
//    double-buffered across sequences).
//  * Eight softmax warps (two per tensor-memory lane quarter, 32 heads each) run the
//    online softmax in fp32.  The running max is lazy: a head's reference max moves
//    only when a score exceeds it by 2^8, so the common tile needs no cross-thread
//    reduction; row sums accumulate per thread and are reduced once per sequence.
//  * e4m3 KV: q.K^T runs as a kind::f8f6f4 MMA on the e4m3 K boxes exactly as TMA
//    wrote them, against q split into e4m3 hi + lo parts (N = 128); four more warps
//    turn each V box into the f16 PV operand, with the token's V scale; K scales
//    multiply the fp32 scores.  A warpgroup register split gives the softmax warps
//    their registers.
//  * The ragged last page is loaded with its valid rows shifted to the end of the
//    box (negative row start; TMA fills the rest with zeros), so NaN or stale data
//    in unused page slots never enters an MMA.
//  * K and V uses share the ring.  With the two MMA streams in different threads, each
//    stream publishes in shared memory how many tiles of its uses have landed, and the
//    other waits on that count before it reuses a slot (an mbarrier parity would be
//    ambiguous for a waiter two phases behind).
//  * Multi-token decode (T new query tokens per sequence, causal among them): each
//    (sequence, token) pair is scheduled as its own sequence of length L - T + 1 + i
//    over the sequence's block-table row; its pages are read once per query token, all
//    but the last token's reads kept in L2 for the next.
//  * mfa_decode_run_host wraps one step with the copies of its host inputs and outputs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>
#include <algorithm>

#include "mfa.h"
#include "mfa_host.h"
#include "ptx.cuh"
#include "mfa_append_row.cuh"

namespace mfa {

constexpr int kH = 64;             // query heads a CTA holds (one unit)
constexpr int kD = 256;            // MFA head width

// Attention shapes.  MFA (the path) and the two designs the Step-3 page sets it against
// (section 5, "Attention Design"; section 7, attention ablation), run by the same kernel:
//   kShapeMfa: 64 query heads of width 256 over one K head and one V head (rows of 256);
//   kShapeGqa: 64 query heads of width 128 over 4 key/value heads (grouped-query attention:
//              cache rows of 4 x 128, query head h reads head h / 16);
//   kShapeMla: 128 query heads of width 512 over one 512-wide latent that is both the key
//              and the value (MLA-style, V = K); a CTA holds one unit of 64 heads, so a
//              sequence is two units.
enum : int { kShapeMfa = 0, kShapeGqa = 1, kShapeMla = 2 };
template <int kShp>
struct ShapeOf;
template <>
struct ShapeOf<kShapeMfa> {
  static constexpr int kRow = 256;      // elements of a cache row (all key/value heads of a token)
  static constexpr int kDq = 256;       // width of q and out per query head
  static constexpr int kGroups = 1;     // key/value heads per cache row
  static constexpr int kUnits = 1;      // 64-head units per sequence (per query token)
  static constexpr int kOBlocks = 2;    // O^T blocks of 128 d lanes x 64 columns per head set
  static constexpr int kOBufs = 2;      // O^T buffers (sequence switches overlap)
};
template <>
struct ShapeOf<kShapeGqa> {
  static constexpr int kRow = 512, kDq = 128, kGroups = 4, kUnits = 1;
  static constexpr int kOBlocks = 1;    // one 64-column block: group g's 16 heads at columns 16 g
  static constexpr int kOBufs = 2;
};
template <>
struct ShapeOf<kShapeMla> {
  static constexpr int kRow = 512, kDq = 512, kGroups = 1, kUnits = 2;
  static constexpr int kOBlocks = 4;    // 512 d = four blocks of 128 lanes: 256 columns
  static constexpr int kOBufs = 1;      // no room for a second buffer in tensor memory
};
constexpr int kPage = 64;          // tokens per KV page
constexpr int kTile = 128;         // tokens per pipeline tile (MMA M)
constexpr int kSoftmaxThreads = 256;  // two warps per TMEM lane quarter, 32 heads each
// bf16 and e4m3 caches: warp 0 TMA, warp 1 QK^T MMAs, warps 2..9 softmax, warp 10 PV MMAs
// (352 threads, 168 registers each).
// MXFP4 cache: warpgroup 0 = warp 0 TMA, warp 1 QK^T MMAs, warp 2 PV MMAs (warp 3 idle);
// warpgroups 1-2 = warps 4..11 softmax; warpgroup 3 = warps 12..15 convert the 4-bit pages
// into the e4m3 operand ring.  Launched with 128 registers per thread and rebalanced to
// 80 / 168 / 168 / 96 (the sum of the four is the launch's 4 x 128).
template <bool kMx>
__host__ __device__ constexpr int threads_of() { return kMx ? 512 : 352; }
template <bool kMx>
__host__ __device__ constexpr int pv_warp() { return kMx ? 2 : 10; }   // issues the PV MMAs
template <bool kMx>
__host__ __device__ constexpr int softmax_warp0() { return kMx ? 4 : 2; }
constexpr int kConvWarp0 = 12;       // MXFP4: first converter warp
constexpr int kConvThreads = 128;
constexpr uint32_t kRegsCtl = 80, kRegsSoftmax = 168, kRegsConv = 96;
static_assert(kRegsCtl + 2 * kRegsSoftmax + kRegsConv == 4 * (65536 / 512),
              "MXFP4 register split must add up to the launch budget (4 warpgroups x 128)");
constexpr int kMaxTilesPerCta = 128;
// Schedule cost units: a 128-token tile weighs kCostTile, a sequence boundary inside a CTA's
// range cost_seq (the next sequence's q and one more epilogue).  Measured per sequence switch:
// under a tile period for bf16, about two tile periods for e4m3 (whose q is converted and
// whose epilogue is not overlapped).
constexpr int kCostTile = 4;
__host__ __device__ constexpr int cost_seq(bool fp8) { return fp8 ? 10 : 3; }
constexpr int kMaxTokensPerSeq = 4;   // new query tokens per sequence (multi-token decode)
constexpr int kMaxSeg = kMaxTilesPerCta;
constexpr uint32_t kTmemCols = 512;
// Lazy running max (log2 domain): a head's reference max moves only when a score exceeds it
// by this much, so p <= 2^8 (bf16 weights) or p <= 2^3 (e4m3: the weight times the token's
// scaled V scale, below 2^5, must stay inside e4m3's 448) between rescales.
template <bool kFp8>
__host__ __device__ constexpr float rescale_threshold() { return kFp8 ? 3.0f : 8.0f; }
// e4m3: each token's V scale s_v is folded into its weights as s_v 2^(kPvShift - E), E the
// segment's reference exponent (every s_v so far below 2^(E + 1)); the output is scaled back by
// 2^(E - kPvShift).  kPvShift = 4 puts typical weights near 1, where both e4m3 parts of the
// weight are normal numbers, and keeps the largest (< 2^3 * 2 * 2^4) under 448.
constexpr int kPvShift = 4;
constexpr int kEMin = -120;   // floor of E (2^(kPvShift - E) stays a normal fp32 number)
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per pipeline wait

constexpr uint64_t kDrainLimitNs = 100000000ull;  // 0.1 s for drains after an abort

// Shared-memory map (offsets from a 1024-byte aligned base).  Both KV formats put the
// barriers at the same offset; they differ below it:
//   bf16 : Q 32 KB | P 16 KB | ring 10 x 16 KB (K/V operand tiles as TMA writes them)
//   e4m3 : Q 32 KB (e4m3 hi and lo parts) | P 16 KB (e4m3 weights: hi part 8 KB, lo part 8 KB) |
//          ring 20 x 8 KB (raw e4m3 boxes: both MMAs read K and V as TMA wrote them); the
//          per-token scales are read from global memory by the threads that apply them
constexpr int kOffQ = 0;                                     // kDq / 64 x [64 heads x 128 B]
constexpr int kOffBar = 212992;                              // mbarriers
// Q (bf16: 64 heads x kDq; e4m3: hi and lo parts, 32 KB), then P (16 KB: bf16 weights
// [128 tokens x 64 heads], or the e4m3 hi and lo parts), then the ring up to the barriers:
//   bf16: slots of 16 KB (a 64-element chunk of both pages of a tile for K; a 128-element
//         block of one page for V), kRow / 64 uses per tile for each of K and V;
//   e4m3: slots of 8 KB (one page's 128-element half row block), four uses each.
//   MXFP4: the e4m3 ring shrinks to 12 slots (K 8, V 4), filled by the converter warps; after
//          it, 8 staging slots of 8 KB hold 4-bit pages as TMA writes them ([64 tokens][128 B]
//          of E2M1 pairs, 128-byte swizzle), two tiles of loads in flight, and their E8M0 scale
//          bytes (512 B a page) sit past the metadata (kOffStageScale).
template <bool kFp8, int kShp, bool kMx = false>
struct Layout {
  using Sh = ShapeOf<kShp>;
  static constexpr int kOffP = kFp8 ? 32768 : 64 * Sh::kDq * 2;
  static constexpr int kOffRing = kOffP + 16384;
  static constexpr int kSlotBytes = kFp8 ? 8192 : 16384;
  static constexpr int kNumSlots = kMx ? 12 : (kOffBar - kOffRing) / kSlotBytes;
  static constexpr int kKU = kFp8 ? 4 : Sh::kRow / 64;   // ring uses per K group and per V group
  static constexpr int kOffStage = kOffRing + kNumSlots * kSlotBytes;   // MXFP4 staging slots
  static constexpr int kStageSlots = 8;
  static constexpr int kStageBytes = 8192;
};
static_assert(Layout<true, kShapeMfa, true>::kOffStage + 8 * 8192 == kOffBar, "MXFP4 staging fills the ring area");
static_assert(Layout<true, kShapeMfa, true>::kNumSlots + Layout<true, kShapeMfa, true>::kStageSlots <= 20,
              "MXFP4: the e4m3 ring and the staging slots share the 20 Full/Empty barrier pairs");
static_assert(Layout<true, kShapeMfa, true>::kNumSlots >= 12, "MXFP4: a K sub-ring of 8 and a V sub-ring of 4 or more");
static_assert(Layout<false, kShapeMfa>::kNumSlots == 10 && Layout<true, kShapeMfa>::kNumSlots == 20 &&
              Layout<false, kShapeGqa>::kNumSlots == 11 && Layout<false, kShapeMla>::kNumSlots == 8, "");
static_assert(Layout<false, kShapeMla>::kNumSlots >= Layout<false, kShapeMla>::kKU, "a ring holds one group");
// The e4m3 QK^T reads a d-half's two pages as one 128-row operand from two adjacent slots
// (uses 2k and 2k + 1 of an aligned group of four): they stay adjacent only for an even count.
static_assert(Layout<true, kShapeMfa>::kNumSlots % 4 == 0, "e4m3 ring: groups must not wrap");
constexpr int kOffMisc = kOffBar + 512;  // int: [0] tmem base [1] abort [2] nseg [3] ntiles [4..19] scan
                                         //      [20..21] CTA tile range [24..31] q maxima
// Ring-order counts.  K and V uses share one ring, and a consumer may only wait on a slot's
// Full barrier once the slot's previous use has landed: a waiter two phases behind would see
// the parity it wants and read a slot still being written.  With the QK^T and PV streams in
// different threads, some slots of tile n's K uses last held the V uses of an earlier tile
// (MFA bf16, 10 slots: V(n - 3); e4m3, 20 slots: V(n - 4)), and with a small ring some slots
// of tile m's V uses last held K uses of tile m + 1 (the 11- and 8-slot rings of the wider
// shapes), with no barrier between the two streams that orders them.  So each stream
// publishes how many tiles of its uses have landed -- cnt[0]: K tiles, by the QK^T issuer
// after its Full waits; cnt[1], cnt[2]: V tiles (page 0 and page 1, written together), by
// the PV issuer after its Full waits -- and waits on the other's count where the slot's
// previous use is not already ordered before it (needs_other: the count is exact -- a larger
// one could wait on a tile that itself waits for this stream's slots).
constexpr int kOffCnt = kOffBar + 448;   // int[4]: K tiles, V tiles of page 0 and of page 1 (one ring), K tiles issued (e4m3)
constexpr int kOffMref = kOffMisc + 128;      // float[64]  reference max per head (log2 domain)
constexpr int kOffAlpha = kOffMref + 256;     // float[64]  rescale factor per head
constexpr int kOffRed = kOffAlpha + 256;      // float[2][4][64] cross-warp reduction scratch
constexpr int kOffLinv = kOffRed + 2048;      // float[2][64]  1 / row sum per O buffer
constexpr int kOffSeg = kOffLinv + 512;       // int4[kMaxSeg] {b, first tile, end tile, L}
constexpr int kOffSegN0 = kOffSeg + 16 * kMaxSeg;       // int[kMaxSeg] CTA-local index of first tile
constexpr int kOffTileInfo = kOffSegN0 + 4 * kMaxSeg;   // int4[kMaxTilesPerCta] {page 0, page 1, rows 0, rows 1}
constexpr int kSmemUsed = kOffTileInfo + 16 * kMaxTilesPerCta;
constexpr int kOffStageScale = kSmemUsed;   // MXFP4: E8M0 bytes of the 8 staged pages, 512 B each
constexpr int smem_bytes(bool mx) { return kSmemUsed + (mx ? 8 * 512 : 0) + 1024; }
static_assert(smem_bytes(true) <= 232448, "shared memory budget");

// MXFP4 uses Full/Empty 0..11 for its e4m3 ring and 12..19 for the staging slots.
enum Bar : int {
  kBarFull = 0,
  kBarEmpty = kBarFull + 20,   // room for the larger ring
  kBarQFull = kBarEmpty + 20,
  kBarQEmpty,
  kBarSFull,   // 2
  kBarSEmpty = kBarSFull + 2,
  kBarPFull = kBarSEmpty + 2,
  kBarPvDone,
  kBarOFull,   // 2
  kBarOEmpty = kBarOFull + 2,
  kBarDrain = kBarOEmpty + 2,
  kBarQReady,   // e4m3: q split in place into e4m3 hi and lo parts
  kBarCount
};
static_assert(kBarCount * 8 <= kOffCnt - kOffBar, "barrier area (the ring-order counts follow it)");

// Tensor-memory columns.
constexpr uint32_t kTmemS = 0;     // S^T buffers [0,64) and [64,128) (e4m3: the hi-part and
                                   // lo-part products of q summed by the tensor core)
template <bool kFp8>
__host__ __device__ constexpr uint32_t s_cols() { return 64u; }
// O^T buffer k, block j: + 64 kOBlocks k + 64 j (MFA: d-halves; MLA: four 128-d blocks; GQA:
// one block whose columns 16 g .. 16 g + 15 hold the heads of key/value head g)
template <bool kFp8>
__host__ __device__ constexpr uint32_t tmem_o() { return kFp8 ? 256u : 128u; }
constexpr uint32_t kTmemL = 384;   // bf16: per-lane row sums of the bf16-rounded weights (normalise O)
constexpr uint32_t kTmemLx = 448;  // bf16: per-lane row sums of the fp32 weights (lse)

struct DecodeParams {
  CUtensorMap tm_q;   // 2-D [B*64 rows, 256] bf16, box 64x64, 128B swizzle
  CUtensorMap tm_k;   // 3-D [num_blocks, 64, 256]: bf16 box {64, 64, 1}, e4m3 box {128, 64, 1};
                      // MXFP4 [num_blocks, 64, 128 B of E2M1 pairs], box {128, 64, 1}; 128B swizzle
  CUtensorMap tm_v;
  const void* k_scale;   // e4m3: fp32 [num_blocks, 64]; MXFP4: E8M0 bytes [num_blocks, 64, 8]
  const void* v_scale;
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
  int tokens;         // new query tokens per sequence T
  int units;          // 64-head units per query token U: batch counts the B * T * U units
  // fused KV append (one new token per sequence, MFA rows; k_new null: none): row b of k_new
  // and v_new goes to slot positions[b] of sequence b, in the cache's format (kv_fmt)
  const uint4* k_new;
  const uint4* v_new;
  const int32_t* positions;
  void* k_cache_w;
  void* v_cache_w;
  void* k_scale_w;
  void* v_scale_w;
  int kv_fmt;
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
  int tokens;         // as DecodeParams::tokens
  int units;          // as DecodeParams::units
  int seq_cost;       // cost_seq of the KV format: the decode kernel's split
};

// ------------------------------------------------------------------ helpers

// tcgen05 shared-memory matrix descriptor: start, leading/stride byte offsets,
// descriptor version 1 (bits 46..47), 128-byte swizzle (bits 61..63 = 2).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// The same with the 64-byte swizzle (layout code 4): 64-byte rows, 8-row atoms of 512 bytes,
// 16-byte chunk c of row r stored at chunk c ^ ((r >> 1) & 3).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (4ull << 61);
}

// tcgen05 instruction descriptor for kind::f16: fp32 D, bf16 or f16 A/B,
// K-major (0) or MN-major (1) operands, N>>3 at bit 17, M>>4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool a_mn, bool b_mn, int m, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// tcgen05 instruction descriptor for kind::f8f6f4 with e4m3 A and B (format code 0),
// fp32 D, K-major (0) or MN-major (1) operands.
__host__ __device__ constexpr uint32_t idesc_e4m3(bool a_mn, bool b_mn, int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ int clamp_len(int L, int cap, bool& bad) {
  if (L < 0) { bad = true; return 0; }
  if (L > cap) { bad = true; return cap; }
  return L;
}

__device__ __forceinline__ int tiles_of(int L) { return (L + kTile - 1) / kTile; }

// Units.  With T new query tokens per sequence (the last T of its L cached tokens) and U
// 64-head units per query token, unit x = (b T + i) U + u is head set u of query token i of
// sequence b: it reads b's block-table row and attends to the cached tokens 0 .. L - T + i
// (length L - T + 1 + i), which is the causal mask among the new tokens.  T = U = 1 is the
// ordinary MFA decode step (x = b, length L).
__device__ __forceinline__ int seq_of(int x, int T, int U) { return (T == 1 && U == 1) ? x : x / (T * U); }
__device__ __forceinline__ int raw_len(const int32_t* lens, int T, int U, int x) { return lens[seq_of(x, T, U)]; }
__device__ __forceinline__ int vlen_from(int L_raw, int T, int U, int x, int cap, bool& bad) {
  const int L = clamp_len(L_raw, cap, bad);
  return T == 1 ? L : max(0, L - (T - 1 - (x / U) % T));
}
// Schedule order.  With R = T U > 1 units reading each sequence's pages, the cost-balanced
// schedule walks the Bv units reader-major: position pos = r (Bv / R) + b holds unit
// x = b R + r.  With readers of equal cost, the CTAs that hold readers r and r' of sequence b
// then sit at the same place in their cost ranges (exactly so for an even split), so a page's
// readers load it at about the same time and all but the first find it in L2.  Partial slots
// are numbered by position (pos + CTA).
__device__ __forceinline__ int unit_at(int pos, int T, int U, int Bv) {
  const int R = T * U;
  if (R == 1) return pos;
  const int Bs = Bv / R;
  return (pos % Bs) * R + pos / Bs;
}
__device__ __forceinline__ int pos_of(int x, int T, int U, int Bv) {
  const int R = T * U;
  return R == 1 ? x : (x % R) * (Bv / R) + x / R;
}

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

// Bounded wait until a monotonic shared-memory count reaches target (see the ring-order
// counts in the kernel); sets the abort flag when it gives up.
__device__ __forceinline__ bool wait_count(const int* count, int target, volatile int* abort_flag) {
  if (ld_acquire_cta(count) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(32);
    if (ld_acquire_cta(count) >= target) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_count_warp(const int* count, int target, volatile int* abort_flag) {
  const bool ok = wait_count(count, target, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Block-wide (kThreads threads) inclusive scan of one value per thread; also returns the total.
template <int kThreads, typename V = int>
__device__ __forceinline__ V block_incl_scan(V v, V* scratch, V& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  V before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const V x = scratch[w];
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

// Two floats to two e4m3 codes (round to nearest even, saturating); lo in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Split two scaled q values x into e4m3 pairs hi + lo with hi = e4m3(x) and lo = e4m3(x - hi).
// x is a bf16 value times a power of two (8 significant bits) and the largest |x| of the
// sequence lies in [64, 128).  x - hi is exact in fp32 and is k * ulp(x) with |k| <= 8, so
// it fits e4m3's 4 significant bits: hi + lo = x exactly when ulp(x) >= 2^-9 (the e4m3
// subnormal step), i.e. for |x| >= 2^-2, which covers every element at least 2^-9 of the
// largest.  Smaller elements err by at most 2^-10, under 2^-16 of the largest.
// (The hi part is read back exactly through the f16 conversion.  A bit-placement read-back,
// the 7 magnitude bits at bit 20 of an fp32 word times 2^120, gives the same bits, but the
// conversion measured faster end to end -- finishing a segment's q split earlier moves the
// CTAs' load streams into a worse phase.)
__device__ __forceinline__ void split_e4m3(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_e4m3_sat(x0, x1);
  uint32_t back;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(back) : "h"(static_cast<uint16_t>(hi)));
  lo = pack_e4m3_sat(x0 - __half2float(__ushort_as_half(static_cast<unsigned short>(back))),
                     x1 - __half2float(__ushort_as_half(static_cast<unsigned short>(back >> 16))));
}

// e4m3: per-token scale of box row ri of page pg of tile `ti` ({page 0, page 1, rows 0,
// rows 1}); 0 for rows past the sequence end and for a page id outside the pool (the last page's valid rows sit at the end of
// the box, so box row ri holds page row ri - (64 - rows)).
__device__ __forceinline__ float token_scale(const float* __restrict__ sc, const int4 ti, int pg, int ri) {
  const int r = pg ? ti.w : ti.z;
  const int blk = pg ? ti.y : ti.x;   // -1: an id outside the pool (its page reads as zeros)
  if (r <= 0 || ri < kPage - r || blk < 0) return 0.f;
  return __ldg(sc + static_cast<size_t>(blk) * kPage + ri - (kPage - r));
}

// MXFP4 (OCP MX FP4: E2M1 elements, one E8M0 scale byte 2^(e - 127) per 32 elements of a
// row).  A token row's reference exponent is its largest scale byte minus 6, at least 1
// (biased).  The converter stores each element as the e4m3 code of its value over
// 2^(ref - 127): an E2M1 value is at most 6 times its block's scale, so the row's codes stay
// at or under 6 x 2^6 = 384, inside e4m3's 448, and the token's scale 2^(ref - 127) is a
// normal fp32 power of two that the softmax applies as it does an e4m3 row scale.
__device__ __forceinline__ int mx_ref_exp(uint2 s8) {
  const uint32_t m = __vmaxu4(s8.x, s8.y);
  const uint32_t m2 = max(max(m & 0xFFu, (m >> 8) & 0xFFu), max((m >> 16) & 0xFFu, m >> 24));
  return max(static_cast<int>(m2) - 6, 1);
}
// A row's scale is loaded one tile ahead as raw bits (e4m3: the fp32 scale; MXFP4: the 8 scale
// bytes, zeros for a row past the sequence end or outside the pool, which the softmax masks)
// and turned into the fp32 scale only where it is used, so that no thread waits on the load.
template <bool kMx>
__device__ __forceinline__ uint2 kv_scale_raw(const void* sc, const int4 ti, int pg, int ri) {
  if constexpr (kMx) {
    const int r = pg ? ti.w : ti.z;
    const int blk = pg ? ti.y : ti.x;
    if (r <= 0 || ri < kPage - r || blk < 0) return make_uint2(0u, 0u);
    return __ldg(reinterpret_cast<const uint2*>(sc) + static_cast<size_t>(blk) * kPage + ri - (kPage - r));
  } else {
    return make_uint2(__float_as_uint(token_scale(static_cast<const float*>(sc), ti, pg, ri)), 0u);
  }
}
template <bool kMx>
__device__ __forceinline__ float kv_scale_of(uint2 raw) {
  if constexpr (kMx)
    return __uint_as_float(static_cast<uint32_t>(mx_ref_exp(raw)) << 23);
  else
    return __uint_as_float(raw.x);
}

// MXFP4 -> e4m3 for one 32-element block: w holds the block's 32 E2M1 codes (element 2i in
// the low nibble of byte i), D = the block's scale byte minus the row's reference exponent
// (at most 6).  Output: 32 e4m3 codes of E2M1(x) * 2^D, element i in byte i.  The magnitude
// of each nibble is looked up by prmt in an 8-byte table (e4m3 codes of 0, 0.5, ..., 6 times
// 2^D) and its sign bit copied to bit 7.  For D >= -5 every nonzero table entry is a normal
// e4m3 number, the code of m 2^D being the code of m plus 8 D; below that the table is built
// by rounding each value to e4m3 (exact down to D = -8; smaller blocks round to e4m3's
// subnormal grid of 2^-9, relative to the row's largest block at most 2^-16 of its scale).
__device__ __forceinline__ void mx_block_to_e4m3(const uint4 w, int D, uint4& out0, uint4& out1) {
  uint32_t l0, l1;
  if (D >= -5) {
    // e4m3 codes of 0, 0.5, 1, 1.5 and of 2, 3, 4, 6, every nonzero byte's exponent moved by D
    l0 = 0x3C383000u + static_cast<uint32_t>(D) * 0x08080800u;
    l1 = 0x4C484440u + static_cast<uint32_t>(D) * 0x08080808u;
  } else {
    const float f = D >= -126 ? __uint_as_float(static_cast<uint32_t>(D + 127) << 23) : 0.f;
    uint16_t a, b, c, d;
    // (the first source goes to the high byte of each pair)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(a) : "f"(0.5f * f), "f"(0.0f));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(b) : "f"(1.5f * f), "f"(1.0f * f));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(3.0f * f), "f"(2.0f * f));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(6.0f * f), "f"(4.0f * f));
    l0 = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);   // bytes: 0, 0.5, 1, 1.5
    l1 = static_cast<uint32_t>(c) | (static_cast<uint32_t>(d) << 16);   // bytes: 2, 3, 4, 6
  }
  auto eight = [&](uint32_t x, uint32_t& lo, uint32_t& hi) {
    // lo: elements 0..3 of x (nibbles 0..3), hi: elements 4..7; the sign of nibble k is bit
    // 4k + 3 of x: the msb of byte k/2 of (x << 4) for even k, of x for odd k, which prmt's
    // sign-replicate selectors (bit 3 set) spread over an output byte
    const uint32_t xs = x << 4;
    uint32_t m0, m1, s0, s1;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(m0) : "r"(l0), "r"(l1), "r"(x & 0x7777u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(m1) : "r"(l0), "r"(l1), "r"((x >> 16) & 0x7777u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s0) : "r"(xs), "r"(x), "r"(0xD9C8u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s1) : "r"(xs), "r"(x), "r"(0xFBEAu));
    lo = m0 | (s0 & 0x80808080u);
    hi = m1 | (s1 & 0x80808080u);
  };
  eight(w.x, out0.x, out0.y);
  eight(w.y, out0.z, out0.w);
  eight(w.z, out1.x, out1.y);
  eight(w.w, out1.z, out1.w);
}

// Ring use index of the first use of the K (is_v = false) or V group of tile t of a CTA with
// `ntiles` tiles, kKU uses per group.  The producer issues K(0), then K(t) and V(t-1) for
// t = 1..N-1, then V(N-1): K(0) = 0.., K(t) = 2 kKU t - kKU.., V(t) = 2 kKU t + 2 kKU.. except
// the last tile's V, which directly follows its K: V(N-1) = 2 kKU N - kKU...
template <int kKU>
__device__ __forceinline__ uint32_t ring_use(int t, int ntiles, bool is_v) {
  constexpr uint32_t U = kKU;
  return is_v ? (t + 1 < ntiles ? 2u * U * t + 2u * U : 2u * U * t + U) : (t == 0 ? 0u : 2u * U * t - U);
}
// The inverse: the tile (and whether V) of the g-th group of uses in the producer's order.
__device__ __forceinline__ int group_owner(int g, int ntiles, bool& is_v) {
  is_v = (g & 1) == 0 ? g > 0 : (g + 1) / 2 >= ntiles;
  return !is_v ? (g + 1) / 2 : ((g & 1) == 0 ? g / 2 - 1 : ntiles - 1);
}
// How many tiles of the other stream (V if want_v, else K) must have landed before the group
// at ring use a may be waited on: the highest such tile among the previous uses of its slots,
// plus one (zero if none).
template <int kKU, int kSlots>
__device__ __forceinline__ int needs_other(int a, int ntiles, bool want_v) {
  const int hi = a + kKU - 1 - kSlots;
  if (hi < 0) return 0;
  int need = 0;
#pragma unroll 1
  for (int g = max(a - kSlots, 0) / kKU; g <= hi / kKU; ++g) {
    bool v;
    const int t = group_owner(g, ntiles, v);
    if (v == want_v) need = max(need, t + 1);
  }
  return need;
}

// The e4m3 operand slots (e4m3 and MXFP4 caches) form two sub-rings: K in slots 0..7 (two
// tiles), V in slots 8..kSlots-1 (e4m3: three tiles, MXFP4: two).  Each stream's uses only
// follow its own earlier uses, so V is issued as soon as PV has released V slots, not when
// QK^T frees K's (V's late arrival bound the e4m3 tile period), and a stream's waiter can
// never be a phase behind (no ring-order counts).  Use u = 4 t + c of tile t: K use c = page
// c & 1, d-half c >> 1 (a d-half's two pages in adjacent slots, one 128-row MMA operand); V
// use c = page c >> 1, d-half c & 1.
constexpr uint32_t kKSub = 8;
template <int kSlots>
constexpr uint32_t kVSub = kSlots > static_cast<int>(kKSub) ? kSlots - kKSub : 1u;   // (only e4m3 rings use it)
template <int kSlots>
__device__ __forceinline__ uint32_t sub_slot(uint32_t u, bool is_v) {
  return is_v ? kKSub + u % kVSub<kSlots> : u % kKSub;
}
template <int kSlots>
__device__ __forceinline__ uint32_t sub_phase(uint32_t u, bool is_v) {
  return (is_v ? u / kVSub<kSlots> : u / kKSub) & 1u;
}

// Fused KV append of sequence b's new row at token t (a warp): the page id, then the K and V
// rows in the cache's format.  A position past the block table or a page id outside the pool
// is reported and the row is skipped, as by the append kernel.
// Sequence b's new K and V rows into slot t % 64 of pool page blk (one warp).
__device__ __noinline__ void append_row_at(const DecodeParams& p, int b, int t, int blk, int lane) {
  const size_t row = static_cast<size_t>(blk) * kPage + (t % kPage);
  const uint4 xk = p.k_new[static_cast<size_t>(b) * (kRowElems / 8) + lane];
  const uint4 xv = p.v_new[static_cast<size_t>(b) * (kRowElems / 8) + lane];
  append_row_warp(p.kv_fmt, xk, lane, p.k_cache_w, p.k_scale_w, row);
  append_row_warp(p.kv_fmt, xv, lane, p.v_cache_w, p.v_scale_w, row);
}
__device__ __noinline__ void fused_append_row(const DecodeParams& p, int b, int t, int lane) {
  if (t >= p.max_pages * kPage) {
    if (lane == 0 && p.status) atomicOr(p.status, MFA_DEV_BAD_LENGTH);
    return;
  }
  const int blk = p.block_table[static_cast<size_t>(b) * p.max_pages + t / kPage];
  if (blk < 0 || blk >= p.num_blocks) {
    if (lane == 0 && p.status) atomicOr(p.status, MFA_DEV_BAD_BLOCK);
    return;
  }
  append_row_at(p, b, t, blk, lane);
}

// kFp8: both contractions on e4m3 operands (an e4m3 cache, or an MXFP4 cache converted to
// e4m3 on chip: kMx).
template <bool kFp8, int kShp, bool kMx = false>
__global__ void __launch_bounds__(threads_of<kMx>(), 1) mfa_decode_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(!kFp8 || kShp == kShapeMfa, "the e4m3 cache is built for the MFA shape");
  static_assert(!kMx || kFp8, "the MXFP4 path runs on the e4m3 MMAs");
  static_assert(threads_of<kMx>() >= kMaxTilesPerCta + kMaxSeg, "page ids and append positions load in one round");
  using Lay = Layout<kFp8, kShp, kMx>;
  using Sh = ShapeOf<kShp>;
  constexpr int kThreads = threads_of<kMx>();
  constexpr int kNumSlots = Lay::kNumSlots;
  constexpr int kSlotBytes = Lay::kSlotBytes;
  constexpr int kOffRing = Lay::kOffRing;
  constexpr int kOffP = Lay::kOffP;
  constexpr int kKU = Lay::kKU;
  constexpr int kQBoxes = Sh::kDq / 64;          // 64-wide q boxes of a unit (bf16)
  constexpr int kVBlocks = Sh::kRow / 128;       // bf16 V uses of one page (128-element blocks)
  constexpr int kNh = 64 / Sh::kGroups;          // query heads per key/value head in a unit
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  int* misc = reinterpret_cast<int*>(smem + kOffMisc);
  int* cnt = reinterpret_cast<int*>(smem + kOffCnt);   // ring-order counts
  volatile int* abort_flag = misc + 1;
  int4* seg = reinterpret_cast<int4*>(smem + kOffSeg);
  int* seg_n0 = reinterpret_cast<int*>(smem + kOffSegN0);
  int4* tile_info = reinterpret_cast<int4*>(smem + kOffTileInfo);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };

  // the unit at schedule position pos (unit_at)
  auto unit_of = [&](int pos) { return unit_at(pos, p.tokens, p.units, p.batch); };
  // With early metadata the lengths are read before anything else: the schedule below
  // waits on them and on nothing the set-up does.
  int L_first = 0;   // raw length of the unit at schedule position tid
  if (p.early_metadata && tid < p.batch) L_first = raw_len(p.seq_lens, p.tokens, p.units, unit_of(tid));

  // ---------------- set-up: barriers (one per lane of warp 0), tensor memory
  if (warp == 0) {
    for (int i = lane; i < kBarCount; i += 32) {
      // arrivals per phase: the softmax threads for the barriers they release, one commit
      // from each MMA issuer for the drain, and one (a commit or an expect_tx arrive) for
      // the others
      uint32_t count = 1;
      if (i == kBarSEmpty || i == kBarSEmpty + 1 || i == kBarOEmpty || i == kBarOEmpty + 1 ||
          i == kBarPFull || i == kBarQReady)
        count = kSoftmaxThreads;
      else if (i == kBarDrain)
        count = 2;
      else if (kMx && i >= kBarFull && i < kBarFull + kNumSlots)
        count = 2;   // MXFP4 e4m3 ring: the two converter warps that write a slot's rows
      else if (kMx && i >= kBarEmpty + kNumSlots && i < kBarEmpty + kNumSlots + Lay::kStageSlots)
        count = kConvThreads / 32;   // MXFP4 staging: every converter warp reads every slot
      mbar_init(bar(i), count);
    }
    if (lane == 0) {
      misc[1] = 0;
      for (int i = 0; i < 4; ++i) cnt[i] = 0;
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32 * 2) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }

  // Launched as a programmatic dependent of the preceding kernel on the stream: nothing
  // that kernel may write is touched before griddepcontrol.wait.  With early metadata
  // the lengths and the block table are read first (the caller guarantees the preceding
  // kernel does not write them); q, K, V and every output wait.
  if (!p.early_metadata) {
    grid_dep_wait();
    if (tid < p.batch) L_first = raw_len(p.seq_lens, p.tokens, p.units, unit_of(tid));
  }

  // ---------------- schedule: this CTA's tile range and its per-sequence segments
  // Cost-balanced split: tile k of sequence b sits at cost 4 (S_b + k) + c N_b, S_b being the
  // tiles and N_b the non-empty sequences before b, c = cost_seq: a sequence boundary inside
  // a CTA's range weighs c/4 of a tile.  CTA g owns the tiles whose cost lies in
  // [floor(g C / G), floor((g + 1) C / G)), C = 4 W + c (N - 1): a contiguous run of tiles, in
  // sequence order across CTAs.  Tile counts and non-empty counts are scanned together (low
  // and high 32 bits).
  constexpr long long kSeqW = cost_seq(kFp8);
  const int cap = p.max_pages * kPage;
  {
    long long* scratch = reinterpret_cast<long long*>(smem + kOffRed);   // idle until the softmax
    int* tb = misc + 20;   // [0] first tile, [1] end tile of this CTA (written by their owners)
    bool bad = false;
    auto packed = [](int T) { return static_cast<long long>(T) | (static_cast<long long>(T > 0) << 32); };
    long long loc = 0;
    // L_first (read above) is reused by the segment scan below
    loc += packed(tiles_of(tid < p.batch ? vlen_from(L_first, p.tokens, p.units, unit_of(tid), cap, bad) : 0));
    for (int b = tid + kThreads; b < p.batch; b += kThreads) {
      const int x = unit_of(b);
      loc += packed(tiles_of(vlen_from(raw_len(p.seq_lens, p.tokens, p.units, x), p.tokens, p.units, x, cap, bad)));
    }
    if (bad) atomicOr(p.status, MFA_DEV_BAD_LENGTH);
    long long tot0 = 0;
    const long long incl0 = block_incl_scan<kThreads, long long>(loc, scratch, tot0);
    const int W = static_cast<int>(tot0 & 0xFFFFFFFFll), N = static_cast<int>(tot0 >> 32);
    const int G = gridDim.x, g = blockIdx.x;
    const long long C = kCostTile * static_cast<long long>(W) + kSeqW * max(N - 1, 0);
    long long X0, X1;
    if (C <= 0x7FFFFFFFll / G) {   // (g + 1) C fits in 32 bits: the short division
      const uint32_t Cu = static_cast<uint32_t>(C), Gu = static_cast<uint32_t>(G), gu = static_cast<uint32_t>(g);
      X0 = (gu * Cu) / Gu;
      X1 = ((gu + 1u) * Cu) / Gu;
    } else {
      X0 = (static_cast<long long>(g) * C) / G;
      X1 = (static_cast<long long>(g + 1) * C) / G;
    }
    // sequence with first-tile cost `base` and T tiles: first of its tiles at cost >= X
    auto first_at = [](long long X, long long base, int T) -> int {
      return X <= base ? 0 : static_cast<int>(min(static_cast<long long>(T), (X - base + kCostTile - 1) / kCostTile));
    };
    // this sequence's contribution to the CTA's [first, end) tiles: the non-empty sequence
    // whose cost span [base, next base) holds X0 (X1) fixes the first (end) tile.  Those spans
    // tile [0, C) exactly, so only X = C (X1 of the last CTA) has no owner: it stands for W.
    auto mark_bounds = [&](long long base, int S, int T) {
      if (T == 0) return;
      const long long nxt = base + kCostTile * static_cast<long long>(T) + kSeqW;
      if (base <= X0 && X0 < nxt) tb[0] = S + first_at(X0, base, T);
      if (base <= X1 && X1 < nxt) tb[1] = S + first_at(X1, base, T);
    };
    int nseg = 0, t0 = 0, t1 = 0;
    if (p.batch <= kThreads) {
      // one sequence per thread: its tiles are [S, S + T) of the first scan; the sequences
      // overlapping the CTA are numbered by a ballot count
      bool dummy = false;
      const int L = (tid < p.batch) ? vlen_from(L_first, p.tokens, p.units, unit_of(tid), cap, dummy) : 0;
      const int T = tiles_of(L);
      const long long ex = incl0 - packed(T);
      const int S = static_cast<int>(ex & 0xFFFFFFFFll), Nb = static_cast<int>(ex >> 32);
      const long long base = kCostTile * static_cast<long long>(S) + kSeqW * Nb;
      if (tid < p.batch) mark_bounds(base, S, T);
      const int k_lo = first_at(X0, base, T), k_hi = first_at(X1, base, T);
      const bool f = (tid < p.batch) && (k_lo < k_hi);
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (lane == 0) misc[4 + warp] = __popc(m);
      __syncthreads();
      t0 = (X0 < C) ? tb[0] : W;
      t1 = (X1 < C) ? tb[1] : W;
      int before = 0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) {
        const int x = misc[4 + w];
        before += (w < warp) ? x : 0;
        nseg += x;
      }
      if (t1 - t0 > kMaxTilesPerCta) {
        if (tid == 0) atomicOr(p.status, MFA_DEV_SCHEDULE);
        nseg = 0;
      } else if (f) {
        const int fidx = before + __popc(m & ((1u << lane) - 1u));
        seg[fidx] = make_int4(unit_of(tid), k_lo, k_hi, L);
        seg_n0[fidx] = S + k_lo - t0;
      }
    } else {
      // pass 1: the CTA's first and end tiles (sequences beyond cost X1 cannot matter)
      long long carry = 0;
      auto cost_of = [](long long pk) { return kCostTile * (pk & 0xFFFFFFFFll) + kSeqW * (pk >> 32); };
      for (int c0 = 0; c0 < p.batch && cost_of(carry) <= X1; c0 += kThreads) {
        const int b = c0 + tid;
        bool dummy = false;
        const int x = unit_of(b);
        const int L = (b < p.batch) ? vlen_from(c0 == 0 ? L_first : raw_len(p.seq_lens, p.tokens, p.units, x), p.tokens, p.units, x, cap, dummy) : 0;
        const int T = tiles_of(L);
        long long tot = 0;
        const long long ex = block_incl_scan<kThreads, long long>(packed(T), scratch, tot) + carry - packed(T);
        if (b < p.batch) mark_bounds(cost_of(ex), static_cast<int>(ex & 0xFFFFFFFFll), T);
        carry += tot;
      }
      __syncthreads();
      t0 = (X0 < C) ? tb[0] : W;
      t1 = (X1 < C) ? tb[1] : W;
      if (t1 - t0 > kMaxTilesPerCta) {
        if (tid == 0) atomicOr(p.status, MFA_DEV_SCHEDULE);
      } else {
        // pass 2: the segments
        carry = 0;
        for (int c0 = 0; c0 < p.batch && (carry & 0xFFFFFFFFll) < t1; c0 += kThreads) {
          const int b = c0 + tid;
          bool dummy = false;
          const int x = unit_of(b);
          const int L = (b < p.batch) ? vlen_from(c0 == 0 ? L_first : raw_len(p.seq_lens, p.tokens, p.units, x), p.tokens, p.units, x, cap, dummy) : 0;
          const int T = tiles_of(L);
          long long tot = 0;
          const long long ex = block_incl_scan<kThreads, long long>(packed(T), scratch, tot) + carry - packed(T);
          const int S = static_cast<int>(ex & 0xFFFFFFFFll);
          const long long base = cost_of(ex);
          const int k_lo = first_at(X0, base, T), k_hi = first_at(X1, base, T);
          const int f = (b < p.batch && k_lo < k_hi) ? 1 : 0;
          int ftot = 0;
          const int fidx = nseg + block_incl_scan<kThreads>(f, misc + 4, ftot) - f;
          if (f) {
            seg[fidx] = make_int4(x, k_lo, k_hi, L);
            seg_n0[fidx] = S + k_lo - t0;
          }
          carry += tot;
          nseg += ftot;
        }
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
  int* app_t = reinterpret_cast<int*>(smem + kOffRed);   // [nseg] fused-append positions (scratch
                                                         // idle until the softmax)
  // ---------------- page ids and valid rows of each of this CTA's tiles (one round of
  // independent loads, one tile per thread).  Rows r of a page: the last page of a sequence
  // has r < 64 (its valid rows land at the end of the box), an absent second page r <= 0.
  {
    bool bad_blk = false;
    for (int n = tid; n < ntiles; n += kThreads) {
      int s = 0;
      while (s + 1 < nseg && seg_n0[s + 1] <= n) ++s;
      const int4 sg = seg[s];
      const int j = sg.y + (n - seg_n0[s]);
      const int r0 = min(kPage, sg.w - kTile * j), r1 = min(kPage, sg.w - kTile * j - kPage);
      const int32_t* row = p.block_table + static_cast<size_t>(seq_of(sg.x, p.tokens, p.units)) * p.max_pages;
      int b0 = row[2 * j];
      int b1 = (r1 > 0) ? row[2 * j + 1] : 0;
      // an id outside the pool is reported and replaced by -1: the TMA box then lies wholly
      // outside the pool and lands as zeros, and an e4m3 page's scales read as 0, so that
      // page contributes zero keys and zero values and no other page's data
      if (b0 < 0 || b0 >= p.num_blocks) { bad_blk = true; b0 = -1; }
      if (r1 > 0 && (b1 < 0 || b1 >= p.num_blocks)) { bad_blk = true; b1 = -1; }
      tile_info[n] = make_int4(b0, b1, r0, r1);
    }
    if (bad_blk) atomicOr(p.status, MFA_DEV_BAD_BLOCK);
    // fused KV append: each segment's new-row position, loaded in the same round by the
    // threads past the page-id ones (with early metadata, before the dependency wait)
    if (p.k_new != nullptr && tid >= kMaxTilesPerCta && tid - kMaxTilesPerCta < nseg)
      app_t[tid - kMaxTilesPerCta] = p.positions[seg[tid - kMaxTilesPerCta].x];
  }
  // ---------------- fused KV append, rows this CTA reads: a sequence's new row at token t <
  // its visible length is written by the CTA that owns tile t / 128 (one segment holds it),
  // before any of that CTA's loads, into the page id the tile already holds.  Warp w takes
  // segments w, w + warps, ...  The rows are fenced to the async proxy, which reads them
  // (TMA), and the block barrier below orders them before the other warps' loads of the
  // per-row scales.  (Rows past the visible length are read by nobody this step; the PV
  // warp writes those.)
  if (p.k_new != nullptr && nseg > 0) {
    __syncthreads();   // app_t and tile_info
    grid_dep_wait();   // the new rows (and the cache) may come from the preceding kernel
    for (int s = warp; s < nseg; s += kThreads / 32) {
      const int4 sg = seg[s];
      const int t = app_t[s];
      if (t >= 0 && t < sg.w && t >= kTile * sg.y && t < kTile * sg.z) {
        const int4 ti = tile_info[seg_n0[s] + t / kTile - sg.y];
        const int blk = ((t / kPage) & 1) ? ti.y : ti.x;
        if (blk >= 0) append_row_at(p, sg.x, t, blk, lane);   // (-1: reported above, page reads as zeros)
      }
    }
    fence_proxy_async_global();
  }
  __syncthreads();

  // MXFP4 warpgroup register split (see threads_of), at the top of each role so that the
  // role's budget covers all of its code: the control warps and the converters give
  // registers up, the softmax warpgroups take them
  if (warp == 0) {
    if constexpr (kMx) reg_dealloc<kRegsCtl>();
    // ---------------- producer: TMA loads of Q, K and V in ring order.  Each group of four
    // ring uses (a tile's K, or a tile's V) is issued by lanes 0..3 together, one use per
    // lane; groups go out strictly in ring order, so every slot's phases stay in step.
    // MXFP4: the groups go to the staging ring instead, two uses (one per page) each, by
    // lanes 0..1: a page's 8 KB of E2M1 pairs by TMA and its 512 scale bytes by a bulk copy.
    if (ntiles > 0) {
      if (p.early_metadata) grid_dep_wait();
      // KV is streamed once: evict first.  Multi-token decode reads a sequence's pages once
      // per query token, the pairs back to back, so all but the last query token's reads keep
      // the lines (evict last) for the next one.
      const uint64_t pol_once = l2_policy_evict_first(), pol_again = l2_policy_evict_last();
      int seg_k = 0, seg_v = 0;   // segment of the producer's current K and V tiles
      const bool act = lane < (kMx ? 2 : kKU);
      const int c = lane;
      bool ok = true;
      int sq = 0, nq = 0;                 // next segment whose q is loaded; q loads issued
      uint32_t mine[3] = {0u, 0u, 0u};    // this lane's last three uses (drain after an abort)
      int nmine = 0;
      // (one ring, bf16) lane c: use c of the group (K: 64-element chunk c of both pages; V:
      // page c / kVBlocks, 128-element block c % kVBlocks); the e4m3 path has its own loop below
      const int reads = p.tokens * p.units;   // units that read one sequence's pages
      auto group = [&](bool is_v, int t) -> bool {
        bool okl = true;
        int& sc_ = is_v ? seg_v : seg_k;
        while (sc_ + 1 < nseg && seg_n0[sc_ + 1] <= t) ++sc_;
        const uint64_t pol = (reads > 1 && seg[sc_].x % reads != reads - 1) ? pol_again : pol_once;
        if constexpr (kMx) {
          if (act) {
            const int4 ti = tile_info[t];
            const uint32_t u = ring_use<2>(t, ntiles, is_v) + c;
            const uint32_t slot = u % Lay::kStageSlots;
            okl = wait_bar(bar(kBarEmpty + kNumSlots + slot), ((u / Lay::kStageSlots) & 1) ^ 1, abort_flag);
            if (okl) {
              const uint32_t fb = bar(kBarFull + kNumSlots + slot);
              const int r = c ? ti.w : ti.z;
              const int blk = c ? ti.y : ti.x;   // -1: outside the pool (codes read as zeros, no scales)
              if (r <= 0) {
                mbar_arrive(fb);
              } else {
                mbar_arrive_expect_tx(fb, Lay::kStageBytes + (blk >= 0 ? 512u : 0u));
                tma_load_3d_hint(sbase + Lay::kOffStage + slot * Lay::kStageBytes, is_v ? &p.tm_v : &p.tm_k, fb, 0,
                                 r - kPage, blk, pol);
                if (blk >= 0)
                  bulk_load_g2s(sbase + kOffStageScale + slot * 512,
                                static_cast<const uint8_t*>(is_v ? p.v_scale : p.k_scale) + static_cast<size_t>(blk) * 512,
                                512, fb);
              }
              mine[nmine % 3] = u;
              ++nmine;
            }
          }
          return __all_sync(0xffffffffu, okl);
        }
        if (act) {
          const int4 ti = tile_info[t];
          const uint32_t u = ring_use<kKU>(t, ntiles, is_v) + c;
          const uint32_t slot = u % kNumSlots;
          okl = wait_bar(bar(kBarEmpty + slot), ((u / kNumSlots) & 1) ^ 1, abort_flag);
          if (okl) {
            const uint32_t dst = sbase + kOffRing + slot * kSlotBytes;
            const uint32_t fb = bar(kBarFull + slot);
            const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
            if (!is_v) {
              mbar_arrive_expect_tx(fb, ti.w > 0 ? 16384 : 8192);
              tma_load_3d_hint(dst, map, fb, 64 * c, ti.z - kPage, ti.x, pol);
              if (ti.w > 0) tma_load_3d_hint(dst + 8192, map, fb, 64 * c, ti.w - kPage, ti.y, pol);
            } else {
              const int pg = c / kVBlocks, dh = c % kVBlocks;
              const int r = pg ? ti.w : ti.z;
              const int blk = pg ? ti.y : ti.x;
              if (r <= 0) {
                mbar_arrive(fb);
              } else {
                mbar_arrive_expect_tx(fb, 16384);
                tma_load_3d_hint(dst, map, fb, 128 * dh, r - kPage, blk, pol);
                tma_load_3d_hint(dst + 8192, map, fb, 128 * dh + 64, r - kPage, blk, pol);
              }
            }
            mine[nmine % 3] = u;
            ++nmine;
          }
        }
        return __all_sync(0xffffffffu, okl);
      };
      if constexpr (kFp8 && !kMx) {
        // e4m3: the K sub-ring by lanes 0..3 and the V sub-ring by lanes 4..7, each stream
        // issued on its own as its slots free (one use a lane per tile: K use c = page c & 1,
        // d-half c >> 1; V use c = page c >> 1, d-half c & 1).  Lane 0 also loads each
        // segment's q, after its K use of the segment's first tile.
        uint32_t mine_bar[3] = {0u, 0u, 0u}, mine_par[3] = {0u, 0u, 0u};
        bool okl = true;
        if (lane < 8) {
          const bool is_v = lane >= 4;
          const int cc = lane & 3;
          const int pg = is_v ? (cc >> 1) : (cc & 1);
          const int dh = is_v ? (cc & 1) : (cc >> 1);
          int segl = 0;
          for (int t = 0; t < ntiles && okl; ++t) {
            while (segl + 1 < nseg && seg_n0[segl + 1] <= t) ++segl;
            const uint64_t pol = (reads > 1 && seg[segl].x % reads != reads - 1) ? pol_again : pol_once;
            // a V lane issues V(t) once lane 0 has issued K(t): at start-up, when every CTA
            // fills its rings at once, the memory queue then holds K(0), V(0), K(1), V(1)
            // first rather than three tiles of V ahead of the first K
            if (is_v && !wait_count(cnt + 3, t + 1, abort_flag)) {
              okl = false;
              break;
            }
            const uint32_t u = 4u * t + cc;
            const uint32_t slot = sub_slot<kNumSlots>(u, is_v);
            okl = wait_bar(bar(kBarEmpty + slot), sub_phase<kNumSlots>(u, is_v) ^ 1, abort_flag);
            if (!okl) break;
            const int4 ti = tile_info[t];
            const int r = pg ? ti.w : ti.z;
            const int blk = pg ? ti.y : ti.x;
            const uint32_t fb = bar(kBarFull + slot);
            if (r <= 0) {
              mbar_arrive(fb);
            } else {
              mbar_arrive_expect_tx(fb, 8192);
              tma_load_3d_hint(sbase + kOffRing + slot * kSlotBytes, is_v ? &p.tm_v : &p.tm_k, fb, 128 * dh, r - kPage,
                               blk, pol);
            }
            mine_bar[nmine % 3] = kBarFull + slot;
            mine_par[nmine % 3] = sub_phase<kNumSlots>(u, is_v);
            ++nmine;
            if (lane == 0) st_release_cta(cnt + 3, t + 1);   // K(t) issued (lane 0's use)
            if (lane == 0 && sq < nseg && t == seg_n0[sq]) {
              if (sq > 0) okl = wait_bar(bar(kBarQEmpty), (sq - 1) & 1, abort_flag);
              if (okl) {
                mbar_arrive_expect_tx(bar(kBarQFull), 4 * 8192);
                for (int q = 0; q < 4; ++q)
                  tma_load_2d(sbase + kOffQ + q * 8192, &p.tm_q, bar(kBarQFull), 64 * q, kH * seg[sq].x);
                ++nq;
                if (sq + 1 < nseg)
                  for (int q = 0; q < 4; ++q) tma_prefetch_2d(&p.tm_q, 64 * q, kH * seg[sq + 1].x);
              }
              ++sq;
            }
          }
        }
        ok = __all_sync(0xffffffffu, okl);
        if (!ok) {
          if (lane == 0) atomicOr(p.status, MFA_DEV_TIMEOUT);
          // let every copy already issued land before the CTA can exit
          for (int i = 0; i < (nmine < 3 ? nmine : 3); ++i) wait_slow(bar(mine_bar[i]), mine_par[i], nullptr, kDrainLimitNs);
          if (lane == 0 && nq > 0) wait_slow(bar(kBarQFull), (nq - 1) & 1, nullptr, kDrainLimitNs);
        }
      } else {
      for (int n = 0; n <= ntiles && ok; ++n) {
        if (n < ntiles) {
          if (ok) ok = group(false, n);
          if (ok && sq < nseg && n == seg_n0[sq]) {
            bool okq = true;
            if (lane == 0) {
              if (sq > 0) okq = wait_bar(bar(kBarQEmpty), (sq - 1) & 1, abort_flag);
              if (okq) {
                constexpr int kQB = kFp8 ? 4 : kQBoxes;
                mbar_arrive_expect_tx(bar(kBarQFull), kQB * 8192);
                for (int q = 0; q < kQB; ++q)
                  tma_load_2d(sbase + kOffQ + q * 8192, &p.tm_q, bar(kBarQFull), 64 * q, kH * seg[sq].x);
                ++nq;
                // the next segment's q waits for this segment's last QK^T; bring it into L2
                // now so that its load then comes from L2
                if (sq + 1 < nseg)
                  for (int q = 0; q < kQB; ++q) tma_prefetch_2d(&p.tm_q, 64 * q, kH * seg[sq + 1].x);
              }
            }
            ok = __all_sync(0xffffffffu, okq);
            ++sq;
          }
        }
        if (ok && n >= 1) ok = group(true, n - 1);
      }
      if (!ok) {
        if (lane == 0) atomicOr(p.status, MFA_DEV_TIMEOUT);
        // let every copy already issued land before the CTA can exit
        constexpr uint32_t kDrainSlots = kMx ? Lay::kStageSlots : kNumSlots;
        constexpr int kDrainBar0 = kMx ? kBarFull + kNumSlots : kBarFull;
        if (act)
          for (int i = 0; i < (nmine < 3 ? nmine : 3); ++i)
            wait_slow(bar(kDrainBar0 + mine[i] % kDrainSlots), (mine[i] / kDrainSlots) & 1, nullptr, kDrainLimitNs);
        if (lane == 0 && nq > 0) wait_slow(bar(kBarQFull), (nq - 1) & 1, nullptr, kDrainLimitNs);
      }
      }
    }
  } else if (warp == 1 || warp == pv_warp<kMx>()) {
    if constexpr (kMx) reg_dealloc<kRegsCtl>();
    if (warp == pv_warp<kMx>() && p.k_new != nullptr) {
      // fused KV append, rows nobody reads this step (token at or past the visible length,
      // including sequences without tokens): sequence b's by CTA b mod G, before its PVs
      grid_dep_wait();
      for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
        const int t = p.positions[b];
        bool dummy = false;
        if (t >= 0 && t >= vlen_from(raw_len(p.seq_lens, p.tokens, p.units, b), p.tokens, p.units, b, cap, dummy))
          fused_append_row(p, b, t, lane);
      }
    }
    // ---------------- MMA issuers: QK^T of tile n, then PV of tile n - 1, so the next tile's
    // scores are computed while the softmax works on the current one.  Warp 1 issues the
    // QK^T stream and warp pv_warp the PV stream (they share no operand, accumulator or
    // barrier), each with its own commits, so that a PV whose operands are ready never
    // waits behind the issue of the next QK^T; both commit to the drain barrier before
    // tensor memory is released.
    if (lane == 0 && ntiles > 0) {
      // N = the query heads that share one key/value head (64; GQA: 16, one MMA per group)
      constexpr uint32_t kIdescQK = idesc_f16(!kFp8, false, false, 128, kNh);
      constexpr uint32_t kIdescQK8 = idesc_e4m3(false, false, 128, 64);
      constexpr uint32_t kIdescPV = idesc_f16(!kFp8, true, true, 128, kNh);
      constexpr uint32_t kIdescPV8 = idesc_e4m3(true, true, 128, 64);
      constexpr int kChunksPerHead = Sh::kDq / 64;   // 64-element K chunks of one key head
      int sk = 0, jk = seg[0].y, sv = 0, jv = seg[0].y;
      bool ok = true;
      for (int n = 0; n <= ntiles && ok; ++n) {
        if (n < ntiles && warp == 1) {
          const int4 sg = seg[sk];
          const bool first = (jk == sg.y), last = (jk == sg.z - 1);
          const uint32_t u0 = kFp8 ? 4u * n : ring_use<kKU>(n, ntiles, false);
          // (one ring) some slots of tile n's K last held an earlier tile's V: it must have landed
          const int nv = kFp8 ? 0 : needs_other<kKU, kNumSlots>(static_cast<int>(u0), ntiles, true);
          if (nv > 0) ok = wait_count(cnt + 1, nv, abort_flag) && wait_count(cnt + 2, nv, abort_flag);
          if (ok && first) ok = wait_bar(bar(kFp8 ? kBarQReady : kBarQFull), sk & 1, abort_flag);
          if (ok && n >= 2) ok = wait_bar(bar(kBarSEmpty + (n & 1)), ((n >> 1) - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + kTmemS + s_cols<kFp8>() * (n & 1);
          if constexpr (!kFp8) {
            // chunk c = 64 elements of the cache row; with grouped heads it belongs to key
            // head g = c / kChunksPerHead, whose query heads are rows 16 g .. 16 g + 15 of q
            // box c % kChunksPerHead and columns 16 g .. of S^T
            for (int c = 0; c < kKU; ++c) {
              const uint32_t slot = (u0 + c) % kNumSlots;
              ok = wait_bar(bar(kBarFull + slot), ((u0 + c) / kNumSlots) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              const int g = c / kChunksPerHead, cq = c % kChunksPerHead;
              const uint32_t a0 = sbase + kOffRing + slot * kSlotBytes;
              const uint32_t b0 = sbase + kOffQ + cq * 8192 + 128 * kNh * (Sh::kGroups > 1 ? g : 0);
              const uint32_t dq = d_tmem + (Sh::kGroups > 1 ? kNh * g : 0);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f16_ss(dq, smem_desc(a0 + 32 * kk, 16, 1024), smem_desc(b0 + 32 * kk, 16, 1024),
                            kIdescQK, ((Sh::kGroups > 1 ? cq : c) | kk) != 0);
              umma_commit(bar(kBarEmpty + slot));
            }
            if (!ok) break;
          } else {
            // e4m3 K boxes as TMA wrote them: the two pages of d-half dh are adjacent slots,
            // one 128-row A operand; per K step (32) one N = 64 MMA against q's e4m3 hi part
            // (rows 0..63 of the q tile) and one against its lo part (rows 64..127), into the
            // same accumulator, so the scores arrive summed
#pragma unroll
            for (int dh = 0; dh < 2; ++dh) {
              for (int c = 2 * dh; c < 2 * dh + 2 && ok; ++c)
                ok = wait_bar(bar(kBarFull + sub_slot<kNumSlots>(u0 + c, false)), sub_phase<kNumSlots>(u0 + c, false),
                              abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint32_t a0 = sbase + kOffRing + sub_slot<kNumSlots>(u0 + 2 * dh, false) * kSlotBytes;
              const uint32_t b0 = sbase + kOffQ + dh * 16384;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = smem_desc(a0 + 32 * kk, 16, 1024);
                umma_f8_ss(d_tmem, ad, smem_desc(b0 + 32 * kk, 16, 1024), kIdescQK8, (dh | kk) != 0);
                umma_f8_ss(d_tmem, ad, smem_desc(b0 + 8192 + 32 * kk, 16, 1024), kIdescQK8, 1u);
              }
              umma_commit(bar(kBarEmpty + sub_slot<kNumSlots>(u0 + 2 * dh, false)));
              umma_commit(bar(kBarEmpty + sub_slot<kNumSlots>(u0 + 2 * dh + 1, false)));
            }
            if (!ok) break;
          }
          st_release_cta(cnt, n + 1);
          umma_commit(bar(kBarSFull + (n & 1)));
          if (last) umma_commit(bar(kBarQEmpty));
          if (++jk == sg.z && ++sk < nseg) jk = seg[sk].y;
        }
        if (n >= 1 && warp == pv_warp<kMx>()) {
          const int m = n - 1;
          const int4 sg = seg[sv];
          const bool first = (jv == sg.y), last = (jv == sg.z - 1);
          constexpr int kOBufs = kFp8 ? 2 : Sh::kOBufs;
          constexpr int kBlocksPerPage = kFp8 ? 2 : kVBlocks;
          const int kb = sv % kOBufs;
          const int4 ti = tile_info[m];
          const uint32_t uv = kFp8 ? 4u * m : ring_use<kKU>(m, ntiles, true);
          ok = wait_bar(bar(kBarPFull), m & 1, abort_flag);
          if (ok && first && sv >= kOBufs)
            ok = wait_bar(bar(kBarOEmpty + kb), ((sv / kOBufs) - 1) & 1, abort_flag);
          // some slots of tile m's V last held a later tile's K (small rings): it must have landed
          const int nk = kFp8 ? 0 : needs_other<kKU, kNumSlots>(static_cast<int>(uv), ntiles, false);
          if (ok && nk > m + 1) ok = wait_count(cnt, nk, abort_flag);
          if (!ok) break;
          tc_fence_after();
          for (int pg = 0; pg < 2 && ok; ++pg) {
            const int r = pg ? ti.w : ti.z;
            for (int hh = 0; hh < kBlocksPerPage; ++hh) {
              const uint32_t u = uv + kBlocksPerPage * pg + hh;
              const uint32_t vslot = kFp8 ? sub_slot<kNumSlots>(u, true) : u % kNumSlots;
              ok = wait_bar(bar(kBarFull + vslot), kFp8 ? sub_phase<kNumSlots>(u, true) : (u / kNumSlots) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
              const uint32_t a0 = sbase + kOffRing + vslot * kSlotBytes;
              // block hh: O^T lanes d of 128-element block hh; with grouped heads it is key
              // head hh's value, for its 16 query heads only (columns 16 hh .., P columns 16 hh ..)
              const uint32_t d_tmem = tmem + tmem_o<kFp8>() + 64u * (kFp8 ? 2 : Sh::kOBlocks) * kb +
                                      (Sh::kGroups > 1 ? static_cast<uint32_t>(kNh) : 64u) * hh;
              if (r > 0) {
                if constexpr (!kFp8) {
                  const uint32_t b0 = sbase + kOffP + pg * 8192 + (Sh::kGroups > 1 ? 2 * kNh * hh : 0);
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    umma_f16_ss(d_tmem, smem_desc(a0 + 2048 * kk, 8192, 1024),
                                smem_desc(b0 + 2048 * kk, 1024, 1024), kIdescPV,
                                !(first && pg == 0 && kk == 0));
                } else {
                  // A = V^T straight from the e4m3 box ([64 tokens][128 d], MN-major, one
                  // 128-element swizzle atom along d); B = the weights' hi part, then their
                  // lo part ([128 tokens][64 heads] each, MN-major, 64-byte swizzle); K = 32
                  // tokens per MMA, both parts into one accumulator
                  const uint32_t bh = sbase + kOffP + pg * 4096;
#pragma unroll
                  for (int kk = 0; kk < 2; ++kk) {
                    const uint64_t ad = smem_desc(a0 + 4096 * kk, 8192, 1024);
                    umma_f8_ss(d_tmem, ad, smem_desc_sw64(bh + 2048 * kk, 4096, 512), kIdescPV8,
                               !(first && pg == 0 && kk == 0));
                    umma_f8_ss(d_tmem, ad, smem_desc_sw64(bh + 8192 + 2048 * kk, 4096, 512), kIdescPV8, 1u);
                  }
                }
              }
              umma_commit(bar(kBarEmpty + vslot));
            }
          }
          if (!ok) break;
          // V(m) has landed
          st_release_cta(cnt + 1, m + 1);
          st_release_cta(cnt + 2, m + 1);
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
  } else if (kMx && warp < softmax_warp0<kMx>()) {
    // MXFP4: warp 3 completes warpgroup 0 and has no role
    if constexpr (kMx) reg_dealloc<kRegsCtl>();
  } else if (kMx && warp >= kConvWarp0) {
    if constexpr (kMx) {
      reg_dealloc<kRegsConv>();
      // ---------------- MXFP4 pages -> e4m3 operand ring (warps 12..15).  Each staging use
      // holds one page (K or V) of a tile; thread dt converts box row ri = dt & 63 of d-half
      // dh = dt >> 6 (warps 12-13: d 0..127, warps 14-15: d 128..255), four 32-element blocks,
      // into the e4m3 slot of that page and d-half, laid out as TMA lays out an e4m3 box
      // ([64 tokens][128 d], 128-byte swizzle), so that the MMAs read both caches alike.  Pages
      // go in the producer's order; each warp releases the staging slot, and the two warps of
      // a d-half together fill an e4m3 slot.
      const int dt = tid - 32 * kConvWarp0;
      const int ri = dt & 63, dh = dt >> 6;
      auto page = [&](bool is_v, int t, int pg) -> bool {
        const uint32_t su = ring_use<2>(t, ntiles, is_v) + pg;
        const uint32_t ss = su % Lay::kStageSlots;
        // the e4m3 use: K use c = 2 dh + pg (page c & 1, d-half c >> 1), V c = 2 pg + dh
        const uint32_t u = 4u * t + (is_v ? 2 * pg + dh : 2 * dh + pg);
        const uint32_t slot = sub_slot<kNumSlots>(u, is_v);
        if (!wait_warp(bar(kBarFull + kNumSlots + ss), (su / Lay::kStageSlots) & 1, abort_flag)) return false;
        if (!wait_warp(bar(kBarEmpty + slot), sub_phase<kNumSlots>(u, is_v) ^ 1, abort_flag)) return false;
        const int4 ti = tile_info[t];
        const int r = pg ? ti.w : ti.z;
        const int blk = pg ? ti.y : ti.x;
        if (r > 0) {   // (an absent page is skipped by the MMAs' masks and the PV)
          uint8_t* dst = smem + kOffRing + slot * kSlotBytes + ri * 128;
          const int pr = ri - (kPage - r);   // page row of box row ri; rows above it read zeros
          if (pr < 0 || blk < 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(dst + (q << 4)) = make_uint4(0u, 0u, 0u, 0u);
          } else {
            const uint8_t* src = smem + Lay::kOffStage + ss * Lay::kStageBytes + ri * 128;
            const uint2 s8 = *reinterpret_cast<const uint2*>(smem + kOffStageScale + ss * 512 + pr * 8);
            const int ref = mx_ref_exp(s8);
            const uint32_t sh = dh ? s8.y : s8.x;   // scale bytes of blocks 4 dh .. 4 dh + 3
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = 4 * dh + k;            // block j: d 32 j .. 32 j + 31, 16-byte chunk j
              const uint4 w = *reinterpret_cast<const uint4*>(src + ((j ^ (ri & 7)) << 4));
              uint4 o0, o1;
              mx_block_to_e4m3(w, static_cast<int>((sh >> (8 * k)) & 0xFFu) - ref, o0, o1);
              *reinterpret_cast<uint4*>(dst + (((2 * k) ^ (ri & 7)) << 4)) = o0;
              *reinterpret_cast<uint4*>(dst + (((2 * k + 1) ^ (ri & 7)) << 4)) = o1;
            }
          }
        }
        fence_proxy_async_smem();   // the rows are read by the tensor cores (async proxy)
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kBarFull + slot));
          mbar_arrive(bar(kBarEmpty + kNumSlots + ss));
        }
        return true;
      };
      // staging use su = page su & 1 of group su >> 1, the groups in the producer's order
      // (ring_use; one call site keeps the loop small)
      bool ok = true;
#pragma unroll 1
      for (int su = 0; su < 4 * ntiles; ++su) {
        bool is_v;
        const int t = group_owner(su >> 1, ntiles, is_v);
        if (!page(is_v, t, su & 1)) {
          ok = false;
          break;
        }
      }
      if (!ok && lane == 0) atomicOr(p.status, MFA_DEV_TIMEOUT);
    }
  } else {
    if constexpr (kMx) reg_alloc<kRegsSoftmax>();
    // ---------------- softmax + epilogue (256 threads: two warps per TMEM lane quarter)
    const int ts = tid - 32 * softmax_warp0<kMx>();   // 0..255
    const int sw = warp - softmax_warp0<kMx>();       // 0..7
    const int grp = sw >> 2;                       // head half [32*grp, +32)
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
    constexpr int kOBufs = kFp8 ? 2 : Sh::kOBufs;
    constexpr int kOBlocks = kFp8 ? 2 : Sh::kOBlocks;
    constexpr int kDq = Sh::kDq;
    float qinv = 1.f, qinv_next = 1.f;              // e4m3: 2^-sigma of the segment's q split

    if (p.early_metadata) grid_dep_wait();
    // sequences with no tokens: out = 0, lse = -inf (one CTA each, round robin)
    for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
      bool dummy = false;
      if (vlen_from(raw_len(p.seq_lens, p.tokens, p.units, b), p.tokens, p.units, b, cap, dummy) != 0) continue;
      const int esz = p.out_f32 ? 4 : 2;
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + static_cast<size_t>(b) * kH * kDq * esz);
      for (int i = ts; i < kH * kDq * esz / 16; i += kSoftmaxThreads) o[i] = make_uint4(0, 0, 0, 0);
      if (p.lse != nullptr && ts < kH) p.lse[b * kH + ts] = -INFINITY;
    }

    bool aborted = false;
    int n = 0;
    const uint32_t l_tmem = tmem + kTmemL + h0 + lane_base;    // bf16: this thread's 32 row-sum partials
    const uint32_t lx_tmem = tmem + kTmemLx + h0 + lane_base;  // bf16: and their fp32-weight twins
    float lreg[32];                                            // e4m3: row-sum partials in registers
    int defer_b[2] = {0, 0}, defer_slot[2] = {0, 0};
    bool defer_whole[2] = {false, false};
    bool prev_written = false;   // the second-to-last segment was written during the last one

    // valid rows of a tile's page pg: the last page's rows sit at the end of the box
    auto page_rows = [&](int L, int j, int pg) { return min(kPage, L - kTile * j - kPage * pg); };

    // Write the finished accumulator of this CTA's segment `sidx` (O buffer sidx % kOBufs),
    // normalised by 1/l from linv, as [head][d] rows.  `direct`: plain stores from
    // registers (the CTA's last two segments, after its last MMA); otherwise the rows are
    // staged in this half's 8 KB of the P buffer and sent by bulk async copies in
    // double-buffered 4 KB rounds, off the threads' critical path (MFA; the other shapes
    // always store directly, one 128-d block at a time).  Returns false if the CTA is aborting.
    auto write_segment = [&](int sidx, int b, int slot_p, bool whole, bool direct) -> bool {
      const int kb = sidx % kOBufs;
      const bool okO = wait_warp(bar(kBarOFull + kb), (sidx / kOBufs) & 1, abort_flag);
      aborted = aborted || !okO;
      if (named_bar_or(1, kSoftmaxThreads, aborted || *abort_flag)) return false;
      tc_fence_after();
      const uint32_t o_tmem = tmem + tmem_o<kFp8>() + 64u * kOBlocks * kb + h0 + lane_base;
      if constexpr (kShp != kShapeMfa) {
        const bool bf16_out = whole && !p.out_f32;
        const int esz = bf16_out ? 2 : 4;
        uint8_t* gdst = whole ? static_cast<uint8_t*>(p.out) + (static_cast<size_t>(b) * kH + h0) * kDq * esz
                              : reinterpret_cast<uint8_t*>(p.part_o) + (static_cast<size_t>(slot_p) * kH + h0) * kDq * 4;
#pragma unroll 1
        for (int blk = 0; blk < kOBlocks; ++blk) {
          uint32_t oa[32];
          tmem_ld32(o_tmem + 64u * blk, oa);
          tmem_ld_wait(oa);
          if (blk == kOBlocks - 1) {
            tc_fence_before();
            mbar_arrive(bar(kBarOEmpty + kb));   // the accumulator is free
          }
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            const float v = __uint_as_float(oa[h]) * linv[kb * kH + h0 + h];
            const size_t e = static_cast<size_t>(h) * kDq + 128 * blk + row;
            if (bf16_out)
              reinterpret_cast<__nv_bfloat16*>(gdst)[e] = __float2bfloat16_rn(v);
            else
              reinterpret_cast<float*>(gdst)[e] = v;
          }
        }
        return true;
      }
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
      if (direct) {
        // straight from registers: for each head a warp writes 32 consecutive d values
#pragma unroll
        for (int h = 0; h < 32; ++h) put(gdst, h, __uint_as_float(oa[h]), __uint_as_float(ob[h]));
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

    // 32 scores of this thread's row (token) for its heads
    auto ld_s32 = [&](uint32_t taddr, uint32_t (&sv)[32]) {
      tmem_ld32(taddr, sv);
      tmem_ld_wait(sv);
    };

    // e4m3: q of segment sidx arrives in bf16 and is split in place into two e4m3 parts,
    // hi = e4m3(2^sigma q) and lo = e4m3(2^sigma q - hi), with one power of two 2^sigma per
    // sequence putting its largest |q| in [64, 128): hi + lo reproduces 2^sigma q (see
    // split_e4m3) and the QK^T MMA runs on e4m3 K as stored.  Thread ts converts row
    // ts & 63 (a head) of bf16 box ts >> 6 (64 d); all reads precede all writes, and each
    // thread reads its row's 16-byte chunks in logical order, which the 128-byte swizzle
    // spreads over the banks (eight rows of a warp hit eight different bank groups).  Done for
    // a later segment right after the previous segment's last scores are read, so its
    // first QK^T can overlap that segment's last PV and epilogue.
    auto convert_q = [&](int sidx) {
      const bool okQ = wait_warp(bar(kBarQFull), sidx & 1, abort_flag);
      const int hq = ts & 63, cq = ts >> 6;
      uint4 w[8];
      float mx = 0.f;
      if (okQ) {
        const uint8_t* src = smem + kOffQ + cq * 8192 + hq * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          w[q] = *reinterpret_cast<const uint4*>(src + 16 * (q ^ (hq & 7)));   // logical chunk q
          const uint32_t* e = reinterpret_cast<const uint32_t*>(&w[q]);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(e[k] << 16)), fabsf(__uint_as_float(e[k] & 0xFFFF0000u))));
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float* qmax = reinterpret_cast<float*>(misc + 24);   // [8] per softmax warp
      if (lane == 0) qmax[sw] = mx;
      named_bar_sync(1, kSoftmaxThreads);
      float M = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) M = fmaxf(M, qmax[i]);
      int sig = 0;
      if (M > 0.f && M <= 3.0e38f) sig = min(126, max(-126, 6 - static_cast<int>((__float_as_uint(M) >> 23) & 0xFFu) + 127));
      const float qs = __uint_as_float(static_cast<uint32_t>(127 + sig) << 23);
      qinv_next = __uint_as_float(static_cast<uint32_t>(127 - sig) << 23);
      if (okQ) {
        uint8_t* dst = smem + kOffQ + (cq >> 1) * 16384 + hq * 128;   // hi part (rows 0..63); lo rows at +8 KB
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int k = q;                                  // logical 16-byte chunk of the bf16 row
          const uint32_t* e = reinterpret_cast<const uint32_t*>(&w[q]);
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            split_e4m3(__uint_as_float(e[i] << 16) * qs, __uint_as_float(e[i] & 0xFFFF0000u) * qs, hi[i], lo[i]);
          // d = 64 cq + 8 k .. +7: bytes 8 (k & 1) of logical e4m3 chunk 4 (cq & 1) + (k >> 1)
          const int ci = 4 * (cq & 1) + (k >> 1);
          const int off = ((ci ^ (hq & 7)) << 4) + 8 * (k & 1);
          *reinterpret_cast<uint2*>(dst + off) = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
          *reinterpret_cast<uint2*>(dst + 8192 + off) = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
        }
        fence_proxy_async_smem();
      } else {
        aborted = true;
      }
      mbar_arrive(bar(kBarQReady));
    };

    uint2 sk_next = make_uint2(0u, 0u), sv_next = make_uint2(0u, 0u);   // e4m3: the row's K and V
                                                                        // scales in the next tile
    int e_ref = kEMin;                              // e4m3: the segment's reference exponent of V scales
    if constexpr (kFp8) {
      if (ntiles > 0) {
        sk_next = kv_scale_raw<kMx>(p.k_scale, tile_info[0], rpg, ri);
        sv_next = kv_scale_raw<kMx>(p.v_scale, tile_info[0], rpg, ri);
        convert_q(0);
      }
    }

    for (int s = 0; s < nseg && !aborted; ++s) {
      const int4 sg = seg[s];
      const int b = sg.x, L = sg.w, kb = s % kOBufs;
      const bool whole = (sg.y == 0) && (sg.z == tiles_of(L));
      const int slot_p = pos_of(b, p.tokens, p.units, p.batch) + static_cast<int>(blockIdx.x);
      const uint32_t o_tmem = tmem + tmem_o<kFp8>() + 64u * kOBlocks * kb + h0 + lane_base;   // + 64 per block
      if (ts < kH) m_ref[ts] = -INFINITY;
      if constexpr (kFp8) {
        qinv = qinv_next;
        e_ref = kEMin;
#pragma unroll
        for (int h = 0; h < 32; ++h) lreg[h] = 0.f;
      }
      named_bar_sync(1, kSoftmaxThreads);
      bool stop = false;
      for (int j = sg.y; j < sg.z; ++j, ++n) {
        const bool first = (j == sg.y);
        const uint32_t s_tmem = tmem + kTmemS + s_cols<kFp8>() * (n & 1) + h0 + lane_base;
        const bool okS = wait_warp(bar(kBarSFull + (n & 1)), (n >> 1) & 1, abort_flag);
        aborted = aborted || !okS;
        bool pv_waited = (n == 0);   // PV of the previous tile must be done before P or O are touched
        const int rp = page_rows(L, j, rpg);
        const bool valid = okS && rp > 0 && ri >= kPage - rp;
        // score multiplier of this row: scale*log2(e), times (e4m3) the token's K scale and
        // the 2^-sigma that undoes q's split scaling; e4m3 also takes the token's V scale
        float ck = c, svt = 0.f;
        int sv_e = kEMin;   // e4m3: unbiased exponent of the token's V scale
        if constexpr (kFp8) {
          ck = c * qinv * kv_scale_of<kMx>(sk_next);   // loaded one tile ahead
          svt = kv_scale_of<kMx>(sv_next);
          if (n + 1 < ntiles) {
            sk_next = kv_scale_raw<kMx>(p.k_scale, tile_info[n + 1], rpg, ri);
            sv_next = kv_scale_raw<kMx>(p.v_scale, tile_info[n + 1], rpg, ri);
          }
          sv_e = static_cast<int>((__float_as_uint(svt) >> 23) & 0xFFu) - 127;
        }
        // --- this row's 32 scores, read from tensor memory once per tile; does any exceed
        //     its head's reference max by more than the threshold (e4m3: or does the token's
        //     V scale reach past the segment's reference exponent)?
        // (bf16 keeps the scores in registers for the exponentials; e4m3, whose row sums
        // already live in registers, reads them again there)
        constexpr float kThr = rescale_threshold<kFp8>();
        bool need = false;
        uint32_t sc[32];
        if (okS) {
          tc_fence_after();
          ld_s32(s_tmem, sc);
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(m_ref + h0 + h);
            need |= (fmaf(__uint_as_float(sc[h + 0]), ck, -m4.x) > kThr) |
                    (fmaf(__uint_as_float(sc[h + 1]), ck, -m4.y) > kThr) |
                    (fmaf(__uint_as_float(sc[h + 2]), ck, -m4.z) > kThr) |
                    (fmaf(__uint_as_float(sc[h + 3]), ck, -m4.w) > kThr);
          }
          if constexpr (kFp8) need |= sv_e > e_ref;
          need = need && valid;
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) sc[h] = 0u;
        }
        const bool any_need = named_bar_or(1, kSoftmaxThreads, need || aborted || *abort_flag);
        if (any_need) {
          if (named_bar_or(1, kSoftmaxThreads, aborted || *abort_flag)) { stop = true; break; }
          // --- rare path: new reference max for heads whose scores jumped past the threshold
          //     (e4m3: and a new reference exponent for the V scales)
          int* red_e = reinterpret_cast<int*>(red + 256);   // e4m3: per-warp maximum exponent
          {
            if constexpr (kFp8) ld_s32(s_tmem, sc);
            float mv[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) mv[h] = valid ? __uint_as_float(sc[h]) * ck : -INFINITY;
            red[wq * 64 + h0 + lane] = warp_reduce_scatter32<true>(mv);
            if constexpr (kFp8) {
              const int em = __reduce_max_sync(0xffffffffu, (valid && svt > 0.f) ? sv_e : kEMin);
              if (lane == 0) red_e[sw] = em;
            }
          }
          named_bar_sync(1, kSoftmaxThreads);
          if (ts < kH) {
            const float mt = fmaxf(fmaxf(red[ts], red[64 + ts]), fmaxf(red[128 + ts], red[192 + ts]));
            const float mo = m_ref[ts];
            float a = 1.f;
            if (mt > mo + kThr) {
              a = exp2f(mo - mt);
              m_ref[ts] = mt;
            }
            alpha_s[ts] = a;
          }
          // e4m3: every thread takes the same new reference exponent; the O accumulated so far
          // was weighted by 2^(kPvShift - e_ref) and is rescaled to the new one
          float o_extra = 1.f;
          if constexpr (kFp8) {
            int em = e_ref;
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) em = max(em, red_e[w8]);
            o_extra = exp2f(static_cast<float>(e_ref - em));
            e_ref = em;
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
            for (int k3 = 0; k3 < kOBlocks + (kFp8 ? 0 : 2); ++k3) {
              uint32_t ov[32];
              const uint32_t ta = (k3 == kOBlocks) ? l_tmem : (k3 == kOBlocks + 1) ? lx_tmem : o_tmem + 64u * k3;
              const float ox = (k3 < kOBlocks) ? o_extra : 1.f;
              tmem_ld32(ta, ov);
              tmem_ld_wait(ov);
#pragma unroll
              for (int h = 0; h < 32; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * (alpha_s[h0 + h] * ox));
              tmem_st32(ta, ov);
            }
            tmem_st_wait();
          }
        }
        // --- probabilities and row sums; the P^T row piece stays in registers until the
        //     previous tile's PV has released the P buffer.  e4m3: the weight times the
        //     token's scaled V scale, u = s_v 2^(kPvShift - e_ref) < 2^(kPvShift + 1), split into
        //     an e4m3 hi part and an e4m3 lo part (pk[0..7] and pk[8..15], four heads a word)
        uint32_t pk[16];
        float u = 0.f;
        uint32_t u2 = 0u;   // e4m3: u in both halves of an f16x2
        if constexpr (kFp8) {
          u = svt * __uint_as_float(static_cast<uint32_t>(127 + kPvShift - e_ref) << 23);
          asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(u2) : "f"(u));
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = 0u;
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t lv[16], lx[16], sf[16];
          const uint32_t* sv = sc + 16 * half;
          if constexpr (kFp8) {
            // (read again: the row sums of e4m3 live in registers, which leaves no room to keep
            // the scores across the vote)
            tmem_ld16(s_tmem + 16 * half, sf);
            tmem_ld_wait(sf);
            sv = sf;
          }
          if (!kFp8 && !first) {
            tmem_ld16(l_tmem + 16 * half, lv);
            tmem_ld16(lx_tmem + 16 * half, lx);
          }
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
            if constexpr (kFp8) {
              // the pair's weights in packed f16 arithmetic: two exponentials per ex2.f16x2, then
              // w = p u split into e4m3 parts hi = e4m3(w) and lo = e4m3(w - hi), with w - hi
              // exact in f16 (hi is within 2^-4 of w).  The exponent's argument x <= 3 is
              // rounded to f16 first (an error under 2^-11 |x|), p and w carry f16's 11 bits,
              // more than hi + lo keep (about 9), and the row sum adds p as rounded.
              const float x0 = fmaf(__uint_as_float(sv[hl]), ck, -m2.x);
              const float x1 = fmaf(__uint_as_float(sv[hl + 1]), ck, -m2.y);
              uint32_t xh, ph;
              asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(xh) : "f"(x1), "f"(x0));
              asm("ex2.approx.f16x2 %0, %1;" : "=r"(ph) : "r"(xh));
              if (!valid) ph = 0u;
              float q0, q1;
              asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
                  : "=f"(q0), "=f"(q1) : "r"(ph));
              lreg[h] += q0;
              lreg[h + 1] += q1;
              uint32_t wh, hb, rh;
              uint16_t hi16, lo16;
              asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(wh) : "r"(ph), "r"(u2));
              asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(hi16) : "r"(wh));
              asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hb) : "h"(hi16));
              asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(rh) : "r"(wh), "r"(hb));
              asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(lo16) : "r"(rh));
              pk[4 * half + (e >> 1)] |= static_cast<uint32_t>(hi16) << (16 * (e & 1));
              pk[8 + 4 * half + (e >> 1)] |= static_cast<uint32_t>(lo16) << (16 * (e & 1));
            } else {
              const float p0 = valid ? ex2_approx(fmaf(__uint_as_float(sv[hl]), ck, -m2.x)) : 0.f;
              const float p1 = valid ? ex2_approx(fmaf(__uint_as_float(sv[hl + 1]), ck, -m2.y)) : 0.f;
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
          // the next segment's q, as soon as this segment's last scores are read
          if (j + 1 == sg.z && s + 1 < nseg) convert_q(s + 1);
        }
        if (!pv_waited && !wait_warp(bar(kBarPvDone), (n - 1) & 1, abort_flag)) aborted = true;
        if constexpr (kFp8) {
          // hi and lo parts: [128 tokens][64 heads] e4m3 each, 64-byte rows with the 64-byte
          // swizzle; this thread's 32 heads are 16-byte chunks 2*grp and 2*grp+1 of its row
          uint8_t* prow = smem + kOffP + row * 64;
          const int swz = (row >> 1) & 3;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int off = ((2 * grp + q) ^ swz) << 4;
            *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            *reinterpret_cast<uint4*>(prow + 8192 + off) =
                make_uint4(pk[8 + 4 * q], pk[9 + 4 * q], pk[10 + 4 * q], pk[11 + 4 * q]);
          }
        } else {
          // this thread's 32 heads are 16-byte chunks 4*grp .. 4*grp+3 of the 128-byte P^T row
          uint8_t* prow = smem + kOffP + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(prow + (((4 * grp + q) ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarPFull));
        // bf16: the second-to-last segment's output, once the last segment's first P is out:
        // its last PV completed before that P could be written, so the stores overlap the
        // remaining tiles instead of adding to the CTA's tail (the e4m3 softmax, which bounds
        // its tile period, keeps both writes for the end)
        if (!kFp8 && kOBufs == 2 && first && s >= 1 && s == nseg - 1) {
          const int ps = s - 1, pkb = ps & 1;
          if (!write_segment(ps, defer_b[pkb], defer_slot[pkb], defer_whole[pkb], true)) { stop = true; break; }
          prev_written = true;
        }
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
        // e4m3: the weights carried 2^(kPvShift - e_ref), undone here
        const float oscale = kFp8 ? __uint_as_float(static_cast<uint32_t>(127 + e_ref - kPvShift) << 23) : 1.f;
        linv[kb * kH + ts] = oscale / l;
        const float lx = kFp8 ? l : (red[256 + ts] + red[320 + ts]) + (red[384 + ts] + red[448 + ts]);
        const float lse_v = (m_ref[ts] + log2f(lx)) * 0.69314718055994531f;
        if (whole) {
          if (p.lse != nullptr) p.lse[b * kH + ts] = lse_v;
        } else {
          p.part_lse[static_cast<size_t>(slot_p) * kH + ts] = lse_v;
        }
      }
      named_bar_sync(1, kSoftmaxThreads);
      if (s + kOBufs < nseg) {
        // the accumulator is needed again by segment s + kOBufs: write it out now
        if (!write_segment(s, b, slot_p, whole, false)) break;
      } else {
        // one of the CTA's last two segments: its accumulator stays in tensor memory and is
        // written from registers after the last tile (bf16: the one before the last during the
        // last segment's first tile)
        defer_b[kb] = b;
        defer_slot[kb] = slot_p;
        defer_whole[kb] = whole;
      }
    }
    if (!aborted && !*abort_flag) {
      // deferred accumulators, newest first, stored straight from registers (uniform:
      // every thread reads the same values)
      // (a CTA whose cost range holds no tile has no segment, and nothing to write)
      const int first_def = (kOBufs == 2 && nseg >= 2 && !prev_written) ? nseg - 2 : nseg - 1;
      for (int s = nseg - 1; s >= 0 && s >= first_def; --s) {
        const int kb = s % kOBufs;
        if (!write_segment(s, defer_b[kb], defer_slot[kb], defer_whole[kb], true)) break;
      }
    }
    if (issuer) bulk_wait_read0();
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

// Largest g with floor(g C / G) <= c: the CTA owning cost position c (see the decode
// kernel's cost-balanced split: tile k of sequence b at cost 4 (S_b + k) + c N_b, N_b the
// non-empty sequences before b, C = 4 W + c (N - 1), c = cost_seq).
__device__ __forceinline__ int cta_of_cost(long long c, long long C, long long G) {
  return static_cast<int>(((c + 1) * G + C - 1) / C - 1);
}

constexpr int kCombineThreads = 256;
constexpr int kCombineMaxParts = 256;        // partials staged per pass

// One CTA per (sequence, group of `heads_per_cta` heads), for MFA's 256-wide rows.  The 256
// threads form four quads of 64 (each thread owns 4 consecutive d, a float4).  With one head
// per CTA the quads split the partials four ways; with four or more heads each
// quad owns a head and the CTA walks its heads in rounds of four.  Partial lse
// values are staged in shared memory; partial O rows stream in with batched
// independent float4 loads.
__global__ void __launch_bounds__(kCombineThreads) mfa_combine_kernel(const __grid_constant__ CombineParams p) {
  grid_dep_wait();
  grid_dep_launch();   // the next kernel may start its own set-up
  __shared__ int red_b[kCombineThreads / 32], red_t[kCombineThreads / 32];
  __shared__ int red_nb[kCombineThreads / 32], red_nt[kCombineThreads / 32];
  __shared__ int slots[kCombineMaxParts];
  __shared__ float wts[16][kCombineMaxParts];   // a single pass: every head's weights; else a round's
  __shared__ float4 part_acc[3][64];
  __shared__ float pass_max[16], pass_sum[16];
  __shared__ int nparts_s;
  const int b = blockIdx.x;
  const int hpc = p.heads_per_cta;
  const int hpr = hpc < 4 ? hpc : 4;          // heads per round
  const int groups = 4 / hpr;                 // quads sharing one head
  const int rounds = hpc / hpr;
  const int cap = p.max_pages * kPage;
  // tiles (and non-empty sequences) before b and in all: the decode kernel's cost positions
  int before = 0, total = 0, nb = 0, nt = 0;
  const int pb = pos_of(b, p.tokens, p.units, p.batch);   // b's schedule position
  for (int i = threadIdx.x; i < p.batch; i += kCombineThreads) {
    bool dummy = false;
    const int x = unit_at(i, p.tokens, p.units, p.batch);
    const int T = tiles_of(vlen_from(raw_len(p.seq_lens, p.tokens, p.units, x), p.tokens, p.units, x, cap, dummy));
    total += T;
    nt += (T > 0);
    before += (i < pb) ? T : 0;
    nb += (i < pb && T > 0);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
    nb += __shfl_xor_sync(0xffffffffu, nb, o);
    nt += __shfl_xor_sync(0xffffffffu, nt, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red_b[threadIdx.x >> 5] = before;
    red_t[threadIdx.x >> 5] = total;
    red_nb[threadIdx.x >> 5] = nb;
    red_nt[threadIdx.x >> 5] = nt;
  }
  __syncthreads();
  before = total = nb = nt = 0;
  for (int w = 0; w < kCombineThreads / 32; ++w) {
    before += red_b[w];
    total += red_t[w];
    nb += red_nb[w];
    nt += red_nt[w];
  }
  bool dummy = false;
  const int Tb = tiles_of(vlen_from(raw_len(p.seq_lens, p.tokens, p.units, b), p.tokens, p.units, b, cap, dummy));
  if (Tb == 0) return;
  const long long sw = p.seq_cost;
  const long long C = kCostTile * static_cast<long long>(total) + sw * max(nt - 1, 0);
  const long long base = kCostTile * static_cast<long long>(before) + sw * nb;   // cost of sequence b's first tile
  const int g0 = cta_of_cost(base, C, p.num_ctas);
  const int g1 = cta_of_cost(base + kCostTile * static_cast<long long>(Tb - 1), C, p.num_ctas);
  if (g0 == g1) return;  // written whole by the decode kernel

  const int quad = threadIdx.x >> 6;
  const int hr = quad / groups;               // head of the round owned by this quad
  const int grp = quad % groups;              // partial group within that head
  const int d4 = threadIdx.x & 63;            // float4 column: d = 4*d4 .. 4*d4+3
  // With all partials in one pass (the usual case) the slots and the weights of all the
  // CTA's heads are found once, before the first round; otherwise pass by pass, round by round.
  const bool one_pass = g1 - g0 + 1 <= kCombineMaxParts;
  for (int r = 0; r < rounds; ++r) {
    const int h = blockIdx.y * hpc + r * hpr + hr;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float run_max = -INFINITY, run_sum = 0.f;
    const bool load_w = r == 0 || !one_pass;
    const int nh = one_pass ? hpc : hpr;                             // heads whose weights a load takes
    const int h_first = blockIdx.y * hpc + (one_pass ? 0 : r * hpr);
    const int hw = (one_pass ? r * hpr : 0) + hr;                    // this quad's row of wts
    // partials come from CTAs g0..g1 (CTAs with an empty tile range hold none)
    for (int gs = g0; gs <= g1; gs += kCombineMaxParts) {
      const int ge = min(g1 + 1, gs + kCombineMaxParts);
      __syncthreads();
      if (threadIdx.x < 32 && load_w) {
        int n = 0;
        for (int g = gs + threadIdx.x; g - static_cast<int>(threadIdx.x) < ge; g += 32) {
          // CTA g holds a tile of b if a tile cost of b lies in its cost range
          bool live = false;
          if (g < ge) {
            const long long x0 = (static_cast<long long>(g) * C) / p.num_ctas;
            const long long x1 = (static_cast<long long>(g + 1) * C) / p.num_ctas;
            const long long k_lo = x0 <= base ? 0 : (x0 - base + kCostTile - 1) / kCostTile;
            const long long k_hi = x1 <= base ? 0 : (x1 - base + kCostTile - 1) / kCostTile;
            live = k_lo < min(k_hi, static_cast<long long>(Tb));
          }
          const unsigned m = __ballot_sync(0xffffffffu, live);
          if (live) slots[n + __popc(m & ((1u << threadIdx.x) - 1))] = pb + g;
          n += __popc(m);
        }
        if (threadIdx.x == 0) nparts_s = n;
      }
      __syncthreads();
      const int n = nparts_s;
      if (load_w) {
        for (int k = threadIdx.x; k < n * nh; k += kCombineThreads) {
          const int kk = k / nh, hh = k % nh;
          wts[hh][kk] = p.part_lse[static_cast<size_t>(slots[kk]) * kH + h_first + hh];
        }
        __syncthreads();
        // warp w turns heads w, w + 8, ... into weights relative to their max
        const int l = threadIdx.x & 31;
#pragma unroll 1
        for (int w = threadIdx.x >> 5; w < nh; w += kCombineThreads / 32) {
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
        __syncthreads();
      }
      if (one_pass && groups == 1 && rounds > 1) {
        // a single pass with one head per quad: every round's partial loads go out together
        // (parts outer, rounds inner), so that the CTA waits for memory once rather than once
        // a round; per head the sums run over the parts in the same order as below
        float4 accr[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) accr[rr] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
        for (int k = 0; k < n; ++k) {
          const float* src0 = p.part_o + (static_cast<size_t>(slots[k]) * kH + blockIdx.y * hpc + hr) * kD;
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            if (rr < rounds) {
              const float4 v = reinterpret_cast<const float4*>(src0 + static_cast<size_t>(rr * hpr) * kD)[d4];
              const float w = wts[rr * hpr + hr][k];
              accr[rr].x = fmaf(w, v.x, accr[rr].x); accr[rr].y = fmaf(w, v.y, accr[rr].y);
              accr[rr].z = fmaf(w, v.z, accr[rr].z); accr[rr].w = fmaf(w, v.w, accr[rr].w);
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          if (rr < rounds) {
            const int hw2 = rr * hpr + hr, h2 = blockIdx.y * hpc + hw2;
            const float4 a = accr[rr];
            const float inv = 1.f / pass_sum[hw2];
            const size_t oi = (static_cast<size_t>(b) * kH + h2) * kD + 4 * d4;
            if (p.out_f32) {
              reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi)[0] =
                  make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
            } else {
              __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * inv, a.y * inv);
              __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * inv, a.w * inv);
              uint2 pk;
              pk.x = *reinterpret_cast<uint32_t*>(&lo);
              pk.y = *reinterpret_cast<uint32_t*>(&hi);
              reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + oi)[0] = pk;
            }
            if (d4 == 0 && p.lse != nullptr) p.lse[b * kH + h2] = pass_max[hw2] + logf(pass_sum[hw2]);
          }
        }
        return;
      }
      // rescale what earlier passes accumulated to this pass's reference
      const float m_new = fmaxf(run_max, pass_max[hw]);
      const float a_old = (run_max == -INFINITY) ? 0.f : expf(run_max - m_new);
      const float a_new = expf(pass_max[hw] - m_new);
      acc.x *= a_old; acc.y *= a_old; acc.z *= a_old; acc.w *= a_old;
      run_sum = run_sum * a_old + pass_sum[hw] * a_new;
      run_max = m_new;
      const float* wrow = wts[hw];
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

// The same merge for the comparison shapes' rows (kDq = 128 or 512).
// One CTA per (unit, group of `heads_per_cta` heads).  The 256 threads form four quads of
// 64; a thread owns 4 consecutive d (a float4) of each 256-d span of the kDq-wide row (for
// kDq = 128 the quad's upper 32 threads hold nothing).  With one head per CTA the quads split
// the partials four ways; with four or more heads each quad owns a head and the CTA walks its
// heads in rounds of four.  Partial lse values are staged in shared memory; partial O rows
// stream in with batched independent float4 loads.
template <int kDq>
__global__ void __launch_bounds__(kCombineThreads) mfa_combine_wide_kernel(const __grid_constant__ CombineParams p) {
  constexpr int kF = (kDq + 255) / 256;          // float4s per thread and row
  constexpr int kRowF4 = kDq / 4;
  grid_dep_wait();
  grid_dep_launch();   // the next kernel may start its own set-up
  __shared__ int red_b[kCombineThreads / 32], red_t[kCombineThreads / 32];
  __shared__ int red_nb[kCombineThreads / 32], red_nt[kCombineThreads / 32];
  __shared__ int slots[kCombineMaxParts];
  __shared__ float wts[4][kCombineMaxParts];
  __shared__ float4 part_acc[3][64 * kF];
  __shared__ float pass_max[4], pass_sum[4];
  __shared__ int nparts_s;
  const int b = blockIdx.x;
  const int hpc = p.heads_per_cta;
  const int hpr = hpc < 4 ? hpc : 4;          // heads per round
  const int groups = 4 / hpr;                 // quads sharing one head
  const int rounds = hpc / hpr;
  const int cap = p.max_pages * kPage;
  // tiles (and non-empty sequences) before b and in all: the decode kernel's cost positions
  int before = 0, total = 0, nb = 0, nt = 0;
  const int pb = pos_of(b, p.tokens, p.units, p.batch);   // b's schedule position
  for (int i = threadIdx.x; i < p.batch; i += kCombineThreads) {
    bool dummy = false;
    const int x = unit_at(i, p.tokens, p.units, p.batch);
    const int T = tiles_of(vlen_from(raw_len(p.seq_lens, p.tokens, p.units, x), p.tokens, p.units, x, cap, dummy));
    total += T;
    nt += (T > 0);
    before += (i < pb) ? T : 0;
    nb += (i < pb && T > 0);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
    nb += __shfl_xor_sync(0xffffffffu, nb, o);
    nt += __shfl_xor_sync(0xffffffffu, nt, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red_b[threadIdx.x >> 5] = before;
    red_t[threadIdx.x >> 5] = total;
    red_nb[threadIdx.x >> 5] = nb;
    red_nt[threadIdx.x >> 5] = nt;
  }
  __syncthreads();
  before = total = nb = nt = 0;
  for (int w = 0; w < kCombineThreads / 32; ++w) {
    before += red_b[w];
    total += red_t[w];
    nb += red_nb[w];
    nt += red_nt[w];
  }
  bool dummy = false;
  const int Tb = tiles_of(vlen_from(raw_len(p.seq_lens, p.tokens, p.units, b), p.tokens, p.units, b, cap, dummy));
  if (Tb == 0) return;
  const long long sw = p.seq_cost;
  const long long C = kCostTile * static_cast<long long>(total) + sw * max(nt - 1, 0);
  const long long base = kCostTile * static_cast<long long>(before) + sw * nb;   // cost of sequence b's first tile
  const int g0 = cta_of_cost(base, C, p.num_ctas);
  const int g1 = cta_of_cost(base + kCostTile * static_cast<long long>(Tb - 1), C, p.num_ctas);
  if (g0 == g1) return;  // written whole by the decode kernel

  const int quad = threadIdx.x >> 6;
  const int hr = quad / groups;               // head of the round owned by this quad
  const int grp = quad % groups;              // partial group within that head
  const int d4 = threadIdx.x & 63;            // float4 columns d4 + 64 f: d = 4 (d4 + 64 f) .. + 3
  const bool live_d = d4 < kRowF4;
  for (int r = 0; r < rounds; ++r) {
    const int h = blockIdx.y * hpc + r * hpr + hr;
    float4 acc[kF];
#pragma unroll
    for (int f = 0; f < kF; ++f) acc[f] = make_float4(0.f, 0.f, 0.f, 0.f);
    float run_max = -INFINITY, run_sum = 0.f;
    // partials come from CTAs g0..g1 (CTAs with an empty tile range hold none)
    for (int gs = g0; gs <= g1; gs += kCombineMaxParts) {
      const int ge = min(g1 + 1, gs + kCombineMaxParts);
      __syncthreads();
      if (threadIdx.x < 32) {
        int n = 0;
        for (int g = gs + threadIdx.x; g - static_cast<int>(threadIdx.x) < ge; g += 32) {
          // CTA g holds a tile of b if a tile cost of b lies in its cost range
          bool live = false;
          if (g < ge) {
            const long long x0 = (static_cast<long long>(g) * C) / p.num_ctas;
            const long long x1 = (static_cast<long long>(g + 1) * C) / p.num_ctas;
            const long long k_lo = x0 <= base ? 0 : (x0 - base + kCostTile - 1) / kCostTile;
            const long long k_hi = x1 <= base ? 0 : (x1 - base + kCostTile - 1) / kCostTile;
            live = k_lo < min(k_hi, static_cast<long long>(Tb));
          }
          const unsigned m = __ballot_sync(0xffffffffu, live);
          if (live) slots[n + __popc(m & ((1u << threadIdx.x) - 1))] = pb + g;
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
#pragma unroll
      for (int f = 0; f < kF; ++f) {
        acc[f].x *= a_old; acc[f].y *= a_old; acc[f].z *= a_old; acc[f].w *= a_old;
      }
      run_sum = run_sum * a_old + pass_sum[hr] * a_new;
      run_max = m_new;
      const float* wrow = wts[hr];
      if (live_d) {
        int k = grp;
        for (; k + 3 * groups < n; k += 4 * groups) {
          float4 v[4][kF];
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int f = 0; f < kF; ++f)
              v[u][f] = reinterpret_cast<const float4*>(
                  p.part_o + (static_cast<size_t>(slots[k + u * groups]) * kH + h) * kDq)[d4 + 64 * f];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float w = wrow[k + u * groups] * a_new;
#pragma unroll
            for (int f = 0; f < kF; ++f) {
              acc[f].x = fmaf(w, v[u][f].x, acc[f].x); acc[f].y = fmaf(w, v[u][f].y, acc[f].y);
              acc[f].z = fmaf(w, v[u][f].z, acc[f].z); acc[f].w = fmaf(w, v[u][f].w, acc[f].w);
            }
          }
        }
        for (; k < n; k += groups) {
          const float w = wrow[k] * a_new;
#pragma unroll
          for (int f = 0; f < kF; ++f) {
            const float4 v =
                reinterpret_cast<const float4*>(p.part_o + (static_cast<size_t>(slots[k]) * kH + h) * kDq)[d4 + 64 * f];
            acc[f].x = fmaf(w, v.x, acc[f].x); acc[f].y = fmaf(w, v.y, acc[f].y);
            acc[f].z = fmaf(w, v.z, acc[f].z); acc[f].w = fmaf(w, v.w, acc[f].w);
          }
        }
      }
    }
    if (groups > 1) {
      __syncthreads();
      if (grp > 0)
#pragma unroll
        for (int f = 0; f < kF; ++f) part_acc[grp - 1][d4 + 64 * f] = acc[f];
      __syncthreads();
      if (grp != 0) continue;
      for (int k = 0; k < groups - 1; ++k)
#pragma unroll
        for (int f = 0; f < kF; ++f) {
          const float4 o = part_acc[k][d4 + 64 * f];
          acc[f].x += o.x; acc[f].y += o.y; acc[f].z += o.z; acc[f].w += o.w;
        }
    }
    const float inv = 1.f / run_sum;
    if (live_d) {
#pragma unroll
      for (int f = 0; f < kF; ++f) {
        const size_t oi = (static_cast<size_t>(b) * kH + h) * kDq + 4 * (d4 + 64 * f);
        if (p.out_f32) {
          reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi)[0] =
              make_float4(acc[f].x * inv, acc[f].y * inv, acc[f].z * inv, acc[f].w * inv);
        } else {
          __nv_bfloat162 lo = __floats2bfloat162_rn(acc[f].x * inv, acc[f].y * inv);
          __nv_bfloat162 hi = __floats2bfloat162_rn(acc[f].z * inv, acc[f].w * inv);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + oi)[0] = pk;
        }
      }
    }
    if (d4 == 0 && p.lse != nullptr) p.lse[b * kH + h] = run_max + logf(run_sum);
  }
}

// ------------------------------------------------------------------ host side

constexpr uint64_t kWsHeader = 256;

// Text of the last CUDA failure seen by this host thread (static strings only).
static thread_local const char* g_last_error = "no error";

mfa_status cuda_fail(cudaError_t e, const char* where) {
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
static uint64_t partial_lse_offset(int num_partials, int dq) {
  return align_up(kWsHeader + static_cast<uint64_t>(num_partials) * kH * dq * 4, 256);
}
static uint64_t workspace_bytes_for(int num_partials, int dq) {
  return align_up(partial_lse_offset(num_partials, dq) + static_cast<uint64_t>(num_partials) * kH * 4, 256);
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

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Most tiles any CTA gets under the decode kernel's cost-balanced split (tile k of sequence b
// at cost 4 (S_b + k) + c N_b, N_b the non-empty sequences before b, c = cost_seq; CTA g owns
// costs [floor(g C / G), floor((g + 1) C / G)), C = 4 W + c (N - 1)) for sequences of T[b]
// tiles: the CTA boundaries walked in order over the non-empty sequences.
static long long max_cta_tiles(const std::vector<long long>& Tall, long long G, long long c) {
  std::vector<long long> T;
  for (long long t : Tall)
    if (t > 0) T.push_back(t);
  const long long B = static_cast<long long>(T.size());
  long long W = 0;
  for (long long t : T) W += t;
  const long long C = kCostTile * W + c * std::max(B - 1, 0ll);
  if (C == 0 || G <= 0) return 0;
  long long b = 0, S = 0;
  // first tile with cost >= X, for non-decreasing X
  auto tile_at = [&](long long X) -> long long {
    if (X >= C) return W;
    while (b + 1 < B && kCostTile * (S + T[b]) + c * (b + 1) <= X) { S += T[b]; ++b; }
    const long long base = kCostTile * S + c * b;
    return S + (X <= base ? 0 : std::min(T[b], (X - base + kCostTile - 1) / kCostTile));
  };
  long long prev = tile_at(0), most = 0;
  for (long long g = 0; g < G; ++g) {
    const long long t1 = tile_at(((g + 1) * C) / G);
    most = std::max(most, t1 - prev);
    prev = t1;
  }
  return most;
}

// The attention shape of a problem (kShapeMfa / kShapeGqa / kShapeMla), or -1.
int problem_shape(const mfa_problem* pr) {
  if (pr->page_size != kPage) return -1;
  if (pr->num_q_heads == 64 && pr->head_dim == 256 && pr->num_kv_heads == 1 && !pr->kv_shared) return kShapeMfa;
  if (pr->num_q_heads == 64 && pr->head_dim == 128 && pr->num_kv_heads == 4 && !pr->kv_shared) return kShapeGqa;
  if (pr->num_q_heads == 128 && pr->head_dim == 512 && pr->num_kv_heads == 1 && pr->kv_shared) return kShapeMla;
  return -1;
}
static int units_of(const mfa_problem* pr) { return problem_shape(pr) == kShapeMla ? 2 : 1; }
static int dq_of(const mfa_problem* pr) { return pr->head_dim; }
static int row_of(const mfa_problem* pr) { return pr->head_dim * pr->num_kv_heads; }

// The units the kernels treat as sequences: (sequence, new query token, 64-head set), B * T * U.
static long long vbatch(const mfa_problem* pr) {
  return static_cast<long long>(pr->batch) * pr->tokens_per_seq * units_of(pr);
}

mfa_status check_problem(const mfa_problem* pr) {
  if (pr == nullptr) return MFA_ERR_INVALID_ARG;
  if (pr->tokens_per_seq < 1 || pr->tokens_per_seq > kMaxTokensPerSeq) return MFA_ERR_INVALID_ARG;
  if (pr->batch < 0 || pr->max_pages_per_seq < 1 || pr->num_blocks < 1) return MFA_ERR_INVALID_ARG;
  if (pr->kv_dtype != MFA_KV_BF16 && pr->kv_dtype != MFA_KV_FP8_E4M3 && pr->kv_dtype != MFA_KV_MXFP4)
    return MFA_ERR_INVALID_ARG;
  if (pr->out_dtype != MFA_OUT_BF16 && pr->out_dtype != MFA_OUT_FP32) return MFA_ERR_INVALID_ARG;
  if (!(std::isfinite(pr->softmax_scale) && pr->softmax_scale > 0.f)) return MFA_ERR_INVALID_ARG;
  if (pr->num_kv_heads < 1 || (pr->kv_shared != 0 && pr->kv_shared != 1)) return MFA_ERR_INVALID_ARG;
  const int shp = problem_shape(pr);
  if (shp < 0) return MFA_ERR_UNSUPPORTED;
  // the grouped-head and shared-latent shapes are built for a bf16 cache and one query token
  if (shp != kShapeMfa && (pr->kv_dtype != MFA_KV_BF16 || pr->tokens_per_seq != 1)) return MFA_ERR_UNSUPPORTED;
  if (static_cast<long long>(pr->max_pages_per_seq) * kPage > INT_MAX / 2) return MFA_ERR_INVALID_ARG;
  if (vbatch(pr) * kH > INT_MAX / 2) return MFA_ERR_INVALID_ARG;
  return MFA_OK;
}

static mfa_status check_plan(const mfa_plan* pl, const mfa_problem* pr) {
  if (pl == nullptr) return MFA_ERR_INVALID_ARG;
  if (pl->batch != pr->batch || pl->kv_dtype != pr->kv_dtype || pl->tokens_per_seq != pr->tokens_per_seq)
    return MFA_ERR_INVALID_ARG;
  if (pl->num_ctas < 1 || pl->num_partials != vbatch(pr) + pl->num_ctas - 1) return MFA_ERR_INVALID_ARG;
  if (pl->workspace_bytes != workspace_bytes_for(pl->num_partials, dq_of(pr))) return MFA_ERR_INVALID_ARG;
  return MFA_OK;
}

static mfa_status encode_maps_uncached(DecodeParams& prm, const mfa_problem* pr, const void* q, const void* k,
                                       const void* v) {
  auto enc = encode_fn();
  if (enc == nullptr) return cuda_fail_msg("cuTensorMapEncodeTiled is not available from the driver");
  const int dq = dq_of(pr), rowlen = row_of(pr);
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(dq), static_cast<cuuint64_t>(vbatch(pr)) * kH};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(dq) * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    if (enc(&prm.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail_msg("cuTensorMapEncodeTiled rejected a tensor map");
  }
  const void* pools[2] = {k, pr->kv_shared ? k : v};   // one latent: the V map reads the K pool
  CUtensorMap* maps[2] = {&prm.tm_k, &prm.tm_v};
  const bool fp8 = pr->kv_dtype != MFA_KV_BF16;   // byte elements: e4m3 codes or MXFP4 code pairs
  const cuuint64_t esz = fp8 ? 1 : 2;
  // an MXFP4 row is rowlen / 2 bytes (two E2M1 codes a byte)
  const cuuint64_t row_elems = pr->kv_dtype == MFA_KV_MXFP4 ? rowlen / 2 : rowlen;
  for (int i = 0; i < 2; ++i) {
    cuuint64_t dims[3] = {row_elems, static_cast<cuuint64_t>(kPage), static_cast<cuuint64_t>(pr->num_blocks)};
    cuuint64_t strides[2] = {row_elems * esz, row_elems * esz * kPage};
    // one 128-byte swizzle row per box row: 64 bf16, 128 e4m3 codes or 256 E2M1 codes
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

// The three tensor maps depend only on the q, K and V addresses and the problem's shapes and
// KV dtype, so a host thread keeps its last few encodings: a decode loop over a handful of
// buffers then encodes each set once.  (Host memory only; it changes no result.)
static mfa_status encode_maps(DecodeParams& prm, const mfa_problem* pr, const void* q, const void* k,
                              const void* v) {
  struct Entry {
    const void* q;
    const void* k;
    const void* v;
    long long rows;
    int num_blocks, kv_dtype, shape;
    CUtensorMap tq, tk, tv;
  };
  constexpr int kEntries = 8;
  static thread_local Entry cache[kEntries];
  static thread_local int used = 0, next = 0;
  const long long rows = vbatch(pr) * kH;
  for (int i = 0; i < used; ++i) {
    const Entry& e = cache[i];
    if (e.q == q && e.k == k && e.v == v && e.rows == rows && e.num_blocks == pr->num_blocks &&
        e.kv_dtype == pr->kv_dtype && e.shape == problem_shape(pr)) {
      prm.tm_q = e.tq;
      prm.tm_k = e.tk;
      prm.tm_v = e.tv;
      return MFA_OK;
    }
  }
  const mfa_status st = encode_maps_uncached(prm, pr, q, k, v);
  if (st != MFA_OK) return st;
  Entry& e = cache[next];
  e.q = q;
  e.k = k;
  e.v = v;
  e.rows = rows;
  e.num_blocks = pr->num_blocks;
  e.kv_dtype = pr->kv_dtype;
  e.shape = problem_shape(pr);
  e.tq = prm.tm_q;
  e.tk = prm.tm_k;
  e.tv = prm.tm_v;
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return MFA_OK;
}

// The decode kernel instance of a problem: bf16 MFA, e4m3 MFA, bf16 GQA, bf16 MLA.
using DecodeKernelFn = void (*)(DecodeParams);
static int kernel_index(const mfa_problem* pr) {
  const int shp = problem_shape(pr);
  if (shp != kShapeMfa) return shp == kShapeGqa ? 2 : 3;
  return pr->kv_dtype == MFA_KV_FP8_E4M3 ? 1 : (pr->kv_dtype == MFA_KV_MXFP4 ? 4 : 0);
}
static int threads_of_kernel(int idx) { return idx == 4 ? threads_of<true>() : threads_of<false>(); }
static DecodeKernelFn decode_kernel_of(int idx) {
  switch (idx) {
    case 1: return mfa_decode_kernel<true, kShapeMfa>;
    case 2: return mfa_decode_kernel<false, kShapeGqa>;
    case 3: return mfa_decode_kernel<false, kShapeMla>;
    case 4: return mfa_decode_kernel<true, kShapeMfa, true>;
    default: return mfa_decode_kernel<false, kShapeMfa>;
  }
}

// cudaFuncSetAttribute for a kernel's dynamic shared memory, once per device and kernel.
static mfa_status ensure_smem_attribute(int idx) {
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> done[5][kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const bool cacheable = dev >= 0 && dev < kMaxDevices;
  if (cacheable && done[idx][dev].load(std::memory_order_acquire)) return MFA_OK;
  e = cudaFuncSetAttribute(decode_kernel_of(idx), cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(idx == 4));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  if (cacheable) done[idx][dev].store(true, std::memory_order_release);
  return MFA_OK;
}

static mfa_status launch_combine(const mfa_plan* pl, const mfa_problem* pr, const void* workspace,
                                 const int32_t* seq_lens, void* out, float* lse, cudaStream_t stream,
                                 bool dependent) {
  CombineParams cp;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  cp.part_o = reinterpret_cast<const float*>(ws + partial_o_offset());
  cp.part_lse = reinterpret_cast<const float*>(ws + partial_lse_offset(pl->num_partials, dq_of(pr)));
  cp.seq_lens = seq_lens;
  cp.out = out;
  cp.out_f32 = pr->out_dtype == MFA_OUT_FP32 ? 1 : 0;
  cp.lse = lse;
  cp.batch = static_cast<int>(vbatch(pr));
  cp.tokens = pr->tokens_per_seq;
  cp.units = units_of(pr);
  cp.seq_cost = cost_seq(pr->kv_dtype != MFA_KV_BF16);
  cp.max_pages = pr->max_pages_per_seq;
  cp.num_ctas = pl->num_ctas;
  cudaLaunchConfig_t cfg = {};
  // about two CTAs per SM: many sequences -> more heads per CTA
  const long long want = 2LL * (pl->num_sms > 0 ? pl->num_sms : 148);
  cp.heads_per_cta = (vbatch(pr) * kH >= 16 * want) ? 16 : (vbatch(pr) * kH >= 4 * want) ? 4 : 1;
  cfg.gridDim = dim3(static_cast<unsigned>(vbatch(pr)), kH / cp.heads_per_cta, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const int dq = dq_of(pr);
  const cudaError_t e = dq == 128   ? cudaLaunchKernelEx(&cfg, mfa_combine_wide_kernel<128>, cp)
                        : dq == 512 ? cudaLaunchKernelEx(&cfg, mfa_combine_wide_kernel<512>, cp)
                                    : cudaLaunchKernelEx(&cfg, mfa_combine_kernel, cp);
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
  const int nt = pr->tokens_per_seq, nu = units_of(pr);
  const long long Bv = vbatch(pr);
  // tiles of each unit (sequence, new token, head set): query token i of a sequence of L
  // tokens attends to its first L - T + 1 + i.  T is in schedule order: reader r = i nu + u
  // of sequence b sits at position r B + b (reader-major, as the kernels walk it)
  std::vector<long long> T(static_cast<size_t>(Bv));
  long long W = 0;
  if (host_seq_lens != nullptr) {
    for (int b = 0; b < pr->batch; ++b) {
      if (host_seq_lens[b] < 0 || host_seq_lens[b] > cap) return MFA_ERR_INVALID_ARG;
      for (int i = 0; i < nt; ++i) {
        const long long L = std::max(0ll, static_cast<long long>(host_seq_lens[b]) - (nt - 1 - i));
        for (int u = 0; u < nu; ++u) {
          const size_t pos = (static_cast<size_t>(i) * nu + u) * pr->batch + b;
          T[pos] = (L + kTile - 1) / kTile;
          W += T[pos];
        }
      }
    }
  } else {
    if (max_seq_len < 0 || max_seq_len > cap) return MFA_ERR_INVALID_ARG;
    for (long long x = 0; x < Bv; ++x) T[static_cast<size_t>(x)] = (max_seq_len + kTile - 1) / kTile;
    W = Bv * ((max_seq_len + kTile - 1) / kTile);
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
    G = std::max(G, (W + kMaxTilesPerCta - 1) / kMaxTilesPerCta);   // then the smallest G that fits
  }
  // planned from a bound, any shorter mix must fit too: a CTA's cost range of at most
  // ceil(C / G) units holds at most ceil(ceil(C / G) / 4) tiles
  const long long cs = cost_seq(pr->kv_dtype != MFA_KV_BF16);
  const long long Cb = kCostTile * W + cs * std::max(Bv - 1, 0ll);
  auto worst = [&](long long g) {
    const long long exact = max_cta_tiles(T, g, cs);
    return host_seq_lens != nullptr ? exact
                                    : std::max(exact, ((Cb + g - 1) / g + kCostTile - 1) / kCostTile);
  };
  long long most = worst(G);
  while (most > kMaxTilesPerCta) {
    if (force_ctas > 0) return MFA_ERR_INVALID_ARG;
    ++G;
    most = worst(G);
  }
  if (G > INT_MAX / 2 || Bv + G - 1 > INT_MAX / 2) return MFA_ERR_INVALID_ARG;
  std::memset(plan, 0, sizeof(*plan));
  plan->num_ctas = static_cast<int32_t>(G);
  plan->tile_tokens = kTile;
  plan->max_tiles_per_cta = static_cast<int32_t>(most);
  plan->num_partials = static_cast<int32_t>(Bv + G - 1);
  plan->batch = pr->batch;
  plan->tokens_per_seq = pr->tokens_per_seq;
  plan->kv_dtype = pr->kv_dtype;
  plan->flags = flags;
  plan->num_sms = num_sms;
  plan->total_tiles = static_cast<uint64_t>(W);
  plan->workspace_bytes = workspace_bytes_for(plan->num_partials, dq_of(pr));
  return MFA_OK;
}

// Host-side checks of one decode step's arguments (everything mfa_decode_run validates).
static mfa_status check_run(const mfa_plan* plan, const mfa_problem* pr, const void* q, const void* k_cache,
                            const void* v_cache, const void* k_scale, const void* v_scale,
                            const int32_t* block_table, const int32_t* seq_lens, const void* out,
                            const float* lse, const void* workspace, uint64_t workspace_bytes) {
  mfa_status st = check_problem(pr);
  if (st != MFA_OK) return st;
  st = check_plan(plan, pr);
  if (st != MFA_OK) return st;
  if (pr->batch == 0) return MFA_OK;
  // a shared latent has no V pool: v_cache is ignored (NULL or the K pool)
  if (pr->kv_shared) v_cache = k_cache;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      seq_lens == nullptr || out == nullptr || workspace == nullptr)
    return MFA_ERR_INVALID_ARG;
  if (pr->kv_dtype != MFA_KV_BF16 &&
      (k_scale == nullptr || v_scale == nullptr || !aligned(k_scale, 16) || !aligned(v_scale, 16)))
    return MFA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (lse != nullptr && !aligned(lse, 4)))
    return MFA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return MFA_ERR_WORKSPACE;
  return MFA_OK;
}

// The fused KV append's arguments (see mfa_decode_append_run); null: a plain decode step.
struct FusedAppend {
  const void* k_new;
  const void* v_new;
  const int32_t* positions;
};

// One decode step after validation: the decode kernel (with the fused append, if given), the
// combine, and the MFA_PLAN_CHECK read-back.  clear_status: clear the status word first (the
// two-kernel append path clears it before its append kernel instead).
static mfa_status decode_step(const mfa_plan* plan, const mfa_problem* pr, const void* q, const void* k_cache,
                              const void* v_cache, const void* k_scale, const void* v_scale,
                              const int32_t* block_table, const int32_t* seq_lens, void* out, float* lse,
                              void* workspace, cudaStream_t stream, const FusedAppend* app, bool clear_status) {
  mfa_status st = MFA_OK;

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
  prm.part_lse = reinterpret_cast<float*>(ws + partial_lse_offset(plan->num_partials, dq_of(pr)));
  prm.status = reinterpret_cast<unsigned int*>(ws);
  prm.batch = static_cast<int>(vbatch(pr));
  prm.tokens = pr->tokens_per_seq;
  prm.units = units_of(pr);
  prm.max_pages = pr->max_pages_per_seq;
  prm.num_blocks = pr->num_blocks;
  prm.scale_log2 = static_cast<float>(static_cast<double>(pr->softmax_scale) * 1.4426950408889634);
  prm.early_metadata = (plan->flags & MFA_PLAN_EARLY_METADATA) ? 1 : 0;
  if (app != nullptr) {
    prm.k_new = static_cast<const uint4*>(app->k_new);
    prm.v_new = static_cast<const uint4*>(app->v_new);
    prm.positions = app->positions;
    prm.k_cache_w = const_cast<void*>(k_cache);
    prm.v_cache_w = const_cast<void*>(v_cache);
    prm.k_scale_w = const_cast<void*>(k_scale);
    prm.v_scale_w = const_cast<void*>(v_scale);
    prm.kv_fmt = pr->kv_dtype;
  }

  const bool check = (plan->flags & MFA_PLAN_CHECK) != 0;
  cudaError_t e = cudaSuccess;
  if (check && clear_status && (e = cudaMemsetAsync(ws, 0, 4, stream)) != cudaSuccess) return cuda_fail(e, "memset");
  const int kidx = kernel_index(pr);
  st = ensure_smem_attribute(kidx);
  if (st != MFA_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan->num_ctas), 1, 1);
  cfg.blockDim = dim3(threads_of_kernel(kidx), 1, 1);
  cfg.dynamicSmemBytes = smem_bytes(kidx == 4);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_kernel_of(kidx), prm);
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

mfa_status mfa_decode_run(const mfa_plan* plan, const mfa_problem* pr, const void* q, const void* k_cache,
                          const void* v_cache, const void* k_scale, const void* v_scale,
                          const int32_t* block_table, const int32_t* seq_lens, void* out, float* lse,
                          void* workspace, uint64_t workspace_bytes, void* stream_ptr) {
  mfa_status st = check_run(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse,
                            workspace, workspace_bytes);
  if (st != MFA_OK || pr->batch == 0) return st;
  return decode_step(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse, workspace,
                     static_cast<cudaStream_t>(stream_ptr), nullptr, true);
}

mfa_status mfa_decode_append_run(const mfa_plan* plan, const mfa_problem* pr, const void* q, void* k_cache,
                                 void* v_cache, void* k_scale, void* v_scale, const int32_t* block_table,
                                 const int32_t* seq_lens, const void* k_new, const void* v_new,
                                 const int32_t* positions, void* out, float* lse, void* workspace,
                                 uint64_t workspace_bytes, void* stream_ptr) {
  mfa_status st = check_run(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse,
                            workspace, workspace_bytes);
  if (st != MFA_OK) return st;
  if (problem_shape(pr) != kShapeMfa) return MFA_ERR_UNSUPPORTED;   // the append writes MFA rows
  if (pr->batch == 0) return MFA_OK;
  if (!k_new || !v_new || !positions || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(positions, 4))
    return MFA_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (pr->tokens_per_seq == 1) {
    const FusedAppend app{k_new, v_new, positions};
    return decode_step(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse, workspace,
                       stream, &app, true);
  }
  // several new tokens per sequence: the rows of one sequence are read by several units (one
  // per query token) on different CTAs, so the append kernel runs first
  if ((plan->flags & MFA_PLAN_CHECK) != 0) {
    const cudaError_t e = cudaMemsetAsync(workspace, 0, 4, stream);
    if (e != cudaSuccess) return cuda_fail(e, "memset");
  }
  st = mfa_kv_append(pr, k_new, v_new, positions, block_table, k_cache, v_cache, k_scale, v_scale,
                     static_cast<uint32_t*>(workspace), stream_ptr);
  if (st != MFA_OK) return st;
  return decode_step(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse, workspace,
                     stream, nullptr, false);
}

mfa_status mfa_decode_run_host(const mfa_plan* plan, const mfa_problem* pr, const void* q_host,
                               const int32_t* block_table_host, const int32_t* seq_lens_host, void* out_host,
                               float* lse_host, void* q_dev, int32_t* block_table_dev, int32_t* seq_lens_dev,
                               void* out_dev, float* lse_dev, const void* k_cache, const void* v_cache,
                               const void* k_scale, const void* v_scale, void* workspace,
                               uint64_t workspace_bytes, void* stream_ptr) {
  // the whole step is validated before anything is enqueued
  mfa_status st = check_run(plan, pr, q_dev, k_cache, v_cache, k_scale, v_scale, block_table_dev, seq_lens_dev,
                            out_dev, lse_dev, workspace, workspace_bytes);
  if (st != MFA_OK || pr->batch == 0) return st;
  if (!q_host || !block_table_host || !seq_lens_host || !out_host) return MFA_ERR_INVALID_ARG;
  if ((lse_host == nullptr) != (lse_dev == nullptr)) return MFA_ERR_INVALID_ARG;
  const size_t B = static_cast<size_t>(pr->batch), Bv = static_cast<size_t>(vbatch(pr));
  const size_t dq = static_cast<size_t>(dq_of(pr));
  const size_t q_bytes = Bv * kH * dq * 2, table_bytes = B * pr->max_pages_per_seq * 4, lens_bytes = B * 4;
  const size_t out_bytes = Bv * kH * dq * (pr->out_dtype == MFA_OUT_FP32 ? 4 : 2), lse_bytes = Bv * kH * 4;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaError_t e;
  if ((e = cudaMemcpyAsync(q_dev, q_host, q_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(block_table_dev, block_table_host, table_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(seq_lens_dev, seq_lens_host, lens_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
    return cuda_fail(e, "host to device copy");
  st = mfa_decode_run(plan, pr, q_dev, k_cache, v_cache, k_scale, v_scale, block_table_dev, seq_lens_dev, out_dev,
                      lse_dev, workspace, workspace_bytes, stream_ptr);
  if (st != MFA_OK) return st;
  if ((e = cudaMemcpyAsync(out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
    return cuda_fail(e, "device to host copy");
  if (lse_host != nullptr &&
      (e = cudaMemcpyAsync(lse_host, lse_dev, lse_bytes, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
    return cuda_fail(e, "device to host copy");
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
    const void* k_scale, const void* v_scale, const int32_t* block_table, const int32_t* seq_lens, void* out,
    float* lse, void* stream_ptr) {
  mfa_status st = check_problem(pr);
  if (st != MFA_OK) return st;
  st = check_plan(plan, pr);
  if (st != MFA_OK) return st;
  if (plan->workspace_bytes > MFA_STATIC_WORKSPACE_BYTES) return MFA_ERR_WORKSPACE;
  // the partials of a split plan live in the library's array, which the caller cannot name:
  // without the combine they could never be merged, so such a plan is refused
  if ((plan->flags & MFA_PLAN_NO_COMBINE) != 0 && plan->num_ctas > 1) return MFA_ERR_INVALID_ARG;
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
  // every argument is validated before anything is enqueued, so a refused call leaves
  // nothing on the stream
  st = check_run(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse, ws,
                 MFA_STATIC_WORKSPACE_BYTES);
  if (st != MFA_OK || pr->batch == 0) return st;
  // the status word is the only part that must start at zero; partial results are
  // always written before they are read
  e = cudaMemsetAsync(ws, 0, 4, static_cast<cudaStream_t>(stream_ptr));
  if (e != cudaSuccess) return cuda_fail(e, "memset");
  return mfa_decode_run(plan, pr, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, lse, ws,
                        MFA_STATIC_WORKSPACE_BYTES, stream_ptr);
}
