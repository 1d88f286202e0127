// KV-cache append for MFA decode (GB300, sm_103a): the step before attention in every
// decode step writes each sequence's new key and value rows into the paged cache.  The
// attention instances own and fill their KV caches (Step-3, paperlayer.ai/abs/2507.19427v1,
// section 7 "Implementation and Results"), which hold 8-bit KV (section 5 "Model-System
// Co-design").  For an FP8 cache the quantisation is fused into the same pass: one fp32
// scale per row, s = absmax / 448 (1 for an all-zero row), and e4m3 codes of x / s, rounded
// to nearest even and saturated to +-448; the format the decode kernel reads.  For an MXFP4
// cache (OCP MX FP4, the 4-bit reading of the page's "further KV quantisation", section 5
// "Quantization and MTP"): per block of 32 elements one E8M0 scale 2^(floor(log2 amax) - 2)
// and E2M1 codes of x over it, rounded to nearest even and saturated to 6.
//
// The work is 2BT independent rows of 256 values, T new tokens per sequence.  Each row is
// 512 bytes of bf16 in and 512 bytes of bf16, or 260 bytes of codes and scale, out, so it
// is a latency-bound scatter: one warp per row, one 16-byte load and one 16- or 8-byte
// store per lane, a warp max for the scale; the row's load is issued before the dependent
// position and page-id loads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mfa.h"
#include "mfa_host.h"
#include "ptx.cuh"

namespace mfa {

constexpr int kAppendRowLen = 256;    // head width d
constexpr int kAppendPage = 64;       // tokens per page
constexpr int kAppendWarps = 8;       // rows per CTA
constexpr float kE4m3Max = 448.0f;    // largest finite e4m3 value

struct AppendParams {
  const uint4* k_new;      // bf16 [B, 256] as 16-byte chunks
  const uint4* v_new;
  const int32_t* positions;
  const int32_t* block_table;
  void* k_cache;
  void* v_cache;
  void* k_scale;           // e4m3: fp32 [nb, 64]; MXFP4: E8M0 bytes [nb, 64, 8]
  void* v_scale;
  unsigned int* status;    // may be null
  int batch;
  int tokens;              // new rows per sequence T: row pairs (b, i) = (x / T, x % T)
  int max_pages;
  int num_blocks;
  int kv;                  // mfa_kv_dtype
};

// Two fp32 values to two e4m3 codes (round to nearest even, saturate to +-448): lo in the
// low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight non-negative fp32 values to eight E2M1 codes (round to nearest even, saturate to 6),
// element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8_rn_sat(const float (&a)[8]) {
  uint32_t r;
  // (the first source of each pair goes to the high nibble)
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(a[0]), "f"(a[1]), "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7]));
  return r;
}

__device__ __forceinline__ float bf16_bits_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_bits_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(32 * kAppendWarps) mfa_kv_append_kernel(const __grid_constant__ AppendParams p) {
  // inputs may come from the preceding kernel; the next kernel (the decode) may start its
  // own prologue now: it reads the cache only after this grid has completed
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);   // row: new token r / 2, K or V
  if (r >= 2 * p.batch * p.tokens) return;
  const int xr = r >> 1, b = xr / p.tokens, i = xr % p.tokens;   // token i of sequence b
  const bool is_v = (r & 1) != 0;
  // lane l holds elements 8l .. 8l+7 of the row; the load is issued first, so that it
  // overlaps the position -> page id chain
  const uint4 x = __ldg((is_v ? p.v_new : p.k_new) + static_cast<size_t>(xr) * (kAppendRowLen / 8) + lane);
  const int t0 = p.positions[b];
  if (t0 < 0) return;                                   // no new token for this sequence
  const int t = t0 + i;
  if (t >= p.max_pages * kAppendPage) {
    if (lane == 0 && !is_v && p.status) atomicOr(p.status, MFA_DEV_BAD_LENGTH);
    return;
  }
  const int blk = p.block_table[static_cast<size_t>(b) * p.max_pages + t / kAppendPage];
  if (blk < 0 || blk >= p.num_blocks) {
    if (lane == 0 && !is_v && p.status) atomicOr(p.status, MFA_DEV_BAD_BLOCK);
    return;
  }
  const size_t row = static_cast<size_t>(blk) * kAppendPage + (t % kAppendPage);
  if (p.kv == MFA_KV_MXFP4) {
    // lanes 4j .. 4j + 3 hold block j (elements 32 j .. 32 j + 31)
    float f[8] = {bf16_bits_lo(x.x), bf16_bits_hi(x.x), bf16_bits_lo(x.y), bf16_bits_hi(x.y),
                  bf16_bits_lo(x.z), bf16_bits_hi(x.z), bf16_bits_lo(x.w), bf16_bits_hi(x.w)};
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    // scale 2^e, e = floor(log2 amax) - 2 = E - 129 for amax's biased exponent E, clamped to
    // -127 (E < 2, zero and subnormal blocks included): the byte e + 127 = max(E - 2, 0)
    const uint32_t E = (__float_as_uint(am) >> 23) & 0xFFu;
    const uint32_t sb = E > 2u ? E - 2u : 0u;
    const float inv = __uint_as_float((254u - sb) << 23);   // 2^-e, a normal number (sb <= 252)
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = fabsf(f[i]) * inv;   // exact, or tiny enough to round to 0
    uint32_t sign = 0;   // bit 3 of each nibble: the sign of its element (-0 included)
#pragma unroll
    for (int i = 0; i < 8; ++i) sign |= (__float_as_uint(f[i]) >> 31) << (4 * i + 3);
    uint8_t* cache = static_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache);
    reinterpret_cast<uint32_t*>(cache + row * (kAppendRowLen / 2))[lane] = e2m1x8_rn_sat(a) | sign;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      lo |= __shfl_sync(0xffffffffu, sb, 4 * j) << (8 * j);
      hi |= __shfl_sync(0xffffffffu, sb, 16 + 4 * j) << (8 * j);
    }
    if (lane == 0)
      reinterpret_cast<uint2*>(static_cast<uint8_t*>(is_v ? p.v_scale : p.k_scale))[row] = make_uint2(lo, hi);
    return;
  }
  if (p.kv == MFA_KV_BF16) {
    uint4* dst = static_cast<uint4*>(is_v ? p.v_cache : p.k_cache) + row * (kAppendRowLen / 8) + lane;
    *dst = x;
    return;
  }
  float f[8] = {bf16_bits_lo(x.x), bf16_bits_hi(x.x), bf16_bits_lo(x.y), bf16_bits_hi(x.y),
                bf16_bits_lo(x.z), bf16_bits_hi(x.z), bf16_bits_lo(x.w), bf16_bits_hi(x.w)};
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const float s = (am > 0.f) ? __fdiv_rn(am, kE4m3Max) : 1.f;
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = e4m3x2_rn_sat(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s));
  uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) + row * kAppendRowLen) + lane;
  *dst = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  if (lane == 0) static_cast<float*>(is_v ? p.v_scale : p.k_scale)[row] = s;
}

}  // namespace mfa

using namespace mfa;

extern "C" mfa_status mfa_kv_append(const mfa_problem* pr, const void* k_new, const void* v_new,
                                    const int32_t* positions, const int32_t* block_table, void* k_cache,
                                    void* v_cache, void* k_scale, void* v_scale, uint32_t* device_status,
                                    void* stream_ptr) {
  const mfa_status st = check_problem(pr);
  if (st != MFA_OK) return st;
  if (problem_shape(pr) != 0) return MFA_ERR_UNSUPPORTED;   // rows of the MFA cache (256 wide)
  if (pr->batch == 0) return MFA_OK;
  const bool fp8 = pr->kv_dtype != MFA_KV_BF16;   // scales: fp32 (e4m3) or E8M0 bytes (MXFP4)
  if (!k_new || !v_new || !positions || !block_table || !k_cache || !v_cache) return MFA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(positions, 4) || !aligned(block_table, 4))
    return MFA_ERR_INVALID_ARG;
  const int sa = pr->kv_dtype == MFA_KV_MXFP4 ? 8 : 4;   // one 8-byte or 4-byte store per row
  if (fp8 && (!k_scale || !v_scale || !aligned(k_scale, sa) || !aligned(v_scale, sa))) return MFA_ERR_INVALID_ARG;
  if (device_status && !aligned(device_status, 4)) return MFA_ERR_INVALID_ARG;
  AppendParams p;
  p.k_new = static_cast<const uint4*>(k_new);
  p.v_new = static_cast<const uint4*>(v_new);
  p.positions = positions;
  p.block_table = block_table;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = fp8 ? k_scale : nullptr;
  p.v_scale = fp8 ? v_scale : nullptr;
  p.status = device_status;
  p.batch = pr->batch;
  p.tokens = pr->tokens_per_seq;
  p.max_pages = pr->max_pages_per_seq;
  p.num_blocks = pr->num_blocks;
  p.kv = pr->kv_dtype;
  cudaLaunchConfig_t cfg = {};
  const long long rows = 2LL * pr->batch * pr->tokens_per_seq;
  cfg.gridDim = dim3(static_cast<unsigned>((rows + kAppendWarps - 1) / kAppendWarps), 1, 1);
  cfg.blockDim = dim3(32 * kAppendWarps, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream_ptr);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mfa_kv_append_kernel, p);
  if (e != cudaSuccess) return cuda_fail(e, "kv append launch");
  return MFA_OK;
}
