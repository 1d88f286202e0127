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
#include "mfa_append_row.cuh"

namespace mfa {

constexpr int kAppendRowLen = 256;    // head width d
constexpr int kAppendPage = 64;       // tokens per page
constexpr int kAppendWarps = 8;       // rows per CTA

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
  append_row_warp(p.kv, x, lane, is_v ? p.v_cache : p.k_cache, is_v ? p.v_scale : p.k_scale, row);
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
