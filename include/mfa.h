/*
 * mfa.h -- C ABI of the MFA decode-attention library (libmfa.so), GB300 / sm_103a.
 *
 * The operation.  Step-3's Multi-Matrix Factorization Attention (MFA) keeps many
 * query heads over a factorised QK circuit with one shared key head and one
 * shared value head (Step-3, paperlayer.ai/abs/2507.19427v1, section 2 "Step-3
 * Model Card").  Section 5 "Model-System Co-design" prints the arithmetic
 * intensity (128 FLOP/B with 8-bit KV) and the effective rank (16,384), which
 * fix H = 64 query heads of width d = 256.  One decode step computes, for every
 * sequence b of a batch and every head h, over the L_b cached tokens t:
 *
 *     s_t        = softmax_scale * dot(q[b,h,:], k_t)
 *     out[b,h,:] = sum_t exp(s_t) v_t / sum_t exp(s_t)
 *     lse[b,h]   = ln sum_t exp(s_t)                      (natural log)
 *
 * with k_t = K[block_table[b][t / 64]][t % 64][:] (V likewise): a paged KV
 * cache of 64-token pages.  Section 4 "Cost Analysis for LLM Decoding" states the
 * cost model that the benchmark reports against: the larger of the compute
 * time and the KV-memory-access time.
 *
 * The work is split along the tokens (split-KV, "flash decoding"): a persistent
 * grid of CTAs divides all 128-token tiles of the batch evenly; each CTA writes
 * either the finished output of a sequence it covers whole, or a partial
 * result (normalised O and lse over its token range) that mfa_combine() merges
 * with the log-sum-exp rule.  The pages give no interface; this one is the
 * plainest carrier of the problem statement above.
 *
 * Conventions for every call:
 *   - All device pointers are caller-owned (allocate them with any allocator);
 *     the library allocates no device memory and keeps no device state between calls
 *     (host-side it remembers, per thread, its last few tensor-map encodings, and sets each
 *     kernel's shared-memory attribute once per device; neither changes any result).
 *   - All tensors are dense, row-major, contiguous, with the strides implied by
 *     their shapes below.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) on the current device; nothing synchronises
 *     unless MFA_PLAN_CHECK is set.
 *   - Host-detectable errors return a status before anything is enqueued.
 *     Launch failures return MFA_ERR_CUDA.  Bad data that only the device sees
 *     (a block id outside the pool, a length outside [0, max_pages*64]) never
 *     faults: the affected loads read zeros, and a bit is set in the device
 *     status word of the workspace (see mfa_read_device_status).
 *   - A sequence with L = 0 yields out = 0 and lse = -inf.
 */
#ifndef MFA_H_
#define MFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MFA_ABI_VERSION 5

typedef enum mfa_status {
    MFA_OK = 0,
    MFA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, inconsistent plan */
    MFA_ERR_UNSUPPORTED = 2,   /* a shape this library does not implement (H!=64, d!=256, page!=64) */
    MFA_ERR_WORKSPACE = 3,     /* workspace smaller than plan->workspace_bytes */
    MFA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    MFA_ERR_DEVICE_CHECK = 5   /* MFA_PLAN_CHECK found a nonzero device status word */
} mfa_status;

typedef enum mfa_kv_dtype {
    MFA_KV_BF16 = 0,           /* K/V cache in bf16 */
    MFA_KV_FP8_E4M3 = 1,       /* K/V cache as OCP e4m3 codes, one fp32 scale per token row */
    MFA_KV_MXFP4 = 2           /* K/V cache in the OCP MX FP4 format: E2M1 codes, two a byte
                                  (element 2i in the low nibble of byte i), and one E8M0
                                  scale byte, 2^(e - 127), per 32 elements of a row
                                  (Step-3 page section 5, "Quantization and MTP", names further
                                  KV quantisation; this format is the reading taken) */
} mfa_kv_dtype;

typedef enum mfa_out_dtype {
    MFA_OUT_BF16 = 0,          /* out in bf16: round to nearest even of the fp32 result */
    MFA_OUT_FP32 = 1           /* out in fp32 (the same fp32 result, unrounded) */
} mfa_out_dtype;

/* Device status word bits (set by the kernels, never cleared by them). */
#define MFA_DEV_TIMEOUT      0x1u  /* a pipeline wait exceeded its time limit; outputs invalid */
#define MFA_DEV_BAD_BLOCK    0x2u  /* a block_table entry outside [0, num_blocks) was used */
#define MFA_DEV_BAD_LENGTH   0x4u  /* a seq_lens entry outside [0, max_pages_per_seq*64] (clamped) */
#define MFA_DEV_SCHEDULE     0x8u  /* device lengths need more tiles per CTA than the plan allows */
#define MFA_DEV_RANGE        0x10u /* reserved: no longer set (e4m3 scales have no range limit) */

/* Plan flags. */
#define MFA_PLAN_CHECK       0x1u  /* run: clear the status word, then read it back (synchronises) */
#define MFA_PLAN_NO_COMBINE  0x2u  /* run: launch only the decode kernel; call mfa_combine() yourself */
/* run: the decode kernel is launched as a programmatic dependent of the preceding
 * kernel on the stream and reads seq_lens and block_table (and, in
 * mfa_decode_append_run, positions) before that kernel has finished.  Set it only if
 * the preceding kernel does not write them (for example, when the host fills them
 * once per decode step).  q, K, V, the new rows and all outputs are always ordered
 * after the preceding kernel. */
#define MFA_PLAN_EARLY_METADATA 0x4u

typedef struct mfa_problem {
    int32_t batch;             /* B >= 0 sequences, one new query token each */
    int32_t num_q_heads;       /* H; this library supports 64 */
    int32_t head_dim;          /* d; this library supports 256 */
    int32_t page_size;         /* tokens per KV page; this library supports 64 */
    int32_t max_pages_per_seq; /* columns of block_table (>= 1) */
    int32_t num_blocks;        /* physical pages in each of the K and V pools (>= 1) */
    int32_t kv_dtype;          /* mfa_kv_dtype */
    float softmax_scale;       /* finite, > 0; 1/sqrt(256) = 0.0625 for MFA */
    int32_t out_dtype;         /* mfa_out_dtype */
    int32_t tokens_per_seq;    /* T new query tokens per sequence, 1..4 (see below) */
    int32_t num_kv_heads;      /* G key/value heads per cache row: 1 (MFA, shared latent) or 4 */
    int32_t kv_shared;         /* 1: one latent serves as keys and values (no V pool), else 0 */
} mfa_problem;

/*
 * Multi-token decode (tokens_per_seq = T > 1, as in multi-token prediction or speculative
 * decoding; Step-3 page section 5 "Model-System Co-design": MTP raises the arithmetic
 * intensity).  The T new tokens of sequence b are the last T of its L_b cached tokens (their
 * K and V already appended), and query token i (0 <= i < T) attends to the cached tokens
 * 0 .. L_b - T + i: each new token sees the cache and the new tokens up to itself (causal).
 * q and out are [B, T, 64, 256] (equivalently [B*T, 64, 256]) and lse is [B, T, 64];
 * block_table and seq_lens stay per sequence.  A query token whose range is empty
 * (L_b - T + i < 0) gets out = 0 and lse = -inf.  The pair (b, i) is computed as its own
 * sequence of length L_b - T + 1 + i over b's block-table row, so its KV pages are read once
 * per query token (mostly from L2, the T pairs being adjacent in the schedule).
 */

typedef struct mfa_plan {
    int32_t num_ctas;          /* decode grid size G (persistent CTAs) */
    int32_t tile_tokens;       /* tokens per pipeline tile (128) */
    int32_t max_tiles_per_cta; /* most tiles one CTA gets for the lengths planned with (<= 128) */
    int32_t num_partials;      /* partial-result slots in the workspace: B*T + G - 1 */
    int32_t batch;             /* copy of problem->batch (checked by run) */
    int32_t kv_dtype;          /* copy of problem->kv_dtype (checked by run) */
    uint32_t flags;            /* MFA_PLAN_* */
    int32_t num_sms;           /* SM count the plan was made for */
    uint64_t total_tiles;      /* 128-token tiles of the batch as planned */
    uint64_t workspace_bytes;  /* device bytes the caller must pass to run/combine */
    int32_t tokens_per_seq;    /* copy of problem->tokens_per_seq (checked by run) */
} mfa_plan;

/*
 * Choose the split of the work (the "plan step": number of CTAs and therefore
 * the number of KV splits per sequence) from the batch size and the context
 * lengths.  Host only: no device memory is touched.
 *   problem        : shapes and dtype (validated here).
 *   host_seq_lens  : host int32 [B] lengths, or NULL to plan for B sequences of
 *                    max_seq_len tokens (an upper bound: any lengths up to it run).
 *   max_seq_len    : used when host_seq_lens is NULL; 0 <= max_seq_len <= max_pages*64.
 *   num_sms        : SMs to plan for; 0 queries the current device.
 *   force_ctas     : 0 = automatic (one CTA per SM, fewer when there are fewer
 *                    tiles); > 0 forces the grid size (tests, tuning).
 *   flags          : MFA_PLAN_* copied into the plan.
 *   plan (out)     : filled on MFA_OK.
 * The work is 128-token tiles laid end to end in sequence order.  Tile k of sequence b
 * sits at cost 4 (S_b + k) + c N_b, with S_b the tiles and N_b the non-empty sequences
 * before b, and CTA g of G takes the tiles whose cost lies in
 * [floor(g*C/G), floor((g+1)*C/G)), C = 4 W + c (N - 1) for W tiles in N non-empty
 * sequences: every CTA gets the same share whatever the length mix, a sequence boundary
 * inside a CTA's range (the next sequence's q and one more epilogue) counting as c/4 of a
 * tile, c = 3 for bf16 KV and c = 10 for e4m3 and MXFP4 KV.  A sequence is split once per CTA
 * boundary that falls inside it.  Where several units read one sequence's pages (T > 1 query
 * tokens, or the shared-latent shape's two head sets: R units a sequence, "readers"), the
 * units are laid end to end reader-major -- reader r of sequence b at position r B + b -- so
 * that a page's readers run at the same time on different CTAs and share its L2 lines.  Planned
 * from a length bound (host_seq_lens NULL), the grid keeps every CTA within 128 tiles
 * for any lengths up to the bound.
 */
mfa_status mfa_decode_plan(const mfa_problem* problem, const int32_t* host_seq_lens,
                           int32_t max_seq_len, int32_t num_sms, int32_t force_ctas,
                           uint32_t flags, mfa_plan* plan);

/*
 * Enqueue one decode step (decode kernel, then the combine kernel when the plan
 * has more than one CTA and MFA_PLAN_NO_COMBINE is not set).
 *   q            : device bf16 [B, 64, 256], 16-byte aligned.
 *   k_cache      : device [num_blocks, 64, 256], bf16 or e4m3 codes (uint8); MXFP4: uint8
 *                  [num_blocks, 64, 128] code pairs; 16-byte aligned.
 *   v_cache      : same layout as k_cache.
 *   k_scale      : MXFP4: device uint8 [num_blocks, 64, 8], the E8M0 byte of each 32-element
 *                  block of a row (byte 255, NaN, gives unspecified results), 16-byte
 *                  aligned.  Each row is converted on chip to e4m3 codes under one
 *                  power-of-two scale per row, 2^(m - 6 - 127) for the row's largest scale
 *                  byte m (at least 2^-126): exact for every block whose scale is at least
 *                  2^-14 of the row's largest; smaller blocks round to e4m3's subnormal grid,
 *                  an absolute error below 2^-16 of the row's largest block scale.  From
 *                  there the path is the e4m3 one.
 *                  e4m3: device fp32 [num_blocks, 64], 16-byte aligned (NULL for bf16):
 *                  value = code * scale, any positive finite scale.  The e4m3 path runs
 *                  both contractions on the e4m3 codes as stored: q.K^T against q split
 *                  exactly into two e4m3 parts under one power-of-two scale per sequence,
 *                  with the K scales applied to the fp32 scores; P.V with each token's V
 *                  scale folded into its weights, which are split into two e4m3 parts under
 *                  one power-of-two reference per sequence segment (fp32 accumulation).
 *   v_scale      : same for V.
 *   block_table  : device int32 [B, max_pages_per_seq]; entries past ceil(L_b/64) are never read.
 *   seq_lens     : device int32 [B].
 *   out          : device [B, 64, 256], 16-byte aligned: bf16 (round to nearest even of
 *                  the fp32 result) or fp32, as problem->out_dtype says.
 *   lse          : device fp32 [B, 64] natural-log log-sum-exp of the scaled scores, or NULL.
 *   workspace    : device buffer of >= plan->workspace_bytes bytes, 256-byte aligned.
 *                  Layout: bytes [0,256) header (uint32 status word at offset 0);
 *                  then partial O fp32 [num_partials, 64, 256]; then partial lse fp32
 *                  [num_partials, 64].  The partial of the unit at position x of the
 *                  order above (x = b for one reader a sequence) from CTA g sits in slot
 *                  x + g.  Contents between calls are scratch, except the status word.
 *   stream       : cudaStream_t.
 * Unused slots of a sequence's last page and unused pool pages may hold any bits
 * (NaN included); they never reach the output.
 */
mfa_status mfa_decode_run(const mfa_plan* plan, const mfa_problem* problem,
                          const void* q, const void* k_cache, const void* v_cache,
                          const void* k_scale, const void* v_scale,
                          const int32_t* block_table, const int32_t* seq_lens,
                          void* out, float* lse, void* workspace, uint64_t workspace_bytes,
                          void* stream);

/*
 * One decode step from host buffers: enqueue on `stream` the copies of q, the block table and
 * the lengths from host memory into the caller's device buffers, the decode step exactly as
 * mfa_decode_run enqueues it (on the device buffers), and the copies of out and lse back to
 * host memory.  Nothing synchronises (MFA_PLAN_CHECK excepted, as for mfa_decode_run); the
 * host outputs are valid once the stream has reached this point.  Host buffers should be
 * page-locked (cudaHostAlloc / pinned), or the copies are not asynchronous.
 *   q_host, block_table_host, seq_lens_host : host, same layouts as mfa_decode_run's q,
 *                  block_table and seq_lens.
 *   out_host, lse_host : host, same layouts as out and lse; lse_host NULL iff lse_dev NULL.
 *   q_dev, block_table_dev, seq_lens_dev, out_dev, lse_dev : the device buffers the step
 *                  runs on (the requirements of mfa_decode_run's arguments); the caller owns
 *                  them and must not reuse them until the stream has passed this step.
 *   k_cache .. workspace_bytes, stream : as for mfa_decode_run.
 * Every argument is validated before anything is enqueued.  Two such steps on two streams,
 * each with its own device buffers and workspace, overlap one step's copies with the other's
 * kernels.
 */
mfa_status mfa_decode_run_host(const mfa_plan* plan, const mfa_problem* problem,
                               const void* q_host, const int32_t* block_table_host,
                               const int32_t* seq_lens_host, void* out_host, float* lse_host,
                               void* q_dev, int32_t* block_table_dev, int32_t* seq_lens_dev,
                               void* out_dev, float* lse_dev,
                               const void* k_cache, const void* v_cache,
                               const void* k_scale, const void* v_scale,
                               void* workspace, uint64_t workspace_bytes, void* stream);

/*
 * Enqueue the log-sum-exp merge of the partial results in `workspace` (the split
 * combine): for every sequence covered by more than one CTA,
 *     lse* = M + ln sum_s exp(lse_s - M),  M = max_s lse_s,
 *     out  = sum_s exp(lse_s - lse*) O_s          (O_s normalised partials)
 * and writes out (in problem->out_dtype) and lse (fp32, if non-NULL).  Sequences covered by one
 * CTA, and empty ones, were written by the decode kernel and are left alone.
 * Arguments as for mfa_decode_run; seq_lens must equal the ones the decode used.
 */
mfa_status mfa_combine(const mfa_plan* plan, const mfa_problem* problem,
                       const void* workspace, uint64_t workspace_bytes,
                       const int32_t* seq_lens, void* out, float* lse, void* stream);

/*
 * Read the device status word of `workspace` into *status_bits (MFA_DEV_* bits),
 * optionally clearing it; synchronises `stream`.
 */
mfa_status mfa_read_device_status(void* workspace, uint32_t* status_bits, int32_t clear,
                                  void* stream);

/* Static description of a status code. */
const char* mfa_status_string(mfa_status status);

/*
 * mfa_decode_run without a caller-supplied workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory: for example a plugin inside a host application whose own
 * allocator owns the GPU's memory (a cudaMalloc from the plugin would bypass the
 * application's accounting), or a latency-critical path where cudaMalloc's
 * implicit device synchronisation is not acceptable.
 *
 * The scratch is a fixed array of MFA_STATIC_WORKSPACE_BYTES inside the library,
 * created on every device that loads it and kept until the process exits.  This
 * call allocates nothing.  Its first call on a device looks the array's device
 * address up (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  Every argument is validated first; a call
 * that is refused enqueues nothing.  A valid call clears the array's status
 * word, then enqueues exactly what mfa_decode_run enqueues (MFA_PLAN_CHECK
 * included).  All calls on a device share the one array and it keeps the last
 * call's contents, so two calls whose kernels may overlap on the GPU (different
 * streams, no ordering between them) race on it: order them on one stream.
 *   - Plans whose workspace_bytes exceed MFA_STATIC_WORKSPACE_BYTES are rejected
 *     with MFA_ERR_WORKSPACE; at the default 24 MiB that covers
 *     batch + num_ctas - 1 <= 382 partial slots (for example B <= 231 on 152 SMs).
 *   - A plan with MFA_PLAN_NO_COMBINE and more than one CTA is rejected with
 *     MFA_ERR_INVALID_ARG: its partial results would stay in the library's
 *     array, which no caller can pass to mfa_combine().
 *   - The array's address is never handed out, so mfa_read_device_status()
 *     cannot read this path's status word.  Its device-side checks (a block id
 *     outside the pool, a bad length, a timed-out wait) are reported only
 *     through MFA_PLAN_CHECK, as MFA_ERR_DEVICE_CHECK.
 * Arguments are those of mfa_decode_run without the workspace.
 */
#define MFA_STATIC_WORKSPACE_BYTES (24u * 1024u * 1024u)
mfa_status mfa_decode_run_static_workspace(const mfa_plan* plan, const mfa_problem* problem,
                                           const void* q, const void* k_cache, const void* v_cache,
                                           const void* k_scale, const void* v_scale,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           void* out, float* lse, void* stream);

/*
 * Enqueue the KV-cache append of one decode step: each sequence's new key row and
 * value row go into the paged cache (the attention instances own and fill their KV
 * caches, Step-3 page section 7 "Implementation and Results"; the cache holds 8-bit
 * KV, section 5 "Model-System Co-design").  With T = problem->tokens_per_seq new tokens
 * per sequence, for every b with positions[b] >= 0 and every i < T, row k_new[b*T + i]
 * goes to K slot t % 64 of page block_table[b][t / 64], t = positions[b] + i, and
 * v_new[b*T + i] to the same V slot:
 *   - bf16 cache: the bf16 bits, unchanged;
 *   - e4m3 cache (quantisation fused in the same pass): the row's scale
 *     s = absmax / 448 in fp32 (s = 1 for an all-zero row) goes to
 *     k_scale/v_scale[page][slot], and each value x to the e4m3 code of x / s
 *     (both divisions fp32, rounded to nearest; the code rounded to nearest even,
 *     magnitudes above 448 saturated to 448; a negative x that rounds to zero gives
 *     the code 0x80).  The row maximum always lands on code +-448;
 *   - MXFP4 cache (quantisation fused in the same pass): per block of 32 elements the
 *     scale byte max(E - 2, 0), E the biased fp32 exponent of the block's largest |x|
 *     (the OCP MX rule: 2^(floor(log2 amax) - 2), clamped to [2^-127, 2^127]; an all-zero
 *     or subnormal block takes byte 0), and each x to the E2M1 code of x / 2^(byte - 127),
 *     rounded to nearest even, saturated to 6, sign kept (a negative x that rounds to zero
 *     gives the code 8).
 *   problem      : the decode's problem description (kv_dtype, batch, table width and
 *                  pool size are used); validated as for mfa_decode_plan.
 *   k_new, v_new : device bf16 [B, T, 256], 16-byte aligned, finite values (non-finite
 *                  values give unspecified codes and scales).
 *   positions    : device int32 [B]: the token index of each sequence's first new row
 *                  (usually its length before the step); a negative entry means no
 *                  new token for that sequence (nothing is written).
 *   block_table  : device int32 [B, max_pages_per_seq]: must already hold the page of
 *                  position t (allocate it before the step).
 *   k_cache, v_cache, k_scale, v_scale : the pools of mfa_decode_run, written in place;
 *                  only the target slots change.  Scales NULL for a bf16 cache; fp32 for
 *                  e4m3, E8M0 bytes for MXFP4.
 *   device_status: device uint32, or NULL.  A position >= max_pages_per_seq * 64 sets
 *                  MFA_DEV_BAD_LENGTH, a page id outside [0, num_blocks) sets
 *                  MFA_DEV_BAD_BLOCK; that token's rows are then not written.  The
 *                  status word of a decode workspace (offset 0) may be passed, so that
 *                  mfa_read_device_status() reports both steps.
 *   stream       : cudaStream_t.  The kernel is launched as a programmatic dependent
 *                  of the preceding kernel and lets the next kernel start early; a
 *                  decode kernel launched next reads the cache only after the append
 *                  has completed.
 */
mfa_status mfa_kv_append(const mfa_problem* problem, const void* k_new, const void* v_new,
                         const int32_t* positions, const int32_t* block_table,
                         void* k_cache, void* v_cache, void* k_scale, void* v_scale,
                         uint32_t* device_status, void* stream);

/*
 * One decode step with the KV append in front of it: the same result as mfa_kv_append()
 * (its status bits going to the workspace's status word) followed by mfa_decode_run() on the
 * same stream, for the MFA shape.  With one new token per sequence it is one kernel launch:
 * the CTA that reads the page of a sequence's new row writes that row first (the caches are
 * written in place, in their format, as by mfa_kv_append), and rows whose position is at or
 * past the sequence's length (read by nobody this step) are written too.  With several new
 * tokens per sequence the append kernel runs first.
 *   k_new, v_new : device bf16 [B, T, 256], 16-byte aligned.
 *   positions    : device int32 [B], 4-byte aligned (as for mfa_kv_append).
 *   k_cache .. k_scale, v_scale : written in place (the pools of mfa_decode_run).
 *   Other arguments as for mfa_decode_run.  seq_lens are the lengths after the append (a
 *   sequence whose new token is at position t has length t + T when it reads it).
 * Every argument is validated before anything is enqueued; other shapes give
 * MFA_ERR_UNSUPPORTED.
 */
mfa_status mfa_decode_append_run(const mfa_plan* plan, const mfa_problem* problem,
                                 const void* q, void* k_cache, void* v_cache,
                                 void* k_scale, void* v_scale,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 const void* k_new, const void* v_new, const int32_t* positions,
                                 void* out, float* lse, void* workspace, uint64_t workspace_bytes,
                                 void* stream);

/* MFA_ABI_VERSION of the loaded library. */
int32_t mfa_abi_version(void);

/* Text of the last CUDA failure behind an MFA_ERR_CUDA on the calling host thread
 * ("no error" if none); a static string, valid until the next call on this thread. */
const char* mfa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MFA_H_ */
