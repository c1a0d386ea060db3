/*
 * rq.h -- C ABI of the B300 (sm_103a) inverse-RoPE + block-FP8 quant library.
 *
 * Two operations, both from the DeepSeek-V4 attention path described on these
 * pages (cited by title and section):
 *
 *  [INV] "[vllm] 한 프로그램이 4개 head를 처리하게 하라: DeepSeek-V4 inverse
 *        RoPE + FP8 quant 커널 3.5배 가속기" (analysis of vLLM PR #63540):
 *        intro (the op and its [token, head, 512] bf16 input), S1 (output
 *        groups of heads_per_group heads, per-head scale slots), S2 (GPT-J
 *        pair rotation of dims 448..511 from a [P, 64] cos|sin cache), S3
 *        (128-element block amax clamped by eps).
 *  [KV]  "[vllm] vLLM DeepSeek-V4 성능 최적화: Eager Break 시 Workspace 재사용
 *        개선" (analysis of vLLM PR #49236), S1-S2: kv [N, 512] is rotated,
 *        quantised and inserted into a paged uint8 k_cache by slot_mapping;
 *        outputs are preallocated by the caller (the `_out` form, void return).
 *  [IDX] "[vllm] vLLM의 GLM5.2 성능 최적화: Triton 커널 융합을 통한 E2E
 *        Throughput 향상" (analysis of vLLM PR #46862), S1: power-of-two
 *        scale exp2(ceil(log2(raw scale))).
 *
 * Numerics shared by both operations (all fp32):
 *   y = float(x)                                   (bf16 -> fp32, exact)
 *   pair j = (y[448+2j], y[449+2j]), c = cache[p][j], s = cache[p][32+j]:
 *     inverse: even' = even*c + odd*s,  odd' = odd*c - even*s
 *     forward: even' = even*c - odd*s,  odd' = odd*c + even*s
 *     (each product and each sum rounded to fp32 separately, no FMA)
 *   per 128-element block b: amax = max(max|y'|, eps),
 *     scale = 2^ceil(log2(fl32(amax / 448))), exactly (a power of two),
 *     code  = e4m3fn(y' / scale): round to nearest even, saturate at +-448.
 *
 * Conventions:
 *  - The caller allocates every buffer; the library allocates nothing and
 *    keeps no state beyond a per-device cache of launch limits.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls
 *    are asynchronous and stream-ordered; nothing synchronises.
 *  - The return value reports host-side argument checks, or a launch error
 *    from cudaGetLastError (RQ_ERR_CUDA; the CUDA error is then cleared).
 *    On any error nothing is launched and no buffer is touched.
 *  - Every device-side wait (the shared-memory pipeline's barriers) is
 *    bounded; one that gives up sets RQ_FLAG_TIMEOUT and its CTA returns.
 *  - Device-side index checks: a token whose position is outside
 *    [0, cache_rows), or whose slot is >= num_blocks * block_size, is
 *    skipped (its outputs are left untouched) and the matching bit is OR-ed
 *    into *error_flags (RQ_FLAG_*) when error_flags is not NULL. No kernel
 *    traps.
 *  - NaN / Inf inputs are outside the contract: results are unspecified
 *    but no memory access depends on them.
 *  - Every pointer is a device pointer (or managed / mapped memory the
 *    device can reach) on the current device.
 *  - No input may overlap an output of the same call: the kernels read
 *    their inputs through the non-coherent read-only path, so bytes written
 *    over an input during the call may or may not be seen.
 */
#ifndef RQ_H_
#define RQ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rq_status {
    RQ_OK = 0,
    RQ_ERR_NULL = 1,     /* a required pointer is NULL                      */
    RQ_ERR_SHAPE = 2,    /* a size or stride is out of range                */
    RQ_ERR_ALIGN = 3,    /* a pointer or stride breaks the 16-byte rule     */
    RQ_ERR_GROUPING = 4, /* heads_per_group < 1 or does not divide n_heads  */
    RQ_ERR_CUDA = 5,     /* the CUDA runtime reported an error              */
    RQ_ERR_ARG = 6       /* eps outside [2^-100, 2^100], or a bad variant or
                            output mode                                     */
} rq_status;

/* device-side error bits (OR-ed into *error_flags) */
#define RQ_FLAG_POSITION_RANGE 1u /* a position was outside [0, cache_rows)   */
#define RQ_FLAG_SLOT_RANGE 2u     /* a slot was >= num_blocks * block_size    */
#define RQ_FLAG_TIMEOUT 4u        /* a pipeline wait gave up (never expected):
                                     the outputs of that launch are incomplete */
#define RQ_FLAG_SLOT_DUPLICATE 8u /* two tokens map to one slot (found only by
                                     rq_validate_indices)                       */

/* Static, NUL-terminated description of a status code. */
const char *rq_status_string(int status);

/* Library ABI version, (major << 16) | minor. */
int rq_version(void);

/*
 * Inverse RoPE + block-FP8 quant ([INV] intro, S1-S3).
 *
 *  x_bf16          [n_tokens, n_heads, 512] bf16; element (t, h, k) at
 *                  x_bf16 + t*x_stride_token + h*x_stride_head + k
 *                  (strides in elements; the last dim is contiguous).
 *                  Base 16-byte aligned, both strides multiples of 8.
 *  positions       [n_tokens] int64, 8-byte aligned; row of the cache.
 *  cos_sin_cache   [cache_rows, 64] fp32 contiguous, 16-byte aligned:
 *                  columns 0..31 cos, 32..63 sin.
 *  heads_per_group >= 1, divides n_heads; G = n_heads / heads_per_group.
 *  eps             lower clamp of every block amax, in [2^-100, 2^100].
 *  out_fp8         [n_tokens, G, heads_per_group*512] e4m3fn codes,
 *                  contiguous, 16-byte aligned: head h = g*hpg + i of token
 *                  t owns bytes [i*512, i*512+512) of row (t, g).
 *  out_scales      [n_tokens, G, heads_per_group*4] fp32, contiguous,
 *                  16-byte aligned: block b of that head at i*4 + b.
 *  error_flags     optional device uint32 (may be NULL), see RQ_FLAG_*.
 *  stream          cudaStream_t.
 *
 * n_tokens == 0 returns RQ_OK with no launch. n_tokens * n_heads must be
 * below 2^31.
 */
rq_status rq_inv_rope_fp8_quant(const void *x_bf16, int64_t n_tokens, int64_t n_heads,
                                int64_t x_stride_token, int64_t x_stride_head,
                                const int64_t *positions, const float *cos_sin_cache,
                                int64_t cache_rows, int64_t heads_per_group, float eps,
                                uint8_t *out_fp8, float *out_scales,
                                uint32_t *error_flags, void *stream);

/*
 * Device workspace, in bytes, that rq_inv_rope_fp8_quant_host needs for
 * chunks of chunk_tokens tokens of n_heads heads (three chunk slots, each
 * holding x, positions, codes and scales). -1 for n_heads < 1,
 * chunk_tokens < 1 or chunk_tokens * n_heads >= 2^31.
 */
int64_t rq_inv_rope_fp8_quant_host_workspace(int64_t n_heads, int64_t chunk_tokens);

/*
 * rq_inv_rope_fp8_quant over HOST buffers (same op, same bytes). The tokens go
 * through the device in chunks of chunk_tokens: each chunk is copied into a
 * slot of the caller's device workspace, processed by the op's kernels on
 * `stream` and copied back. Two copy streams owned by the library run the
 * copies: while one chunk is processed, the next is copied in and the
 * previous one out, so both directions of the host link are busy at once.
 * The call is stream-ordered on `stream` like every other: the copies start
 * after the work enqueued on `stream` before the call, and work enqueued
 * after it starts once the last copy-out has finished. The host outputs are
 * complete when `stream` has synchronised.
 *  x_bf16_host      [N, H, 512] bf16, contiguous, host memory (page-locked
 *                   for the copies to overlap; pageable memory works, slowly).
 *  positions_host   [N] int64, host memory.
 *  cos_sin_cache    [cache_rows, 64] fp32, DEVICE memory (as in
 *                   rq_inv_rope_fp8_quant).
 *  out_fp8_host     [N, G, hpg*512] uint8, host memory.
 *  out_scales_host  [N, G, hpg*4] fp32, host memory.
 *  workspace        device memory, 256-byte aligned, owned by the caller, at
 *                   least rq_inv_rope_fp8_quant_host_workspace(H, chunk_tokens)
 *                   bytes (else RQ_ERR_SHAPE); must not be reused until `stream`
 *                   passes this call.
 *  error_flags      device memory or NULL, as in rq_inv_rope_fp8_quant.
 * Other arguments and errors as in rq_inv_rope_fp8_quant, except that the
 * host outputs of a token whose position is out of range are unspecified
 * (chunks are copied back whole; the flag is still set). On an RQ_ERR_CUDA
 * return part of the pipeline may have been enqueued; the outputs are then
 * unspecified. Calls from several host threads are serialised per device.
 */
rq_status rq_inv_rope_fp8_quant_host(const void *x_bf16_host, int64_t n_tokens, int64_t n_heads,
                                     const int64_t *positions_host, const float *cos_sin_cache,
                                     int64_t cache_rows, int64_t heads_per_group, float eps,
                                     uint8_t *out_fp8_host, float *out_scales_host,
                                     void *workspace, int64_t workspace_bytes,
                                     int64_t chunk_tokens, uint32_t *error_flags, void *stream);

/*
 * TEST ONLY: fault injection for the bounded waits of the TMA / tensor-core
 * kernels, for calls made afterwards from the calling host thread. Each
 * selected kernel skips one of its own copies, so a wait on a barrier that
 * nothing will complete runs out after spin_limit polls (0 = the default,
 * 2^22); the kernel then sets RQ_FLAG_TIMEOUT in error_flags, lets its
 * copies in flight land, frees what it holds and exits, leaving the context
 * usable. Outputs of an injected call are unspecified. mask 0 and
 * spin_limit 0 restore normal operation.
 *   RQ_DEBUG_STREAM_STAGE  the TMA-ring inverse kernel (RQ_INV_STREAM):
 *                          warp 0 leaves its first tile unarmed
 *   RQ_DEBUG_GEMM_LOADS    rq_grouped_fp8_gemm and rq_grouped_fp8_gemm_ue8m0:
 *                          the first CTA's TMA producer issues no copy
 */
#define RQ_DEBUG_STREAM_STAGE 1u
#define RQ_DEBUG_GEMM_LOADS 2u
void rq_debug_inject(uint32_t mask, uint32_t spin_limit);

/*
 * TEST ONLY: the kernels' own per-block arithmetic over a range of fp32 bit
 * patterns, so that it can be checked exhaustively against an independent
 * statement of it. Neither is part of the op; both are stream-ordered and
 * asynchronous, allocate nothing and write only the caller's arrays.
 *
 * rq_debug_block_scale: for i in [0, count), with amax = the fp32 value of
 * bit pattern first_bits + i, writes the block scale every quantising kernel
 * takes, 2^ceil(log2(fl32(max(amax, eps) / 448))) (the power-of-two scale of
 * the GLM5.2 page, S1, applied to the block absmax of the inverse-RoPE page,
 * S3), to scales[i] and its exact reciprocal to inv_scales[i] (both device
 * fp32 [count], 4-byte aligned). Defined for finite amax; eps as in
 * rq_inv_rope_fp8_quant. first_bits + count <= 2^32, else RQ_ERR_SHAPE.
 *
 * rq_debug_quant_codes: for i in [0, count), writes to codes[i] the e4m3
 * code the kernels store for the fp32 value v of bit pattern first_bits + i
 * in a block whose scale is 2^scale_exp: v times the exact inverse scale
 * (round to nearest even), converted with round-to-nearest-even and
 * saturation to +-448 (inverse-RoPE page, S3). count a multiple of 16;
 * codes device, 16-byte aligned; scale_exp in [-126, 126] (else RQ_ERR_ARG).
 */
rq_status rq_debug_block_scale(uint32_t first_bits, int64_t count, float eps, float *scales,
                               float *inv_scales, void *stream);
rq_status rq_debug_quant_codes(uint32_t first_bits, int64_t count, int scale_exp,
                               uint8_t *codes, void *stream);

/*
 * Debug helper: checks the device-side preconditions of the ops, which the
 * ops themselves only partly check (a repeated slot goes unnoticed there),
 * without running them. One non-trapping kernel on `stream`, then the result
 * word is copied to the host and `stream` is synchronised.
 *  positions      [n_tokens] int64, device: each must be in [0, cache_rows)
 *                 (else RQ_FLAG_POSITION_RANGE).
 *  slot_mapping   [n_tokens] int64, device, or NULL to check positions only:
 *                 each must be negative (the token is skipped) or below
 *                 num_slots (else RQ_FLAG_SLOT_RANGE), and no two tokens may
 *                 share a slot (else RQ_FLAG_SLOT_DUPLICATE).
 *  num_slots      num_blocks * block_size of the paged cache (>= 1 when
 *                 slot_mapping is given).
 *  workspace      device, 16-byte aligned, at least
 *                 rq_validate_indices_workspace(num_slots) bytes (a bitmap of
 *                 num_slots bits and the result word); owned by the caller.
 *  result         host uint32: the RQ_FLAG_* bits found (0 = all valid).
 * positions and slot_mapping 8-byte aligned. n_tokens >= 0 (0 writes 0).
 */
int64_t rq_validate_indices_workspace(int64_t num_slots);
rq_status rq_validate_indices(const int64_t *positions, const int64_t *slot_mapping,
                              int64_t n_tokens, int64_t cache_rows, int64_t num_slots,
                              void *workspace, int64_t workspace_bytes, uint32_t *result,
                              void *stream);

/*
 * rq_validate_indices for callers that cannot allocate device memory: a
 * program that links only this library and has no device allocator, or an
 * engine whose free device memory is all given to its KV cache and that must
 * not allocate mid-step. The pages have no counterpart; this is a library
 * convenience. Same checks, arguments and result as rq_validate_indices,
 * without the workspace: the slot bitmap and result word live in a fixed
 * device array of the library (131,328 bytes on every GPU that loads it, held
 * until the process exits). num_slots above 1,048,576 (2^20) returns
 * RQ_ERR_SHAPE. Nothing is allocated. The first call on a device looks up
 * the array's device address (make that first call before any stream
 * capture); that address belongs to the device's primary context, so after a
 * cudaDeviceReset the entry point must not be called again in the process.
 * A CUDA failure returns RQ_ERR_CUDA and clears the runtime's sticky error,
 * as the other entry points do. Every call clears the part of the array it uses; calls whose
 * work overlaps on the GPU (other streams or host threads) race on the
 * shared array. The call synchronises `stream` before it returns.
 */
rq_status rq_validate_indices_noalloc(const int64_t *positions, const int64_t *slot_mapping,
                                      int64_t n_tokens, int64_t cache_rows, int64_t num_slots,
                                      uint32_t *result, void *stream);

/* Kernel variants of rq_inv_rope_fp8_quant; all produce identical bytes. */
typedef enum rq_inv_variant {
    RQ_INV_AUTO = 0,          /* the default: warp rows (measured the faster of the
                                 two at every size on B300)                          */
    RQ_INV_WARP_ROWS = 1,     /* persistent warps, rows loaded straight to registers */
    RQ_INV_STREAM = 2         /* every warp streams 8-head tiles through a private
                                 two-stage ring of shared memory filled by 1-D bulk
                                 copies (TMA), re-arming each stage once read        */
} rq_inv_variant;

/* rq_inv_rope_fp8_quant with an explicit kernel variant (rq_inv_variant);
 * any other value returns RQ_ERR_ARG. Same arguments and behaviour. */
rq_status rq_inv_rope_fp8_quant_ex(const void *x_bf16, int64_t n_tokens, int64_t n_heads,
                                   int64_t x_stride_token, int64_t x_stride_head,
                                   const int64_t *positions, const float *cos_sin_cache,
                                   int64_t cache_rows, int64_t heads_per_group, float eps,
                                   uint8_t *out_fp8, float *out_scales,
                                   uint32_t *error_flags, void *stream, int variant);

/* What rq_inv_rope_quant_layout writes for each head. */
typedef enum rq_out_mode {
    RQ_OUT_FP8_SCALE_F32 = 0,   /* 512 e4m3 codes + 4 fp32 block scales               */
    RQ_OUT_FP8_SCALE_UE8M0 = 1, /* 512 e4m3 codes + one uint32 of packed UE8M0 scales:
                                   byte b (bits 8b..8b+7) = the biased exponent of
                                   block b's power-of-two scale (value 2^(byte-127))  */
    RQ_OUT_BF16 = 2             /* no quantisation: the 512 inverse-rotated values as
                                   bf16, each rounded to nearest even                 */
} rq_out_mode;

/*
 * Inverse RoPE with a choice of output kind and any output layout ([INV]
 * S1-S4: the page's kernel has a non-quantising variant (CompileKey.quantize,
 * S4) and packs scales as UE8M0 as well (S3)). Inputs and numerics are those
 * of rq_inv_rope_fp8_quant; only the outputs differ:
 *
 *  out        head i (0 <= i < heads_per_group) of group g of token t starts at
 *               out + t*out_stride_token + g*out_stride_group + i*W  (bytes),
 *             W = 512 (codes) or 1024 (bf16); its W bytes are contiguous.
 *             16-byte aligned; both strides >= 0 and multiples of 16.
 *             The contiguous [N, G, hpg*512] layout of rq_inv_rope_fp8_quant is
 *             out_stride_token = G*hpg*W, out_stride_group = hpg*W; a
 *             group-major [G, N, hpg*W] buffer is out_stride_group = N*hpg*W,
 *             out_stride_token = hpg*W.
 *  scales     element j of group g of token t sits at
 *               scales + t*scale_stride_token + g*scale_stride_group
 *                      + j*scale_stride_elem          (in elements),
 *             j = 4i + b (fp32, RQ_OUT_FP8_SCALE_F32) or j = i (uint32,
 *             RQ_OUT_FP8_SCALE_UE8M0). 4-byte aligned, strides >= 0.
 *             Ignored (may be NULL) for RQ_OUT_BF16.
 *  out_mode   an rq_out_mode; any other value returns RQ_ERR_ARG.
 *
 * Outputs that overlap give unspecified bytes. Positions outside
 * [0, cache_rows) are skipped and flagged as in rq_inv_rope_fp8_quant.
 * The kernel is chosen from the layout, the mode and the size; all choices
 * write the same bytes. Row-linear token-major quantised outputs (head r =
 * t*H + h at out + r*512, its scales at r*4 or its word at r) and contiguous
 * group-major ones ([G, N, hpg*512] codes with [G, N, hpg*4] fp32 scales or
 * [G, N, hpg] words, 16-byte aligned) take the warp-rows kernel of
 * rq_inv_rope_fp8_quant. fp32 scales stored token-contiguous
 * (scale_stride_token == 1, e.g. transposed [G, hpg*4, N]) take a
 * token-tiled kernel that stores 8 tokens' scales at once, when the call is
 * large enough (at least 6 tiles of 8 tokens per warp). Other layouts take
 * the warp-rows layout kernel (quantising modes with each warp on fixed
 * heads, bf16 by a row walk).
 */
rq_status rq_inv_rope_quant_layout(const void *x_bf16, int64_t n_tokens, int64_t n_heads,
                                   int64_t x_stride_token, int64_t x_stride_head,
                                   const int64_t *positions, const float *cos_sin_cache,
                                   int64_t cache_rows, int64_t heads_per_group, float eps,
                                   int out_mode, void *out, int64_t out_stride_token,
                                   int64_t out_stride_group, void *scales,
                                   int64_t scale_stride_token, int64_t scale_stride_group,
                                   int64_t scale_stride_elem, uint32_t *error_flags,
                                   void *stream);

/*
 * Forward RoPE + block-FP8 quant + paged insert ([KV] S1, numerics as above
 * with the forward rotation).
 *
 *  kv_bf16         [n_tokens, 512] bf16, token stride kv_stride_token
 *                  elements (multiple of 8), base 16-byte aligned.
 *  positions       [n_tokens] int64; cos_sin_cache as above.
 *  slot_mapping    [n_tokens] int64: slot s < 0 skips the token; otherwise
 *                  the token's 528-byte record (512 codes, then the four
 *                  fp32 block scales) goes to
 *                  k_cache + (s / block_size) * block_stride_bytes
 *                          + (s % block_size) * 528.
 *                  Slots of different tokens must differ (a repeated slot
 *                  gets one of the writers' bytes, unspecified which).
 *  k_cache         [num_blocks, block_stride_bytes] uint8, 16-byte aligned;
 *                  bytes outside the mapped records are never written.
 *  block_stride_bytes >= block_size * 528 and a multiple of 16.
 *  error_flags     optional device uint32 (may be NULL).
 */
rq_status rq_rope_fp8_quant_insert(const void *kv_bf16, int64_t n_tokens,
                                   int64_t kv_stride_token, const int64_t *positions,
                                   const float *cos_sin_cache, int64_t cache_rows,
                                   const int64_t *slot_mapping, uint8_t *k_cache,
                                   int64_t num_blocks, int64_t block_size,
                                   int64_t block_stride_bytes, float eps,
                                   uint32_t *error_flags, void *stream);

/*
 * The fused q/kv op of [KV] S1-S2 (the `_out` form: q_out is preallocated by
 * the caller, nothing is returned). In one launch, for every token t:
 *  - each q head h < n_heads_q (bf16 [N, n_heads_q, 512], strides in
 *    elements, multiples of 8, base 16-byte aligned) is RMS-normalised over
 *    its 512 values, y_k = x_k / sqrt(mean(x^2) + norm_eps) * w_k, then
 *    forward-rotated on dims 448..511 with row positions[t] of the cache,
 *    and written as bf16 (round to nearest even) to q_out[t, h, :];
 *  - heads n_heads_q <= h < q_head_padded of q_out are written as zeros;
 *  - kv row t is rotated, quantised and inserted exactly as
 *    rq_rope_fp8_quant_insert does (quant_eps is its block-amax clamp).
 *  q_out           bf16 [N, q_head_padded, 512], contiguous, 16-byte aligned.
 *  q_head_padded   >= n_heads_q.
 *  norm_eps        >= 0 and finite (arithmetic in fp32: fp32 sum of squares,
 *                  correctly rounded reciprocal square root).
 *  q_norm_weight   bf16 [512] device vector w, 16-byte aligned, shared by all
 *                  heads; NULL means w = 1 (the page's op takes no weight).
 *                  It multiplies the normalised values before the rotation.
 * The paged-cache arguments and rules are those of rq_rope_fp8_quant_insert.
 * A token whose position is outside [0, cache_rows) leaves its q heads and
 * its record untouched (its pad heads are still zeroed) and sets
 * RQ_FLAG_POSITION_RANGE. n_tokens * (q_head_padded + 1) must be below 2^31.
 */
rq_status rq_qnorm_rope_kv_rope_quant_insert(
    const void *q_bf16, int64_t n_tokens, int64_t n_heads_q, int64_t q_stride_token,
    int64_t q_stride_head, const void *kv_bf16, int64_t kv_stride_token, void *q_out_bf16,
    int64_t q_head_padded, const int64_t *positions, const float *cos_sin_cache,
    int64_t cache_rows, const int64_t *slot_mapping, uint8_t *k_cache, int64_t num_blocks,
    int64_t block_size, int64_t block_stride_bytes, float norm_eps, const void *q_norm_weight,
    float quant_eps, uint32_t *error_flags, void *stream);

/* Which dims of the indexer head's rotary part form a rotation pair. */
typedef enum rq_rope_style {
    RQ_ROPE_NEOX = 0,   /* dim j with dim 32 + j, j = 0..31 (halves)        */
    RQ_ROPE_GPTJ = 1    /* dim 2j with dim 2j + 1, j = 0..31 (interleaved)  */
} rq_rope_style;

/*
 * The indexer q op of [IDX] S1 (RoPE + FP8 quant + scale fold in one pass).
 * For every 128-wide head (t, h) of q:
 *  - dims 0..63 are rotated forward with row positions[t] of the [P, 64]
 *    cache (cos in columns 0..31, sin in 32..63, pair j uses column j):
 *    r0 = x0*c - x1*s, r1 = x1*c + x0*s, each product and sum rounded to
 *    fp32, then rounded to bf16 and back to fp32 (round to nearest even);
 *  - one block per head: amax = max(max|y|, eps), q_scale =
 *    2^ceil(log2(fl32(amax / 448))), out_fp8[t, h, k] = e4m3(y_k / q_scale);
 *  - out_weights[t, h] = ((weights[t, h] * q_scale) * softmax_scale)
 *    * head_scale, in fp32, in that order.
 *  q_bf16       [N, H, 128] bf16, strides in elements (multiples of 8), base
 *               16-byte aligned.
 *  rope_style   an rq_rope_style; any other value returns RQ_ERR_ARG.
 *  weights      [N, H] fp32, contiguous.
 *  eps          in [2^-100, 2^100].
 *  out_fp8      [N, H, 128] e4m3 codes, contiguous, 16-byte aligned.
 *  out_weights  [N, H] fp32, contiguous.
 * A head whose position is outside [0, cache_rows) is skipped (outputs
 * untouched) and RQ_FLAG_POSITION_RANGE is set. N * H must be below 2^31.
 */
rq_status rq_indexer_q_rope_fp8_quant(const void *q_bf16, int64_t n_tokens, int64_t n_heads,
                                      int64_t q_stride_token, int64_t q_stride_head,
                                      const int64_t *positions, const float *cos_sin_cache,
                                      int64_t cache_rows, int rope_style, const float *weights,
                                      float softmax_scale, float head_scale, float eps,
                                      uint8_t *out_fp8, float *out_weights,
                                      uint32_t *error_flags, void *stream);

/*
 * The consumer of the block-FP8 output: a grouped FP8 GEMM on the tensor
 * cores ([INV] intro: each output group's quantised attention output feeds
 * that group's wo_a projection). For every group g and token m:
 *   y[m, g, n] = sum over 128-wide K blocks kt of
 *                a_scales[m, g, kt] * w_scales[g, n / 128, kt]
 *                * sum_{k in kt} e4m3(a_codes[m, g, k]) * e4m3(w_codes[g, n, k])
 * in fp32, written as bf16 (round to nearest even).
 *  a_codes     [n_tokens, groups, k_per_group] e4m3 codes (the layout
 *              rq_inv_rope_fp8_quant writes), 16-byte aligned.
 *  a_scales    [n_tokens, groups, k_per_group / 128] fp32 (idem).
 *  w_codes     [groups, n_out, k_per_group] e4m3 codes (K contiguous),
 *              16-byte aligned.
 *  w_scales    [groups, n_out / 128, k_per_group / 128] fp32, one per
 *              128 x 128 block.
 *  y_bf16      [n_tokens, groups, n_out] bf16, 16-byte aligned.
 *  k_per_group, n_out: multiples of 128. Any n_tokens >= 0.
 * A bounded wait that gives up sets RQ_FLAG_TIMEOUT (never expected).
 * Up to 64 tokens with k_per_group a multiple of 512 (decode) the call runs
 * a split-K kernel on clusters of 8 CTAs (4 when k_per_group is not a
 * multiple of 1024): one fp32 accumulator per 128-wide K block, the block's
 * a_scales * w_scales folded per block in K order, the clusters' partials
 * summed in a fixed order (deterministic, within the same accumulation
 * error). It is launched with programmatic dependent launch and may
 * prefetch w_codes into L2 before the previous kernel in the stream has
 * finished (a prefetch reads no data into the kernel).
 */
rq_status rq_grouped_fp8_gemm(const uint8_t *a_codes, const float *a_scales, int64_t n_tokens,
                              int64_t groups, int64_t k_per_group, const uint8_t *w_codes,
                              const float *w_scales, int64_t n_out, uint16_t *y_bf16,
                              uint32_t *error_flags, void *stream);

/*
 * The same grouped FP8 GEMM with UE8M0 block scales (power-of-two scales
 * stored as 8-bit biased exponents, the encoding of the op's packed-scale
 * output, [INV] S3), computed by the block-scaled tensor-core MMA, which
 * applies both scales inside the K loop:
 *   y[m, g, n] = sum over 128-wide K blocks kt of
 *                2^(ea(m, g, kt) - 127) * 2^(ew(g, n / 128, kt) - 127)
 *                * sum_{k in kt} e4m3(a_codes[m, g, k]) * e4m3(w_codes[g, n, k])
 * accumulated in fp32 by the tensor cores, written as bf16 (round to
 * nearest even). The order of the fp32 additions is the hardware's, so
 * results agree with rq_grouped_fp8_gemm to fp32 accumulation error, not
 * bit for bit.
 *  a_codes     [n_tokens, groups, k_per_group] e4m3 codes, 16-byte aligned.
 *  a_sf        [n_tokens, groups, k_per_group / 512] uint32, 4-byte aligned:
 *              byte b (bits 8b..8b+7) of word (m, g, h) is ea(m, g, 4h + b),
 *              i.e. the token-major scales of rq_inv_rope_quant_layout in
 *              RQ_OUT_FP8_SCALE_UE8M0 mode (one word per 512-wide head).
 *  w_codes     [groups, n_out, k_per_group] e4m3 codes, 16-byte aligned.
 *  w_sf        [groups, n_out / 128, k_per_group / 128] uint8, one code ew
 *              per 128 x 128 block.
 *  y_bf16      [n_tokens, groups, n_out] bf16, 16-byte aligned.
 *  k_per_group a multiple of 512, at most 4096; n_out a multiple of 128.
 * Code 255 (NaN in the UE8M0 encoding) gives unspecified outputs. Any
 * n_tokens >= 0. A bounded wait that gives up sets RQ_FLAG_TIMEOUT (never
 * expected).
 * Up to 64 tokens (decode) the call runs a split-K kernel: clusters of 8 CTAs
 * (4 when k_per_group is not a multiple of 1024) each accumulate a run of K
 * blocks in fp32 and the partials are summed in fp32 in a fixed order, so
 * results are deterministic and within the same fp32 accumulation error. It
 * is launched with programmatic dependent launch: while the previous kernel
 * in the stream finishes it may prefetch w_codes into L2 (a prefetch reads
 * no data into the kernel); every read of the call's data happens after
 * that kernel has completed.
 */
rq_status rq_grouped_fp8_gemm_ue8m0(const uint8_t *a_codes, const uint32_t *a_sf,
                                    int64_t n_tokens, int64_t groups, int64_t k_per_group,
                                    const uint8_t *w_codes, const uint8_t *w_sf, int64_t n_out,
                                    uint16_t *y_bf16, uint32_t *error_flags, void *stream);

/*
 * The inverse RoPE + block-FP8 quant fused into its consumer: the grouped
 * FP8 GEMM of rq_grouped_fp8_gemm, whose A operand (group g's 128-wide K
 * blocks = its heads' quantisation blocks) is produced inside the GEMM from
 * x with exactly the arithmetic of rq_inv_rope_fp8_quant; the codes and
 * scales never reach HBM. The result equals rq_inv_rope_fp8_quant followed
 * by rq_grouped_fp8_gemm, bit for bit.
 * It is NOT the fast path: every A tile is produced again by each of the
 * n_out / 128 CTAs that need it, and measured on B300 (16384 tokens, 4
 * groups, K 4096, n_out 1024) it takes about 2.5 ms against about 336 us for
 * rq_inv_rope_quant_layout in RQ_OUT_FP8_SCALE_UE8M0 mode followed by
 * rq_grouped_fp8_gemm_ue8m0, the recommended pair; at one token, about
 * 86 us against about 7 us for that pair or for rq_inv_rope_fp8_quant
 * followed by rq_grouped_fp8_gemm (both GEMMs then run split over K).
 *  x_bf16 .. eps   as in rq_inv_rope_fp8_quant, with heads_per_group <= 8
 *                  and both strides > 0 (the input is read by tensor-map TMA).
 *  w_codes, w_scales, n_out, y_bf16   as in rq_grouped_fp8_gemm, with
 *                  groups = n_heads / heads_per_group and
 *                  K = heads_per_group * 512.
 * A token whose position is outside [0, cache_rows) sets
 * RQ_FLAG_POSITION_RANGE; its y rows are then unspecified.
 */
rq_status rq_inv_rope_fp8_quant_gemm(const void *x_bf16, int64_t n_tokens, int64_t n_heads,
                                     int64_t x_stride_token, int64_t x_stride_head,
                                     const int64_t *positions, const float *cos_sin_cache,
                                     int64_t cache_rows, int64_t heads_per_group, float eps,
                                     const uint8_t *w_codes, const float *w_scales, int64_t n_out,
                                     uint16_t *y_bf16, uint32_t *error_flags, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* RQ_H_ */
