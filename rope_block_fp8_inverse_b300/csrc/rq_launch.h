// rq_launch.h -- internal interface between the C-ABI layer (rq_api.cpp) and
// the kernel launchers (rq_kernels.cu). Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "rq.h"

namespace rq {

// Launch `kernel` with programmatic stream serialization: it may be scheduled
// while the stream's previous kernel drains (the kernel's pdl_wait() keeps
// stream order for memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Polls of an mbarrier before a wait gives up and the kernel reports
// RQ_FLAG_TIMEOUT (never expected in normal operation).
constexpr uint32_t kSpinLimit = 1u << 22;

// Test-only fault injection (rq_debug_inject): a kernel skips one of its own
// copies so that a bounded wait runs out; the values are RQ_DEBUG_* of rq.h.
constexpr uint32_t kInjectStreamStage = 1u;  // TMA-ring inverse: warp 0 leaves tile 0 unarmed
constexpr uint32_t kInjectGemmLoads = 2u;    // grouped GEMMs: CTA 0's producer issues nothing

struct WaitCtl {
    uint32_t spin_limit = kSpinLimit;  // polls per wait
    uint32_t inject = 0;               // kInject* bits
};

constexpr int kInvThreads = 256;  // 8 warps per CTA
constexpr int kInsThreads = 256;
constexpr int64_t kRecordBytesABI = 528;  // paged record: 512 codes + 4 fp32 scales
constexpr int64_t kHeadDimABI = 512;

struct DeviceInfo {
    int ordinal;
    int sm_count;
};

// Output of the layout entry point (rq_inv_rope_quant_layout): what is written
// and where. Head i of group g of token t starts at
//   out + t*ot + g*og + i*head_bytes   (head_bytes 512 for codes, 1024 for bf16),
// and scale element j of that group (j = 4i + b for fp32 scales, j = i for
// packed UE8M0 words) sits at scales + t*st + g*sg + j*se.
enum OutMode { kOutFp8F32 = 0, kOutFp8Ue8m0 = 1, kOutBf16 = 2 };
struct OutLayout {
    int mode;
    uint32_t hpg;
    int64_t ot, og;       // bytes
    int64_t st, sg, se;   // scale elements (fp32 or uint32)
};

// Arguments of the inverse kernel, validated on the host (rq_api.cpp).
struct InvParams {
    const void* x;            // bf16 [N, H, 512], strides sx_t / sx_h elements
    int64_t sx_t, sx_h;
    uint32_t n_rows;          // N * H (< 2^31)
    uint32_t n_heads;
    uint32_t n_tokens;
    const int64_t* positions;
    const float* cache;       // [cache_rows, 64]
    int64_t cache_rows;
    float eps;
    uint8_t* out;             // [N*H, 512] codes
    float* scales;            // [N*H, 4]
    uint32_t* error_flags;    // may be null
    // warp-rows kernels (set by their launchers, >= 1): tokens per sweep of
    // the grid; a sweep is whole tokens, so that every warp keeps its heads
    uint32_t sweep_tokens;
    OutLayout lay;            // used by the layout kernel only
    WaitCtl wait;             // used by the stream kernel only
};

struct InsParams {
    const void* kv;           // bf16 [N, 512], token stride skv elements
    int64_t skv;
    uint32_t n_tokens;
    const int64_t* positions;
    const float* cache;
    int64_t cache_rows;
    const int64_t* slot_mapping;
    uint8_t* k_cache;
    int64_t num_blocks, block_size, block_stride;
    float eps;
    uint32_t* error_flags;
};

// Arguments of the fused q/kv kernel (rq_qnorm_rope_kv_rope_quant_insert).
struct FusedParams {
    const void* q;            // bf16 [N, Hq, 512], strides sq_t / sq_h elements
    int64_t sq_t, sq_h;
    uint32_t n_heads_q, q_head_padded;
    const void* kv;           // bf16 [N, 512], token stride skv elements
    int64_t skv;
    uint16_t* q_out;          // bf16 [N, q_head_padded, 512] contiguous
    uint32_t n_tokens;
    uint32_t n_units;         // n_tokens * (q_head_padded + 1) < 2^31
    const int64_t* positions;
    const float* cache;
    int64_t cache_rows;
    const int64_t* slot_mapping;
    uint8_t* k_cache;
    int64_t num_blocks, block_size, block_stride;
    float norm_eps, quant_eps;
    const uint16_t* norm_w;   // bf16 [512] RMSNorm weight, or null for none
    uint32_t* error_flags;
};

// Arguments of the index check (rq_validate_indices).
struct ValParams {
    const int64_t* positions;     // [n_tokens]
    const int64_t* slot_mapping;  // [n_tokens] or null
    int64_t n_tokens, cache_rows, num_slots;
    uint32_t* bitmap;             // num_slots bits, zeroed
    uint32_t* result;             // RQ_FLAG_* bits, zeroed
};

// Arguments of the indexer q kernel (rq_indexer_q_rope_fp8_quant).
struct IdxParams {
    const void* q;            // bf16 [N, H, 128], strides sq_t / sq_h elements
    int64_t sq_t, sq_h;
    uint32_t n_rows, n_heads; // n_rows = N * H < 2^31
    const int64_t* positions;
    const float* cache;       // [cache_rows, 64]
    int64_t cache_rows;
    bool neox;                // NeoX halves (true) or GPT-J pairs of dims 0..63
    const float* weights;     // [N, H] fp32
    float softmax_scale, head_scale, eps;
    uint8_t* out;             // [N, H, 128] e4m3 codes
    float* weights_out;       // [N, H] fp32
    uint32_t* error_flags;
    // tokens per sweep of the grid when a sweep is whole tokens (set by the
    // launcher; every 8-lane head slot then keeps its head), else 0
    uint32_t sweep_tokens;
};

// Arguments of the grouped FP8 GEMM (rq_grouped_fp8_gemm).
struct GemmParams {
    int m, groups, k, n_out;  // k = per-group K (multiple of 128), n_out multiple of 128
    const float* a_scales;    // [m, groups, k / 128]
    const float* w_scales;    // [groups, n_out / 128, k / 128]
    uint16_t* y;              // bf16 [m, groups, n_out]
    uint32_t* error_flags;
    WaitCtl wait;
};

// Arguments of the grouped FP8 GEMM with UE8M0 block scales.
struct MxGemmParams {
    int m, groups, k, n_out;  // k = per-group K (multiple of 512, at most 4096), n_out % 128 == 0
    const uint32_t* a_sf;     // [m, groups, k / 512] packed UE8M0 words (byte b = block 4h + b)
    const uint8_t* w_sf;      // [groups, n_out / 128, k / 128] UE8M0 codes
    uint16_t* y;              // bf16 [m, groups, n_out]
    uint32_t* error_flags;
    WaitCtl wait;
};

// Arguments of the fused inverse-RoPE + quant + grouped GEMM.
struct FusedGemmParams {
    const void* x;            // bf16 [m, groups * hpg, 512], strides sx_t / sx_h elements
    int64_t sx_t, sx_h;
    const int64_t* positions;
    const float* cache;
    int64_t cache_rows;
    int m, groups, hpg, k, n_out;   // k = hpg * 512
    float eps;
    const float* w_scales;    // [groups, n_out / 128, k / 128]
    uint16_t* y;              // bf16 [m, groups, n_out]
    uint32_t* error_flags;
    WaitCtl wait;             // spin limit only
};

// Kernel variants of the inverse op (all bit-identical in output).
enum InvVariant {
    kInvAuto = 0,        // chosen from the problem size
    kInvWarpRows = 1,    // persistent warps, register loads (rq_kernels.cu)
    kInvStream = 2       // one TMA ring per warp (rq_stream.cu)
};



cudaError_t launch_inv_rope_fp8_quant(const InvParams& p, const DeviceInfo& dev, int variant,
                                      cudaStream_t stream);
// The inverse op into a row-linear layout (row r's codes at out + r*512; its
// scales at scales + r*4 (fp32) or its packed UE8M0 word at scales + r), on
// the warp-rows kernel. mode: kOutFp8F32 or kOutFp8Ue8m0. Row r = t*H + h
// (token-major), or with group_major r = (g*N + t)*hpg + i for head
// h = g*hpg + i (the contiguous group-major layout; p.lay.hpg set).
cudaError_t launch_inv_rope_rows(const InvParams& p, const DeviceInfo& dev, int mode,
                                 bool group_major, cudaStream_t stream);
cudaError_t launch_inv_rope_quant_layout(const InvParams& p, const DeviceInfo& dev,
                                         cudaStream_t stream);
// The TMA-ring kernel (RQ_INV_STREAM) into the plain op's contiguous output.
cudaError_t launch_inv_rope_fp8_quant_stream(const InvParams& p, const DeviceInfo& dev,
                                             cudaStream_t stream);
cudaError_t launch_rope_fp8_quant_insert(const InsParams& p, const DeviceInfo& dev,
                                         cudaStream_t stream);
cudaError_t launch_qnorm_rope_kv_insert(const FusedParams& p, const DeviceInfo& dev,
                                        cudaStream_t stream);
cudaError_t launch_indexer_q_rope_quant(const IdxParams& p, const DeviceInfo& dev,
                                        cudaStream_t stream);
cudaError_t launch_grouped_fp8_gemm(const GemmParams& p, const uint8_t* a_codes,
                                    const uint8_t* w_codes, int dev_ordinal, cudaStream_t stream);
// The fp32-scale GEMM's decode-size split-K kernel (p.m <= 64, p.k % 512 == 0).
cudaError_t launch_grouped_fp8_gemm_small(const GemmParams& p, const uint8_t* a_codes,
                                          const uint8_t* w_codes, int dev_ordinal,
                                          cudaStream_t stream);
cudaError_t launch_fused_inv_rope_quant_gemm(const FusedGemmParams& p, const uint8_t* w_codes,
                                             int dev_ordinal, cudaStream_t stream);
cudaError_t launch_validate_indices(const ValParams& p, const DeviceInfo& dev,
                                    cudaStream_t stream);
cudaError_t launch_grouped_fp8_gemm_ue8m0(const MxGemmParams& p, const uint8_t* a_codes,
                                          const uint8_t* w_codes, const DeviceInfo& dev,
                                          cudaStream_t stream);

// Tensor map of a 2-D uint8 tensor [rows, inner] with row stride `stride`
// bytes: boxes of 128 bytes x box_rows rows, 128-byte swizzle, rows past the
// end read as zeros. False when the driver rejects it (or has no encoder).
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride,
              uint32_t box_rows);

}  // namespace rq
