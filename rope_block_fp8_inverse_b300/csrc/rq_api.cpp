// rq_api.cpp -- the C ABI declared in include/rq.h: host-side argument
// checks, device lookup and dispatch to the kernel launchers. Every check
// runs before any CUDA call, so an invalid call launches nothing and
// touches no buffer.
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "rq.h"
#include "rq_launch.h"

#define RQ_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kVersionMajor = 1;
constexpr int kVersionMinor = 0;
constexpr int64_t kMaxRows = int64_t(1) << 31;

// rq_debug_inject's settings for calls from this host thread.
thread_local rq::WaitCtl g_wait;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool eps_ok(float eps) {
    // 2^-100 <= eps <= 2^100 keeps amax / 448 a normal fp32 and the
    // power-of-two scale and its inverse representable for every finite amax.
    return std::isfinite(eps) && eps >= 0x1p-100f && eps <= 0x1p100f;
}

// Current device and its SM count (cached per device, per thread).
cudaError_t current_device(rq::DeviceInfo* info) {
    constexpr int kMax = 64;
    static thread_local int sm_count[kMax] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int slot = (dev >= 0 && dev < kMax) ? dev : -1;
    int n = slot >= 0 ? sm_count[slot] : 0;
    if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (slot >= 0) sm_count[slot] = n;
    }
    info->ordinal = dev;
    info->sm_count = n;
    return cudaSuccess;
}

rq_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return RQ_OK;
    (void)cudaGetLastError();  // clear this runtime's sticky launch error
    return RQ_ERR_CUDA;
}

}  // namespace

RQ_EXPORT const char* rq_status_string(int status) {
    switch (status) {
        case RQ_OK: return "ok";
        case RQ_ERR_NULL: return "a required pointer is NULL";
        case RQ_ERR_SHAPE: return "a size or stride is out of range";
        case RQ_ERR_ALIGN: return "a pointer or stride breaks the 16-byte alignment rule";
        case RQ_ERR_GROUPING: return "heads_per_group must be >= 1 and divide n_heads";
        case RQ_ERR_CUDA: return "the CUDA runtime reported an error";
        case RQ_ERR_ARG: return "eps must be finite and within [2^-100, 2^100]; variant must be known";
        default: return "unknown status";
    }
}

RQ_EXPORT int rq_version(void) { return (kVersionMajor << 16) | kVersionMinor; }

RQ_EXPORT int64_t rq_validate_indices_workspace(int64_t num_slots) {
    if (num_slots < 0 || num_slots > (int64_t(1) << 40)) return -1;
    const int64_t bitmap = ((num_slots + 31) / 32 * 4 + 15) / 16 * 16;
    return bitmap + 16;  // then the result word, in its own 16 bytes
}

RQ_EXPORT rq_status rq_validate_indices(const int64_t* positions, const int64_t* slot_mapping,
                                        int64_t n_tokens, int64_t cache_rows, int64_t num_slots,
                                        void* workspace, int64_t workspace_bytes, uint32_t* result,
                                        void* stream) {
    if (n_tokens < 0 || cache_rows < 1 || num_slots < 0 || (slot_mapping && num_slots < 1))
        return RQ_ERR_SHAPE;
    if (!result) return RQ_ERR_NULL;
    const int64_t need = rq_validate_indices_workspace(slot_mapping ? num_slots : 0);
    if (need < 0) return RQ_ERR_SHAPE;
    if (n_tokens == 0) {
        *result = 0;
        return RQ_OK;
    }
    if (!positions || !workspace) return RQ_ERR_NULL;
    if (workspace_bytes < need) return RQ_ERR_SHAPE;
    if (!aligned(positions, 8) || (slot_mapping && !aligned(slot_mapping, 8)) ||
        !aligned(workspace, 16))
        return RQ_ERR_ALIGN;
    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    rq::ValParams p;
    p.positions = positions;
    p.slot_mapping = slot_mapping;
    p.n_tokens = n_tokens;
    p.cache_rows = cache_rows;
    p.num_slots = num_slots;
    p.bitmap = reinterpret_cast<uint32_t*>(ws);
    p.result = reinterpret_cast<uint32_t*>(ws + need - 16);
    uint32_t word = 0;
    if ((e = cudaMemsetAsync(ws, 0, size_t(need), st)) != cudaSuccess ||
        (e = rq::launch_validate_indices(p, dev, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(&word, p.result, 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaStreamSynchronize(st)) != cudaSuccess)
        return from_cuda(e);
    *result = word;
    return RQ_OK;
}

RQ_EXPORT void rq_debug_inject(uint32_t mask, uint32_t spin_limit) {
    g_wait.inject = mask;
    g_wait.spin_limit = spin_limit ? spin_limit : rq::kSpinLimit;
}

RQ_EXPORT rq_status rq_inv_rope_fp8_quant_ex(const void* x_bf16, int64_t n_tokens,
                                             int64_t n_heads, int64_t x_stride_token,
                                             int64_t x_stride_head, const int64_t* positions,
                                             const float* cos_sin_cache, int64_t cache_rows,
                                             int64_t heads_per_group, float eps, uint8_t* out_fp8,
                                             float* out_scales, uint32_t* error_flags,
                                             void* stream, int variant) {
    if (variant < RQ_INV_AUTO || variant > RQ_INV_STREAM) return RQ_ERR_ARG;
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1) return RQ_ERR_SHAPE;
    if (heads_per_group < 1 || n_heads % heads_per_group != 0) return RQ_ERR_GROUPING;
    if (!eps_ok(eps)) return RQ_ERR_ARG;
    if (n_heads >= kMaxRows || n_tokens >= kMaxRows / n_heads) return RQ_ERR_SHAPE;
    if (n_tokens == 0) return RQ_OK;
    if (!x_bf16 || !positions || !cos_sin_cache || !out_fp8 || !out_scales) return RQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || x_stride_token % 8 != 0 || x_stride_head % 8 != 0 ||
        !aligned(positions, 8) || !aligned(cos_sin_cache, 16) || !aligned(out_fp8, 16) ||
        !aligned(out_scales, 16) || (error_flags && !aligned(error_flags, 4)))
        return RQ_ERR_ALIGN;

    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);

    rq::InvParams p;
    p.wait = g_wait;
    p.x = x_bf16;
    p.sx_t = x_stride_token;
    p.sx_h = x_stride_head;
    p.n_rows = static_cast<uint32_t>(n_tokens * n_heads);
    p.n_heads = static_cast<uint32_t>(n_heads);
    p.n_tokens = static_cast<uint32_t>(n_tokens);
    p.positions = positions;
    p.cache = cos_sin_cache;
    p.cache_rows = cache_rows;
    p.eps = eps;
    p.out = out_fp8;
    p.scales = out_scales;
    p.error_flags = error_flags;
    // contiguous [N, G, hpg*512] output is [N, 1, H*512]: one group per token
    p.lay.mode = rq::kOutFp8F32;
    p.lay.hpg = static_cast<uint32_t>(n_heads);
    p.lay.ot = n_heads * rq::kHeadDimABI;
    p.lay.og = 0;
    p.lay.st = n_heads * 4;
    p.lay.sg = 0;
    p.lay.se = 1;
    return from_cuda(
        rq::launch_inv_rope_fp8_quant(p, dev, variant, static_cast<cudaStream_t>(stream)));
}

RQ_EXPORT rq_status rq_inv_rope_fp8_quant(const void* x_bf16, int64_t n_tokens, int64_t n_heads,
                                          int64_t x_stride_token, int64_t x_stride_head,
                                          const int64_t* positions, const float* cos_sin_cache,
                                          int64_t cache_rows, int64_t heads_per_group, float eps,
                                          uint8_t* out_fp8, float* out_scales,
                                          uint32_t* error_flags, void* stream) {
    return rq_inv_rope_fp8_quant_ex(x_bf16, n_tokens, n_heads, x_stride_token, x_stride_head,
                                    positions, cos_sin_cache, cache_rows, heads_per_group, eps,
                                    out_fp8, out_scales, error_flags, stream, RQ_INV_AUTO);
}

RQ_EXPORT rq_status rq_inv_rope_quant_layout(
    const void* x_bf16, int64_t n_tokens, int64_t n_heads, int64_t x_stride_token,
    int64_t x_stride_head, const int64_t* positions, const float* cos_sin_cache,
    int64_t cache_rows, int64_t heads_per_group, float eps, int out_mode, void* out,
    int64_t out_stride_token, int64_t out_stride_group, void* scales, int64_t scale_stride_token,
    int64_t scale_stride_group, int64_t scale_stride_elem, uint32_t* error_flags, void* stream) {
    if (out_mode < RQ_OUT_FP8_SCALE_F32 || out_mode > RQ_OUT_BF16) return RQ_ERR_ARG;
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1) return RQ_ERR_SHAPE;
    if (heads_per_group < 1 || n_heads % heads_per_group != 0) return RQ_ERR_GROUPING;
    if (!eps_ok(eps)) return RQ_ERR_ARG;
    if (n_heads >= kMaxRows || n_tokens >= kMaxRows / n_heads) return RQ_ERR_SHAPE;
    if (out_stride_token < 0 || out_stride_group < 0 || scale_stride_token < 0 ||
        scale_stride_group < 0 || scale_stride_elem < 0)
        return RQ_ERR_SHAPE;
    if (n_tokens == 0) return RQ_OK;
    const bool quant = out_mode != RQ_OUT_BF16;
    if (!x_bf16 || !positions || !cos_sin_cache || !out || (quant && !scales)) return RQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || x_stride_token % 8 != 0 || x_stride_head % 8 != 0 ||
        !aligned(positions, 8) || !aligned(cos_sin_cache, 16) || !aligned(out, 16) ||
        out_stride_token % 16 != 0 || out_stride_group % 16 != 0 ||
        (quant && !aligned(scales, 4)) || (error_flags && !aligned(error_flags, 4)))
        return RQ_ERR_ALIGN;

    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);

    rq::InvParams p;
    p.wait = g_wait;
    p.x = x_bf16;
    p.sx_t = x_stride_token;
    p.sx_h = x_stride_head;
    p.n_rows = static_cast<uint32_t>(n_tokens * n_heads);
    p.n_heads = static_cast<uint32_t>(n_heads);
    p.n_tokens = static_cast<uint32_t>(n_tokens);
    p.positions = positions;
    p.cache = cos_sin_cache;
    p.cache_rows = cache_rows;
    p.eps = eps;
    p.out = static_cast<uint8_t*>(out);
    p.scales = static_cast<float*>(scales);
    p.error_flags = error_flags;
    p.lay.mode = out_mode;
    p.lay.hpg = static_cast<uint32_t>(heads_per_group);
    p.lay.ot = out_stride_token;
    p.lay.og = out_stride_group;
    p.lay.st = scale_stride_token;
    p.lay.sg = scale_stride_group;
    p.lay.se = scale_stride_elem;
    // A quantising layout that is row-linear (token-major, contiguous: head r =
    // t*H + h at out + r*512, its scales at r*4 or its word at r) takes the
    // warp-rows kernel of rq_inv_rope_fp8_quant with that scale encoding.
    const int64_t groups = n_heads / heads_per_group;
    const int64_t spe = out_mode == RQ_OUT_FP8_SCALE_F32 ? 4 : 1;  // scale elements per head
    const bool row_linear =
        quant && out_stride_token == n_heads * rq::kHeadDimABI &&
        (groups == 1 || out_stride_group == heads_per_group * rq::kHeadDimABI) &&
        scale_stride_elem == 1 && scale_stride_token == n_heads * spe &&
        (groups == 1 || scale_stride_group == heads_per_group * spe) && aligned(scales, 16);
    if (row_linear)
        return from_cuda(
            rq::launch_inv_rope_rows(p, dev, out_mode, false, static_cast<cudaStream_t>(stream)));
    // The contiguous group-major layout ([G, N, hpg*512] codes, [G, N, hpg*spe]
    // scales) is row-linear in the output row (g*N + t)*hpg + i: the same
    // kernel, storing each row there.
    const bool group_linear =
        quant && groups > 1 && out_stride_token == heads_per_group * rq::kHeadDimABI &&
        out_stride_group == n_tokens * heads_per_group * rq::kHeadDimABI &&
        scale_stride_elem == 1 && scale_stride_token == heads_per_group * spe &&
        scale_stride_group == n_tokens * heads_per_group * spe && aligned(scales, 16);
    if (group_linear)
        return from_cuda(
            rq::launch_inv_rope_rows(p, dev, out_mode, true, static_cast<cudaStream_t>(stream)));
    // any other layout: the warp-rows layout kernel (each warp on fixed heads
    // for the quantising modes, the row walk for bf16)
    return from_cuda(
        rq::launch_inv_rope_quant_layout(p, dev, static_cast<cudaStream_t>(stream)));
}

RQ_EXPORT rq_status rq_rope_fp8_quant_insert(const void* kv_bf16, int64_t n_tokens,
                                             int64_t kv_stride_token, const int64_t* positions,
                                             const float* cos_sin_cache, int64_t cache_rows,
                                             const int64_t* slot_mapping, uint8_t* k_cache,
                                             int64_t num_blocks, int64_t block_size,
                                             int64_t block_stride_bytes, float eps,
                                             uint32_t* error_flags, void* stream) {
    if (n_tokens < 0 || n_tokens >= kMaxRows || cache_rows < 1 || num_blocks < 1 ||
        block_size < 1 || block_size > (int64_t(1) << 40) / rq::kRecordBytesABI)
        return RQ_ERR_SHAPE;
    if (block_stride_bytes < block_size * rq::kRecordBytesABI ||
        num_blocks > (int64_t(1) << 62) / block_stride_bytes)
        return RQ_ERR_SHAPE;
    if (block_stride_bytes % 16 != 0) return RQ_ERR_ALIGN;
    if (!eps_ok(eps)) return RQ_ERR_ARG;
    if (n_tokens == 0) return RQ_OK;
    if (!kv_bf16 || !positions || !cos_sin_cache || !slot_mapping || !k_cache) return RQ_ERR_NULL;
    if (!aligned(kv_bf16, 16) || kv_stride_token % 8 != 0 || !aligned(positions, 8) ||
        !aligned(cos_sin_cache, 16) || !aligned(slot_mapping, 8) || !aligned(k_cache, 16) ||
        (error_flags && !aligned(error_flags, 4)))
        return RQ_ERR_ALIGN;

    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);

    rq::InsParams p;
    p.kv = kv_bf16;
    p.skv = kv_stride_token;
    p.n_tokens = static_cast<uint32_t>(n_tokens);
    p.positions = positions;
    p.cache = cos_sin_cache;
    p.cache_rows = cache_rows;
    p.slot_mapping = slot_mapping;
    p.k_cache = k_cache;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.block_stride = block_stride_bytes;
    p.eps = eps;
    p.error_flags = error_flags;
    return from_cuda(
        rq::launch_rope_fp8_quant_insert(p, dev, static_cast<cudaStream_t>(stream)));
}

RQ_EXPORT rq_status rq_qnorm_rope_kv_rope_quant_insert(
    const void* q_bf16, int64_t n_tokens, int64_t n_heads_q, int64_t q_stride_token,
    int64_t q_stride_head, const void* kv_bf16, int64_t kv_stride_token, void* q_out_bf16,
    int64_t q_head_padded, const int64_t* positions, const float* cos_sin_cache,
    int64_t cache_rows, const int64_t* slot_mapping, uint8_t* k_cache, int64_t num_blocks,
    int64_t block_size, int64_t block_stride_bytes, float norm_eps, const void* q_norm_weight,
    float quant_eps, uint32_t* error_flags, void* stream) {
    if (n_tokens < 0 || n_heads_q < 1 || q_head_padded < n_heads_q || cache_rows < 1 ||
        num_blocks < 1 || block_size < 1 ||
        block_size > (int64_t(1) << 40) / rq::kRecordBytesABI)
        return RQ_ERR_SHAPE;
    if (q_head_padded >= kMaxRows - 1 || n_tokens >= kMaxRows / (q_head_padded + 1))
        return RQ_ERR_SHAPE;
    if (block_stride_bytes < block_size * rq::kRecordBytesABI ||
        num_blocks > (int64_t(1) << 62) / block_stride_bytes)
        return RQ_ERR_SHAPE;
    if (block_stride_bytes % 16 != 0) return RQ_ERR_ALIGN;
    if (!std::isfinite(norm_eps) || norm_eps < 0.0f || !eps_ok(quant_eps)) return RQ_ERR_ARG;
    if (n_tokens == 0) return RQ_OK;
    if (!q_bf16 || !kv_bf16 || !q_out_bf16 || !positions || !cos_sin_cache || !slot_mapping ||
        !k_cache)
        return RQ_ERR_NULL;
    if (!aligned(q_bf16, 16) || q_stride_token % 8 != 0 || q_stride_head % 8 != 0 ||
        !aligned(kv_bf16, 16) || kv_stride_token % 8 != 0 || !aligned(q_out_bf16, 16) ||
        !aligned(positions, 8) || !aligned(cos_sin_cache, 16) || !aligned(slot_mapping, 8) ||
        !aligned(k_cache, 16) || (error_flags && !aligned(error_flags, 4)) ||
        (q_norm_weight && !aligned(q_norm_weight, 16)))
        return RQ_ERR_ALIGN;

    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);

    rq::FusedParams p;
    p.norm_w = static_cast<const uint16_t*>(q_norm_weight);
    p.q = q_bf16;
    p.sq_t = q_stride_token;
    p.sq_h = q_stride_head;
    p.n_heads_q = static_cast<uint32_t>(n_heads_q);
    p.q_head_padded = static_cast<uint32_t>(q_head_padded);
    p.kv = kv_bf16;
    p.skv = kv_stride_token;
    p.q_out = static_cast<uint16_t*>(q_out_bf16);
    p.n_tokens = static_cast<uint32_t>(n_tokens);
    p.n_units = static_cast<uint32_t>(n_tokens * (q_head_padded + 1));
    p.positions = positions;
    p.cache = cos_sin_cache;
    p.cache_rows = cache_rows;
    p.slot_mapping = slot_mapping;
    p.k_cache = k_cache;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.block_stride = block_stride_bytes;
    p.norm_eps = norm_eps;
    p.quant_eps = quant_eps;
    p.error_flags = error_flags;
    return from_cuda(rq::launch_qnorm_rope_kv_insert(p, dev, static_cast<cudaStream_t>(stream)));
}

RQ_EXPORT rq_status rq_indexer_q_rope_fp8_quant(
    const void* q_bf16, int64_t n_tokens, int64_t n_heads, int64_t q_stride_token,
    int64_t q_stride_head, const int64_t* positions, const float* cos_sin_cache,
    int64_t cache_rows, int rope_style, const float* weights, float softmax_scale,
    float head_scale, float eps, uint8_t* out_fp8, float* out_weights, uint32_t* error_flags,
    void* stream) {
    if (rope_style != RQ_ROPE_NEOX && rope_style != RQ_ROPE_GPTJ) return RQ_ERR_ARG;
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1) return RQ_ERR_SHAPE;
    if (n_heads >= kMaxRows || n_tokens >= kMaxRows / n_heads) return RQ_ERR_SHAPE;
    if (!eps_ok(eps) || !std::isfinite(softmax_scale) || !std::isfinite(head_scale))
        return RQ_ERR_ARG;
    if (n_tokens == 0) return RQ_OK;
    if (!q_bf16 || !positions || !cos_sin_cache || !weights || !out_fp8 || !out_weights)
        return RQ_ERR_NULL;
    if (!aligned(q_bf16, 16) || q_stride_token % 8 != 0 || q_stride_head % 8 != 0 ||
        !aligned(positions, 8) || !aligned(cos_sin_cache, 16) || !aligned(weights, 4) ||
        !aligned(out_fp8, 16) || !aligned(out_weights, 4) ||
        (error_flags && !aligned(error_flags, 4)))
        return RQ_ERR_ALIGN;

    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);

    rq::IdxParams p;
    p.q = q_bf16;
    p.sq_t = q_stride_token;
    p.sq_h = q_stride_head;
    p.n_rows = static_cast<uint32_t>(n_tokens * n_heads);
    p.n_heads = static_cast<uint32_t>(n_heads);
    p.positions = positions;
    p.cache = cos_sin_cache;
    p.cache_rows = cache_rows;
    p.neox = rope_style == RQ_ROPE_NEOX;
    p.weights = weights;
    p.softmax_scale = softmax_scale;
    p.head_scale = head_scale;
    p.eps = eps;
    p.out = out_fp8;
    p.weights_out = out_weights;
    p.error_flags = error_flags;
    return from_cuda(rq::launch_indexer_q_rope_quant(p, dev, static_cast<cudaStream_t>(stream)));
}

RQ_EXPORT rq_status rq_grouped_fp8_gemm(const uint8_t* a_codes, const float* a_scales,
                                        int64_t n_tokens, int64_t groups, int64_t k_per_group,
                                        const uint8_t* w_codes, const float* w_scales,
                                        int64_t n_out, uint16_t* y_bf16, uint32_t* error_flags,
                                        void* stream) {
    if (n_tokens < 0 || groups < 1 || k_per_group < 128 || n_out < 128) return RQ_ERR_SHAPE;
    if (k_per_group % 128 != 0 || n_out % 128 != 0) return RQ_ERR_SHAPE;
    if (n_tokens >= kMaxRows || groups * k_per_group >= kMaxRows || groups * n_out >= kMaxRows ||
        n_tokens * groups >= kMaxRows / n_out)
        return RQ_ERR_SHAPE;
    if (n_tokens == 0) return RQ_OK;
    if (!a_codes || !a_scales || !w_codes || !w_scales || !y_bf16) return RQ_ERR_NULL;
    if (!aligned(a_codes, 16) || !aligned(w_codes, 16) || !aligned(y_bf16, 16) ||
        !aligned(a_scales, 4) || !aligned(w_scales, 4) || (error_flags && !aligned(error_flags, 4)))
        return RQ_ERR_ALIGN;
    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);
    rq::GemmParams p;
    p.wait = g_wait;
    p.m = static_cast<int>(n_tokens);
    p.groups = static_cast<int>(groups);
    p.k = static_cast<int>(k_per_group);
    p.n_out = static_cast<int>(n_out);
    p.a_scales = a_scales;
    p.w_scales = w_scales;
    p.y = y_bf16;
    p.error_flags = error_flags;
    return from_cuda(rq::launch_grouped_fp8_gemm(p, a_codes, w_codes, dev.ordinal,
                                                 static_cast<cudaStream_t>(stream)));
}

RQ_EXPORT rq_status rq_grouped_fp8_gemm_ue8m0(const uint8_t* a_codes, const uint32_t* a_sf,
                                              int64_t n_tokens, int64_t groups,
                                              int64_t k_per_group, const uint8_t* w_codes,
                                              const uint8_t* w_sf, int64_t n_out,
                                              uint16_t* y_bf16, uint32_t* error_flags,
                                              void* stream) {
    if (n_tokens < 0 || groups < 1 || k_per_group < 512 || k_per_group > 4096 || n_out < 128)
        return RQ_ERR_SHAPE;
    if (k_per_group % 512 != 0 || n_out % 128 != 0) return RQ_ERR_SHAPE;
    if (n_tokens >= kMaxRows || groups * k_per_group >= kMaxRows || groups * n_out >= kMaxRows ||
        n_tokens * groups >= kMaxRows / n_out)
        return RQ_ERR_SHAPE;
    if (n_tokens == 0) return RQ_OK;
    if (!a_codes || !a_sf || !w_codes || !w_sf || !y_bf16) return RQ_ERR_NULL;
    if (!aligned(a_codes, 16) || !aligned(w_codes, 16) || !aligned(y_bf16, 16) ||
        !aligned(a_sf, 4) || (error_flags && !aligned(error_flags, 4)))
        return RQ_ERR_ALIGN;
    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);
    rq::MxGemmParams p;
    p.wait = g_wait;
    p.m = static_cast<int>(n_tokens);
    p.groups = static_cast<int>(groups);
    p.k = static_cast<int>(k_per_group);
    p.n_out = static_cast<int>(n_out);
    p.a_sf = a_sf;
    p.w_sf = w_sf;
    p.y = y_bf16;
    p.error_flags = error_flags;
    return from_cuda(rq::launch_grouped_fp8_gemm_ue8m0(p, a_codes, w_codes, dev,
                                                       static_cast<cudaStream_t>(stream)));
}

RQ_EXPORT rq_status rq_inv_rope_fp8_quant_gemm(
    const void* x_bf16, int64_t n_tokens, int64_t n_heads, int64_t x_stride_token,
    int64_t x_stride_head, const int64_t* positions, const float* cos_sin_cache,
    int64_t cache_rows, int64_t heads_per_group, float eps, const uint8_t* w_codes,
    const float* w_scales, int64_t n_out, uint16_t* y_bf16, uint32_t* error_flags, void* stream) {
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1 || n_out < 128 || n_out % 128 != 0)
        return RQ_ERR_SHAPE;
    if (heads_per_group < 1 || n_heads % heads_per_group != 0) return RQ_ERR_GROUPING;
    if (heads_per_group > 8) return RQ_ERR_SHAPE;  // K = heads_per_group * 512 <= 4096
    if (!eps_ok(eps)) return RQ_ERR_ARG;
    const int64_t groups = n_heads / heads_per_group;
    if (n_tokens >= kMaxRows || groups * n_out >= kMaxRows ||
        n_tokens * groups >= kMaxRows / n_out)
        return RQ_ERR_SHAPE;
    if (n_tokens == 0) return RQ_OK;
    if (!x_bf16 || !positions || !cos_sin_cache || !w_codes || !w_scales || !y_bf16)
        return RQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || x_stride_token % 8 != 0 || x_stride_head % 8 != 0 ||
        x_stride_token <= 0 || x_stride_head <= 0 || !aligned(positions, 8) ||
        !aligned(cos_sin_cache, 16) || !aligned(w_codes, 16) || !aligned(w_scales, 4) ||
        !aligned(y_bf16, 16) || (error_flags && !aligned(error_flags, 4)))
        return RQ_ERR_ALIGN;
    rq::DeviceInfo dev;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return from_cuda(e);
    rq::FusedGemmParams p;
    p.wait = g_wait;
    p.x = x_bf16;
    p.sx_t = x_stride_token;
    p.sx_h = x_stride_head;
    p.positions = positions;
    p.cache = cos_sin_cache;
    p.cache_rows = cache_rows;
    p.m = static_cast<int>(n_tokens);
    p.groups = static_cast<int>(groups);
    p.hpg = static_cast<int>(heads_per_group);
    p.k = static_cast<int>(heads_per_group * 512);
    p.n_out = static_cast<int>(n_out);
    p.eps = eps;
    p.w_scales = w_scales;
    p.y = y_bf16;
    p.error_flags = error_flags;
    return from_cuda(rq::launch_fused_inv_rope_quant_gemm(p, w_codes, dev.ordinal,
                                                          static_cast<cudaStream_t>(stream)));
}
