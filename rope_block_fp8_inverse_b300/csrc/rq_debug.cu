// rq_debug.cu -- test-only entry points that run the kernels' own per-block
// scale rule and quantisation step over ranges of fp32 bit patterns, so that
// both can be checked exhaustively against an independent statement of the
// arithmetic (every positive finite block amax; every fp32 value through the
// e4m3 conversion). They are not part of the op.
//
// What they evaluate is exactly the device code every quantising kernel of
// the library runs (rq_device.cuh):
//   scale  = scale_bits(fmaxf(amax, eps))      the power-of-two block scale
//            2^ceil(log2(fl32(amax / 448))) ("[vllm] vLLM의 GLM5.2 성능
//            최적화", S1; the block absmax of "[vllm] 한 프로그램이 4개 head를
//            처리하게 하라", S3), and inv_scale(scale), its exact reciprocal;
//   codes  = quant16(values, inv_scale(2^e))  the exact power-of-two scaling
//            (mul.rn.f32x2) followed by cvt.rn.satfinite.e4m3x2, sixteen
//            values per thread in the lane layout of a row.
// Both entry points are stream-ordered and asynchronous, allocate nothing and
// write only the caller's output arrays.
#include "rq_device.cuh"
#include "rq_launch.h"

#define RQ_EXPORT extern "C" __attribute__((visibility("default")))

namespace rq {
namespace {

// Bit pattern first + i (mod 2^32) as an fp32 value.
__device__ __forceinline__ float pattern(uint32_t first, uint64_t i) {
    return __uint_as_float(first + static_cast<uint32_t>(i));
}

__global__ void debug_block_scale_kernel(uint32_t first, uint64_t count, float eps,
                                         float* __restrict__ scales, float* __restrict__ inv) {
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride) {
        const uint32_t sb = scale_bits(fmaxf(pattern(first, i), eps));
        scales[i] = __uint_as_float(sb);
        inv[i] = inv_scale(sb);
    }
}

// Thread j handles patterns first + 16 j .. first + 16 j + 15, as the 16
// values (two 8-element chunks) one lane quantises in a row.
__global__ void debug_quant_codes_kernel(uint32_t first, uint64_t groups, uint32_t sbits,
                                         uint4* __restrict__ codes) {
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    const float inv = inv_scale(sbits);
    for (uint64_t j = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; j < groups; j += stride) {
        const uint64_t i0 = 16 * j;
        Pairs p;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // element order of unpack(): 4k, 4k+1, 4k+2, 4k+3
            p.ev[k] = make_float2(pattern(first, i0 + 4 * k), pattern(first, i0 + 4 * k + 2));
            p.od[k] = make_float2(pattern(first, i0 + 4 * k + 1), pattern(first, i0 + 4 * k + 3));
        }
        codes[j] = quant16(p, inv);
    }
}

int grid_for(uint64_t work, int sm_count) {
    const uint64_t need = (work + 255) / 256;
    const uint64_t cap = uint64_t(sm_count) * 8;
    return static_cast<int>(need < cap ? need : cap);
}

rq_status status_of(cudaError_t e) {
    if (e == cudaSuccess) return RQ_OK;
    (void)cudaGetLastError();
    return RQ_ERR_CUDA;
}

cudaError_t sm_count_of_current(int* n) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
}

}  // namespace
}  // namespace rq

RQ_EXPORT rq_status rq_debug_block_scale(uint32_t first_bits, int64_t count, float eps,
                                         float* scales, float* inv_scales, void* stream) {
    if (count < 0 || uint64_t(first_bits) + uint64_t(count) > (uint64_t(1) << 32))
        return RQ_ERR_SHAPE;
    if (!(eps >= 0x1p-100f && eps <= 0x1p100f)) return RQ_ERR_ARG;
    if (count == 0) return RQ_OK;
    if (!scales || !inv_scales) return RQ_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(scales) | reinterpret_cast<uintptr_t>(inv_scales)) & 3u)
        return RQ_ERR_ALIGN;
    int sms = 0;
    cudaError_t e = rq::sm_count_of_current(&sms);
    if (e != cudaSuccess) return rq::status_of(e);
    rq::debug_block_scale_kernel<<<rq::grid_for(uint64_t(count), sms), 256, 0,
                                   static_cast<cudaStream_t>(stream)>>>(
        first_bits, uint64_t(count), eps, scales, inv_scales);
    return rq::status_of(cudaGetLastError());
}

RQ_EXPORT rq_status rq_debug_quant_codes(uint32_t first_bits, int64_t count, int scale_exp,
                                         uint8_t* codes, void* stream) {
    if (count < 0 || count % 16 || uint64_t(first_bits) + uint64_t(count) > (uint64_t(1) << 32))
        return RQ_ERR_SHAPE;
    if (scale_exp < -126 || scale_exp > 126) return RQ_ERR_ARG;
    if (count == 0) return RQ_OK;
    if (!codes) return RQ_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(codes) & 15u) return RQ_ERR_ALIGN;
    int sms = 0;
    cudaError_t e = rq::sm_count_of_current(&sms);
    if (e != cudaSuccess) return rq::status_of(e);
    // the bit pattern of 2^scale_exp, as scale_bits() produces it
    const uint32_t sbits = uint32_t(scale_exp + 127) << 23;
    const uint64_t groups = uint64_t(count) / 16;
    rq::debug_quant_codes_kernel<<<rq::grid_for(groups, sms), 256, 0,
                                   static_cast<cudaStream_t>(stream)>>>(
        first_bits, groups, sbits, reinterpret_cast<uint4*>(codes));
    return rq::status_of(cudaGetLastError());
}
