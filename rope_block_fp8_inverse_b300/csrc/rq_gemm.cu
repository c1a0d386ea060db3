// rq_gemm.cu -- the consumer of the block-FP8 output: a grouped FP8 GEMM on
// the 5th-generation tensor cores (tcgen05, accumulators in TMEM), as in the
// DeepSeek-V4 path of "[vllm] 한 프로그램이 4개 head를 처리하게 하라: DeepSeek-V4
// inverse RoPE + FP8 quant 커널 3.5배 가속기" (vLLM PR #63540 analysis), intro:
// the inverse-RoPE'd, block-quantised attention output of each output group
// feeds that group's wo_a projection.
//
// For every group g:  Y[:, g, :] = dequant(A_g) @ dequant(W_g)^T  with
//   A_g  the codes [M, K] of group g (K = heads_per_group * 512), scale
//        sa[m, g, kt] for row m and 128-wide K block kt (the op's own scales);
//   W_g  e4m3 weights [n_out, K] (K-major), scale sw[g, nb, kt] for each
//        128 x 128 block (nb = n / 128);
//   Y    bf16 [M, G, n_out].
// A 128-wide K tile is exactly one scale block of A and of W, so each tile's
// product is accumulated by the tensor cores into a fresh fp32 TMEM
// accumulator and then folded into fp32 registers with sa * sw (one fused
// multiply-add per element): the per-block scales never meet inside the MMA.
//
// CTA: 128 x 128 output tile. Warp 0 (one lane) loads the A and W tiles of
// each K step with tensor-map TMA (128-byte swizzle) into a 4-stage ring;
// warp 1 owns TMEM (two 128-column accumulators) and one lane issues the
// MMAs (4 x K=32 per tile) and commits them to mbarriers; warps 2..5 (one
// thread per output row = TMEM lane) fold each finished accumulator into
// registers and write the row at the end. Every wait is bounded.
#include "rq_device.cuh"
#include "rq_launch.h"
#include "rq_tma.cuh"
#include "rq_umma.cuh"

namespace rq {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 128;
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kTileBytes = kBM * kBK;                  // 128 rows x 128 bytes
constexpr uint32_t kOffB = kGemmStages * kTileBytes;
constexpr uint32_t kOffBar = 2 * kGemmStages * kTileBytes;
constexpr uint32_t kNumBars = 2 * kGemmStages + 2 + 2 + 1;  // full, empty, tfull, tempty, done
constexpr uint32_t kOffTmem = kOffBar + 8 * kNumBars;
constexpr uint32_t kGemmSmem = kOffTmem + 16 + 1024;        // + room to align the base to 1 KiB
constexpr uint32_t kTmemCols = 2 * kBN;

}  // namespace

__global__ void __launch_bounds__(kGemmThreads, 1)
grouped_fp8_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                        const __grid_constant__ CUtensorMap tma_w, GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1 KiB alignment
    const uint32_t a0 = base, w0 = base + kOffB, bar0 = base + kOffBar;
    const uint32_t full0 = bar0, empty0 = bar0 + 8 * kGemmStages;
    const uint32_t tfull0 = bar0 + 16 * kGemmStages, tempty0 = tfull0 + 16;
    const uint32_t done = tempty0 + 16;
    const uint32_t tmem_slot = base + kOffTmem;
    volatile uint32_t* tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - raw));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN, g = blockIdx.z;
    const int n_kt = p.k / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 128);
        }
        mbar_init(done, 1);
        mbar_init_fence();
    }
    if (warp == 1) {
        umma::tmem_alloc(tmem_slot, kTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot_ptr;

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            for (int kt = 0; kt < n_kt; ++kt) {
                const int s = kt % kGemmStages;
                const uint32_t ph = (kt / kGemmStages) & 1;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * s, 2 * kTileBytes);
                umma::tma_load_2d(a0 + s * kTileBytes, &tma_a, g * p.k + kt * kBK, m0, full0 + 8 * s);
                umma::tma_load_2d(w0 + s * kTileBytes, &tma_w, kt * kBK, g * p.n_out + n0,
                                  full0 + 8 * s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma::idesc_e4m3_f32(kBM, kBN);
            for (int kt = 0; kt < n_kt; ++kt) {
                const int s = kt % kGemmStages;
                const uint32_t ph = (kt / kGemmStages) & 1;
                const int buf = kt & 1;
                const uint32_t bph = (kt >> 1) & 1;
                if (!mbar_wait(full0 + 8 * s, ph) || !mbar_wait(tempty0 + 8 * buf, bph ^ 1u)) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
                const uint64_t ad = umma::smem_desc_sw128(a0 + s * kTileBytes);
                const uint64_t wd = umma::smem_desc_sw128(w0 + s * kTileBytes);
#pragma unroll
                for (int k = 0; k < kBK / 32; ++k)  // K = 32 bytes of e4m3 per MMA
                    umma::mma_f8f6f4(tmem + buf * kBN, ad + 2 * k, wd + 2 * k, idesc, k > 0);
                umma::commit(empty0 + 8 * s);   // the smem stage is free once these finish
                umma::commit(tfull0 + 8 * buf); // and the accumulator is ready
            }
            umma::commit(done);
            if (!mbar_wait(done, 0)) ok = false;  // nothing in flight before teardown
        }
    } else {
        // epilogue: thread = output row = TMEM lane 32 * (warp % 4) + lane
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int gm = m0 + row;
        const int cm = gm < p.m ? gm : p.m - 1;  // rows past M hold zeros; read a valid scale
        const float* sa = p.a_scales + (int64_t(cm) * p.groups + g) * n_kt;
        const float* sw = p.w_scales + (int64_t(g) * (p.n_out / kBN) + blockIdx.y) * n_kt;
        float acc[kBN];
#pragma unroll
        for (int j = 0; j < kBN; ++j) acc[j] = 0.f;
        for (int kt = 0; kt < n_kt; ++kt) {
            const int buf = kt & 1;
            const uint32_t bph = (kt >> 1) & 1;
            const float sc = __fmul_rn(__ldg(sa + kt), __ldg(sw + kt));
            // the warp leaves together: the TMEM loads below are warp-collective
            if (!__all_sync(kFull, mbar_wait(tfull0 + 8 * buf, bph))) {
                ok = false;
                break;
            }
            umma::fence_after_sync();
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                float d[32];
                umma::ld32(tmem + (uint32_t(quad * 32) << 16) + buf * kBN + c * 32, d);
                umma::wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[c * 32 + j] = __fmaf_rn(d[j], sc, acc[c * 32 + j]);
            }
            umma::fence_before_sync();
            mbar_arrive(tempty0 + 8 * buf);
        }
        if (ok && gm < p.m) {
            uint16_t* y = p.y + (int64_t(gm) * p.groups + g) * p.n_out + n0;
#pragma unroll
            for (int j = 0; j < kBN; j += 8) {
                const uint4 v = make_uint4(bf16x2(acc[j], acc[j + 1]), bf16x2(acc[j + 2], acc[j + 3]),
                                           bf16x2(acc[j + 4], acc[j + 5]),
                                           bf16x2(acc[j + 6], acc[j + 7]));
                *reinterpret_cast<uint4*>(y + j) = v;
            }
        }
    }
    if (!ok && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_TIMEOUT);
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kTmemCols);
    }
}

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(ptr);
    }
    return fn;
}

// 2-D uint8 tensor [rows, inner] with row stride `stride` bytes, boxes of
// 128 x 128 bytes, 128-byte swizzle; rows past the end read as zeros.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride) {
    EncodeTiled fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_grouped_fp8_gemm(const GemmParams& p, const uint8_t* a_codes,
                                    const uint8_t* w_codes, int dev_ordinal, cudaStream_t stream) {
    CUtensorMap ma, mw;
    if (!make_map(&ma, a_codes, uint64_t(p.groups) * p.k, uint64_t(p.m), uint64_t(p.groups) * p.k) ||
        !make_map(&mw, w_codes, uint64_t(p.k), uint64_t(p.groups) * p.n_out, uint64_t(p.k)))
        return cudaErrorInvalidValue;
    constexpr int kMax = 64;
    static thread_local bool attr_done[kMax] = {};
    const int d = (dev_ordinal >= 0 && dev_ordinal < kMax) ? dev_ordinal : 0;
    if (!attr_done[d]) {
        const cudaError_t e = cudaFuncSetAttribute(
            grouped_fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kGemmSmem));
        if (e != cudaSuccess) return e;
        attr_done[d] = true;
    }
    const dim3 grid((p.m + kBM - 1) / kBM, p.n_out / kBN, p.groups);
    grouped_fp8_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, stream>>>(ma, mw, p);
    return cudaGetLastError();
}

}  // namespace rq
