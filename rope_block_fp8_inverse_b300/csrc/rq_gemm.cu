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
// MMAs (4 x K=32 per tile) and commits them to mbarriers; warps 2..9 (one
// thread per output row = TMEM lane and 64 of the 128 columns) fold each
// finished accumulator into registers and write their part of the row at the
// end. Every wait is bounded.
#include "rq_device.cuh"
#include "rq_launch.h"
#include "rq_tma.cuh"
#include "rq_umma.cuh"

namespace rq {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 128;  // the fused kernel's tile
constexpr int kGemmStages = 4;
constexpr uint32_t kTileBytes = kBM * kBK;                  // 128 rows x 128 bytes
constexpr uint32_t kOffB = kGemmStages * kTileBytes;
constexpr uint32_t kNumBars = 2 * kGemmStages + 2 + 2 + 1;  // full, empty, tfull, tempty, done
constexpr uint32_t kTmemCols = 2 * kBN;

// the unfused kernel's tile: 128 x 256 (one MMA of N = 256 per K = 32 step),
// two 256-column accumulators = all 512 TMEM columns
constexpr int kGBN = 256;
// epilogue warps: a multiple of 4 (one per TMEM lane quadrant per column slice).
// 8 warps of 128 columns; 16 warps of 64 columns measured slower on B300 (436
// vs 294 us at M = 16384: 96 registers with spills at 576 threads, and the
// same 128 KiB TMEM readback per K tile)
#ifndef RQ_GEMM_EPI_WARPS
#define RQ_GEMM_EPI_WARPS 8
#endif
constexpr int kGEpiWarps = RQ_GEMM_EPI_WARPS;
constexpr int kGEpiCols = kGBN / (kGEpiWarps / 4);          // accumulator columns per warp
constexpr int kGemmThreads = 64 + 32 * kGEpiWarps;          // warp 0 TMA, warp 1 MMA, epilogue
static_assert(kGEpiWarps % 4 == 0 && kGEpiCols % 32 == 0 && 128 % kGEpiCols == 0,
              "epilogue slices must tile the 256 columns in 32-column loads within 128-blocks");
constexpr uint32_t kGWTile = kGBN * kBK;                     // 256 rows x 128 bytes
constexpr uint32_t kGOffW = kGemmStages * kTileBytes;
constexpr uint32_t kGOffBar = kGOffW + kGemmStages * kGWTile;
constexpr uint32_t kGOffTmem = kGOffBar + 8 * kNumBars;
constexpr uint32_t kGemmSmem = kGOffTmem + 16 + 1024;        // + room to align the base to 1 KiB
constexpr uint32_t kGTmemCols = 2 * kGBN;

}  // namespace

__global__ void __launch_bounds__(kGemmThreads, 1)
grouped_fp8_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                        const __grid_constant__ CUtensorMap tma_w, GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1 KiB alignment
    const uint32_t a0 = base, w0 = base + kGOffW, bar0 = base + kGOffBar;
    const uint32_t full0 = bar0, empty0 = bar0 + 8 * kGemmStages;
    const uint32_t tfull0 = bar0 + 16 * kGemmStages, tempty0 = tfull0 + 16;
    const uint32_t done = tempty0 + 16;
    const uint32_t tmem_slot = base + kGOffTmem;
    volatile uint32_t* tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - raw));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kGBN, g = blockIdx.z;
    const int n_kt = p.k / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 32 * kGEpiWarps);
        }
        mbar_init(done, 1);
        mbar_init_fence();
    }
    if (warp == 1) {
        umma::tmem_alloc(tmem_slot, kGTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot_ptr;

    bool ok = true;
    const uint32_t lim = p.wait.spin_limit;
    // test-only fault injection: CTA 0's producer issues nothing
    const bool starve = (p.wait.inject & kInjectGemmLoads) && blockIdx.x == 0 && blockIdx.y == 0 &&
                        blockIdx.z == 0;
    if (warp == 0) {
        if (lane == 0 && !starve) {
            for (int kt = 0; kt < n_kt; ++kt) {
                const int s = kt % kGemmStages;
                const uint32_t ph = (kt / kGemmStages) & 1;
                if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * s, kTileBytes + kGWTile);
                umma::tma_load_2d(a0 + s * kTileBytes, &tma_a, g * p.k + kt * kBK, m0, full0 + 8 * s);
                umma::tma_load_2d(w0 + s * kGWTile, &tma_w, kt * kBK, g * p.n_out + n0,
                                  full0 + 8 * s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma::idesc_e4m3_f32(kBM, kGBN);
            for (int kt = 0; kt < n_kt; ++kt) {
                const int s = kt % kGemmStages;
                const uint32_t ph = (kt / kGemmStages) & 1;
                const int buf = kt & 1;
                const uint32_t bph = (kt >> 1) & 1;
                if (!mbar_wait(full0 + 8 * s, ph, lim) || !mbar_wait(tempty0 + 8 * buf, bph ^ 1u, lim)) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
                const uint64_t ad = umma::smem_desc_sw128(a0 + s * kTileBytes);
                const uint64_t wd = umma::smem_desc_sw128(w0 + s * kGWTile);
#pragma unroll
                for (int k = 0; k < kBK / 32; ++k)  // K = 32 bytes of e4m3 per MMA
                    umma::mma_f8f6f4(tmem + buf * kGBN, ad + 2 * k, wd + 2 * k, idesc, k > 0);
                umma::commit(empty0 + 8 * s);   // the smem stage is free once these finish
                umma::commit(tfull0 + 8 * buf); // and the accumulator is ready
            }
            umma::commit(done);
            if (!mbar_wait(done, 0, lim)) ok = false;  // nothing in flight before teardown
        }
    } else {
        // epilogue (warps 2 ..): thread = output row = TMEM lane 32 * (warp % 4) + lane,
        // columns col0 .. col0 + kGEpiCols - 1 of the tile, col0 = kGEpiCols * ((warp - 2) / 4)
        const int quad = warp & 3;
        const int col0 = kGEpiCols * ((warp - 2) >> 2);
        const int row = quad * 32 + lane;
        const int gm = m0 + row;
        const int cm = gm < p.m ? gm : p.m - 1;  // rows past M hold zeros; read a valid scale
        const float* sa = p.a_scales + (int64_t(cm) * p.groups + g) * n_kt;
        // weight scales: one per 128 x 128 block; this slice lies in block
        // 2 * blockIdx.y + col0 / 128 (when n_out is an odd multiple of 128 the
        // last tile's second half is past the end: computed, never stored)
        const bool live = n0 + col0 < p.n_out;
        const float* sw = p.w_scales + (int64_t(g) * (p.n_out / 128) +
                                        (live ? 2 * blockIdx.y + col0 / 128 : 0)) * n_kt;
        float acc[kGEpiCols];
#pragma unroll
        for (int j = 0; j < kGEpiCols; ++j) acc[j] = 0.f;
        for (int kt = 0; kt < n_kt; ++kt) {
            const int buf = kt & 1;
            const uint32_t bph = (kt >> 1) & 1;
            const float sc = __fmul_rn(__ldg(sa + kt), __ldg(sw + kt));
            // the warp leaves together: the TMEM loads below are warp-collective
            if (!__all_sync(kFull, mbar_wait(tfull0 + 8 * buf, bph, lim))) {
                ok = false;
                break;
            }
            umma::fence_after_sync();
#pragma unroll
            for (int c = 0; c < kGEpiCols / 32; ++c) {
                float d[32];
                umma::ld32(tmem + (uint32_t(quad * 32) << 16) + buf * kGBN + col0 + c * 32, d);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[c * 32 + j] = __fmaf_rn(d[j], sc, acc[c * 32 + j]);
            }
            umma::fence_before_sync();
            mbar_arrive(tempty0 + 8 * buf);
        }
        if (ok && gm < p.m && live) {
            uint16_t* y = p.y + (int64_t(gm) * p.groups + g) * p.n_out + n0 + col0;
#pragma unroll
            for (int j = 0; j < kGEpiCols; j += 8) {
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
        umma::tmem_dealloc(tmem, kGTmemCols);
    }
}

// ------------------------------------------------------------------ fused

// The same GEMM with its A operand produced inside the kernel from the bf16
// attention output: producer warps apply the inverse RoPE and the block-FP8
// quantisation of the inverse-RoPE page (S1-S3), with the arithmetic of
// rq_inv_rope_fp8_quant, to each 128-wide K tile (head kt / 4, block kt % 4
// of the group's heads) and write the e4m3 codes straight into the swizzled
// shared-memory layout the MMA reads, and the row's scale into a shared
// array the epilogue reads. The codes never go to HBM.
//
// The bf16 input tiles (128 tokens x 128 elements = 32 KiB) come in by 3-D
// tensor-map TMA (dims 512 x heads x tokens, so any token / head strides
// work) into a double-buffered ring, ahead of the producers.
//
// Warps: 0 TMA (x tiles and W tiles), 1 TMEM + MMA, 2..9 epilogue (8 warps:
// TMEM lane quadrant warp % 4, column half (warp - 2) / 4), 10..13 A
// producers (32 rows each). The grid runs the N tiles of an M tile next to
// each other, so their x tiles are L2 hits after the first.
namespace {

constexpr int kFusThreads = 448;
constexpr int kFusEpiWarp0 = 2, kFusProdWarp0 = 10;
constexpr uint32_t kXTileBytes = kBM * kBK * 2;                 // bf16 input tile
constexpr uint32_t kFusOffX = 2 * kGemmStages * kTileBytes;     // after A and W stages (128 x 128)
constexpr uint32_t kFusMaxKt = 32;                              // K up to 4096
constexpr uint32_t kFusOffSa = kFusOffX + 2 * kXTileBytes;      // sa[kt][128] fp32
constexpr uint32_t kFusOffBar = kFusOffSa + kFusMaxKt * 128 * 4;
constexpr uint32_t kFusNumBars = kNumBars + 4;                  // + xfull[2], xempty[2]
constexpr uint32_t kFusOffTmem = kFusOffBar + 8 * kFusNumBars;
constexpr uint32_t kFusSmem = kFusOffTmem + 16 + 1024;

}  // namespace

__global__ void __launch_bounds__(kFusThreads, 1)
fused_inv_rope_quant_gemm_kernel(const __grid_constant__ CUtensorMap tma_x,
                                 const __grid_constant__ CUtensorMap tma_w, FusedGemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t a0 = base, w0 = base + kOffB, x0 = base + kFusOffX, sa0 = base + kFusOffSa;
    const uint32_t bar0 = base + kFusOffBar;
    const uint32_t full0 = bar0, empty0 = bar0 + 8 * kGemmStages;
    const uint32_t tfull0 = bar0 + 16 * kGemmStages, tempty0 = tfull0 + 16;
    const uint32_t done = tempty0 + 16;
    const uint32_t xfull0 = done + 8, xempty0 = xfull0 + 16;
    const uint32_t tmem_slot = base + kFusOffTmem;
    volatile uint32_t* tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t*>(smem_raw + (tmem_slot - raw));
    const float* sa_smem = reinterpret_cast<const float*>(smem_raw + (sa0 - raw));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM, g = blockIdx.z;
    const int n_kt = p.k / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(full0 + 8 * s, 1 + 4);   // W's expect_tx arrival + 4 producer warps
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 256);
            mbar_init(xfull0 + 8 * b, 1);
            mbar_init(xempty0 + 8 * b, 4);
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
    const uint32_t lim = p.wait.spin_limit;
    if (warp == 0) {
        if (lane == 0) {
            for (int kt = 0; kt < n_kt; ++kt) {
                const int sx = kt & 1;
                if (!mbar_wait(xempty0 + 8 * sx, ((kt >> 1) & 1) ^ 1u, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(xfull0 + 8 * sx, kXTileBytes);
                umma::tma_load_3d(x0 + sx * kXTileBytes, &tma_x, (kt & 3) * kBK, g * p.hpg + kt / 4,
                                  m0, xfull0 + 8 * sx);
                const int s = kt % kGemmStages;
                if (!mbar_wait(empty0 + 8 * s, ((kt / kGemmStages) & 1) ^ 1u, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * s, kTileBytes);
                umma::tma_load_2d(w0 + s * kTileBytes, &tma_w, kt * kBK, g * p.n_out + n0,
                                  full0 + 8 * s);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma::idesc_e4m3_f32(kBM, kBN);
            for (int kt = 0; kt < n_kt; ++kt) {
                const int s = kt % kGemmStages;
                const int buf = kt & 1;
                if (!mbar_wait(full0 + 8 * s, (kt / kGemmStages) & 1, lim) ||
                    !mbar_wait(tempty0 + 8 * buf, ((kt >> 1) & 1) ^ 1u, lim)) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
                const uint64_t ad = umma::smem_desc_sw128(a0 + s * kTileBytes);
                const uint64_t wd = umma::smem_desc_sw128(w0 + s * kTileBytes);
#pragma unroll
                for (int k = 0; k < kBK / 32; ++k)
                    umma::mma_f8f6f4(tmem + buf * kBN, ad + 2 * k, wd + 2 * k, idesc, k > 0);
                umma::commit(empty0 + 8 * s);
                umma::commit(tfull0 + 8 * buf);
            }
            umma::commit(done);
            if (!mbar_wait(done, 0, lim)) ok = false;
        }
    } else if (warp < kFusProdWarp0) {
        // epilogue: row = TMEM lane, 64 of the tile's 128 columns
        const int quad = warp & 3;
        const int half = (warp - kFusEpiWarp0) >> 2;
        const int row = quad * 32 + lane;
        const int gm = m0 + row;
        const float* sw = p.w_scales + (int64_t(g) * (p.n_out / kBN) + blockIdx.x) * n_kt;
        float acc[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) acc[j] = 0.f;
        for (int kt = 0; kt < n_kt; ++kt) {
            const int buf = kt & 1;
            const float swk = __ldg(sw + kt);
            if (!__all_sync(kFull, mbar_wait(tfull0 + 8 * buf, (kt >> 1) & 1, lim))) {
                ok = false;
                break;
            }
            umma::fence_after_sync();
            const float sc = __fmul_rn(sa_smem[kt * 128 + row], swk);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float d[32];
                umma::ld32(tmem + (uint32_t(quad * 32) << 16) + buf * kBN + half * 64 + c * 32, d);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[c * 32 + j] = __fmaf_rn(d[j], sc, acc[c * 32 + j]);
            }
            umma::fence_before_sync();
            mbar_arrive(tempty0 + 8 * buf);
        }
        if (ok && gm < p.m) {
            uint16_t* y = p.y + (int64_t(gm) * p.groups + g) * p.n_out + n0 + half * 64;
#pragma unroll
            for (int j = 0; j < 64; j += 8) {
                const uint4 v = make_uint4(bf16x2(acc[j], acc[j + 1]), bf16x2(acc[j + 2], acc[j + 3]),
                                           bf16x2(acc[j + 4], acc[j + 5]),
                                           bf16x2(acc[j + 6], acc[j + 7]));
                *reinterpret_cast<uint4*>(y + j) = v;
            }
        }
    } else {
        // A producers: warp (warp - 10) owns rows 32 * (warp - 10) .. + 31 of the tile.
        // Lane l holds elements 4l .. 4l+3 of the row's 128-wide block; in the last
        // block of a head (dims 384..511) lanes 16..31 hold dims 448..511, two whole
        // (even, odd) pairs each: pairs 2(l-16), 2(l-16)+1 of the RoPE tail.
        const int pw = warp - kFusProdWarp0;
        const int my_t = m0 + pw * 32 + lane;   // positions of this warp's rows, one per lane
        const int64_t my_pos = my_t < p.m ? __ldg(p.positions + my_t) : 0;
        const bool my_pos_ok = static_cast<uint64_t>(my_pos) < static_cast<uint64_t>(p.cache_rows);
        if (!__all_sync(kFull, my_pos_ok) && lane == 0 && p.error_flags)
            atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
        const bool rope_lane = lane >= 16;
        const int pair0 = rope_lane ? 2 * (lane - 16) : 0;
        for (int kt = 0; kt < n_kt; ++kt) {
            const int s = kt % kGemmStages;
            const int sx = kt & 1;
            if (!__all_sync(kFull, mbar_wait(xfull0 + 8 * sx, (kt >> 1) & 1, lim) &&
                                       mbar_wait(empty0 + 8 * s, ((kt / kGemmStages) & 1) ^ 1u, lim))) {
                ok = false;
                break;
            }
            const bool rope_blk = (kt & 3) == 3;
            const uint32_t tile = a0 + s * kTileBytes;
            const uint32_t xt = x0 + sx * kXTileBytes;
#pragma unroll 1
            for (int b8 = 0; b8 < 4; ++b8) {
                float cc[8][2], ss[8][2];
                if (rope_blk) {  // warp-uniform: the batch's cos/sin reads, all in flight together
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int64_t pos = __shfl_sync(kFull, my_pos, b8 * 8 + i);
                        const bool pos_ok = static_cast<uint64_t>(pos) <
                                            static_cast<uint64_t>(p.cache_rows);
                        const float* cs = p.cache + (pos_ok ? pos : 0) * kCacheWidth + pair0;
                        float2 c2 = make_float2(1.f, 1.f), s2 = make_float2(0.f, 0.f);
                        if (rope_lane) {
                            c2 = __ldg(reinterpret_cast<const float2*>(cs));
                            s2 = __ldg(reinterpret_cast<const float2*>(cs + kHalfRope));
                        }
                        cc[i][0] = c2.x;
                        cc[i][1] = c2.y;
                        ss[i][0] = s2.x;
                        ss[i][1] = s2.y;
                    }
                }
                // 8 rows at a time, in phases: all loads, then the arithmetic with the
                // 8 warp reductions interleaved, then all stores
                uint32_t raw[8][2];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = pw * 32 + b8 * 8 + i;
                    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                 : "=r"(raw[i][0]), "=r"(raw[i][1])
                                 : "r"(xt + r * (kBK * 2) + 8 * lane));
                }
                float v[8][4], am[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[i][0] = __uint_as_float(raw[i][0] << 16);
                    v[i][1] = __uint_as_float(raw[i][0] & 0xffff0000u);
                    v[i][2] = __uint_as_float(raw[i][1] << 16);
                    v[i][3] = __uint_as_float(raw[i][1] & 0xffff0000u);
                    if (rope_blk && rope_lane) {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {  // inverse: e' = e*c + o*s, o' = o*c - e*s
                            const float e = v[i][2 * q], o = v[i][2 * q + 1];
                            v[i][2 * q] = __fadd_rn(__fmul_rn(e, cc[i][q]), __fmul_rn(o, ss[i][q]));
                            v[i][2 * q + 1] =
                                __fsub_rn(__fmul_rn(o, cc[i][q]), __fmul_rn(e, ss[i][q]));
                        }
                    }
                    am[i] = fmaxf(fmaxf(fabsf(v[i][0]), fabsf(v[i][1])),
                                  fmaxf(fabsf(v[i][2]), fabsf(v[i][3])));
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) am[i] = fmaxf(am[i], __shfl_xor_sync(kFull, am[i], off));
                }
                uint32_t q4[8], sbits[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    sbits[i] = scale_bits(fmaxf(am[i], p.eps));
                    const float inv = inv_scale(sbits[i]);
                    q4[i] = e4m3x2(__fmul_rn(v[i][0], inv), __fmul_rn(v[i][1], inv)) |
                            (e4m3x2(__fmul_rn(v[i][2], inv), __fmul_rn(v[i][3], inv)) << 16);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = pw * 32 + b8 * 8 + i;
                    // K-major, 128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8)
                    const uint32_t chunk = uint32_t(lane >> 2) ^ uint32_t(r & 7);
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(tile + r * 128 + chunk * 16 +
                                                                 (lane & 3) * 4),
                                 "r"(q4[i])
                                 : "memory");
                    if (lane == 0)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(sa0 + (kt * 128 + r) * 4),
                                     "f"(__uint_as_float(sbits[i]))
                                     : "memory");
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xempty0 + 8 * sx);   // the bf16 tile is consumed
            fence_proxy_async_smem();                        // the codes, visible to the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(full0 + 8 * s);
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

}  // namespace

bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride,
              uint32_t box_rows) {
    EncodeTiled fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// The bf16 input as a 3-D tensor [tokens, heads, 512] with free token / head
// strides; boxes of 128 elements x 1 head x 128 tokens, no swizzle.
bool make_x_map(CUtensorMap* map, const FusedGemmParams& p) {
    EncodeTiled fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {512, uint64_t(p.groups) * p.hpg, uint64_t(p.m)};
    const cuuint64_t strides[2] = {uint64_t(p.sx_h) * 2, uint64_t(p.sx_t) * 2};
    const cuuint32_t box[3] = {128, 1, 128};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.x), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_grouped_fp8_gemm(const GemmParams& p, const uint8_t* a_codes,
                                    const uint8_t* w_codes, int dev_ordinal, cudaStream_t stream) {
    // up to 64 tokens with K a multiple of 512: the split-K decode kernel
    if (p.m <= 64 && p.k % 512 == 0)
        return launch_grouped_fp8_gemm_small(p, a_codes, w_codes, dev_ordinal, stream);
    CUtensorMap ma, mw;
    if (!make_map(&ma, a_codes, uint64_t(p.groups) * p.k, uint64_t(p.m), uint64_t(p.groups) * p.k,
                  128) ||
        !make_map(&mw, w_codes, uint64_t(p.k), uint64_t(p.groups) * p.n_out, uint64_t(p.k), kGBN))
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
    const dim3 grid((p.m + kBM - 1) / kBM, (p.n_out + kGBN - 1) / kGBN, p.groups);
    grouped_fp8_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, stream>>>(ma, mw, p);
    return cudaGetLastError();
}

cudaError_t launch_fused_inv_rope_quant_gemm(const FusedGemmParams& p, const uint8_t* w_codes,
                                             int dev_ordinal, cudaStream_t stream) {
    CUtensorMap mw, mx;
    if (!make_map(&mw, w_codes, uint64_t(p.k), uint64_t(p.groups) * p.n_out, uint64_t(p.k), 128) ||
        !make_x_map(&mx, p))
        return cudaErrorInvalidValue;
    constexpr int kMax = 64;
    static thread_local bool attr_done[kMax] = {};
    const int d = (dev_ordinal >= 0 && dev_ordinal < kMax) ? dev_ordinal : 0;
    if (!attr_done[d]) {
        const cudaError_t e =
            cudaFuncSetAttribute(fused_inv_rope_quant_gemm_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(kFusSmem));
        if (e != cudaSuccess) return e;
        attr_done[d] = true;
    }
    const dim3 grid(p.n_out / kBN, (p.m + kBM - 1) / kBM, p.groups);
    fused_inv_rope_quant_gemm_kernel<<<grid, kFusThreads, kFusSmem, stream>>>(mx, mw, p);
    return cudaGetLastError();
}

}  // namespace rq
