// rq_kernels.cu -- sm_103a kernels of the inverse-RoPE + block-FP8 quant op
// and of its forward-RoPE + paged-insert sibling, with their launchers.
//
// Both are HBM-bound streams (about 1.5 bytes moved per fp32 op), so the
// design goal is bytes in flight, not arithmetic: a persistent grid of warps
// sized to the SM count, each warp owning whole 512-wide rows
// (rq_device.cuh) and issuing the loads of kRows rows before it computes any
// of them. The pages' Triton kernel (one program per 1 to 4 heads) is prior
// art: here a warp is the program, and the number of rows in flight per SM
// is set by kRows x resident warps instead of by BLOCK_H.
#include "rq_device.cuh"
#include "rq_launch.h"
#include "rq_tma.cuh"

namespace rq {

// ------------------------------------------------------------------ inverse

// Row r = t * n_heads + h. Output row r (512 codes) sits at out + r*512 and
// its 4 scales at scales + r*4: with contiguous [N, G, hpg*512] /
// [N, G, hpg*4] outputs this is exactly the grouped layout of the inverse
// RoPE page, S1 (head h = g*hpg + i of token t at row (t, g), offset i*512),
// so the grouping never changes an address.
template <int kRows>
__global__ void __launch_bounds__(kInvThreads)
inv_rope_fp8_quant_kernel(InvParams p) {
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
    const int cs_col = (lane >= kRopeLane0 ? lane - kRopeLane0 : 0) * 4;

    for (uint32_t r0 = warp * kRows; r0 < p.n_rows; r0 += n_warps * kRows) {
        RowRegs in[kRows];
        bool live[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const uint32_t r = r0 + i;
            live[i] = false;
            if (r < p.n_rows) {  // warp-uniform
                const uint32_t t = r / p.n_heads;
                const uint32_t h = r - t * p.n_heads;
                const int64_t pos = __ldg(p.positions + t);
                live[i] = static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
                if (live[i]) {
                    const uint16_t* row = x + static_cast<int64_t>(t) * p.sx_t +
                                          static_cast<int64_t>(h) * p.sx_h;
                    in[i].a = ld_stream16(row + 8 * lane);
                    in[i].b = ld_stream16(row + kHalf + 8 * lane);
                    if (lane >= kRopeLane0) {
                        const float* cs = p.cache + pos * kCacheWidth + cs_col;
                        in[i].c = ld_shared_ro16(cs);
                        in[i].s = ld_shared_ro16(cs + kHalfRope);
                    }
                } else if (lane == 0 && p.error_flags) {
                    atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            if (!live[i]) continue;
            const uint32_t r = r0 + i;
            const RowOut o = rope_quant_row<true>(in[i], lane, p.eps);
            uint8_t* dst = p.out + static_cast<int64_t>(r) * kHeadDim;
            st_stream8(dst + 8 * lane, o.qa.x, o.qa.y);
            st_stream8(dst + kHalf + 8 * lane, o.qb.x, o.qb.y);
            const float s1 = __shfl_sync(kFull, o.sa, 16);
            const float s3 = __shfl_sync(kFull, o.sb, 16);
            if (lane == 0) st_stream16f(p.scales + static_cast<int64_t>(r) * 4, o.sa, s1, o.sb, s3);
        }
    }
}

// ------------------------------------------------------------------ inverse, TMA pipeline

// Shared-memory pipeline: one producer warp streams tiles of kRows head rows
// (one token, heads h0 .. h0+kRows-1) into a ring of kStages stages with 1-D
// bulk copies (TMA), together with the token's 256-byte cos|sin row. kGroups
// groups of kRows consumer warps take the stages in turn (group g the tiles
// it = g mod kGroups); warp k of a group takes row k, releases the stage as
// soon as the row is in registers, then rotates, quantises and stores it.
// Bytes in flight per SM are set by the ring (kStages x ~8.25 KiB per CTA),
// not by the number of resident warps; the consumer groups only have to
// cover the arithmetic latency. Tiles are dealt round-robin over a
// persistent grid, so at any moment all SMs stream neighbouring regions.
template <int kRows, int kStages, int kGroups>
struct TmaLayout {
    static constexpr uint32_t kRowBytes = kHeadDim * 2;
    static constexpr uint32_t kCsBytes = kCacheWidth * 4;
    static constexpr uint32_t kStageBytes = kRows * kRowBytes + kCsBytes;
    static constexpr uint32_t kMetaOffset = kStages * kStageBytes;
    static constexpr uint32_t kBarOffset = (kMetaOffset + 4 * kStages + 7) & ~7u;
    static constexpr uint32_t kBytes = kBarOffset + 16 * kStages;
    static constexpr int kConsumerWarps = kGroups * kRows;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;
};

template <int kRows, int kStages, int kGroups>
__global__ void __launch_bounds__(TmaLayout<kRows, kStages, kGroups>::kThreads)
inv_rope_fp8_quant_tma_kernel(InvParams p) {
    using L = TmaLayout<kRows, kStages, kGroups>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t base = smem_addr(smem);
    const uint32_t full0 = base + L::kBarOffset;
    const uint32_t empty0 = full0 + 8 * kStages;
    volatile int32_t* meta = reinterpret_cast<volatile int32_t*>(smem + L::kMetaOffset);
    const uint32_t n_chunks = (p.n_heads + kRows - 1) / kRows;
    const uint64_t n_tiles = uint64_t(p.n_tokens) * n_chunks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kRows);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == L::kConsumerWarps) {
        // ---------------- producer warp (lane 0 issues; all lanes prefetch positions)
        const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
        const bool contiguous_heads = p.sx_h == kHeadDim;
        const uint64_t pol = policy_evict_first();
        auto load_pos = [&](uint64_t it) -> int64_t {
            const uint64_t tile = blockIdx.x + it * gridDim.x;
            return tile < n_tiles ? __ldg(p.positions + tile / n_chunks) : 0;
        };
        int64_t pos_cur = 0, pos_next = 0;
        uint32_t it = 0;
        bool ok = true;
        for (uint64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            if ((it & 31u) == 0) {
                pos_cur = it == 0 ? load_pos(lane) : pos_next;
                pos_next = load_pos(uint64_t(it) + 32 + lane);
            }
            const int64_t pos = __shfl_sync(kFull, pos_cur, it & 31u);
            const uint32_t s = it % kStages;
            const uint32_t ph = (it / kStages) & 1u;
            if (lane == 0) {
                ok = mbar_wait(empty0 + 8 * s, ph ^ 1u);
                if (ok) {
                    const uint32_t t = static_cast<uint32_t>(tile / n_chunks);
                    const uint32_t h0 = static_cast<uint32_t>(tile - uint64_t(t) * n_chunks) * kRows;
                    const uint32_t nrows = min(uint32_t(kRows), p.n_heads - h0);
                    const bool pos_ok =
                        static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
                    const uint32_t stage = base + s * L::kStageBytes;
                    meta[s] = pos_ok ? int32_t(nrows) : 0;
                    if (pos_ok) {
                        mbar_arrive_expect_tx(full0 + 8 * s, nrows * L::kRowBytes + L::kCsBytes);
                        const uint16_t* row0 =
                            x + int64_t(t) * p.sx_t + int64_t(h0) * p.sx_h;
                        if (contiguous_heads) {
                            bulk_g2s_hint(stage, row0, nrows * L::kRowBytes, full0 + 8 * s, pol);
                        } else {
                            for (uint32_t k = 0; k < nrows; ++k)
                                bulk_g2s_hint(stage + k * L::kRowBytes, row0 + int64_t(k) * p.sx_h,
                                              L::kRowBytes, full0 + 8 * s, pol);
                        }
                        bulk_g2s(stage + kRows * L::kRowBytes, p.cache + pos * kCacheWidth,
                                 L::kCsBytes, full0 + 8 * s);
                    } else {
                        if (p.error_flags) atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
                        mbar_arrive(full0 + 8 * s);  // phase completes with no data
                    }
                }
            }
            ok = __shfl_sync(kFull, ok, 0);
            if (!ok) break;
        }
        if (!ok) {
            if (lane == 0) {
                if (p.error_flags) atomicOr(p.error_flags, RQ_FLAG_TIMEOUT);
                // no copy may still be landing in this CTA's shared memory on exit
                const uint32_t first = it >= kStages ? it - kStages : 0;
                for (uint32_t j = first; j < it; ++j)
                    (void)mbar_wait(full0 + 8 * (j % kStages), (j / kStages) & 1u);
            }
        }
        return;
    }

    // ---------------- consumer warps: warp k of group g takes row k of the
    // stages of iterations g, g + kGroups, ...
    const int group = warp / kRows;
    const int k = warp - group * kRows;
    const int cs_off = (lane >= kRopeLane0 ? lane - kRopeLane0 : 0) * 16;
    uint32_t it = group;
    for (uint64_t tile = blockIdx.x + uint64_t(group) * gridDim.x; tile < n_tiles;
         tile += uint64_t(kGroups) * gridDim.x, it += kGroups) {
        const uint32_t s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        const bool got = mbar_wait(full0 + 8 * s, ph);
        if (!__all_sync(kFull, got)) {
            if (lane == 0 && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_TIMEOUT);
            return;
        }
        const int nrows = meta[s];
        const bool live = k < nrows;
        const uint32_t stage = base + s * L::kStageBytes;
        RowRegs in;
        if (live) {
            const uint32_t row = stage + k * L::kRowBytes;
            in.a = lds16(row + 16 * lane);
            in.b = lds16(row + 512 + 16 * lane);
            if (lane >= kRopeLane0) {
                const uint32_t cs = stage + kRows * L::kRowBytes;
                in.c = lds16f(cs + cs_off);
                in.s = lds16f(cs + 128 + cs_off);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);  // stage free: the row is in registers
        if (live) {
            const uint32_t t = static_cast<uint32_t>(tile / n_chunks);
            const uint32_t h = static_cast<uint32_t>(tile - uint64_t(t) * n_chunks) * kRows + k;
            const int64_t r = int64_t(t) * p.n_heads + h;
            const RowOut o = rope_quant_row<true>(in, lane, p.eps);
            uint8_t* dst = p.out + r * kHeadDim;
            st_stream8(dst + 8 * lane, o.qa.x, o.qa.y);
            st_stream8(dst + kHalf + 8 * lane, o.qb.x, o.qb.y);
            const float s1 = __shfl_sync(kFull, o.sa, 16);
            const float s3 = __shfl_sync(kFull, o.sb, 16);
            if (lane == 0) st_stream16f(p.scales + r * 4, o.sa, s1, o.sb, s3);
        }
    }
}

// ------------------------------------------------------------------ insert

template <int kRows>
__global__ void __launch_bounds__(kInsThreads)
rope_fp8_quant_insert_kernel(InsParams p) {
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    const uint16_t* __restrict__ kv = static_cast<const uint16_t*>(p.kv);
    const int cs_col = (lane >= kRopeLane0 ? lane - kRopeLane0 : 0) * 4;
    const int64_t n_slots = p.num_blocks * p.block_size;

    for (uint32_t t0 = warp * kRows; t0 < p.n_tokens; t0 += n_warps * kRows) {
        RowRegs in[kRows];
        int64_t slot[kRows];
        bool live[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const uint32_t t = t0 + i;
            live[i] = false;
            slot[i] = -1;
            if (t < p.n_tokens) {
                const int64_t pos = __ldg(p.positions + t);
                slot[i] = __ldg(p.slot_mapping + t);
                const bool pos_ok =
                    static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
                const bool slot_ok = slot[i] < n_slots;
                live[i] = pos_ok && slot_ok && slot[i] >= 0;
                if (live[i]) {
                    const uint16_t* row = kv + static_cast<int64_t>(t) * p.skv;
                    in[i].a = ld_stream16(row + 8 * lane);
                    in[i].b = ld_stream16(row + kHalf + 8 * lane);
                    if (lane >= kRopeLane0) {
                        const float* cs = p.cache + pos * kCacheWidth + cs_col;
                        in[i].c = ld_shared_ro16(cs);
                        in[i].s = ld_shared_ro16(cs + kHalfRope);
                    }
                } else if (lane == 0 && p.error_flags && (!pos_ok || !slot_ok)) {
                    atomicOr(p.error_flags,
                             (pos_ok ? 0u : RQ_FLAG_POSITION_RANGE) |
                                 (slot_ok ? 0u : RQ_FLAG_SLOT_RANGE));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            if (!live[i]) continue;
            const RowOut o = rope_quant_row<false>(in[i], lane, p.eps);
            const int64_t blk = slot[i] / p.block_size;
            const int64_t off = slot[i] - blk * p.block_size;
            uint8_t* rec = p.k_cache + blk * p.block_stride + off * kRecordBytes;
            st_stream8(rec + 8 * lane, o.qa.x, o.qa.y);
            st_stream8(rec + kHalf + 8 * lane, o.qb.x, o.qb.y);
            const float s1 = __shfl_sync(kFull, o.sa, 16);
            const float s3 = __shfl_sync(kFull, o.sb, 16);
            if (lane == 0) st_stream16f(rec + kHeadDim, o.sa, s1, o.sb, s3);
        }
    }
}

// ------------------------------------------------------------------ launchers

namespace {

// Resident CTAs per SM of each kernel variant, queried once per device and
// variant (thread-local: no locking on the launch path).
constexpr int kMaxDevices = 64;
enum Variant { kInv1, kInv2, kIns2, kVariants };

template <typename K>
int resident_blocks(int device, Variant v, K kernel, int threads) {
    static thread_local int cache[kMaxDevices][kVariants];
    if (device < 0 || device >= kMaxDevices) device = 0;
    int& n = cache[device][v];
    if (n == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess ||
            n < 1)
            n = 1;
    }
    return n;
}

// Persistent grid: enough CTAs for the work, at most one full wave.
int grid_size(int64_t units, int units_per_block, int sm_count, int resident) {
    const int64_t need = (units + units_per_block - 1) / units_per_block;
    const int64_t cap = int64_t(sm_count) * resident;
    return static_cast<int>(need < cap ? need : cap);
}

}  // namespace

namespace {

constexpr int kTmaRows = 8;
constexpr int kTmaStages = 12;
constexpr int kTmaGroups = 2;
using TmaL = TmaLayout<kTmaRows, kTmaStages, kTmaGroups>;
#define RQ_TMA_KERNEL inv_rope_fp8_quant_tma_kernel<kTmaRows, kTmaStages, kTmaGroups>

// Dynamic shared memory above 48 KiB must be enabled per device.
cudaError_t enable_tma_smem(int device) {
    static thread_local bool done[kMaxDevices] = {false};
    const int d = (device >= 0 && device < kMaxDevices) ? device : 0;
    if (done[d]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(RQ_TMA_KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TmaL::kBytes);
    // ask for the largest shared-memory carveout so two CTAs fit per SM
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(RQ_TMA_KERNEL, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess) done[d] = true;
    return e;
}

int tma_resident_blocks(int device) {
    static thread_local int cache[kMaxDevices] = {0};
    const int d = (device >= 0 && device < kMaxDevices) ? device : 0;
    if (cache[d] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, RQ_TMA_KERNEL, TmaL::kThreads,
                                                          TmaL::kBytes) != cudaSuccess ||
            n < 1)
            n = 1;
        cache[d] = n;
    }
    return cache[d];
}

}  // namespace

cudaError_t launch_inv_rope_fp8_quant(const InvParams& p, const DeviceInfo& dev, int variant,
                                      cudaStream_t stream) {
    constexpr int kWarps = kInvThreads / 32;
    if (variant == kInvAuto)
        variant = int64_t(p.n_rows) >= int64_t(dev.sm_count) * 64 ? kInvTmaPipeline : kInvWarpRows;
    if (variant == kInvTmaPipeline) {
        cudaError_t e = enable_tma_smem(dev.ordinal);
        if (e != cudaSuccess) return e;
        const int64_t tiles = int64_t(p.n_tokens) * ((p.n_heads + kTmaRows - 1) / kTmaRows);
        const int grid = grid_size(tiles, 1, dev.sm_count, tma_resident_blocks(dev.ordinal));
        RQ_TMA_KERNEL<<<grid, TmaL::kThreads, TmaL::kBytes, stream>>>(p);
        return cudaGetLastError();
    }
    // warp-rows kernel: two rows in flight per warp when the grid fills the
    // GPU, one otherwise (decode-sized calls spread over more warps)
    if (int64_t(p.n_rows) >= int64_t(dev.sm_count) * kWarps * 4) {
        auto k = inv_rope_fp8_quant_kernel<2>;
        const int res = resident_blocks(dev.ordinal, kInv2, k, kInvThreads);
        k<<<grid_size(p.n_rows, kWarps * 2, dev.sm_count, res), kInvThreads, 0, stream>>>(p);
    } else {
        auto k = inv_rope_fp8_quant_kernel<1>;
        const int res = resident_blocks(dev.ordinal, kInv1, k, kInvThreads);
        k<<<grid_size(p.n_rows, kWarps * 1, dev.sm_count, res), kInvThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_rope_fp8_quant_insert(const InsParams& p, const DeviceInfo& dev,
                                         cudaStream_t stream) {
    constexpr int kWarps = kInsThreads / 32;
    auto k = rope_fp8_quant_insert_kernel<2>;
    const int res = resident_blocks(dev.ordinal, kIns2, k, kInsThreads);
    k<<<grid_size(p.n_tokens, kWarps * 2, dev.sm_count, res), kInsThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rq
