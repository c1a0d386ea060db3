// rq_stream.cu -- the inverse-RoPE + block-FP8 quant kernel built as one
// independent TMA stream per warp (sm_103a), and its launcher: the
// RQ_INV_STREAM variant of the plain op (contiguous [N, G, hpg*512] codes and
// [N, G, hpg*4] fp32 scales). The default kernel of the plain op, and of
// every layout, is the warp-rows kernel in rq_kernels.cu.
//
// Every warp owns a private ring of kStages shared-memory stages. A stage
// holds one tile -- kRows consecutive heads of one token (1 KiB each) plus
// the token's 256-byte cos|sin row -- brought in by 1-D bulk copies (TMA,
// cp.async.bulk) that complete on the stage's mbarrier. The warp keeps
// kStages tiles in flight: it waits for the oldest stage, computes and
// stores its rows, then re-arms that same stage with the tile kStages ahead.
// A tile's codes and scales are gathered in one of two shared-memory output
// buffers and leave with two bulk stores (4 KiB of codes and 128 bytes of
// scales for an 8-head tile), so the writes too are large contiguous copies.
// There is no producer warp and no barrier shared between warps, so the
// bytes in flight per SM (resident warps x kStages x kRows KiB) cost no
// registers and no cross-warp handshakes.
//
// Arithmetic per row follows "[vllm] 한 프로그램이 4개 head를 처리하게 하라:
// DeepSeek-V4 inverse RoPE + FP8 quant 커널 3.5배 가속기" (vLLM PR #63540
// analysis): S2 for the rotation (partner in registers), S3 for the block
// amax; the scale is 2^ceil(log2(amax/448)) as in "[vllm] vLLM의 GLM5.2 성능
// 최적화" S1. Lane layout: the block-interleaved layout of rq_device.cuh.
#include "rq_device.cuh"
#include "rq_launch.h"
#include "rq_tma.cuh"

#ifndef RQ_STREAM_ROWS
#define RQ_STREAM_ROWS 8
#endif
#ifndef RQ_STREAM_STAGES
#define RQ_STREAM_STAGES 2
#endif

namespace rq {

namespace {

#ifndef RQ_STREAM_WARPS
#define RQ_STREAM_WARPS 8
#endif
constexpr int kStreamWarps = RQ_STREAM_WARPS;  // warps per CTA; each runs its own ring

template <int kRows, int kStages>
struct Ring {
    static constexpr uint32_t kRowBytes = kHeadDim * 2;       // one head row of bf16
    static constexpr uint32_t kCsBytes = kCacheWidth * 4;     // cos | sin row
    static constexpr uint32_t kStageBytes = kRows * kRowBytes + kCsBytes;
    static constexpr uint32_t kBarBytes = 128;                // the ring's mbarriers, padded
    static constexpr uint32_t kOutBytes = kRows * (kHeadDim + 16);  // a tile's codes + scales
    static constexpr uint32_t kWarpBytes = kBarBytes + kStages * kStageBytes + 2 * kOutBytes;
    static constexpr uint32_t kCtaBytes = kStreamWarps * kWarpBytes;
    static_assert(kStages * 8 <= int(kBarBytes), "too many stages for the barrier block");
    static_assert(kStageBytes % 128 == 0, "stages must stay 128-byte aligned");
    static_assert(kOutBytes % 16 == 0, "output buffers must stay 16-byte aligned");
};

// A warp's tiles are warp, warp + n_warps, warp + 2 n_warps, ...; this walks
// them as (token t, head chunk c) without dividing per tile.
struct TileWalk {
    uint32_t t, c, dt, dc, n_chunks;
    __device__ __forceinline__ TileWalk(uint32_t first, uint32_t n_warps, uint32_t chunks)
        : n_chunks(chunks) {
        t = first / chunks;
        c = first - t * chunks;
        dt = n_warps / chunks;
        dc = n_warps - dt * chunks;
    }
    __device__ __forceinline__ void next() {
        c += dc;
        t += dt;
        if (c >= n_chunks) {
            c -= n_chunks;
            ++t;
        }
    }
};

}  // namespace

// kRows heads per tile (n_heads need not be a multiple: the last tile of a
// token is short), kStages tiles in flight per warp.
template <int kRows, int kStages>
__global__ void __launch_bounds__(kStreamWarps * 32)
inv_rope_fp8_quant_stream_kernel(InvParams p) {
    pdl_wait();
    pdl_launch_dependents();
    using R = Ring<kRows, kStages>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const uint32_t wib = threadIdx.x >> 5;
    const uint32_t warp = blockIdx.x * kStreamWarps + wib;
    const uint32_t n_warps = gridDim.x * kStreamWarps;
    const uint32_t n_chunks = (p.n_heads + kRows - 1) / kRows;
    const uint32_t n_tiles = p.n_tokens * n_chunks;  // <= n_tokens * n_heads < 2^31
    if (warp >= n_tiles) return;
    const uint32_t n_mine = (n_tiles - warp + n_warps - 1) / n_warps;
    const uint32_t bar0 = smem_addr(smem) + wib * R::kWarpBytes;
    const uint32_t stage0 = bar0 + R::kBarBytes;
    const uint32_t out0 = stage0 + kStages * R::kStageBytes;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();

    const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
    const bool contiguous = p.sx_h == kHeadDim;
    const uint64_t pol = policy_evict_first();

    // ---- issue side: tile j of this warp into stage j % kStages
    TileWalk iw(warp, n_warps, n_chunks);
    int64_t pos_pf = 0;   // lane i: position of the tile i issues after the last refresh
    uint32_t valid = 0;   // bit s: stage s holds a tile whose position is in range
    auto issue = [&](uint32_t j) {
        if ((j & 31u) == 0) {
            const uint64_t ahead = uint64_t(warp) + (uint64_t(j) + uint64_t(lane)) * n_warps;
            pos_pf = ahead < n_tiles ? __ldg(p.positions + uint32_t(ahead) / n_chunks) : 0;
        }
        const int64_t pos = __shfl_sync(kFull, pos_pf, j & 31u);
        const uint32_t s = j % kStages;
        const bool ok = static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
        valid = ok ? (valid | (1u << s)) : (valid & ~(1u << s));
        // test-only fault injection: warp 0 leaves its first tile's stage
        // unarmed, so the wait for it runs out
        const bool starve = (p.wait.inject & kInjectStreamStage) && warp == 0 && j == 0;
        if (lane == 0 && !starve) {
            const uint32_t bar = bar0 + 8 * s;
            if (ok) {
                const uint32_t h0 = iw.c * kRows;
                const uint32_t nrows = min(uint32_t(kRows), p.n_heads - h0);
                const uint32_t dst = stage0 + s * R::kStageBytes;
                mbar_arrive_expect_tx(bar, nrows * R::kRowBytes + R::kCsBytes);
                const uint16_t* row0 = x + int64_t(iw.t) * p.sx_t + int64_t(h0) * p.sx_h;
                if (contiguous) {
                    bulk_g2s_hint(dst, row0, nrows * R::kRowBytes, bar, pol);
                } else {
                    for (uint32_t k = 0; k < nrows; ++k)
                        bulk_g2s_hint(dst + k * R::kRowBytes, row0 + int64_t(k) * p.sx_h,
                                      R::kRowBytes, bar, pol);
                }
                bulk_g2s(dst + kRows * R::kRowBytes, p.cache + pos * kCacheWidth, R::kCsBytes, bar);
            } else {
                if (p.error_flags) atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
                mbar_arrive(bar);  // the phase completes with no data
            }
        }
        iw.next();
    };
    const uint32_t prologue = n_mine < uint32_t(kStages) ? n_mine : uint32_t(kStages);
    for (uint32_t j = 0; j < prologue; ++j) issue(j);

    // ---- consume side
    TileWalk cw(warp, n_warps, n_chunks);
    const int ca = chunk_a(lane);
    const bool rope_lane = lane >= kRopeLane0;
    const uint32_t cs_off = uint32_t(rope_lane ? lane - kRopeLane0 : 0) * 16;
    uint32_t j = 0;
    bool ok = true;
    for (; j < n_mine; ++j) {
        const uint32_t s = j % kStages;
        ok = mbar_wait(bar0 + 8 * s, (j / kStages) & 1u, p.wait.spin_limit);
        if (!__all_sync(kFull, ok)) {
            ok = false;
            break;
        }
        if ((valid >> s) & 1u) {
            const uint32_t st = stage0 + s * R::kStageBytes;
            const uint32_t h0 = cw.c * kRows;
            const uint32_t nrows = min(uint32_t(kRows), p.n_heads - h0);
            float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f), s4 = c4;
            if (rope_lane) {
                c4 = lds16f(st + kRows * R::kRowBytes + cs_off);
                s4 = lds16f(st + kRows * R::kRowBytes + kHalfRope * 4 + cs_off);
            }
            // contiguous output: the tile's codes and scales are contiguous
            uint8_t* head0 = p.out + (int64_t(cw.t) * p.n_heads + h0) * kHeadDim;
            float* scale0 = p.scales + (int64_t(cw.t) * p.n_heads + h0) * 4;
            // the tile's codes and scales are gathered in output buffer j % 2
            // and leave with two bulk stores: the buffer's previous stores
            // (tile j - 2, one commit group older than the newest) must have
            // finished reading it
            const uint32_t ob = out0 + (j & 1u) * R::kOutBytes;
            const uint32_t osc = ob + kRows * kHeadDim;
            if (lane == 0) bulk_wait_read_all_but_newest();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                if (uint32_t(i) < nrows) {
                    const uint32_t row = st + i * R::kRowBytes;
                    const uint4 a = lds16(row + 16 * ca);
                    const uint4 b = lds16(row + 16 * (ca + 8));
                    float scale;
                    const uint4 q = rope_quant_row<true>(a, b, rope_lane, c4, s4, p.eps, &scale);
                    const uint32_t o = ob + i * kHeadDim;
                    sts8(o + 8 * ca, q.x, q.y);
                    sts8(o + 8 * (ca + 8), q.z, q.w);
                    if ((lane & 7) == 0) sts4f(osc + i * 16 + (lane >> 3) * 4, scale);
                }
            }
            fence_proxy_async_smem();  // this lane's writes, visible to the bulk stores
            __syncwarp();
            if (lane == 0) {
                bulk_s2g(head0, ob, nrows * kHeadDim);
                bulk_s2g(scale0, osc, nrows * 16);
            }
        }
        if (lane == 0) bulk_commit();  // one group per tile (empty if skipped)
        cw.next();
        __syncwarp();  // every lane has read stage s: it may be refilled
        if (j + kStages < n_mine) issue(j + kStages);
    }
    if (lane == 0) bulk_wait_all();  // no bulk store may read smem at exit
    __syncwarp();
    if (!ok) {
        // a wait gave up (never expected): report it, and let no copy still
        // land in this warp's stages after the CTA exits
        if (lane == 0) {
            if (p.error_flags) atomicOr(p.error_flags, RQ_FLAG_TIMEOUT);
            const uint32_t end = j + kStages < n_mine ? j + kStages : n_mine;
            for (uint32_t d = j; d < end; ++d)
                (void)mbar_wait(bar0 + 8 * (d % kStages), (d / kStages) & 1u, p.wait.spin_limit);
        }
        __syncwarp();
    }
}

namespace {

using StreamRing = Ring<RQ_STREAM_ROWS, RQ_STREAM_STAGES>;
constexpr int kMaxDevices = 64;

// Opt in to more than 48 KiB of dynamic shared memory (once per device and
// kernel instance) and read the resulting residency.
cudaError_t stream_setup(int device, int* resident) {
    auto kernel = inv_rope_fp8_quant_stream_kernel<RQ_STREAM_ROWS, RQ_STREAM_STAGES>;
    static thread_local int cache[kMaxDevices] = {0};
    const int d = (device >= 0 && device < kMaxDevices) ? device : 0;
    if (cache[d] == 0) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(StreamRing::kCtaBytes));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     int(cudaSharedmemCarveoutMaxShared));
        if (e != cudaSuccess) return e;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kStreamWarps * 32,
                                                          StreamRing::kCtaBytes) != cudaSuccess ||
            n < 1)
            n = 1;
        cache[d] = n;
    }
    *resident = cache[d];
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_inv_rope_fp8_quant_stream(const InvParams& p, const DeviceInfo& dev,
                                             cudaStream_t stream) {
    int resident = 1;
    cudaError_t e = stream_setup(dev.ordinal, &resident);
    if (e != cudaSuccess) return e;
    const int64_t chunks = (p.n_heads + RQ_STREAM_ROWS - 1) / RQ_STREAM_ROWS;
    const int64_t warps_needed = int64_t(p.n_tokens) * chunks;
    const int64_t ctas_needed = (warps_needed + kStreamWarps - 1) / kStreamWarps;
    const int64_t cap = int64_t(dev.sm_count) * resident;
    const int grid = static_cast<int>(ctas_needed < cap ? ctas_needed : cap);
    return launch_pdl(inv_rope_fp8_quant_stream_kernel<RQ_STREAM_ROWS, RQ_STREAM_STAGES>, grid,
                      kStreamWarps * 32, StreamRing::kCtaBytes, stream, p);
}

}  // namespace rq
