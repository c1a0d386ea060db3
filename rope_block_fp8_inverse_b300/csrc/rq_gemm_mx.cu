// rq_gemm_mx.cu -- the consumer grouped FP8 GEMM with UE8M0 block scales on
// the block-scaled 5th-generation tensor-core MMA (tcgen05.mma
// kind::mxf8f6f4, one UE8M0 scale code per row and 32-wide K step).
//
// The inverse-RoPE page's packed-scale output ("[vllm] 한 프로그램이 4개 head를
// 처리하게 하라: DeepSeek-V4 inverse RoPE + FP8 quant 커널 3.5배 가속기", S3:
// four UE8M0 codes per head in one 32-bit word) is exactly the scale operand
// this MMA reads: the word of head h covers the group's K blocks 4h..4h+3,
// and the instruction descriptor's scale-factor byte (kt % 4) picks block kt's
// code out of it. Weight scales are one code per 128 x 128 block. The tensor
// cores apply both scales inside the K loop, so the whole K reduction of a
// tile accumulates in TMEM and is read back once, by the epilogue: nothing is
// folded in registers per K tile (which is what bounds the fp32-scale GEMM of
// rq_gemm.cu).
//
// For every group g:  Y[:, g, :] = (A_g * 2^(sa - 127)) @ (W_g * 2^(sw - 127))^T,
// Y bf16 [M, G, n_out].
//
// Persistent CTAs (one per SM) walk the 128 x 256 output tiles t =
// blockIdx.x, blockIdx.x + gridDim.x, ...; the N tiles of one (M tile,
// group) are neighbours in the walk, so CTAs running at the same time read
// the same A rows, and the few W tiles of a group, from L2. Each CTA loads
// its own operands with plain tensor-map copies into its own shared memory.
//   warp 0   one lane: tensor-map TMA of each 128-wide K step of A (16 KiB)
//            and W (32 KiB) into a 4-stage ring;
//   warp 1   allocates TMEM; one lane copies each tile's scale codes from
//            shared memory to TMEM (tcgen05.cp) and issues the MMAs
//            (M = 128, N = 256, 4 x K = 32 per K step);
//   warp 2   builds each tile's scale-code atoms in shared memory (double
//            buffered), one tile ahead of the MMA;
//   warps 4..11  epilogue: thread = output row (TMEM lane 32 * (warp % 4) +
//            lane), 128 of the 256 columns; reads the finished accumulator,
//            releases it to the next tile's MMAs, then stores bf16.
// TMEM (512 columns): accumulator 0..255, A scale codes 256..319 (two tiles),
// W scale codes 320..447 (two tiles). Every wait is bounded; a role that gives
// up raises a shared abort flag that the others poll, so the CTA still drains
// its copies, frees TMEM and exits, and the call reports RQ_FLAG_TIMEOUT.
#include "rq_device.cuh"
#include "rq_launch.h"
#include "rq_tma.cuh"
#include "rq_umma.cuh"

namespace rq {

namespace {

constexpr int kMxBM = 128, kMxBN = 256, kMxBK = 128;
constexpr int kMxStages = 4;
constexpr int kMxMaxHeads = 8;                                  // K up to 8 x 512 = 4096
constexpr uint32_t kMxATile = kMxBM * kMxBK;                    // 16 KiB
constexpr uint32_t kMxWTile = kMxBN * kMxBK;                    // 32 KiB
constexpr uint32_t kSfAtom = 512;                               // 32 rows x 16 bytes
constexpr uint32_t kSfaBytes = kMxMaxHeads * kSfAtom;           // one atom per head
constexpr uint32_t kSfbBytes = 2 * kMxMaxHeads * kSfAtom;       // per head: two N halves
constexpr uint32_t kSfBufBytes = kSfaBytes + kSfbBytes;
constexpr uint32_t kMxOffW = kMxStages * kMxATile;
constexpr uint32_t kMxOffSf = kMxOffW + kMxStages * kMxWTile;
constexpr uint32_t kMxOffBar = kMxOffSf + 2 * kSfBufBytes;
// full[S], empty[S], sf_full[2], sf_empty[2], tfull, tempty, done
constexpr uint32_t kMxNumBars = 2 * kMxStages + 4 + 3;
constexpr uint32_t kMxOffSlot = kMxOffBar + 8 * kMxNumBars;     // TMEM base, abort flag
constexpr uint32_t kMxSmem = kMxOffSlot + 16 + 1024;            // + room to align to 1 KiB
constexpr int kMxThreads = 384;
constexpr int kMxEpiWarp0 = 4;
constexpr int kMxEpiThreads = kMxThreads - 32 * kMxEpiWarp0;    // 256
constexpr uint32_t kTmemSfa = 256;     // + 32 per buffer: 4 columns per head word
constexpr uint32_t kTmemSfb = 320;     // + 64 per buffer: 8 columns per head word
constexpr uint32_t kMxTmemCols = 512;
constexpr uint32_t kUe8m0One4 = 0x7f7f7f7fu;                    // four codes of 1.0

static_assert(kMxSmem <= 232448, "shared memory per CTA");
static_assert(kTmemSfb + 2 * 8 * kMxMaxHeads <= kMxTmemCols, "TMEM columns");

// Poll an mbarrier phase; give up after `limit` polls (raising `abort`)
// or as soon as another role has raised it.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile uint32_t* abort, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort) return false;
    }
    *abort = 1u;
    return false;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                      uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

struct MxTile {
    int mt, g, nt;
};

// Tile t of the walk: N tiles innermost, then groups, then M tiles.
__device__ __forceinline__ MxTile mx_tile(int t, int n_nt, int groups) {
    MxTile x;
    x.nt = t % n_nt;
    const int r = t / n_nt;
    x.g = r % groups;
    x.mt = r / groups;
    return x;
}

}  // namespace

__global__ void __launch_bounds__(kMxThreads, 1)
grouped_fp8_gemm_ue8m0_kernel(const __grid_constant__ CUtensorMap tma_a,
                              const __grid_constant__ CUtensorMap tma_w, MxGemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t a0 = base, w0 = base + kMxOffW, sf0 = base + kMxOffSf, bar0 = base + kMxOffBar;
    const uint32_t full0 = bar0, empty0 = bar0 + 8 * kMxStages;
    const uint32_t sfull0 = bar0 + 16 * kMxStages, sempty0 = sfull0 + 16;
    const uint32_t tfull = sempty0 + 16, tempty = tfull + 8, done = tempty + 8;
    uint8_t* slot = smem_raw + (base + kMxOffSlot - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(slot);
    volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(slot + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_kt = p.k / kMxBK, n_heads = p.k / 512;
    const int n_nt = (p.n_out + kMxBN - 1) / kMxBN;
    const int n_tiles = ((p.m + kMxBM - 1) / kMxBM) * p.groups * n_nt;
    const uint32_t lim = p.wait.spin_limit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sfull0 + 8 * b, 1);
            mbar_init(sempty0 + 8 * b, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, kMxEpiThreads);
        mbar_init(done, 1);
        *abort = 0u;
        mbar_init_fence();
    }
    if (warp == 1) {
        umma::tmem_alloc(base + kMxOffSlot, kMxTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // test-only fault injection: CTA 0's producer issues nothing
        const bool starve = (p.wait.inject & kInjectGemmLoads) && blockIdx.x == 0;
        if (lane == 0 && !starve) {
            uint32_t it = 0;  // K steps issued
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const MxTile x = mx_tile(t, n_nt, p.groups);
                for (int kt = 0; kt < n_kt; ++kt) {
                    const uint32_t s = it % kMxStages, ph = (it / kMxStages) & 1u;
                    if (!wait_or_abort(empty0 + 8 * s, ph ^ 1u, abort, lim)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full0 + 8 * s, kMxATile + kMxWTile);
                    umma::tma_load_2d(a0 + s * kMxATile, &tma_a, x.g * p.k + kt * kMxBK,
                                      x.mt * kMxBM, full0 + 8 * s);
                    umma::tma_load_2d(w0 + s * kMxWTile, &tma_w, kt * kMxBK,
                                      x.g * p.n_out + x.nt * kMxBN, full0 + 8 * s);
                    ++it;
                }
            }
            // Let the copies still in flight land before the CTA exits (on the
            // normal path every one of them was already consumed).
            for (uint32_t j = it > uint32_t(kMxStages) ? it - kMxStages : 0u; j < it; ++j)
                if (!mbar_wait(full0 + 8 * (j % kMxStages), (j / kMxStages) & 1u, lim)) *abort = 1u;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0, i = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++i) {
                const uint32_t b = i & 1u;
                if (!wait_or_abort(sfull0 + 8 * b, (i >> 1) & 1u, abort, lim) ||
                    !wait_or_abort(tempty, (i & 1u) ^ 1u, abort, lim))
                    break;
                umma::fence_after_sync();
                const uint32_t sfa_t = tmem + kTmemSfa + 32 * b, sfb_t = tmem + kTmemSfb + 64 * b;
                const uint32_t sfa = sf0 + b * kSfBufBytes, sfb = sfa + kSfaBytes;
                for (int h = 0; h < n_heads; ++h) {
                    umma::cp_32x128b_warpx4(sfa_t + 4 * h, umma::smem_desc_plain(sfa + h * kSfAtom));
                    umma::cp_32x128b_warpx4(sfb_t + 8 * h,
                                            umma::smem_desc_plain(sfb + 2 * h * kSfAtom));
                    umma::cp_32x128b_warpx4(sfb_t + 8 * h + 4,
                                            umma::smem_desc_plain(sfb + (2 * h + 1) * kSfAtom));
                }
                umma::commit(sempty0 + 8 * b);  // the atoms are free once copied
                for (int kt = 0; kt < n_kt; ++kt) {
                    const uint32_t s = it % kMxStages, ph = (it / kMxStages) & 1u;
                    if (!wait_or_abort(full0 + 8 * s, ph, abort, lim)) {
                        ok = false;
                        break;
                    }
                    umma::fence_after_sync();
                    const uint64_t ad = umma::smem_desc_sw128(a0 + s * kMxATile);
                    const uint64_t wd = umma::smem_desc_sw128(w0 + s * kMxWTile);
                    const uint32_t idesc = umma::idesc_mx_e4m3_ue8m0(kMxBM, kMxBN, uint32_t(kt & 3));
                    const uint32_t h = uint32_t(kt >> 2);
#pragma unroll
                    for (int k = 0; k < kMxBK / 32; ++k)  // K = 32 bytes of e4m3 per MMA
                        umma::mma_mxf8f6f4(tmem, ad + 2 * k, wd + 2 * k, idesc, sfa_t + 4 * h,
                                           sfb_t + 8 * h, (kt | k) != 0);
                    umma::commit(empty0 + 8 * s);
                    ++it;
                }
                if (ok) umma::commit(tfull);
            }
            umma::commit(done);
            if (!mbar_wait(done, 0, lim)) *abort = 1u;  // nothing in flight before teardown
        }
    } else if (warp == 2) {
        uint32_t i = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            const MxTile x = mx_tile(t, n_nt, p.groups);
            const uint32_t b = i & 1u;
            if (!__all_sync(kFull, wait_or_abort(sempty0 + 8 * b, ((i >> 1) & 1u) ^ 1u, abort, lim)))
                break;
            const uint32_t sfa = sf0 + b * kSfBufBytes, sfb = sfa + kSfaBytes;
            // A: atom h, 16-byte row `lane` = the words of rows lane + 32c, c = 0..3
            uint32_t wa[kMxMaxHeads][4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int row = x.mt * kMxBM + lane + 32 * c;
                const uint32_t* src = p.a_sf + (int64_t(row) * p.groups + x.g) * n_heads;
#pragma unroll
                for (int h = 0; h < kMxMaxHeads; ++h)
                    wa[h][c] = (h < n_heads && row < p.m) ? __ldg(src + h) : kUe8m0One4;
            }
#pragma unroll
            for (int h = 0; h < kMxMaxHeads; ++h)
                if (h < n_heads)
                    sts16(sfa + h * kSfAtom + 16 * lane, wa[h][0], wa[h][1], wa[h][2], wa[h][3]);
            // W: one code per 128 x 128 block, the same for every row of an atom;
            // bytes b of the word = K blocks 4h + b
            const int n_blk = p.n_out / 128;
            for (int h = 0; h < n_heads; ++h) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int nb = 2 * x.nt + half;
                    uint32_t w = kUe8m0One4;
                    if (nb < n_blk) {
                        const uint8_t* src = p.w_sf + (int64_t(x.g) * n_blk + nb) * n_kt + 4 * h;
                        w = uint32_t(__ldg(src)) | (uint32_t(__ldg(src + 1)) << 8) |
                            (uint32_t(__ldg(src + 2)) << 16) | (uint32_t(__ldg(src + 3)) << 24);
                    }
                    sts16(sfb + (2 * h + half) * kSfAtom + 16 * lane, w, w, w, w);
                }
            }
            fence_proxy_async_smem();  // generic-proxy writes -> tcgen05.cp reads
            __syncwarp();
            if (lane == 0) mbar_arrive(sfull0 + 8 * b);
        }
    } else if (warp >= kMxEpiWarp0) {
        const int quad = warp & 3;
        const int half = (warp - kMxEpiWarp0) >> 2;
        uint32_t i = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            const MxTile x = mx_tile(t, n_nt, p.groups);
            // the warp leaves together: the TMEM loads below are warp-collective
            if (!__all_sync(kFull, wait_or_abort(tfull, i & 1u, abort, lim))) break;
            umma::fence_after_sync();
            uint32_t packed[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float d[32];
                umma::ld32(tmem + (uint32_t(quad * 32) << 16) + half * 128 + c * 32, d);
#pragma unroll
                for (int j = 0; j < 16; ++j) packed[c * 16 + j] = bf16x2(d[2 * j], d[2 * j + 1]);
            }
            umma::fence_before_sync();
            mbar_arrive(tempty);  // the accumulator may take the next tile's MMAs
            const int row = x.mt * kMxBM + quad * 32 + lane;
            const int col = x.nt * kMxBN + half * 128;
            if (row < p.m && col < p.n_out) {
                uint16_t* y = p.y + (int64_t(row) * p.groups + x.g) * p.n_out + col;
#pragma unroll
                for (int j = 0; j < 64; j += 4)
                    *reinterpret_cast<uint4*>(y + 2 * j) =
                        make_uint4(packed[j], packed[j + 1], packed[j + 2], packed[j + 3]);
            }
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_TIMEOUT);
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kMxTmemCols);
    }
}

// ------------------------------------------------------------------ few tokens

// Decode-sized calls (few tokens): the 128 x 256 tiles above leave all but a
// handful of SMs idle (one M tile x groups x N tiles CTAs), each streaming its
// W tiles at one SM's feed rate. This kernel swaps the operands and splits K:
//   MMA A = W (128 output rows of one group), MMA B = the tokens (N = up to 64
//   tokens, padded to a multiple of 16 with rows the tensor map reads as
//   zeros), D[output row, token] in TMEM; the UE8M0 scales are applied in the
//   MMA as above, with the roles of the two scale operands exchanged;
//   a cluster of kSplit CTAs shares one (token tile, group, 128-row) tile,
//   CTA r taking the r-th of kSplit equal runs of K steps, so the call spreads
//   over kSplit times as many CTAs;
//   launched with programmatic dependent launch: barriers, TMEM and an L2
//   prefetch of the CTA's W tiles are set up while the previous kernel
//   finishes; after the dependency wait every CTA issues all of its K steps'
//   copies at once (no ring reuse), one thread issues the MMAs, and the four
//   warps read the partial tile from TMEM; after a cluster barrier (every
//   CTA's operands consumed) each thread stores its row of the partial into
//   the shared memory of the CTA that owns the row (128 / kSplit rows each;
//   slot = this CTA's rank) with remote stores, and after a second one each
//   CTA sums its rows' kSplit partials, in rank order, from its own shared
//   memory and stores them as bf16.
// Every mbarrier wait is bounded (as above, a timeout raises RQ_FLAG_TIMEOUT);
// each CTA's path to both cluster barriers is straight-line code.
constexpr int kSmRows = 128;                      // W rows per tile (the MMA's M)
constexpr int kSmMaxTok = 64;                     // tokens per tile (the MMA's N, at most)
constexpr int kSmMaxHeads = 3;                    // scale words a CTA's K steps touch, at most
constexpr uint32_t kSmWTile = kSmRows * kMxBK;    // 16 KiB
constexpr uint32_t kSmStage = kSmWTile + kSmMaxTok * kMxBK;  // + 8 KiB of tokens
constexpr int kSmThreads = 128;
constexpr uint32_t kSmTmemCols = 128;             // accumulator 0..63, W codes 64.., tokens' 96..
constexpr uint32_t kSmTmemSfw = 64, kSmTmemSfx = 96;

template <int kSplit>
struct SmLayout {
    static constexpr int kMaxSteps = 4096 / kMxBK / kSplit;           // K steps per CTA, at most
    static constexpr int kRowsPer = kSmRows / kSplit;                  // rows each CTA sums
    static constexpr uint32_t kOffSf = kMaxSteps * kSmStage;
    static constexpr uint32_t kOffBar = kOffSf + 2 * kSmMaxHeads * kSfAtom;
    static constexpr uint32_t kOffSlot = kOffBar + 8 * (kMaxSteps + 1);  // full[], done
    static constexpr uint32_t kSmem = kOffSlot + 16 + 1024;
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static_assert(uint32_t(kSplit) * kSmMaxTok * kRowsPer * 4 <= kOffSf,
                  "received partials fit in the stage region");
    static_assert((kMaxSteps + 3) / 4 + 1 <= kSmMaxHeads, "scale words per CTA");
};

// The split-K kernels' reduction (128 threads; every CTA of the cluster
// calls it). Thread (w, l) holds its row 32w + l of this CTA's partial tile
// for tokens 0 .. n_tok - 1 in d0 (tokens 0-31) and d1 (32-63). After a
// cluster barrier (every CTA's stage region is free) it stores the row into
// the shared memory of the CTA that owns it (CTA (32w + l) / kRowsPer, slot =
// this CTA's rank, laid out [token][row within that CTA's rows]); after a
// second one each CTA sums its rows' kSplit partials in rank order and
// stores them as bf16: y_tile[token * y_token_stride + row], for the first
// tok_here tokens.
template <int kSplit>
__device__ __forceinline__ void small_reduce_store(uint32_t base, uint32_t rank,
                                                   const float (&d0)[32], const float (&d1)[32],
                                                   int n_tok, int tok_here, uint16_t* y_tile,
                                                   int64_t y_token_stride) {
    using L = SmLayout<kSplit>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    umma::cluster_sync();  // every CTA's stage region is free
    const uint32_t slot_bytes = uint32_t(n_tok) * L::kRowsPer * 4;
    {
        const int row = warp * 32 + lane;
        const uint32_t dst = umma::cluster_addr(
            base + rank * slot_bytes + uint32_t(row % L::kRowsPer) * 4, uint32_t(row / L::kRowsPer));
#pragma unroll
        for (int c = 0; c < kSmMaxTok; ++c)
            if (c < n_tok)
                umma::st_cluster_f32(dst + uint32_t(c * L::kRowsPer * 4), c < 32 ? d0[c] : d1[c - 32]);
    }
    umma::cluster_sync();  // every partial has arrived
    const int r = threadIdx.x % L::kRowsPer;
    constexpr int kTokStep = kSmThreads / L::kRowsPer;
    uint16_t* y = y_tile + int(rank) * L::kRowsPer + r;
    for (int c = threadIdx.x / L::kRowsPer; c < min(n_tok, tok_here); c += kTokStep) {
        const uint32_t a = base + uint32_t(c * L::kRowsPer + r) * 4;
        float sum = lds4f(a);
#pragma unroll
        for (int q = 1; q < kSplit; ++q) sum = __fadd_rn(sum, lds4f(a + q * slot_bytes));
        y[int64_t(c) * y_token_stride] = uint16_t(bf16x2(sum, 0.f));
    }
}

template <int kSplit>
__global__ void __launch_bounds__(kSmThreads, 1)
grouped_fp8_gemm_ue8m0_small_kernel(const __grid_constant__ CUtensorMap tma_x,
                                    const __grid_constant__ CUtensorMap tma_w, MxGemmParams p,
                                    int n_tok) {
    using L = SmLayout<kSplit>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sf0 = base + L::kOffSf, full0 = base + L::kOffBar;
    const uint32_t done = full0 + 8 * L::kMaxSteps;
    uint8_t* slot = smem_raw + (base + L::kOffSlot - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(slot);
    volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(slot + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = umma::cluster_ctarank();
    // tile = (token tile, group, 128 output rows), output rows fastest
    const int n_rt = p.n_out / kSmRows;
    const int tile = blockIdx.x / kSplit;
    const int rt = tile % n_rt, g = (tile / n_rt) % p.groups, tt = tile / (n_rt * p.groups);
    const int n_kt = p.k / kMxBK, n_words = p.k / 512;
    const int steps = n_kt / kSplit;              // >= 1 (the launcher checks)
    const int kt0 = int(rank) * steps;
    const int h_first = kt0 / 4, h_last = (kt0 + steps - 1) / 4;
    const uint32_t lim = p.wait.spin_limit;
    const uint32_t tok_bytes = uint32_t(n_tok) * kMxBK;
    // test-only fault injection: cluster 0's first CTA issues no copies
    const bool starve = (p.wait.inject & kInjectGemmLoads) && blockIdx.x == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < steps; ++s) mbar_init(full0 + 8 * s, 1);
        mbar_init(done, 1);
        *abort = 0u;
        mbar_init_fence();
        // Launched with programmatic dependent launch, the CTA gets here while
        // the previous kernel (typically the op that wrote the activations)
        // may still run. Only a prefetch of W into L2, which returns no data,
        // runs before the dependency wait; the copies after it read whatever
        // that kernel wrote.
        for (int s = 0; s < steps; ++s)
            umma::tma_prefetch_l2_2d(&tma_w, (kt0 + s) * kMxBK, g * p.n_out + rt * kSmRows);
    }
    if (warp == 1) {
        umma::tmem_alloc(base + L::kOffSlot, kSmTmemCols);
        umma::tmem_relinquish();
    }
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0 && !starve) {  // all K steps' copies at once (this thread made the barriers)
        for (int s = 0; s < steps; ++s) {
            const uint32_t st = base + s * kSmStage;
            const int kt = kt0 + s;
            mbar_arrive_expect_tx(full0 + 8 * s, kSmWTile + tok_bytes);
            umma::tma_load_2d(st, &tma_w, kt * kMxBK, g * p.n_out + rt * kSmRows, full0 + 8 * s);
            umma::tma_load_2d(st + kSmWTile, &tma_x, g * p.k + kt * kMxBK, tt * kSmMaxTok,
                              full0 + 8 * s);
        }
    }
    // Scale-code atoms (one per scale word the K steps touch): W's code of
    // this 128 x 128 block is the same for all 128 rows; the tokens' words sit
    // at row i + 32c of the atom as 16-byte row i, column c (rows past the
    // last token hold codes of 1.0; their operand rows are zero).
    for (int h = h_first; h <= h_last; ++h) {
        const int j = h - h_first;
        const uint8_t* ws = p.w_sf + (int64_t(g) * (p.n_out / 128) + rt) * n_kt + 4 * h;
        const uint32_t w = uint32_t(__ldg(ws)) | (uint32_t(__ldg(ws + 1)) << 8) |
                           (uint32_t(__ldg(ws + 2)) << 16) | (uint32_t(__ldg(ws + 3)) << 24);
        if (warp == 0) sts16(sf0 + (2 * j) * kSfAtom + 16 * lane, w, w, w, w);
        if (warp == 1) {
            uint32_t x[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int tok = tt * kSmMaxTok + lane + 32 * c;
                x[c] = (lane + 32 * c < kSmMaxTok && tok < p.m)
                           ? __ldg(p.a_sf + (int64_t(tok) * p.groups + g) * n_words + h)
                           : kUe8m0One4;
            }
            sts16(sf0 + (2 * j + 1) * kSfAtom + 16 * lane, x[0], x[1], x[2], x[3]);
        }
    }
    fence_proxy_async_smem();  // generic-proxy atom writes -> tcgen05.cp reads
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 1 && lane == 0) {
        for (int h = h_first; h <= h_last; ++h) {
            const int j = h - h_first;
            umma::cp_32x128b_warpx4(tmem + kSmTmemSfw + 4 * j,
                                    umma::smem_desc_plain(sf0 + (2 * j) * kSfAtom));
            umma::cp_32x128b_warpx4(tmem + kSmTmemSfx + 4 * j,
                                    umma::smem_desc_plain(sf0 + (2 * j + 1) * kSfAtom));
        }
        for (int s = 0; s < steps; ++s) {
            if (!wait_or_abort(full0 + 8 * s, 0, abort, lim)) break;
            umma::fence_after_sync();
            const uint32_t st = base + s * kSmStage;
            const uint64_t wd = umma::smem_desc_sw128(st);
            const uint64_t xd = umma::smem_desc_sw128(st + kSmWTile);
            const int kt = kt0 + s, j = kt / 4 - h_first;
            const uint32_t idesc = umma::idesc_mx_e4m3_ue8m0(kSmRows, n_tok, uint32_t(kt & 3));
#pragma unroll
            for (int k = 0; k < kMxBK / 32; ++k)
                umma::mma_mxf8f6f4(tmem, wd + 2 * k, xd + 2 * k, idesc, tmem + kSmTmemSfw + 4 * j,
                                   tmem + kSmTmemSfx + 4 * j, (s | k) != 0);
        }
        umma::commit(done);  // also after an abort: every issued MMA completes first
    }
    // the accumulator is final (or the wait gave up and the call is flagged)
    if (!mbar_wait(done, 0, lim)) *abort = 1u;
    if (warp == 0 && lane == 0 && !starve) {
        // the copies in flight land before the stage region is reused
        for (int s = 0; s < steps; ++s)
            if (!mbar_wait(full0 + 8 * s, 0, lim)) *abort = 1u;
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    // this thread's row of the partial tile (TMEM lane 32w + l)
    float d0[32], d1[32];
    umma::ld32(tmem + (uint32_t(warp * 32) << 16), d0);
    if (n_tok > 32) umma::ld32(tmem + (uint32_t(warp * 32) << 16) + 32u, d1);
    umma::fence_before_sync();
    small_reduce_store<kSplit>(base, rank, d0, d1, n_tok, p.m - tt * kSmMaxTok,
                               p.y + int64_t(tt) * kSmMaxTok * p.groups * p.n_out +
                                   int64_t(g) * p.n_out + rt * kSmRows,
                               int64_t(p.groups) * p.n_out);
    if (threadIdx.x == 0 && *abort && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_TIMEOUT);
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, kSmTmemCols);
    }
}

// The same decode-size split-K kernel for fp32 block scales (the op's default
// output, rq_grouped_fp8_gemm): the plain kind::f8f6f4 MMA into one TMEM
// accumulator per K step (128 x n_tok fp32 each, n_tmem columns in all, at
// most 512 per SM: 256 per CTA and two CTAs per SM with the 8-way split, 512
// and one CTA per SM with the 4-way split), then each thread folds its row:
//   part[token] = sum over its K steps s, in order, of
//                 (w_scale[s] * a_scale[token, s]) * D_s[row, token]
// and the cluster sums the parts as in the UE8M0 kernel. The A scales of the
// tile's tokens and K steps are staged in shared memory; W's scale of a K step
// is the same for the tile's 128 rows.
template <int kSplit>
__global__ void __launch_bounds__(kSmThreads, 1)
grouped_fp8_gemm_f32_small_kernel(const __grid_constant__ CUtensorMap tma_x,
                                  const __grid_constant__ CUtensorMap tma_w, GemmParams p,
                                  int n_tok, uint32_t n_tmem) {
    using L = SmLayout<kSplit>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sa0 = base + L::kOffSf, full0 = base + L::kOffBar;
    const uint32_t done = full0 + 8 * L::kMaxSteps;
    uint8_t* slot = smem_raw + (base + L::kOffSlot - raw);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(slot);
    volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(slot + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = umma::cluster_ctarank();
    const int n_rt = p.n_out / kSmRows;
    const int tile = blockIdx.x / kSplit;
    const int rt = tile % n_rt, g = (tile / n_rt) % p.groups, tt = tile / (n_rt * p.groups);
    const int n_kt = p.k / kMxBK;
    const int steps = n_kt / kSplit;              // >= 1 (the launcher checks)
    const int kt0 = int(rank) * steps;
    const uint32_t lim = p.wait.spin_limit;
    const uint32_t tok_bytes = uint32_t(n_tok) * kMxBK;
    const bool starve = (p.wait.inject & kInjectGemmLoads) && blockIdx.x == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < steps; ++s) mbar_init(full0 + 8 * s, 1);
        mbar_init(done, 1);
        *abort = 0u;
        mbar_init_fence();
        // only a prefetch of W (no data returned) before the dependency wait
        for (int s = 0; s < steps; ++s)
            umma::tma_prefetch_l2_2d(&tma_w, (kt0 + s) * kMxBK, g * p.n_out + rt * kSmRows);
    }
    if (warp == 1) {
        umma::tmem_alloc(base + L::kOffSlot, n_tmem);
        umma::tmem_relinquish();
    }
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0 && !starve) {  // all K steps' copies at once
        for (int s = 0; s < steps; ++s) {
            const uint32_t st = base + s * kSmStage;
            const int kt = kt0 + s;
            mbar_arrive_expect_tx(full0 + 8 * s, kSmWTile + tok_bytes);
            umma::tma_load_2d(st, &tma_w, kt * kMxBK, g * p.n_out + rt * kSmRows, full0 + 8 * s);
            umma::tma_load_2d(st + kSmWTile, &tma_x, g * p.k + kt * kMxBK, tt * kSmMaxTok,
                              full0 + 8 * s);
        }
    }
    // the tile's A scales, [K step][token] (0 past the last token)
    for (int i = threadIdx.x; i < steps * n_tok; i += kSmThreads) {
        const int s = i / n_tok, c = i - s * n_tok, tok = tt * kSmMaxTok + c;
        sts4f(sa0 + 4u * uint32_t(i),
              tok < p.m ? __ldg(p.a_scales + (int64_t(tok) * p.groups + g) * n_kt + kt0 + s) : 0.f);
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 1 && lane == 0) {
        const uint32_t idesc = umma::idesc_e4m3_f32(kSmRows, n_tok);
        for (int s = 0; s < steps; ++s) {
            if (!wait_or_abort(full0 + 8 * s, 0, abort, lim)) break;
            umma::fence_after_sync();
            const uint32_t st = base + s * kSmStage;
            const uint64_t wd = umma::smem_desc_sw128(st);
            const uint64_t xd = umma::smem_desc_sw128(st + kSmWTile);
#pragma unroll
            for (int k = 0; k < kMxBK / 32; ++k)
                umma::mma_f8f6f4(tmem + uint32_t(s * n_tok), wd + 2 * k, xd + 2 * k, idesc, k != 0);
        }
        umma::commit(done);  // also after an abort: every issued MMA completes first
    }
    if (!mbar_wait(done, 0, lim)) *abort = 1u;
    if (warp == 0 && lane == 0 && !starve) {
        for (int s = 0; s < steps; ++s)
            if (!mbar_wait(full0 + 8 * s, 0, lim)) *abort = 1u;
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    // fold this thread's row over the K steps, in order
    float d0[32], d1[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) d0[c] = d1[c] = 0.f;
    const float* ws = p.w_scales + (int64_t(g) * n_rt + rt) * n_kt + kt0;
    for (int s = 0; s < steps; ++s) {
        const float sw = __ldg(ws + s);
        const uint32_t col = tmem + (uint32_t(warp * 32) << 16) + uint32_t(s * n_tok);
        float d[32];
        umma::ld32(col, d);
#pragma unroll
        for (int c = 0; c < 32; ++c)
            if (c < n_tok)
                d0[c] = __fadd_rn(d0[c], __fmul_rn(__fmul_rn(sw, lds4f(sa0 + 4u * uint32_t(s * n_tok + c))), d[c]));
        if (n_tok > 32) {
            umma::ld32(col + 32u, d);
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (32 + c < n_tok)
                    d1[c] = __fadd_rn(d1[c], __fmul_rn(__fmul_rn(sw, lds4f(sa0 + 4u * uint32_t(s * n_tok + 32 + c))), d[c]));
        }
    }
    umma::fence_before_sync();
    small_reduce_store<kSplit>(base, rank, d0, d1, n_tok, p.m - tt * kSmMaxTok,
                               p.y + int64_t(tt) * kSmMaxTok * p.groups * p.n_out +
                                   int64_t(g) * p.n_out + rt * kSmRows,
                               int64_t(p.groups) * p.n_out);
    if (threadIdx.x == 0 && *abort && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_TIMEOUT);
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, n_tmem);
    }
}

namespace {

// The split-K decode kernel: one cluster of kSplit CTAs per (token tile,
// group, 128 output rows).
template <int kSplit>
cudaError_t launch_small(const MxGemmParams& p, const uint8_t* a_codes, const uint8_t* w_codes,
                         const DeviceInfo& dev, cudaStream_t stream) {
    using L = SmLayout<kSplit>;
    const int n_tok = p.m >= kSmMaxTok ? kSmMaxTok : (p.m + 15) / 16 * 16;
    CUtensorMap mx, mw;
    if (!make_map(&mx, a_codes, uint64_t(p.groups) * p.k, uint64_t(p.m), uint64_t(p.groups) * p.k,
                  uint32_t(n_tok)) ||
        !make_map(&mw, w_codes, uint64_t(p.k), uint64_t(p.groups) * p.n_out, uint64_t(p.k),
                  kSmRows))
        return cudaErrorInvalidValue;
    auto k = grouped_fp8_gemm_ue8m0_small_kernel<kSplit>;
    constexpr int kMax = 64;
    static thread_local bool attr_done[kMax] = {};
    const int d = (dev.ordinal >= 0 && dev.ordinal < kMax) ? dev.ordinal : 0;
    if (!attr_done[d]) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(L::kSmem));
        if (e != cudaSuccess) return e;
        attr_done[d] = true;
    }
    const int64_t tiles = int64_t((p.m + kSmMaxTok - 1) / kSmMaxTok) * p.groups * (p.n_out / kSmRows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(tiles * kSplit));
    cfg.blockDim = dim3(kSmThreads);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k, mx, mw, p, n_tok);
}

// K split 8 ways when K is a multiple of 1024 (two CTAs fit on an SM), else
// 4 ways (K is a multiple of 512). Measured on B300 at 4 groups x K 4096 x
// 1024 outputs, one token: 6.6 us (8 ways) against 7.1 us (4 ways) per call,
// 13.2 us on the 128 x 256 tile kernel.
cudaError_t launch_grouped_fp8_gemm_ue8m0_small(const MxGemmParams& p, const uint8_t* a_codes,
                                               const uint8_t* w_codes, const DeviceInfo& dev,
                                               cudaStream_t stream) {
    if ((p.k / kMxBK) % 8 == 0) return launch_small<8>(p, a_codes, w_codes, dev, stream);
    return launch_small<4>(p, a_codes, w_codes, dev, stream);
}

// The fp32-scale decode kernel; n_tmem covers one accumulator per K step
// plus the columns a 32-wide TMEM read past the last one touches.
template <int kSplit>
cudaError_t launch_f32_small(const GemmParams& p, const uint8_t* a_codes, const uint8_t* w_codes,
                             int dev_ordinal, cudaStream_t stream) {
    using L = SmLayout<kSplit>;
    const int n_tok = p.m >= kSmMaxTok ? kSmMaxTok : (p.m + 15) / 16 * 16;
    const int steps = p.k / kMxBK / kSplit;
    const uint32_t need = uint32_t(steps * n_tok + (n_tok % 32 ? 32 - n_tok % 32 : 0));
    uint32_t n_tmem = 32;
    while (n_tmem < need) n_tmem <<= 1;
    // The CTAs that fit on an SM (228 KiB of shared memory, 1 KiB reserved per
    // CTA) must never ask for more than its 512 TMEM columns together, so an
    // allocation never waits on a CTA that is itself waiting at a cluster
    // barrier: 256 columns at most with the 8-way split (two CTAs per SM),
    // 512 with the 4-way split (one). Always true for K <= 4096.
    const uint32_t ctas_per_sm = 233472u / (L::kSmem + 1024u);
    if (n_tmem * ctas_per_sm > 512u) return cudaErrorInvalidValue;
    CUtensorMap mx, mw;
    if (!make_map(&mx, a_codes, uint64_t(p.groups) * p.k, uint64_t(p.m), uint64_t(p.groups) * p.k,
                  uint32_t(n_tok)) ||
        !make_map(&mw, w_codes, uint64_t(p.k), uint64_t(p.groups) * p.n_out, uint64_t(p.k),
                  kSmRows))
        return cudaErrorInvalidValue;
    auto k = grouped_fp8_gemm_f32_small_kernel<kSplit>;
    constexpr int kMax = 64;
    static thread_local bool attr_done[kMax] = {};
    const int d = (dev_ordinal >= 0 && dev_ordinal < kMax) ? dev_ordinal : 0;
    if (!attr_done[d]) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   int(L::kSmem));
        if (e != cudaSuccess) return e;
        attr_done[d] = true;
    }
    const int64_t tiles = int64_t((p.m + kSmMaxTok - 1) / kSmMaxTok) * p.groups * (p.n_out / kSmRows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(tiles * kSplit));
    cfg.blockDim = dim3(kSmThreads);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k, mx, mw, p, n_tok, n_tmem);
}

}  // namespace

// fp32 block scales, up to 64 tokens, K a multiple of 512 (the 8-way split
// when K is a multiple of 1024).
cudaError_t launch_grouped_fp8_gemm_small(const GemmParams& p, const uint8_t* a_codes,
                                          const uint8_t* w_codes, int dev_ordinal,
                                          cudaStream_t stream) {
    if ((p.k / kMxBK) % 8 == 0) return launch_f32_small<8>(p, a_codes, w_codes, dev_ordinal, stream);
    return launch_f32_small<4>(p, a_codes, w_codes, dev_ordinal, stream);
}

cudaError_t launch_grouped_fp8_gemm_ue8m0(const MxGemmParams& p, const uint8_t* a_codes,
                                          const uint8_t* w_codes, const DeviceInfo& dev,
                                          cudaStream_t stream) {
    CUtensorMap ma, mw;
    if (!make_map(&ma, a_codes, uint64_t(p.groups) * p.k, uint64_t(p.m), uint64_t(p.groups) * p.k,
                  kMxBM) ||
        !make_map(&mw, w_codes, uint64_t(p.k), uint64_t(p.groups) * p.n_out, uint64_t(p.k),
                  kMxBN))
        return cudaErrorInvalidValue;
    constexpr int kMax = 64;
    static thread_local bool attr_done[kMax] = {};
    const int d = (dev.ordinal >= 0 && dev.ordinal < kMax) ? dev.ordinal : 0;
    if (!attr_done[d]) {
        const cudaError_t e = cudaFuncSetAttribute(
            grouped_fp8_gemm_ue8m0_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kMxSmem));
        if (e != cudaSuccess) return e;
        attr_done[d] = true;
    }
    // up to 64 tokens: the split-K kernel (measured faster at every such size;
    // at 96 and 128 tokens the two are within 5% of each other)
    if (p.m <= kSmMaxTok) return launch_grouped_fp8_gemm_ue8m0_small(p, a_codes, w_codes, dev, stream);
    const int64_t tiles = int64_t((p.m + kMxBM - 1) / kMxBM) * p.groups *
                          ((p.n_out + kMxBN - 1) / kMxBN);
    if (tiles == 0) return cudaSuccess;
    const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
    grouped_fp8_gemm_ue8m0_kernel<<<grid, kMxThreads, kMxSmem, stream>>>(ma, mw, p);
    return cudaGetLastError();
}

}  // namespace rq
