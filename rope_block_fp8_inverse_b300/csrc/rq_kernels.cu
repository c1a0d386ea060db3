// rq_kernels.cu -- the warp-rows kernels (sm_103a) and their launchers: the
// inverse-RoPE + block-FP8 quant op (also into row-linear UE8M0 and
// contiguous group-major layouts), the same op into any strided layout
// (fixed heads per warp, or token tiles per warp for token-contiguous fp32
// scales) or as bf16, its forward-RoPE + paged-insert sibling, and the fused
// q RMS norm + RoPE + kv insert op. (The TMA-ring variant of the inverse op
// is in rq_stream.cu.)
//
// All are HBM-bound streams (about 1.5 bytes moved per fp32 op), so the
// design goal is bytes in flight, not arithmetic: a persistent grid of warps
// sized to the SM count, each warp owning whole 512-wide rows
// (rq_device.cuh) and issuing the loads of kRows rows before it computes any
// of them. The pages' Triton kernel (one program per 1 to 4 heads) is prior
// art: here a warp is the program, and the number of rows in flight per SM
// is set by kRows x resident warps instead of by BLOCK_H.
#include <algorithm>

#include "rq_device.cuh"
#include "rq_launch.h"

namespace rq {

// ------------------------------------------------------------------ inverse

// Row r = t * n_heads + h. Output row r (512 codes) sits at out + r*512 and
// its 4 scales at scales + r*4: with contiguous [N, G, hpg*512] /
// [N, G, hpg*4] outputs this is exactly the grouped layout of the inverse
// RoPE page, S1 (head h = g*hpg + i of token t at row (t, g), offset i*512),
// so the grouping never changes an address.
// Held to 4 CTAs per SM (64 registers), measured 1% faster than the
// compiler's free choice of 73 registers (3 CTAs). kMode picks the scale
// encoding: fp32 scales at scales + r*4, or (kOutFp8Ue8m0) one packed UE8M0
// word per row at scales + r -- the row-linear token-major layouts of the
// layout call, which takes this kernel for them. kGroupMajor writes the
// contiguous group-major layout instead ([G, N, hpg*512] codes and
// [G, N, hpg*4] / [G, N, hpg] scales): the same rows, each stored at its
// output row q = (g*N + t)*hpg + i.
// The launcher sizes the grid so that one sweep of it (all warps, kRows rows
// each) is a whole number of tokens (p.sweep_tokens): every warp then keeps
// the same heads from sweep to sweep, and each of its rows advances by
// constant steps in the input, the positions and the output. (A walk that
// moved each warp to new (token, head) pairs cost 14% more instructions per
// row with group-major output, measured on B300.)
template <int kRows, int kMode = kOutFp8F32, bool kGroupMajor = false>
__global__ void __launch_bounds__(kInvThreads, 4)
inv_rope_fp8_quant_kernel(InvParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
    const int ca = chunk_a(lane);
    const bool rope_lane = lane >= kRopeLane0;
    const int cs_col = (rope_lane ? lane - kRopeLane0 : 0) * 4;

    // A sweep of the grid is p.sweep_tokens (>= 1) whole tokens and n_heads
    // is a multiple of kRows, so warp w keeps heads h0 .. h0 + kRows - 1 of
    // one token in every sweep (rows w*kRows + j), the token advancing by
    // sweep_tokens. Input, position and output then advance by constants (no
    // row walk, no per-row multiply).
    const uint32_t sweep_rows = p.sweep_tokens * p.n_heads;
    if (warp * kRows >= sweep_rows) return;  // warp-uniform: idle warps of the grid
    const uint32_t r0 = warp * kRows;
    uint32_t t = r0 / p.n_heads;
    const uint32_t h0 = r0 - t * p.n_heads;
    const uint16_t* row = x + static_cast<int64_t>(t) * p.sx_t + static_cast<int64_t>(h0) * p.sx_h;
    // output row of head h0 (token-major r0; group-major q), and the offset of
    // head h0 + j from it (group-major: + (N - 1) * hpg once the heads cross
    // into the next group)
    uint32_t orow = r0;
    uint32_t cross = kRows;  // first j in the next group
    if (kGroupMajor) {
        const uint32_t g = h0 / p.lay.hpg, i = h0 - g * p.lay.hpg;
        orow = (g * p.n_tokens + t) * p.lay.hpg + i;
        cross = p.lay.hpg - i;
    }
    const int64_t dx = static_cast<int64_t>(p.sweep_tokens) * p.sx_t;
    const uint32_t dorow = kGroupMajor ? p.sweep_tokens * p.lay.hpg : sweep_rows;
    for (; t < p.n_tokens; t += p.sweep_tokens, row += dx, orow += dorow) {
        uint4 a[kRows], b[kRows];
        float4 c, s;
        // the rows' reads do not wait for the position: only cos/sin do
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            a[j] = ld_stream16(row + j * p.sx_h + 8 * ca);
            b[j] = ld_stream16(row + j * p.sx_h + 8 * (ca + 8));
        }
        const int64_t pos = __ldg(p.positions + t);
        if (static_cast<uint64_t>(pos) >= static_cast<uint64_t>(p.cache_rows)) {  // warp-uniform
            if (lane == 0 && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
            continue;
        }
        if (rope_lane) {  // one cos/sin row serves the token's kRows heads
            const float* cs = p.cache + pos * kCacheWidth + cs_col;
            c = ld_ro16(cs);
            s = ld_ro16(cs + kHalfRope);
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const int64_t r = int64_t(orow) + j +
                              (kGroupMajor && uint32_t(j) >= cross
                                   ? int64_t(p.n_tokens - 1) * p.lay.hpg
                                   : 0);
            float scale;
            const uint4 qc = rope_quant_row<true>(a[j], b[j], rope_lane, c, s, p.eps, &scale);
            if (kMode == kOutFp8F32) {
                store_row(p.out + r * kHeadDim, p.scales + r * 4, lane, ca, qc, scale);
            } else {
                uint8_t* codes = p.out + r * kHeadDim;
                st_stream8(codes + 8 * ca, qc.x, qc.y);
                st_stream8(codes + 8 * (ca + 8), qc.z, qc.w);
                // byte b of the row's word: block b's biased exponent
                if ((lane & 7) == 0)
                    st_stream1(reinterpret_cast<uint8_t*>(reinterpret_cast<uint32_t*>(p.scales) +
                                                          r) +
                                   (lane >> 3),
                               __float_as_uint(scale) >> 23);
            }
        }
    }
}

// ------------------------------------------------------------------ inverse, any output layout

// The warp-rows kernel with the output addressed through OutLayout: fp32 or
// packed UE8M0 scales, or (kMode == kOutBf16) the rotated head as bf16 with
// no quantisation, into token-major, group-major or any other strided
// layout. Loads and arithmetic are those of inv_rope_fp8_quant_kernel. Rows
// are walked without division (RowPos), and the kernel is held to 4 CTAs per
// SM (64 registers): on B300 that took the fp8 layouts from 0.86 to 0.92 of
// the copy peak.
template <int kRows, int kMode>
__global__ void __launch_bounds__(kInvThreads, 4)
inv_rope_quant_layout_kernel(InvParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
    const int ca = chunk_a(lane);
    const bool rope_lane = lane >= kRopeLane0;
    const int cs_col = (rope_lane ? lane - kRopeLane0 : 0) * 4;
    constexpr int64_t kHeadBytes = kMode == kOutBf16 ? 2 * kHeadDim : kHeadDim;
    const uint32_t hpg = p.lay.hpg, groups = p.n_heads / hpg;
    const RowStride step = row_stride(n_warps * kRows, p.n_heads, hpg);
    const RowStride next = row_stride(1, p.n_heads, hpg);
    RowPos base = row_pos(warp * kRows, p.n_heads, hpg);

    for (uint32_t r0 = warp * kRows; r0 < p.n_rows;
         r0 += n_warps * kRows, row_advance(base, step, p.n_heads, hpg, groups)) {
        uint4 a[kRows], b[kRows];
        float4 c[kRows], s[kRows];
        RowPos w[kRows];
        bool live[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const uint32_t r = r0 + i;
            w[i] = base;
            if (i > 0) {
                w[i] = w[i - 1];
                row_advance(w[i], next, p.n_heads, hpg, groups);
            }
            live[i] = false;
            if (r < p.n_rows) {  // warp-uniform
                const uint32_t t = w[i].t;
                const uint16_t* row = x + static_cast<int64_t>(t) * p.sx_t +
                                      static_cast<int64_t>(w[i].h) * p.sx_h;
                a[i] = ld_stream16(row + 8 * ca);
                b[i] = ld_stream16(row + 8 * (ca + 8));
                const int64_t pos = __ldg(p.positions + t);
                live[i] = static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
                if (live[i]) {
                    if (rope_lane) {
                        const float* cs = p.cache + pos * kCacheWidth + cs_col;
                        c[i] = ld_ro16(cs);
                        s[i] = ld_ro16(cs + kHalfRope);
                    }
                } else if (lane == 0 && p.error_flags) {
                    atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            if (!live[i]) continue;
            const uint32_t g = w[i].g, hig = w[i].i;
            uint8_t* head = p.out + int64_t(w[i].t) * p.lay.ot + int64_t(g) * p.lay.og +
                            int64_t(hig) * kHeadBytes;
            if (kMode == kOutBf16) {
                uint4 qa, qb;
                rope_row_bf16<true>(a[i], b[i], rope_lane, c[i], s[i], &qa, &qb);
                st_stream16(head + 16 * ca, qa);
                st_stream16(head + 16 * (ca + 8), qb);
                continue;
            }
            float scale;
            const uint4 q = rope_quant_row<true>(a[i], b[i], rope_lane, c[i], s[i], p.eps, &scale);
            st_stream8(head + 8 * ca, q.x, q.y);
            st_stream8(head + 8 * (ca + 8), q.z, q.w);
            const int64_t sbase = int64_t(w[i].t) * p.lay.st + int64_t(g) * p.lay.sg;
            if (kMode == kOutFp8F32) {
                if ((lane & 7) == 0)
                    st_stream4f(p.scales + sbase + (int64_t(hig) * 4 + (lane >> 3)) * p.lay.se,
                                scale);
            } else if ((lane & 7) == 0) {
                // UE8M0: the biased exponent of the power-of-two scale, one
                // byte per block, block b in bits 8b..8b+7 of the head's word
                // (little-endian: byte b), written by block b's first lane
                const uint32_t e = __float_as_uint(scale) >> 23;
                st_stream1(reinterpret_cast<uint8_t*>(reinterpret_cast<uint32_t*>(p.scales) +
                                                      sbase + int64_t(hig) * p.lay.se) +
                               (lane >> 3),
                           e);
            }
        }
    }
}

// The layout kernel's fixed-head form (what the layout call launches when a
// sweep of the grid holds at least one whole token): as in
// inv_rope_fp8_quant_kernel, warp w keeps heads h0 .. h0 + kRows - 1 of one
// token (n_heads a multiple of kRows) in every sweep of p.sweep_tokens
// tokens, and its output and scale addresses advance by sweep_tokens times
// the layout's token strides. The heads' offsets from head h0 within a token
// are constants of the warp.
template <int kRows, int kMode>
__global__ void __launch_bounds__(kInvThreads, 4)
inv_rope_quant_layout_fixed_kernel(InvParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
    const int ca = chunk_a(lane);
    const bool rope_lane = lane >= kRopeLane0;
    const int cs_col = (rope_lane ? lane - kRopeLane0 : 0) * 4;
    constexpr int64_t kHeadBytes = kMode == kOutBf16 ? 2 * kHeadDim : kHeadDim;
    // scale elements per head: 4 fp32 block scales, or one packed UE8M0 word
    constexpr int64_t kScalesPerHead = kMode == kOutFp8F32 ? 4 : 1;
    const uint32_t sweep_rows = p.sweep_tokens * p.n_heads;
    if (warp * kRows >= sweep_rows) return;  // warp-uniform: idle warps of the grid
    const uint32_t r0 = warp * kRows;
    uint32_t t = r0 / p.n_heads;
    const uint32_t h0 = r0 - t * p.n_heads;
    const uint16_t* row = x + static_cast<int64_t>(t) * p.sx_t + static_cast<int64_t>(h0) * p.sx_h;
    // head h of token t: codes at out + t*ot + g*og + i*kHeadBytes, its scale
    // elements from scales + t*st + g*sg + i*kScalesPerHead*se
    int64_t oo[kRows], so[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const uint32_t h = h0 + j, g = h / p.lay.hpg, i = h - g * p.lay.hpg;
        oo[j] = int64_t(t) * p.lay.ot + int64_t(g) * p.lay.og + int64_t(i) * kHeadBytes;
        so[j] = int64_t(t) * p.lay.st + int64_t(g) * p.lay.sg + int64_t(i) * kScalesPerHead * p.lay.se;
    }
    const int64_t dx = static_cast<int64_t>(p.sweep_tokens) * p.sx_t;
    const int64_t doo = static_cast<int64_t>(p.sweep_tokens) * p.lay.ot;
    const int64_t dso = static_cast<int64_t>(p.sweep_tokens) * p.lay.st;
    for (; t < p.n_tokens; t += p.sweep_tokens, row += dx) {
        uint4 a[kRows], b[kRows];
        float4 c, s;
        // the rows' reads do not wait for the position: only cos/sin do
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            a[j] = ld_stream16(row + j * p.sx_h + 8 * ca);
            b[j] = ld_stream16(row + j * p.sx_h + 8 * (ca + 8));
        }
        const int64_t pos = __ldg(p.positions + t);
        const bool live = static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
        if (live) {  // warp-uniform
            if (rope_lane) {  // one cos/sin row serves the token's kRows heads
                const float* cs = p.cache + pos * kCacheWidth + cs_col;
                c = ld_ro16(cs);
                s = ld_ro16(cs + kHalfRope);
            }
        } else if (lane == 0 && p.error_flags) {
            atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            if (live) {
                uint8_t* head = p.out + oo[j];
                if (kMode == kOutBf16) {
                    uint4 qa, qb;
                    rope_row_bf16<true>(a[j], b[j], rope_lane, c, s, &qa, &qb);
                    st_stream16(head + 16 * ca, qa);
                    st_stream16(head + 16 * (ca + 8), qb);
                } else {
                    float scale;
                    const uint4 q = rope_quant_row<true>(a[j], b[j], rope_lane, c, s, p.eps, &scale);
                    st_stream8(head + 8 * ca, q.x, q.y);
                    st_stream8(head + 8 * (ca + 8), q.z, q.w);
                    if ((lane & 7) == 0) {
                        if (kMode == kOutFp8F32) {
                            st_stream4f(p.scales + so[j] + (lane >> 3) * p.lay.se, scale);
                        } else {
                            // UE8M0: byte b of the head's word = block b's biased exponent
                            st_stream1(reinterpret_cast<uint8_t*>(
                                           reinterpret_cast<uint32_t*>(p.scales) + so[j]) +
                                           (lane >> 3),
                                       __float_as_uint(scale) >> 23);
                        }
                    }
                }
            }
            oo[j] += doo;
            so[j] += dso;
        }
    }
}

// ------------------------------------------------------------------ inverse, token-contiguous scales

// The layout kernel for fp32 scales whose elements of consecutive tokens are
// adjacent (scale token stride 1: [G, hpg*4, N], the scales stored
// transposed, as an M-major GEMM scale operand takes them). Stored row by row
// such scales cost four partial 32-byte sectors per row, a quarter more
// write sectors than the codes. Here warp w keeps head h = w % n_heads and
// walks tiles of kScaleTile consecutive tokens of it, two rows at a time;
// lane 8b + k keeps block b's scale of the tile's token k, and the tile's 32
// scales leave in one store of four whole sectors. Loads, arithmetic and
// code stores are those of the other warp-rows kernels; each row fetches its
// own cos/sin (its token differs from the other row's), after the previous
// row's arithmetic, which keeps the kernel within 64 registers.
constexpr uint32_t kScaleTile = 8;

__global__ void __launch_bounds__(kInvThreads, 4)
inv_rope_quant_layout_tiled_kernel(InvParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
    const int ca = chunk_a(lane);
    const bool rope_lane = lane >= kRopeLane0;
    const int cs_col = (rope_lane ? lane - kRopeLane0 : 0) * 4;
    // A sweep of the grid is p.sweep_tokens tokens (whole tiles) of every
    // head: warp w has head w % n_heads and, in each sweep, tile w / n_heads.
    const uint32_t tile = warp / p.n_heads;
    if (tile * kScaleTile >= p.sweep_tokens) return;  // warp-uniform: idle warps of the grid
    const uint32_t h = warp - tile * p.n_heads;
    const uint32_t g = h / p.lay.hpg, i = h - g * p.lay.hpg;
    const uint16_t* xh = x + static_cast<int64_t>(h) * p.sx_h;
    uint8_t* oh = p.out + int64_t(g) * p.lay.og + int64_t(i) * kHeadDim;
    // the tile token k and block b of the scale this lane stores, and that
    // scale's element for token 0
    const uint32_t kk = lane & 7;
    float* sl = p.scales + int64_t(g) * p.lay.sg + (int64_t(i) * 4 + (lane >> 3)) * p.lay.se;
    for (uint32_t t0 = tile * kScaleTile; t0 < p.n_tokens; t0 += p.sweep_tokens) {
        const uint32_t n_here = min(kScaleTile, p.n_tokens - t0);
        // the tile's positions, lane k holding token t0 + k's (-1 past the end)
        int64_t tpos = -1;
        if (uint32_t(lane) < n_here) tpos = __ldg(p.positions + t0 + lane);
        float keep = 0.f;  // block (lane >> 3)'s scale of token t0 + kk
        bool have = false;
        for (uint32_t k = 0; k < n_here; k += 2) {  // warp-uniform
            const bool second = k + 1 < n_here;
            const uint16_t* row = xh + static_cast<int64_t>(t0 + k) * p.sx_t;
            uint4 a[2], b[2];
            // the rows' reads do not wait for the positions: only cos/sin do
            a[0] = ld_stream16(row + 8 * ca);
            b[0] = ld_stream16(row + 8 * (ca + 8));
            if (second) {
                a[1] = ld_stream16(row + p.sx_t + 8 * ca);
                b[1] = ld_stream16(row + p.sx_t + 8 * (ca + 8));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                if (j == 1 && !second) break;  // warp-uniform
                const int64_t pos = __shfl_sync(kFull, tpos, k + j);
                if (static_cast<uint64_t>(pos) >= static_cast<uint64_t>(p.cache_rows)) {
                    if (lane == 0 && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
                    continue;  // warp-uniform: the row is skipped
                }
                float4 c, s;
                if (rope_lane) {
                    const float* cs = p.cache + pos * kCacheWidth + cs_col;
                    c = ld_ro16(cs);
                    s = ld_ro16(cs + kHalfRope);
                }
                float scale;
                const uint4 q = rope_quant_row<true>(a[j], b[j], rope_lane, c, s, p.eps, &scale);
                uint8_t* head = oh + int64_t(t0 + k + j) * p.lay.ot;
                st_stream8(head + 8 * ca, q.x, q.y);
                st_stream8(head + 8 * (ca + 8), q.z, q.w);
                if (kk == k + j) {
                    keep = scale;
                    have = true;
                }
            }
        }
        if (have) st_stream4f(sl + t0 + kk, keep);  // token stride 1
    }
}

// ------------------------------------------------------------------ insert

template <int kRows>
__global__ void __launch_bounds__(kInsThreads)
rope_fp8_quant_insert_kernel(InsParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    const uint16_t* __restrict__ kv = static_cast<const uint16_t*>(p.kv);
    const int ca = chunk_a(lane);
    const bool rope_lane = lane >= kRopeLane0;
    const int cs_col = (rope_lane ? lane - kRopeLane0 : 0) * 4;
    const int64_t n_slots = p.num_blocks * p.block_size;

    for (uint32_t t0 = warp * kRows; t0 < p.n_tokens; t0 += n_warps * kRows) {
        uint4 a[kRows], b[kRows];
        float4 c[kRows], s[kRows];
        int64_t slot[kRows];
        bool live[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const uint32_t t = t0 + i;
            live[i] = false;
            slot[i] = -1;
            if (t < p.n_tokens) {
                // the row's reads do not wait for its position or slot
                const uint16_t* row = kv + static_cast<int64_t>(t) * p.skv;
                a[i] = ld_stream16(row + 8 * ca);
                b[i] = ld_stream16(row + 8 * (ca + 8));
                const int64_t pos = __ldg(p.positions + t);
                slot[i] = __ldg(p.slot_mapping + t);
                const bool pos_ok =
                    static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
                const bool slot_ok = slot[i] < n_slots;
                live[i] = pos_ok && slot_ok && slot[i] >= 0;
                if (live[i]) {
                    if (rope_lane) {
                        const float* cs = p.cache + pos * kCacheWidth + cs_col;
                        c[i] = ld_ro16(cs);
                        s[i] = ld_ro16(cs + kHalfRope);
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
            float scale;
            const uint4 q = rope_quant_row<false>(a[i], b[i], rope_lane, c[i], s[i], p.eps, &scale);
            const int64_t blk = slot[i] / p.block_size;
            const int64_t off = slot[i] - blk * p.block_size;
            uint8_t* rec = p.k_cache + blk * p.block_stride + off * kRecordBytes;
            store_row(rec, reinterpret_cast<float*>(rec + kHeadDim), lane, ca, q, scale);
        }
    }
}

// ------------------------------------------------------------------ fused q + kv

// The fused op of the Eager-Break workspace page (S1) in one launch: unit u
// of token t = u / (Hpad + 1) is q head k = u % (Hpad + 1) for k < Hq (RMS
// norm + forward RoPE -> bf16 into q_out), a pad head for Hq <= k < Hpad
// (zeros), and the token's kv row for k == Hpad (forward RoPE + FP8 quant +
// paged insert). A token whose position is out of range leaves its q heads
// and its record untouched (pad heads are still zeroed) and sets the flag.
template <int kRows>
__global__ void __launch_bounds__(kInvThreads)
qnorm_rope_kv_insert_kernel(FusedParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    const uint16_t* __restrict__ q = static_cast<const uint16_t*>(p.q);
    const uint16_t* __restrict__ kv = static_cast<const uint16_t*>(p.kv);
    const int ca = chunk_a(lane);
    const bool rope_lane = lane >= kRopeLane0;
    const int cs_col = (rope_lane ? lane - kRopeLane0 : 0) * 4;
    const uint32_t per_token = p.q_head_padded + 1;
    const int64_t n_slots = p.num_blocks * p.block_size;
    // units walked without division (unit u = t * per_token + k)
    const RowStride step = row_stride(n_warps * kRows, per_token, per_token);
    const RowStride next = row_stride(1, per_token, per_token);
    RowPos base = row_pos(warp * kRows, per_token, per_token);

    for (uint32_t u0 = warp * kRows; u0 < p.n_units;
         u0 += n_warps * kRows, row_advance(base, step, per_token, per_token, 1)) {
        uint4 a[kRows], b[kRows];
        float4 c[kRows], s[kRows];
        uint32_t tt[kRows], kk[kRows];
        int64_t slot[kRows];
        bool live[kRows];
        RowPos w = base;
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const uint32_t u = u0 + i;
            if (i > 0) row_advance(w, next, per_token, per_token, 1);
            live[i] = false;
            if (u >= p.n_units) continue;  // warp-uniform
            const uint32_t t = w.t;
            const uint32_t k = w.h;
            tt[i] = t;
            kk[i] = k;
            const bool is_kv = k == p.q_head_padded;
            if (!is_kv && k >= p.n_heads_q) {  // pad head: zeros, no input
                live[i] = true;
                continue;
            }
            const uint16_t* row = is_kv ? kv + int64_t(t) * p.skv
                                        : q + int64_t(t) * p.sq_t + int64_t(k) * p.sq_h;
            a[i] = ld_stream16(row + 8 * ca);
            b[i] = ld_stream16(row + 8 * (ca + 8));
            const int64_t pos = __ldg(p.positions + t);
            const bool pos_ok = static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
            bool slot_ok = true;
            if (is_kv) {
                slot[i] = __ldg(p.slot_mapping + t);
                slot_ok = slot[i] < n_slots;
                live[i] = pos_ok && slot_ok && slot[i] >= 0;
            } else {
                live[i] = pos_ok;
            }
            if (live[i]) {
                if (rope_lane) {
                    const float* cs = p.cache + pos * kCacheWidth + cs_col;
                    c[i] = ld_ro16(cs);
                    s[i] = ld_ro16(cs + kHalfRope);
                }
            } else if (lane == 0 && p.error_flags && (!pos_ok || !slot_ok)) {
                atomicOr(p.error_flags, (pos_ok ? 0u : RQ_FLAG_POSITION_RANGE) |
                                            (slot_ok ? 0u : RQ_FLAG_SLOT_RANGE));
            }
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            if (!live[i]) continue;
            const uint32_t t = tt[i], k = kk[i];
            if (k == p.q_head_padded) {
                float scale;
                const uint4 qv =
                    rope_quant_row<false>(a[i], b[i], rope_lane, c[i], s[i], p.quant_eps, &scale);
                const int64_t blk = slot[i] / p.block_size;
                const int64_t off = slot[i] - blk * p.block_size;
                uint8_t* rec = p.k_cache + blk * p.block_stride + off * kRecordBytes;
                store_row(rec, reinterpret_cast<float*>(rec + kHeadDim), lane, ca, qv, scale);
                continue;
            }
            uint8_t* dst = reinterpret_cast<uint8_t*>(
                p.q_out + (int64_t(t) * p.q_head_padded + k) * kHeadDim);
            uint4 qa = make_uint4(0, 0, 0, 0), qb = qa;
            if (k < p.n_heads_q)
                qnorm_rope_row_bf16(a[i], b[i], rope_lane, c[i], s[i], p.norm_eps, p.norm_w, ca,
                                    &qa, &qb);
            st_stream16(dst + 16 * ca, qa);
            st_stream16(dst + 16 * (ca + 8), qb);
        }
    }
}

// ------------------------------------------------------------------ launchers

namespace {

// Resident CTAs per SM of each kernel variant, queried once per device and
// variant (thread-local: no locking on the launch path).
constexpr int kMaxDevices = 64;
// (kLay: 2 entries per output mode, one row or two rows per warp)
// (kRowsVariant: 4 entries per scale encoding: one or two rows per warp,
// token-major or group-major rows)
// (kLayFixed: the same for the layout kernel's fixed-head form)
// (kLayTiled: the token-tiled layout kernel)
enum Variant { kInv1, kInv2, kIns1, kFus1, kLay, kLayFixed = kLay + 6, kRowsVariant = kLayFixed + 6,
               kLayTiled = kRowsVariant + 8, kVariants = kLayTiled + 1 };

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

// The fixed-head inverse kernels run at most 4 CTAs (32 warps) per SM: an
// instance whose registers would allow a fifth (the bf16 layout, 48
// registers) measured 3% slower with it on B300.
constexpr int kMaxCtasPerSm = 4;

// Persistent grid: enough CTAs for the work, at most one full wave.
int grid_size(int64_t units, int units_per_block, int sm_count, int resident) {
    const int64_t need = (units + units_per_block - 1) / units_per_block;
    const int64_t cap = int64_t(sm_count) * resident;
    return static_cast<int>(need < cap ? need : cap);
}

}  // namespace

// The warp-rows kernel with kRows rows per warp and iteration: a persistent
// grid of at most one full wave, and, when a sweep of that grid holds at
// least one whole token, the sweep cut down to whole tokens (p.sweep_tokens)
// so that every warp keeps its heads (the warps past the last whole token,
// fewer than one token's rows per sweep, stay idle).
template <int kRows, int kMode, bool kGroupMajor>
cudaError_t launch_warp_rows(InvParams p, const DeviceInfo& dev, Variant slot,
                             cudaStream_t stream) {
    constexpr int kWarps = kInvThreads / 32;
    auto k = inv_rope_fp8_quant_kernel<kRows, kMode, kGroupMajor>;
    const int res = std::min(resident_blocks(dev.ordinal, slot, k, kInvThreads), kMaxCtasPerSm);
    const int grid = grid_size(p.n_rows, kWarps * kRows, dev.sm_count, res);
    const int64_t tokens = int64_t(grid) * kWarps * kRows / p.n_heads;
    // more heads per token than one sweep holds (thousands): the layout
    // kernel, which walks the rows, writes the same layout (p.lay)
    if (tokens < 1) return launch_inv_rope_quant_layout(p, dev, stream);
    p.sweep_tokens = static_cast<uint32_t>(tokens);
    return launch_pdl(k, grid, kInvThreads, 0, stream, p);
}

cudaError_t launch_inv_rope_fp8_quant(const InvParams& p, const DeviceInfo& dev, int variant,
                                      cudaStream_t stream) {
    constexpr int kWarps = kInvThreads / 32;
    // The automatic choice is the warp-rows kernel at every size: launched with
    // programmatic serialization, its CTAs (no shared memory) are scheduled
    // into an SM while the previous kernel's CTAs drain, which the stream
    // kernel's one 204 KB CTA per SM cannot be; measured on B300 it is the
    // faster of the two from 2048 tokens x 32 heads up (0.98 vs 0.95 of the
    // copy peak at 16384 tokens).
    if (variant == kInvStream) return launch_inv_rope_fp8_quant_stream(p, dev, stream);
    // warp-rows kernel: two rows (heads of one token) in flight per warp when
    // the grid fills the GPU and the head count is even, one otherwise
    // (decode-sized calls spread over more warps)
    if (int64_t(p.n_rows) >= int64_t(dev.sm_count) * kWarps * 4 && p.n_heads % 2 == 0)
        return launch_warp_rows<2, kOutFp8F32, false>(p, dev, kInv2, stream);
    return launch_warp_rows<1, kOutFp8F32, false>(p, dev, kInv1, stream);
}

template <int kMode>
cudaError_t launch_layout(const InvParams& p, const DeviceInfo& dev, cudaStream_t stream) {
    constexpr int kWarps = kInvThreads / 32;
    // Quantising modes: each warp on fixed heads (two heads of one token when
    // the call fills the GPU and the head count is even), when a sweep of the
    // grid holds a whole token. Measured on B300 at 16384 x 32 heads: fp8 /
    // UE8M0 with transposed scales 134.0 / 126.6 us, group-major with a padded
    // group stride 127.1 / 126.8 us, against 148.6 / 149.4 and 134.7 / 134.7
    // us on the TMA-ring kernel. bf16 output keeps the row walk at one row per
    // warp (166.9 us against 170.2 us with fixed heads, and 0.95 of the copy
    // peak with two rows per warp).
    if (kMode == kOutFp8F32 && p.lay.st == 1) {
        // fp32 scales stored token-contiguous: the token-tiled kernel, when
        // every warp gets at least 6 tiles. Measured on B300 against the
        // fixed-head kernel (us): 16384 x 32 heads 126.3 / 133.2, 12288 x 32
        // 96.8 / 102.1, 8192 x 32 64.5 / 67.3, 16384 x 24 96.9 / 100.8, 8192 x
        // 64 126.8 / 133.9; with fewer tiles per warp its coarser last sweep
        // costs more than the sectors save (8192 x 24, 5.2 tiles per warp:
        // 51.9 / 51.2; 4096 x 32: 33.0 / 31.1). UE8M0 words stay on the
        // fixed-head kernel, whose one word per row already fills a single
        // sector (equal or faster at every size measured).
        auto k = inv_rope_quant_layout_tiled_kernel;
        const int res =
            std::min(resident_blocks(dev.ordinal, kLayTiled, k, kInvThreads), kMaxCtasPerSm);
        const int64_t n_tiles = (int64_t(p.n_tokens) + kScaleTile - 1) / kScaleTile;
        int grid = grid_size(n_tiles * p.n_heads, kWarps, dev.sm_count, res);
        int64_t tiles = int64_t(grid) * kWarps / p.n_heads;  // per sweep
        if (tiles >= 1 && n_tiles >= 6 * tiles) {
            // the same number of sweeps with the tiles spread evenly over them
            const int64_t sweeps = (n_tiles + tiles - 1) / tiles;
            tiles = (n_tiles + sweeps - 1) / sweeps;
            grid = static_cast<int>((tiles * p.n_heads + kWarps - 1) / kWarps);
            InvParams q = p;
            q.sweep_tokens = static_cast<uint32_t>(tiles * kScaleTile);
            return launch_pdl(k, grid, kInvThreads, 0, stream, q);
        }
    }
    if (kMode != kOutBf16) {
        InvParams q = p;
        const bool two = int64_t(p.n_rows) >= int64_t(dev.sm_count) * kWarps * 4 && p.n_heads % 2 == 0;
        if (two) {
            auto k = inv_rope_quant_layout_fixed_kernel<2, kMode>;
            const int res = std::min(
                resident_blocks(dev.ordinal, Variant(kLayFixed + 2 * kMode + 1), k, kInvThreads),
                kMaxCtasPerSm);
            const int grid = grid_size(p.n_rows, kWarps * 2, dev.sm_count, res);
            const int64_t tokens = int64_t(grid) * kWarps * 2 / p.n_heads;
            if (tokens >= 1) {
                q.sweep_tokens = static_cast<uint32_t>(tokens);
                return launch_pdl(k, grid, kInvThreads, 0, stream, q);
            }
        } else {
            auto k = inv_rope_quant_layout_fixed_kernel<1, kMode>;
            const int res = std::min(
                resident_blocks(dev.ordinal, Variant(kLayFixed + 2 * kMode), k, kInvThreads),
                kMaxCtasPerSm);
            const int grid = grid_size(p.n_rows, kWarps, dev.sm_count, res);
            const int64_t tokens = int64_t(grid) * kWarps / p.n_heads;
            if (tokens >= 1) {
                q.sweep_tokens = static_cast<uint32_t>(tokens);
                return launch_pdl(k, grid, kInvThreads, 0, stream, q);
            }
        }
        // more heads per token than a sweep holds: walk the rows
    }
    if (kMode != kOutBf16 && int64_t(p.n_rows) >= int64_t(dev.sm_count) * kWarps * 4) {
        auto k = inv_rope_quant_layout_kernel<2, kMode>;
        const int res = resident_blocks(dev.ordinal, Variant(kLay + 2 * kMode + 1), k, kInvThreads);
        return launch_pdl(k, grid_size(p.n_rows, kWarps * 2, dev.sm_count, res), kInvThreads, 0,
                          stream, p);
    }
    auto k = inv_rope_quant_layout_kernel<1, kMode>;
    const int res = resident_blocks(dev.ordinal, Variant(kLay + 2 * kMode), k, kInvThreads);
    return launch_pdl(k, grid_size(p.n_rows, kWarps * 1, dev.sm_count, res), kInvThreads, 0,
                      stream, p);
}

template <int kMode, bool kGroupMajor>
cudaError_t launch_rows(const InvParams& p, const DeviceInfo& dev, cudaStream_t stream) {
    constexpr int kWarps = kInvThreads / 32;
    constexpr int kSlot = kRowsVariant + 4 * kMode + (kGroupMajor ? 2 : 0);
    if (int64_t(p.n_rows) >= int64_t(dev.sm_count) * kWarps * 4 && p.n_heads % 2 == 0)
        return launch_warp_rows<2, kMode, kGroupMajor>(p, dev, Variant(kSlot + 1), stream);
    return launch_warp_rows<1, kMode, kGroupMajor>(p, dev, Variant(kSlot), stream);
}

cudaError_t launch_inv_rope_rows(const InvParams& p, const DeviceInfo& dev, int mode,
                                 bool group_major, cudaStream_t stream) {
    if (group_major)
        return mode == kOutFp8F32 ? launch_rows<kOutFp8F32, true>(p, dev, stream)
                                  : launch_rows<kOutFp8Ue8m0, true>(p, dev, stream);
    if (mode == kOutFp8F32) return launch_inv_rope_fp8_quant(p, dev, kInvWarpRows, stream);
    return launch_rows<kOutFp8Ue8m0, false>(p, dev, stream);
}

cudaError_t launch_inv_rope_quant_layout(const InvParams& p, const DeviceInfo& dev,
                                         cudaStream_t stream) {
    switch (p.lay.mode) {
        case kOutFp8F32: return launch_layout<kOutFp8F32>(p, dev, stream);
        case kOutFp8Ue8m0: return launch_layout<kOutFp8Ue8m0>(p, dev, stream);
        default: return launch_layout<kOutBf16>(p, dev, stream);
    }
}

cudaError_t launch_rope_fp8_quant_insert(const InsParams& p, const DeviceInfo& dev,
                                         cudaStream_t stream) {
    constexpr int kWarps = kInsThreads / 32;
    // one token per warp and iteration (44 registers, more CTAs per SM): the
    // 30 MB op is latency-bound, and on B300 this ran it in 4.9 us against
    // 5.7 us with two tokens per warp (CUDA-graph replays)
    auto k = rope_fp8_quant_insert_kernel<1>;
    const int res = resident_blocks(dev.ordinal, kIns1, k, kInsThreads);
    return launch_pdl(k, grid_size(p.n_tokens, kWarps * 1, dev.sm_count, res), kInsThreads, 0,
                      stream, p);
}

cudaError_t launch_qnorm_rope_kv_insert(const FusedParams& p, const DeviceInfo& dev,
                                        cudaStream_t stream) {
    constexpr int kWarps = kInvThreads / 32;
    // one unit per warp and iteration at every size: 63 registers, 4 CTAs per
    // SM; two units per warp need 80 registers (3 CTAs) and measured 7% slower
    auto k = qnorm_rope_kv_insert_kernel<1>;
    const int res = resident_blocks(dev.ordinal, kFus1, k, kInvThreads);
    return launch_pdl(k, grid_size(p.n_units, kWarps * 1, dev.sm_count, res), kInvThreads, 0,
                      stream, p);
}

}  // namespace rq
