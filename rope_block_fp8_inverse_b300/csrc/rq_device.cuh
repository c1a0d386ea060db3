// rq_device.cuh -- per-row device arithmetic shared by every kernel of the
// library (sm_103a).
//
// Work unit: one 512-wide head row (one (token, head) of the inverse op, one
// token of the insert op), owned by one warp, in the "block-interleaved" lane
// layout: lane l owns two 8-element chunks,
//     A = 16 * (l / 8) + l % 8   and   B = A + 8,
// both inside 128-element block l / 8. So
//  * each lane has exactly one block scale, and a block's amax is a 3-step
//    xor reduction over 8 lanes;
//  * a warp-wide 16-byte access to every lane's A chunk (or B chunk) touches
//    four whole 128-byte segments: coalesced in global memory, free of bank
//    conflicts in shared memory;
//  * dims 448..511 are the B chunks of lanes 24..31, and a chunk holds four
//    whole (even, odd) pairs, so the RoPE partner is in the same thread's
//    registers (no shuffle, no second read): lane l rotates pairs
//    4(l-24) .. 4(l-24)+3.
//
// Arithmetic follows "[vllm] 한 프로그램이 4개 head를 처리하게 하라: DeepSeek-V4
// inverse RoPE + FP8 quant 커널 3.5배 가속기" (vLLM PR #63540 analysis):
// S2 for the pair rotation, S3 for the block amax; the power-of-two scale
// 2^ceil(log2(amax/448)) follows "[vllm] vLLM의 GLM5.2 성능 최적화" S1.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rq {

constexpr int kHeadDim = 512;
constexpr int kRopeLane0 = 24;      // first lane whose B chunk is >= dim 448
constexpr int kCacheWidth = 64;     // cos | sin
constexpr int kHalfRope = 32;
constexpr int kRecordBytes = 528;   // paged record: 512 codes + 4 fp32 scales
constexpr unsigned kFull = 0xffffffffu;

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream drains;
// pdl_wait() blocks until that kernel has completed and its memory is
// visible, so it must come before the first global access. Without PDL
// both are no-ops. pdl_launch_dependents() lets the next such kernel be
// scheduled (its own pdl_wait() still waits for this one to finish).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Position of row r = t * n_heads + h of the [N, H] row space, with head h =
// g * hpg + i (group g, head i within it), advanced by a fixed row stride with
// no division: the persistent warp-rows kernels step every warp by the same
// stride, so only the set-up divides.
struct RowPos {
    uint32_t t, h, g, i;
};

struct RowStride {
    uint32_t dt, dh, dg, di;
};

__device__ __forceinline__ RowPos row_pos(uint32_t r, uint32_t n_heads, uint32_t hpg) {
    RowPos w;
    w.t = r / n_heads;
    w.h = r - w.t * n_heads;
    w.g = w.h / hpg;
    w.i = w.h - w.g * hpg;
    return w;
}

__device__ __forceinline__ RowStride row_stride(uint32_t d, uint32_t n_heads, uint32_t hpg) {
    const RowPos q = row_pos(d, n_heads, hpg);
    return RowStride{q.t, q.h, q.g, q.i};
}

// w += s rows (n_heads = groups * hpg).
__device__ __forceinline__ void row_advance(RowPos& w, const RowStride& s, uint32_t n_heads,
                                            uint32_t hpg, uint32_t groups) {
    w.t += s.dt;
    w.h += s.dh;
    w.g += s.dg;
    w.i += s.di;
    if (w.i >= hpg) {
        w.i -= hpg;
        ++w.g;
    }
    if (w.h >= n_heads) {
        w.h -= n_heads;
        ++w.t;
        w.g -= groups;
    }
}

// Index (in 8-element chunks) of lane l's A chunk; its B chunk is A + 8.
__device__ __forceinline__ int chunk_a(int lane) { return 16 * (lane >> 3) + (lane & 7); }

// Streaming 16-byte read of data touched once: read-only path, no L1 line.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte read of data re-read by other warps (cos/sin rows): read-only path.
__device__ __forceinline__ float4 ld_ro16(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ uint4 ld_ro16u(const uint16_t* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

// Streaming stores (evict-first in L2: written once, read by a later op).
__device__ __forceinline__ void st_stream8(void* p, uint32_t lo, uint32_t hi) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(lo), "r"(hi) : "memory");
}

__device__ __forceinline__ void st_stream4f(void* p, float v) {
    asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// The lane's 16 elements as 8 (even, odd) pairs, two pairs per packed
// register: ev[i] = (even of pair 2i, even of pair 2i+1), od[i] likewise.
// Pairs 0-3 are chunk A, pairs 4-7 chunk B. bf16 -> fp32 is exact (bf16 is
// the top half of an fp32).
struct Pairs {
    float2 ev[4], od[4];
};

__device__ __forceinline__ Pairs unpack(uint4 a, uint4 b) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    Pairs p;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        p.ev[i] = make_float2(__uint_as_float(w[2 * i] << 16), __uint_as_float(w[2 * i + 1] << 16));
        p.od[i] = make_float2(__uint_as_float(w[2 * i] & 0xffff0000u),
                              __uint_as_float(w[2 * i + 1] & 0xffff0000u));
    }
    return p;
}

// Rotate the four pairs of chunk B with cos c4 and sin s4 (one value per
// pair). Every product and every sum is rounded on its own, in the page's
// order (S2): inverse  even' = even*c + odd*s,  odd' = odd*c - even*s;
//             forward  even' = even*c - odd*s,  odd' = odd*c + even*s.
// Scalar __fmul_rn / __fadd_rn / __fsub_rn are never contracted into an FMA;
// packed fp32x2 arithmetic is not used here because ptxas may fuse it, which
// moves values that sit exactly on an e4m3 rounding tie.
template <bool kInverse>
__device__ __forceinline__ void rotate_b(Pairs& p, float4 c4, float4 s4) {
    const float c[4] = {c4.x, c4.y, c4.z, c4.w};
    const float s[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float& e = (k & 1) ? p.ev[2 + k / 2].y : p.ev[2 + k / 2].x;
        float& o = (k & 1) ? p.od[2 + k / 2].y : p.od[2 + k / 2].x;
        const float ec = __fmul_rn(e, c[k]), os = __fmul_rn(o, s[k]);
        const float oc = __fmul_rn(o, c[k]), es = __fmul_rn(e, s[k]);
        if (kInverse) {
            e = __fadd_rn(ec, os);
            o = __fsub_rn(oc, es);
        } else {
            e = __fsub_rn(ec, os);
            o = __fadd_rn(oc, es);
        }
    }
}

__device__ __forceinline__ float absmax(const Pairs& p) {
    float m0 = fmaxf(fabsf(p.ev[0].x), fabsf(p.ev[0].y));
    float m1 = fmaxf(fabsf(p.od[0].x), fabsf(p.od[0].y));
#pragma unroll
    for (int i = 1; i < 4; ++i) {
        m0 = fmaxf(m0, fmaxf(fabsf(p.ev[i].x), fabsf(p.ev[i].y)));
        m1 = fmaxf(m1, fmaxf(fabsf(p.od[i].x), fabsf(p.od[i].y)));
    }
    return fmaxf(m0, m1);
}

// max over the 8 lanes of this lane's block (xor offsets stay in aligned
// 8-lane groups)
__device__ __forceinline__ float block_max(float m) {
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    return m;
}

// Bit pattern of the block scale 2^e, e = ceil(log2(fl32(amax / 448))), read
// off amax's bits without dividing. With amax = 1.m * 2^E normal, round-to-
// nearest-even gives fl32(amax/448) <= 2^k exactly when amax/448 <=
// 2^k (1 + 2^-24), and since no fp32 value lies in (1.75 * 2^(k+8),
// 1.75 * 2^(k+8) (1 + 2^-24)] that is amax <= 1.75 * 2^(k+8). So e = E - 8
// when the mantissa field is <= 0x600000 and E - 7 otherwise. Adding 0x1fffff
// to amax's bits carries into the exponent field exactly when the mantissa
// field exceeds 0x600000, so the masked sum holds the biased E or E + 1, and
// subtracting 8 << 23 rebiases it to e. Valid for normal amax >= 0 (the ABI
// keeps amax >= eps >= 2^-100, and e stays within [-108, 120]).
__device__ __forceinline__ uint32_t scale_bits(float amax) {
    return ((__float_as_uint(amax) + 0x1fffffu) & 0x7f800000u) - (8u << 23);
}

// 2^-e from the bits of 2^e (both normal for e in [-108, 120]).
__device__ __forceinline__ float inv_scale(uint32_t sbits) {
    return __uint_as_float((254u << 23) - sbits);
}

// cvt.rn.satfinite.e4m3x2.f32 d, a, b puts a in the upper byte and b in the
// lower byte: pass (odd, even) so the even element lands at the lower address.
__device__ __forceinline__ uint32_t e4m3x2(float even, float odd) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(odd), "f"(even));
    return r;
}

// Exact power-of-two scaling of two values at once (mul.rn.f32x2). The result
// feeds only the e4m3 conversion, so no contraction can change it.
__device__ __forceinline__ float2 mul2_exact(float2 a, float2 b) { return __fmul2_rn(a, b); }

// 16 values times an exact power-of-two inverse scale -> 16 e4m3 codes in
// element order (even of pair k at byte 2k, odd at byte 2k+1): x, y hold
// chunk A's 8 codes, z, w chunk B's.
__device__ __forceinline__ uint4 quant16(const Pairs& p, float inv) {
    const float2 iv = make_float2(inv, inv);
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 e = mul2_exact(p.ev[i], iv);
        const float2 o = mul2_exact(p.od[i], iv);
        q[i] = e4m3x2(e.x, o.x) | (e4m3x2(e.y, o.y) << 16);
    }
    return make_uint4(q[0], q[1], q[2], q[3]);
}

// One row for one lane: chunks a (A) and b (B) as bf16 x8; rope lanes pass
// the cos / sin of their four pairs. Returns the 16 codes and sets *scale to
// the lane's block scale.
template <bool kInverse>
__device__ __forceinline__ uint4 rope_quant_row(uint4 a, uint4 b, bool rope_lane, float4 c4,
                                                float4 s4, float eps, float* scale) {
    Pairs p = unpack(a, b);
    if (rope_lane) rotate_b<kInverse>(p, c4, s4);
    const uint32_t sb = scale_bits(fmaxf(block_max(absmax(p)), eps));
    *scale = __uint_as_float(sb);
    return quant16(p, inv_scale(sb));
}

// Two fp32 values -> one bf16x2 word, each rounded to nearest even (the
// first value at the lower address). cvt.rn.bf16x2.f32 d, a, b puts a in the
// upper half.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The non-quantising row: rotation only, then bf16. Returns chunk A's 8
// values in *qa and chunk B's in *qb, in element order.
template <bool kInverse>
__device__ __forceinline__ void rope_row_bf16(uint4 a, uint4 b, bool rope_lane, float4 c4,
                                              float4 s4, uint4* qa, uint4* qb) {
    Pairs p = unpack(a, b);
    if (rope_lane) rotate_b<kInverse>(p, c4, s4);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w[2 * i] = bf16x2(p.ev[i].x, p.od[i].x);
        w[2 * i + 1] = bf16x2(p.ev[i].y, p.od[i].y);
    }
    *qa = make_uint4(w[0], w[1], w[2], w[3]);
    *qb = make_uint4(w[4], w[5], w[6], w[7]);
}

// Sum over the whole warp (xor butterfly).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
    return v;
}

// One q head of the fused q/kv op: RMS norm over its 512 values (no weight),
// then the forward rotation of the RoPE tail, then bf16 (round to nearest
// even). fp32 throughout: sum of squares with fused multiply-adds, a
// correctly rounded reciprocal square root. Returns chunk A's 8 values in
// *qa and chunk B's in *qb.
__device__ __forceinline__ void qnorm_rope_row_bf16(uint4 a, uint4 b, bool rope_lane, float4 c4,
                                                    float4 s4, float eps, const uint16_t* weight,
                                                    int ca, uint4* qa, uint4* qb) {
    Pairs p = unpack(a, b);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ss = __fmaf_rn(p.ev[i].x, p.ev[i].x, ss);
        ss = __fmaf_rn(p.ev[i].y, p.ev[i].y, ss);
        ss = __fmaf_rn(p.od[i].x, p.od[i].x, ss);
        ss = __fmaf_rn(p.od[i].y, p.od[i].y, ss);
    }
    ss = warp_sum(ss);
    const float r = __frsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / kHeadDim), eps));
    const float2 rr = make_float2(r, r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        p.ev[i] = __fmul2_rn(p.ev[i], rr);
        p.od[i] = __fmul2_rn(p.od[i], rr);
    }
    if (weight) {  // the norm's per-dimension weight (same chunks as the row), before the rotation
        const Pairs w = unpack(ld_ro16u(weight + 8 * ca), ld_ro16u(weight + 8 * (ca + 8)));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            p.ev[i] = __fmul2_rn(p.ev[i], w.ev[i]);
            p.od[i] = __fmul2_rn(p.od[i], w.od[i]);
        }
    }
    if (rope_lane) rotate_b<false>(p, c4, s4);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w[2 * i] = bf16x2(p.ev[i].x, p.od[i].x);
        w[2 * i + 1] = bf16x2(p.ev[i].y, p.od[i].y);
    }
    *qa = make_uint4(w[0], w[1], w[2], w[3]);
    *qb = make_uint4(w[4], w[5], w[6], w[7]);
}

__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream1(void* p, uint32_t v) {
    asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Store one quantised row: 8 codes of chunk A, 8 of chunk B, and (from the
// first lane of each block) the block's fp32 scale.
__device__ __forceinline__ void store_row(uint8_t* codes, float* scales4, int lane, int ca,
                                          uint4 q, float scale) {
    st_stream8(codes + 8 * ca, q.x, q.y);
    st_stream8(codes + 8 * (ca + 8), q.z, q.w);
    if ((lane & 7) == 0) st_stream4f(scales4 + (lane >> 3), scale);
}

}  // namespace rq
