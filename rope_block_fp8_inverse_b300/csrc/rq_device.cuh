// rq_device.cuh -- per-row device arithmetic shared by the inverse and the
// insert kernels (sm_103a).
//
// Work unit: one 512-wide head row (one (token, head) of the inverse op, one
// token of the insert op), owned by one warp. Lane l holds elements
// [8l, 8l+8) ("half A", blocks 0-1) and [256+8l, 256+8l+8) ("half B",
// blocks 2-3), so each 16-byte load instruction of the warp reads 512
// contiguous bytes and each 8-byte store writes 256 contiguous bytes. A
// lane's 8 elements are 4 whole (even, odd) pairs, so the RoPE partner is
// in the same thread's registers (no shuffle, no second read). Lanes 24-31
// of half B hold dims 448..511, the 32 rotated pairs: lane l rotates pairs
// 4(l-24) .. 4(l-24)+3. A 128-element block is 16 lanes of one half, so the
// block amax is a 4-step xor-shuffle within 16 lanes.
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
constexpr int kHalf = 256;          // elements per half-row
constexpr int kRopeLane0 = 24;      // first lane whose half-B elements are >= 448
constexpr int kCacheWidth = 64;     // cos | sin
constexpr int kHalfRope = 32;
constexpr int kRecordBytes = 528;   // paged record: 512 codes + 4 fp32 scales
constexpr unsigned kFull = 0xffffffffu;

// Streaming 16-byte read of data touched once: read-only path, no L1 line.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte read of data re-read by other warps (cos/sin rows): read-only path.
__device__ __forceinline__ float4 ld_shared_ro16(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

// Streaming 8-byte store (evict-first in L2: written once, read by a later op).
__device__ __forceinline__ void st_stream8(void* p, uint32_t lo, uint32_t hi) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(lo), "r"(hi) : "memory");
}

__device__ __forceinline__ void st_stream16f(void* p, float a, float b, float c, float d) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

// bf16 pair in one 32-bit word -> two fp32 (exact: bf16 is the top half).
__device__ __forceinline__ void unpack_bf16x8(const uint4 w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// Rotate the 4 (even, odd) pairs of f with cos c[i], sin s[i]; every product
// and every sum is rounded on its own (no FMA contraction).
template <bool kInverse>
__device__ __forceinline__ void rotate4(float (&f)[8], const float4 c4, const float4 s4) {
    const float c[4] = {c4.x, c4.y, c4.z, c4.w};
    const float s[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float e = f[2 * i], o = f[2 * i + 1];
        const float ec = __fmul_rn(e, c[i]), os = __fmul_rn(o, s[i]);
        const float oc = __fmul_rn(o, c[i]), es = __fmul_rn(e, s[i]);
        if (kInverse) {
            f[2 * i] = __fadd_rn(ec, os);
            f[2 * i + 1] = __fsub_rn(oc, es);
        } else {
            f[2 * i] = __fsub_rn(ec, os);
            f[2 * i + 1] = __fadd_rn(oc, es);
        }
    }
}

__device__ __forceinline__ float absmax8(const float (&f)[8]) {
    float m = fabsf(f[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    return m;
}

// max over the 16 lanes of this lane's half-warp (xor offsets stay inside
// aligned 16-lane groups).
__device__ __forceinline__ float halfwarp_max(float m) {
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    return m;
}

// Exponent of the block scale, e = ceil(log2(fl32(amax / 448))), read off
// amax's bits without dividing. With amax = 1.m * 2^E normal and k an
// integer, round-to-nearest-even gives fl32(amax/448) <= 2^k exactly when
// amax/448 <= 2^k * (1 + 2^-24), and since no fp32 value lies in
// (1.75 * 2^(k+8), 1.75 * 2^(k+8) * (1 + 2^-24)] that is amax <= 1.75 * 2^(k+8).
// So e = E - 8 when 1.m <= 1.75 (mantissa field <= 0x600000), else E - 7.
// Valid for normal amax (the ABI keeps amax >= eps >= 2^-100).
__device__ __forceinline__ int scale_exponent(float amax) {
    const uint32_t u = __float_as_uint(amax);
    const int E = static_cast<int>((u >> 23) & 0xffu) - 127;
    return E - 8 + ((u & 0x7fffffu) > 0x600000u ? 1 : 0);
}

__device__ __forceinline__ float pow2f(int e) {  // e in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// cvt.rn.satfinite.e4m3x2.f32 d, a, b puts a in the upper byte and b in the
// lower byte: pass (odd, even) so the even element lands at the lower address.
__device__ __forceinline__ uint32_t e4m3x2(float even, float odd) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(odd), "f"(even));
    return r;
}

// 8 fp32 values times an exact power-of-two inverse scale -> 8 e4m3 codes.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float inv) {
    uint2 q;
    q.x = e4m3x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv)) |
          (e4m3x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv)) << 16);
    q.y = e4m3x2(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv)) |
          (e4m3x2(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv)) << 16);
    return q;
}

// Loaded operands of one row for one lane.
struct RowRegs {
    uint4 a, b;      // half A / half B bf16 x8
    float4 c, s;     // cos / sin of this lane's 4 pairs (lanes 24..31 only)
};

// Quantised result of one row for one lane.
struct RowOut {
    uint2 qa, qb;    // 8 codes of half A, 8 of half B
    float sa, sb;    // this lane's block scales (block lane/16, 2 + lane/16)
};

template <bool kInverse>
__device__ __forceinline__ RowOut rope_quant_row(const RowRegs& in, int lane, float eps) {
    float fa[8], fb[8];
    unpack_bf16x8(in.a, fa);
    unpack_bf16x8(in.b, fb);
    if (lane >= kRopeLane0) rotate4<kInverse>(fb, in.c, in.s);
    float ma = halfwarp_max(absmax8(fa));
    float mb = halfwarp_max(absmax8(fb));
    ma = fmaxf(ma, eps);
    mb = fmaxf(mb, eps);
    const int ea = scale_exponent(ma);
    const int eb = scale_exponent(mb);
    RowOut o;
    o.qa = quant8(fa, pow2f(-ea));
    o.qb = quant8(fb, pow2f(-eb));
    o.sa = pow2f(ea);
    o.sb = pow2f(eb);
    return o;
}

}  // namespace rq
