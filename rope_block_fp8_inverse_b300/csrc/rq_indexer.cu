// rq_indexer.cu -- the indexer q op of "[vllm] vLLM의 GLM5.2 성능 최적화: Triton
// 커널 융합을 통한 E2E Throughput 향상" (vLLM PR #46862 analysis), S1: RoPE on
// the rotary dims of each 128-wide q head, the rotated values rounded through
// bf16, one power-of-two FP8 scale per head, and that scale folded into the
// head's indexer weight, weight * q_scale * softmax_scale * head_scale.
//
// Lane layout: a head is 16 chunks of 8 elements; 8 lanes own one head and a
// warp holds 4 heads. Lane m (0..7) of a head owns chunks A = m and B = m + 4
// when m < 4 (the 64 rotary dims) and A = m + 4, B = m + 8 when m >= 4, so
//  * NeoX pairs (dim j with dim 32 + j) are element k of A and element k of
//    B of the same lane (j = 8m + k), and GPT-J pairs (2j, 2j + 1) sit inside
//    one chunk: the partner is always in the thread's registers;
//  * the head's amax is a 3-step xor reduction over its 8 lanes.
#include "rq_device.cuh"
#include "rq_launch.h"

namespace rq {

namespace {

constexpr int kIdxDim = 128;

// Round to bf16 and back (the page's .to(bfloat16).to(float32)), two values.
__device__ __forceinline__ void round_bf16_pair(float& a, float& b) {
    const uint32_t w = bf16x2(a, b);
    a = __uint_as_float(w << 16);
    b = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ void unpack8(uint4 w, float (&v)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// Forward rotation of one pair, each product and sum rounded on its own.
__device__ __forceinline__ void rot(float& x0, float& x1, float c, float s) {
    const float r0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
    const float r1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
    x0 = r0;
    x1 = r1;
}

__device__ __forceinline__ uint2 quant8(const float (&v)[8], float inv) {
    uint2 q;
    q.x = e4m3x2(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv)) |
          (e4m3x2(__fmul_rn(v[2], inv), __fmul_rn(v[3], inv)) << 16);
    q.y = e4m3x2(__fmul_rn(v[4], inv), __fmul_rn(v[5], inv)) |
          (e4m3x2(__fmul_rn(v[6], inv), __fmul_rn(v[7], inv)) << 16);
    return q;
}

}  // namespace

template <bool kNeox>
__global__ void __launch_bounds__(kInvThreads)
indexer_q_rope_quant_kernel(IdxParams p) {
    const int lane = threadIdx.x & 31;
    const int rs = lane >> 3;           // head slot within the warp
    const int m = lane & 7;             // lane within the head
    const bool rope_lane = m < 4;
    const int ca = rope_lane ? m : m + 4;
    const int cb = ca + 4;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    const uint16_t* __restrict__ q = static_cast<const uint16_t*>(p.q);
    const uint32_t n_groups = (p.n_rows + 3) / 4;

    for (uint32_t g0 = warp; g0 < n_groups; g0 += n_warps) {
        const uint32_t r = g0 * 4 + rs;
        const bool row_ok = r < p.n_rows;  // uniform within the head's 8 lanes
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0, s0 = c0, s1 = c0;
        bool live = false;
        if (row_ok) {
            const uint32_t t = r / p.n_heads;
            const uint32_t h = r - t * p.n_heads;
            const uint16_t* row = q + int64_t(t) * p.sq_t + int64_t(h) * p.sq_h;
            a = ld_stream16(row + 8 * ca);
            b = ld_stream16(row + 8 * cb);
            const int64_t pos = __ldg(p.positions + t);
            live = static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
            if (live && rope_lane) {
                const float* cs = p.cache + pos * kCacheWidth;
                // NeoX: pairs j = 8m .. 8m+7; GPT-J: chunk A pairs 4m .. 4m+3,
                // chunk B pairs 16 + 4m .. 16 + 4m + 3
                const int j0 = kNeox ? 8 * m : 4 * m;
                const int j1 = kNeox ? 8 * m + 4 : 16 + 4 * m;
                c0 = ld_ro16(cs + j0);
                c1 = ld_ro16(cs + j1);
                s0 = ld_ro16(cs + kHalfRope + j0);
                s1 = ld_ro16(cs + kHalfRope + j1);
            } else if (!live && m == 0 && p.error_flags) {
                atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
            }
        }
        float va[8], vb[8];
        unpack8(a, va);
        unpack8(b, vb);
        if (rope_lane) {
            const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
            if (kNeox) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    rot(va[k], vb[k], c[k], s[k]);
                    round_bf16_pair(va[k], vb[k]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    rot(va[2 * i], va[2 * i + 1], c[i], s[i]);
                    rot(vb[2 * i], vb[2 * i + 1], c[4 + i], s[4 + i]);
                    round_bf16_pair(va[2 * i], va[2 * i + 1]);
                    round_bf16_pair(vb[2 * i], vb[2 * i + 1]);
                }
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fmaxf(fabsf(va[k]), fabsf(vb[k])));
        const uint32_t sb = scale_bits(fmaxf(block_max(amax), p.eps));
        const float inv = inv_scale(sb);
        const uint2 qa = quant8(va, inv), qb = quant8(vb, inv);
        if (live) {
            uint8_t* dst = p.out + int64_t(r) * kIdxDim;
            st_stream8(dst + 8 * ca, qa.x, qa.y);
            st_stream8(dst + 8 * cb, qb.x, qb.y);
            if (m == 0) {
                const float w0 = __fmul_rn(__ldg(p.weights + r), __uint_as_float(sb));
                st_stream4f(p.weights_out + r,
                            __fmul_rn(__fmul_rn(w0, p.softmax_scale), p.head_scale));
            }
        }
    }
}

namespace {

// Resident CTAs per SM of each style's kernel, queried once per device.
int idx_resident(int device, bool neox) {
    constexpr int kMax = 64;
    static thread_local int cache[kMax][2] = {};
    const int d = (device >= 0 && device < kMax) ? device : 0;
    int& n = cache[d][neox ? 1 : 0];
    if (n == 0) {
        const cudaError_t e =
            neox ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &n, indexer_q_rope_quant_kernel<true>, kInvThreads, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &n, indexer_q_rope_quant_kernel<false>, kInvThreads, 0);
        if (e != cudaSuccess || n < 1) n = 1;
    }
    return n;
}

}  // namespace

cudaError_t launch_indexer_q_rope_quant(const IdxParams& p, const DeviceInfo& dev,
                                        cudaStream_t stream) {
    constexpr int kWarps = kInvThreads / 32;
    const int64_t groups = (int64_t(p.n_rows) + 3) / 4;
    const int64_t need = (groups + kWarps - 1) / kWarps;
    const int64_t cap = int64_t(dev.sm_count) * idx_resident(dev.ordinal, p.neox);
    const int grid = static_cast<int>(need < cap ? need : cap);
    if (p.neox)
        indexer_q_rope_quant_kernel<true><<<grid, kInvThreads, 0, stream>>>(p);
    else
        indexer_q_rope_quant_kernel<false><<<grid, kInvThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rq
