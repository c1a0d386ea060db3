// rq_indexer.cu -- the indexer q op of "[vllm] vLLM의 GLM5.2 성능 최적화: Triton
// 커널 융합을 통한 E2E Throughput 향상" (vLLM PR #46862 analysis), S1: RoPE on
// the rotary dims of each 128-wide q head, the rotated values rounded through
// bf16, one power-of-two FP8 scale per head, and that scale folded into the
// head's indexer weight, weight * q_scale * softmax_scale * head_scale.
//
// Lane layout: 8 lanes own one head and a warp holds 4 heads. Half of a
// head's 128 dims are rotary (dims 0..63, 32 pairs), so the rotation is
// spread over all 8 lanes: lane m (0..7) owns the four pairs j = 4m .. 4m+3
// (NeoX: dims j and 32 + j, two 8-byte pieces; GPT-J: dims 2j and 2j + 1,
// one 16-byte chunk) and the 8 non-rotary dims 64 + 8m .. 64 + 8m + 7. Every
// lane rotates the same number of pairs (no divergence) with the partner in
// its own registers, and the head's amax is a 3-step xor reduction over its
// 8 lanes.
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

// A warp takes kIdxGroups x 4 consecutive heads per iteration and issues all
// their loads and position reads before computing any; cos/sin rows are read
// in the compute phase (after the first head of a token they hit L1). Memory
// parallelism comes from occupancy rather than depth: one group per warp
// keeps the kernel at 32 registers, so 8 CTAs (64 warps) fit on an SM, which
// measured faster than 2 or 4 groups at lower occupancy (every such variant
// wrote the same bytes). The launcher takes the fixed-head form of the kernel
// whenever a sweep of the grid can be cut to whole tokens (measured on B300
// at 16384 x 64 heads: 66.7 against 67.4 us with a division per row); the
// row-walk form remains for the shapes where it cannot.
constexpr int kIdxGroups = 1;
constexpr int kIdxMinBlocks = 8;

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream4(void* p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// One 128-wide head, 8 lanes: rotation, bf16 rounding, the head's scale,
// codes, and the folded weight (lane m == 0). x0 / x1: the lane's four
// rotary pairs as loaded; nv: its 8 non-rotary values.
template <bool kNeox>
__device__ __forceinline__ void indexer_head(const IdxParams& p, uint4 rp, uint4 np, int64_t pos,
                                             bool live, int m, int nc, uint8_t* dst,
                                             const float* weight, float* weight_out) {
    float x0[4], x1[4], nv[8];
    if (kNeox) {
        float lo[4], hi[4];
        const uint32_t w[4] = {rp.x, rp.y, rp.z, rp.w};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            lo[2 * i] = __uint_as_float(w[i] << 16);
            lo[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            hi[2 * i] = __uint_as_float(w[2 + i] << 16);
            hi[2 * i + 1] = __uint_as_float(w[2 + i] & 0xffff0000u);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x0[i] = lo[i];
            x1[i] = hi[i];
        }
    } else {
        float v[8];
        unpack8(rp, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x0[i] = v[2 * i];
            x1[i] = v[2 * i + 1];
        }
    }
    unpack8(np, nv);
    if (live) {
        const float* cs = p.cache + pos * kCacheWidth + 4 * m;
        const float4 c4 = ld_ro16(cs), s4 = ld_ro16(cs + kHalfRope);
        const float c[4] = {c4.x, c4.y, c4.z, c4.w};
        const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            rot(x0[i], x1[i], c[i], sn[i]);
            round_bf16_pair(x0[i], x1[i]);
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(x0[i]), fabsf(x1[i])));
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(nv[i]));
    const uint32_t sb = scale_bits(fmaxf(block_max(amax), p.eps));
    const float inv = inv_scale(sb);
    const uint2 qn = quant8(nv, inv);
    if (live) {
        if (kNeox) {
            const uint32_t q0 = e4m3x2(__fmul_rn(x0[0], inv), __fmul_rn(x0[1], inv)) |
                                (e4m3x2(__fmul_rn(x0[2], inv), __fmul_rn(x0[3], inv)) << 16);
            const uint32_t q1 = e4m3x2(__fmul_rn(x1[0], inv), __fmul_rn(x1[1], inv)) |
                                (e4m3x2(__fmul_rn(x1[2], inv), __fmul_rn(x1[3], inv)) << 16);
            st_stream4(dst + 4 * m, q0);
            st_stream4(dst + 32 + 4 * m, q1);
        } else {
            const float v[8] = {x0[0], x1[0], x0[1], x1[1], x0[2], x1[2], x0[3], x1[3]};
            const uint2 qr = quant8(v, inv);
            st_stream8(dst + 8 * m, qr.x, qr.y);
        }
        st_stream8(dst + 8 * nc, qn.x, qn.y);
        if (m == 0) {
            const float w0 = __fmul_rn(__ldg(weight), __uint_as_float(sb));
            st_stream4f(weight_out, __fmul_rn(__fmul_rn(w0, p.softmax_scale), p.head_scale));
        }
    }
}

// The kernel with every 8-lane head slot on a fixed head: a sweep of the
// grid is p.sweep_tokens whole tokens, so slot rs of warp w keeps head h of
// row w * 4 + rs in every sweep, its token advancing by sweep_tokens, and
// its input, position and outputs by constant steps (no per-row division).
template <bool kNeox>
__global__ void __launch_bounds__(kInvThreads, kIdxMinBlocks)
indexer_q_rope_quant_fixed_kernel(IdxParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int rs = lane >> 3;           // head slot within a group of 4
    const int m = lane & 7;             // lane within the head: pairs 4m .. 4m+3
    const int nc = 8 + m;               // the lane's non-rotary chunk
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t sweep_rows = p.sweep_tokens * p.n_heads;  // a multiple of 4
    if (warp * 4 >= sweep_rows) return;  // warp-uniform: idle warps of the grid
    const uint32_t n_tokens = p.n_rows / p.n_heads;
    uint32_t r = warp * 4 + rs;
    uint32_t t = r / p.n_heads;
    const uint16_t* row = static_cast<const uint16_t*>(p.q) + int64_t(t) * p.sq_t +
                          int64_t(r - t * p.n_heads) * p.sq_h;
    const int64_t drow = int64_t(p.sweep_tokens) * p.sq_t;
    // slot 0 has the smallest token: the warp has work while it is in range
    for (; __shfl_sync(kFull, t, 0) < n_tokens;
         t += p.sweep_tokens, row += drow, r += sweep_rows) {
        const bool in = t < n_tokens;  // uniform within the head's 8 lanes
        uint4 rp = make_uint4(0, 0, 0, 0), np = rp;
        int64_t pos = 0;
        bool live = false;
        if (in) {
            if (kNeox) {
                const uint2 lo = ld_stream8(row + 4 * m);          // dims 4m .. 4m+3
                const uint2 hi = ld_stream8(row + 32 + 4 * m);     // dims 32+4m .. 32+4m+3
                rp = make_uint4(lo.x, lo.y, hi.x, hi.y);
            } else {
                rp = ld_stream16(row + 8 * m);                     // dims 8m .. 8m+7
            }
            np = ld_stream16(row + 8 * nc);
            pos = __ldg(p.positions + t);
            live = static_cast<uint64_t>(pos) < static_cast<uint64_t>(p.cache_rows);
            if (!live && m == 0 && p.error_flags) atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
        }
        indexer_head<kNeox>(p, rp, np, pos, live, m, nc, p.out + int64_t(r) * kIdxDim,
                            p.weights + r, p.weights_out + r);
    }
}

template <bool kNeox>
__global__ void __launch_bounds__(kInvThreads, kIdxMinBlocks)
indexer_q_rope_quant_kernel(IdxParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int rs = lane >> 3;           // head slot within a group of 4
    const int m = lane & 7;             // lane within the head: pairs 4m .. 4m+3
    const int nc = 8 + m;               // the lane's non-rotary chunk
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
    const uint16_t* __restrict__ q = static_cast<const uint16_t*>(p.q);
    constexpr uint32_t kRowsPerIter = 4 * kIdxGroups;

    for (uint32_t base = warp * kRowsPerIter; base < p.n_rows; base += n_warps * kRowsPerIter) {
        uint4 rp[kIdxGroups], np[kIdxGroups];  // rotary words (NeoX: x = lo, y = hi), other chunk
        int64_t pos[kIdxGroups];
        bool live[kIdxGroups];
#pragma unroll
        for (int k = 0; k < kIdxGroups; ++k) {
            const uint32_t r = base + 4 * k + rs;
            rp[k] = make_uint4(0, 0, 0, 0);
            np[k] = rp[k];
            pos[k] = 0;
            live[k] = false;
            if (r < p.n_rows) {  // uniform within the head's 8 lanes
                const uint32_t t = r / p.n_heads;
                const uint32_t h = r - t * p.n_heads;
                const uint16_t* row = q + int64_t(t) * p.sq_t + int64_t(h) * p.sq_h;
                if (kNeox) {
                    const uint2 lo = ld_stream8(row + 4 * m);          // dims 4m .. 4m+3
                    const uint2 hi = ld_stream8(row + 32 + 4 * m);     // dims 32+4m .. 32+4m+3
                    rp[k] = make_uint4(lo.x, lo.y, hi.x, hi.y);
                } else {
                    rp[k] = ld_stream16(row + 8 * m);                  // dims 8m .. 8m+7
                }
                np[k] = ld_stream16(row + 8 * nc);
                pos[k] = __ldg(p.positions + t);
                live[k] = static_cast<uint64_t>(pos[k]) < static_cast<uint64_t>(p.cache_rows);
                if (!live[k] && m == 0 && p.error_flags)
                    atomicOr(p.error_flags, RQ_FLAG_POSITION_RANGE);
            }
        }
#pragma unroll
        for (int k = 0; k < kIdxGroups; ++k) {
            const uint32_t r = base + 4 * k + rs;
            indexer_head<kNeox>(p, rp[k], np[k], pos[k], live[k], m, nc,
                                p.out + int64_t(r) * kIdxDim, p.weights + r, p.weights_out + r);
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
    const int64_t per_warp = 4 * kIdxGroups;
    const int64_t warps = (int64_t(p.n_rows) + per_warp - 1) / per_warp;
    const int64_t need = (warps + kWarps - 1) / kWarps;
    const int64_t cap = int64_t(dev.sm_count) * idx_resident(dev.ordinal, p.neox);
    const int grid = static_cast<int>(need < cap ? need : cap);
    // every head slot on a fixed head when a sweep of the grid (4 heads per
    // warp) can be cut to whole tokens with a whole number of warps
    int64_t tokens = int64_t(grid) * kWarps * 4 / p.n_heads;
    while (tokens > 0 && (tokens * p.n_heads) % 4 != 0) --tokens;
    if (tokens > 0) {
        IdxParams q = p;
        q.sweep_tokens = static_cast<uint32_t>(tokens);
        if (p.neox)
            return launch_pdl(indexer_q_rope_quant_fixed_kernel<true>, grid, kInvThreads, 0, stream, q);
        return launch_pdl(indexer_q_rope_quant_fixed_kernel<false>, grid, kInvThreads, 0, stream, q);
    }
    if (p.neox) return launch_pdl(indexer_q_rope_quant_kernel<true>, grid, kInvThreads, 0, stream, p);
    return launch_pdl(indexer_q_rope_quant_kernel<false>, grid, kInvThreads, 0, stream, p);
}

}  // namespace rq
