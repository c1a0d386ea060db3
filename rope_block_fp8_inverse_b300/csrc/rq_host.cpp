// rq_host.cpp -- the inverse op over host buffers: a chunked copy-in /
// kernel / copy-out pipeline on the caller's stream plus two copy streams.
//
// Chunk c of the tokens goes through workspace slot c % 3:
//   copy-in stream   waits until slot c % 3 is free (copy-out of chunk c - 3
//                    done), copies x and positions host -> device
//   caller's stream  waits for that copy, runs the op's kernels on the slot
//   copy-out stream  waits for the kernels, copies codes and scales device ->
//                    host
// so at any time one chunk is coming in, one is being processed and one is
// going out; host -> device and device -> host copies use the two directions
// of the link at once. The copy streams first wait for everything enqueued on
// the caller's stream before the call, and the caller's stream finally waits
// for the last copy-out, so the call is ordered on `stream` like any other
// and its host outputs are complete once `stream` is.
//
// The streams and events are created once per device and reused; a mutex per
// device keeps calls from different host threads from interleaving their
// enqueues on them. No memory is allocated: the slots live in the caller's
// workspace.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "rq.h"

#define RQ_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kSlots = 3;
constexpr int kMaxDevices = 64;
constexpr int64_t kHeadDim = 512;

int64_t align256(int64_t b) { return (b + 255) & ~int64_t(255); }

// Byte sizes of one slot's four buffers for chunk_tokens tokens of n_heads heads.
struct SlotLayout {
    int64_t x, pos, codes, scales, total;
    SlotLayout(int64_t n_heads, int64_t chunk_tokens) {
        x = align256(chunk_tokens * n_heads * kHeadDim * 2);
        pos = align256(chunk_tokens * 8);
        codes = align256(chunk_tokens * n_heads * kHeadDim);
        scales = align256(chunk_tokens * n_heads * 16);
        total = x + pos + codes + scales;
    }
};

struct Pipeline {
    std::mutex mu;
    bool ready = false;
    cudaStream_t cin = nullptr, cout = nullptr;
    cudaEvent_t entry = nullptr, in[kSlots] = {}, done[kSlots] = {}, out[kSlots] = {};

    cudaError_t init() {
        if (ready) return cudaSuccess;
        cudaError_t e = cudaStreamCreateWithFlags(&cin, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&cout, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&entry, cudaEventDisableTiming);
        for (int s = 0; s < kSlots && e == cudaSuccess; ++s) {
            e = cudaEventCreateWithFlags(&in[s], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&done[s], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&out[s], cudaEventDisableTiming);
        }
        ready = e == cudaSuccess;
        return e;
    }
};

Pipeline g_pipes[kMaxDevices];

rq_status status_of(cudaError_t e) {
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

RQ_EXPORT int64_t rq_inv_rope_fp8_quant_host_workspace(int64_t n_heads, int64_t chunk_tokens) {
    if (n_heads < 1 || chunk_tokens < 1 || n_heads > (int64_t(1) << 20) ||
        chunk_tokens > (int64_t(1) << 31) / n_heads)
        return -1;
    return kSlots * SlotLayout(n_heads, chunk_tokens).total;
}

RQ_EXPORT rq_status rq_inv_rope_fp8_quant_host(
    const void* x_bf16_host, int64_t n_tokens, int64_t n_heads, const int64_t* positions_host,
    const float* cos_sin_cache, int64_t cache_rows, int64_t heads_per_group, float eps,
    uint8_t* out_fp8_host, float* out_scales_host, void* workspace, int64_t workspace_bytes,
    int64_t chunk_tokens, uint32_t* error_flags, void* stream) {
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1 || chunk_tokens < 1) return RQ_ERR_SHAPE;
    if (heads_per_group < 1 || n_heads % heads_per_group != 0) return RQ_ERR_GROUPING;
    const int64_t need = rq_inv_rope_fp8_quant_host_workspace(n_heads, chunk_tokens);
    if (need < 0 || n_tokens >= (int64_t(1) << 31) / n_heads) return RQ_ERR_SHAPE;
    if (n_tokens == 0) return RQ_OK;
    if (!x_bf16_host || !positions_host || !cos_sin_cache || !out_fp8_host || !out_scales_host ||
        !workspace)
        return RQ_ERR_NULL;
    if (workspace_bytes < need) return RQ_ERR_SHAPE;
    if (!aligned(workspace, 256)) return RQ_ERR_ALIGN;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return RQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RQ_ERR_ARG;
    Pipeline& pl = g_pipes[dev];
    std::lock_guard<std::mutex> lock(pl.mu);
    if ((e = pl.init()) != cudaSuccess) return RQ_ERR_CUDA;

    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const SlotLayout lay(n_heads, chunk_tokens);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* xh = static_cast<const uint8_t*>(x_bf16_host);
    const int64_t x_row = n_heads * kHeadDim * 2, code_row = n_heads * kHeadDim,
                  scale_row = n_heads * 16;

    if ((e = cudaEventRecord(pl.entry, st)) != cudaSuccess) return RQ_ERR_CUDA;
    if ((e = cudaStreamWaitEvent(pl.cin, pl.entry, 0)) != cudaSuccess) return RQ_ERR_CUDA;
    if ((e = cudaStreamWaitEvent(pl.cout, pl.entry, 0)) != cudaSuccess) return RQ_ERR_CUDA;

    int64_t c = 0;
    for (int64_t t0 = 0; t0 < n_tokens; t0 += chunk_tokens, ++c) {
        const int s = static_cast<int>(c % kSlots);
        const int64_t nt = (n_tokens - t0) < chunk_tokens ? (n_tokens - t0) : chunk_tokens;
        uint8_t* base = ws + s * lay.total;
        uint8_t* dx = base;
        int64_t* dpos = reinterpret_cast<int64_t*>(base + lay.x);
        uint8_t* dcodes = base + lay.x + lay.pos;
        float* dscales = reinterpret_cast<float*>(base + lay.x + lay.pos + lay.codes);
        // copy in, once the slot's previous chunk has left
        if (c >= kSlots && (e = cudaStreamWaitEvent(pl.cin, pl.out[s], 0)) != cudaSuccess)
            return RQ_ERR_CUDA;
        if ((e = cudaMemcpyAsync(dx, xh + t0 * x_row, nt * x_row, cudaMemcpyHostToDevice,
                                 pl.cin)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dpos, positions_host + t0, nt * 8, cudaMemcpyHostToDevice,
                                 pl.cin)) != cudaSuccess ||
            (e = cudaEventRecord(pl.in[s], pl.cin)) != cudaSuccess)
            return RQ_ERR_CUDA;
        // the op on the caller's stream
        if ((e = cudaStreamWaitEvent(st, pl.in[s], 0)) != cudaSuccess) return RQ_ERR_CUDA;
        const rq_status rs = rq_inv_rope_fp8_quant(dx, nt, n_heads, n_heads * kHeadDim, kHeadDim,
                                                   dpos, cos_sin_cache, cache_rows,
                                                   heads_per_group, eps, dcodes, dscales,
                                                   error_flags, stream);
        if (rs != RQ_OK) return rs;
        if ((e = cudaEventRecord(pl.done[s], st)) != cudaSuccess) return RQ_ERR_CUDA;
        // copy out
        if ((e = cudaStreamWaitEvent(pl.cout, pl.done[s], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(out_fp8_host + t0 * code_row, dcodes, nt * code_row,
                                 cudaMemcpyDeviceToHost, pl.cout)) != cudaSuccess ||
            (e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(out_scales_host) + t0 * scale_row,
                                 dscales, nt * scale_row, cudaMemcpyDeviceToHost, pl.cout)) !=
                cudaSuccess ||
            (e = cudaEventRecord(pl.out[s], pl.cout)) != cudaSuccess)
            return RQ_ERR_CUDA;
    }
    // the caller's stream continues after the last copy-out (the copy-out
    // stream is in order, so that covers every chunk)
    const int last = static_cast<int>((c - 1) % kSlots);
    return status_of(cudaStreamWaitEvent(st, pl.out[last], 0));
}
