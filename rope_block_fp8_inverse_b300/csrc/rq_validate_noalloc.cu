// rq_validate_noalloc.cu -- rq_validate_indices without a caller workspace.
//
// Some callers cannot hand the index check a device buffer: a plain C or C++
// host program that links only this library and has no device allocator of
// its own, or a serving engine that has given every free byte of the GPU to
// its KV cache and must not allocate in the middle of a step (an allocation
// there can fail, or stall the stream while memory is reclaimed). For them
// this entry point keeps its scratch -- the slot bitmap and the result word --
// in a file-scope device array of fixed size, which every GPU that loads the
// library holds from load until the process exits. It allocates nothing.
//
// The array is shared by every call on a device and keeps the previous call's
// bits, so each call clears the part it uses before the check. Two calls
// whose work overlaps on the GPU (two streams, or two host threads) race on
// it; the call synchronises its stream before returning, so calls made one
// after another from one host thread never overlap.
#include <mutex>

#include "rq_launch.h"

#define RQ_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// Slots the bitmap can cover: 2^20 (128 KiB of bits), then the result word.
constexpr int64_t kNoallocMaxSlots = int64_t(1) << 20;
constexpr int64_t kBitmapBytes = kNoallocMaxSlots / 8;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_validate_scratch[kBitmapBytes + 256];

// Device address of the array, looked up once per device (host code cannot
// use the array's name as a device pointer). The address stays valid for the
// life of the device's primary context: after a cudaDeviceReset (which
// destroys that context and the module's copy of the array) this entry point
// must not be called again in the same process.
uint8_t* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_for_device(int device, uint8_t** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[device]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_validate_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[device] = static_cast<uint8_t*>(ptr);
    }
    *out = g_scratch_addr[device];
    return cudaSuccess;
}

bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// A CUDA failure as the other entry points report it: clear this runtime's
// sticky launch error, return RQ_ERR_CUDA.
rq_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return RQ_OK;
    (void)cudaGetLastError();
    return RQ_ERR_CUDA;
}

}  // namespace

RQ_EXPORT rq_status rq_validate_indices_noalloc(const int64_t* positions,
                                                const int64_t* slot_mapping, int64_t n_tokens,
                                                int64_t cache_rows, int64_t num_slots,
                                                uint32_t* result, void* stream) {
    if (n_tokens < 0 || cache_rows < 1 || num_slots < 0 || (slot_mapping && num_slots < 1))
        return RQ_ERR_SHAPE;
    if (slot_mapping && num_slots > kNoallocMaxSlots) return RQ_ERR_SHAPE;  // beyond the array
    if (!result) return RQ_ERR_NULL;
    if (n_tokens == 0) {
        *result = 0;
        return RQ_OK;
    }
    if (!positions) return RQ_ERR_NULL;
    if (!aligned8(positions) || (slot_mapping && !aligned8(slot_mapping))) return RQ_ERR_ALIGN;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return RQ_ERR_ARG;
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_status(e);
    uint8_t* scratch = nullptr;
    if ((e = scratch_for_device(dev, &scratch)) != cudaSuccess) return cuda_status(e);

    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t bitmap = slot_mapping ? ((num_slots + 31) / 32) * 4 : 0;
    rq::ValParams p;
    p.positions = positions;
    p.slot_mapping = slot_mapping;
    p.n_tokens = n_tokens;
    p.cache_rows = cache_rows;
    p.num_slots = num_slots;
    p.bitmap = reinterpret_cast<uint32_t*>(scratch);
    p.result = reinterpret_cast<uint32_t*>(scratch + kBitmapBytes);
    rq::DeviceInfo info;
    info.ordinal = dev;
    info.sm_count = sms;
    uint32_t word = 0;
    // clear the bits this call reads and the result word, then check
    if ((bitmap && (e = cudaMemsetAsync(scratch, 0, size_t(bitmap), st)) != cudaSuccess) ||
        (e = cudaMemsetAsync(p.result, 0, 4, st)) != cudaSuccess ||
        (e = rq::launch_validate_indices(p, info, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(&word, p.result, 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaStreamSynchronize(st)) != cudaSuccess)
        return cuda_status(e);
    *result = word;
    return RQ_OK;
}
