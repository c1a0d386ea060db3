// rq_validate.cu -- the debug helper that checks the device-side
// preconditions of the insert and fused ops (and the positions of every op)
// without running them: one non-trapping pass over the tokens, then a host
// readback of the result word.
//
// Slots are checked for range and for reuse. A repeated slot is found with a
// bitmap of num_slots bits in the caller's workspace: each token sets its
// slot's bit with atomicOr, and a bit that was already set marks a second
// writer. That is one pass over the tokens whatever their number.
#include "rq_device.cuh"
#include "rq_launch.h"

namespace rq {

__global__ void __launch_bounds__(256)
validate_indices_kernel(ValParams p) {
    uint32_t found = 0;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < p.n_tokens; t += stride) {
        const int64_t pos = p.positions[t];
        if (pos < 0 || pos >= p.cache_rows) found |= RQ_FLAG_POSITION_RANGE;
        if (p.slot_mapping) {
            const int64_t s = p.slot_mapping[t];
            if (s >= p.num_slots) {
                found |= RQ_FLAG_SLOT_RANGE;
            } else if (s >= 0) {
                const uint32_t bit = 1u << (s & 31);
                if (atomicOr(p.bitmap + (s >> 5), bit) & bit) found |= RQ_FLAG_SLOT_DUPLICATE;
            }
        }
    }
    // one atomic per warp at most
    found = __reduce_or_sync(0xffffffffu, found);
    if ((threadIdx.x & 31) == 0 && found) atomicOr(p.result, found);
}

cudaError_t launch_validate_indices(const ValParams& p, const DeviceInfo& dev,
                                    cudaStream_t stream) {
    const int64_t blocks = (p.n_tokens + 255) / 256;
    const int64_t cap = int64_t(dev.sm_count) * 8;
    validate_indices_kernel<<<int(blocks < cap ? blocks : cap), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace rq
