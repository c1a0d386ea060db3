// rq_umma.cuh -- 5th-generation tensor core (tcgen05) and tensor-map TMA
// primitives for sm_103a, as inline PTX, plus the two descriptors the MMA
// takes. Used by the grouped FP8 GEMM (rq_gemm.cu).
//
// Shared-memory matrix descriptor (64 bits) for an operand tile stored
// K-major with the 128-byte swizzle (each row of the tile is 128 bytes of K;
// 8-row groups of 1024 bytes; inside a group the 16-byte chunk c of row r sits
// at chunk position c ^ (r % 8), which is what a TMA load with
// CU_TENSOR_MAP_SWIZZLE_128B writes into a 1024-byte aligned buffer):
//   bits  0..13  start address >> 4
//   bits 16..29  leading-dimension byte offset >> 4 (unused for this layout: 1)
//   bits 32..45  stride byte offset >> 4 (distance between 8-row groups: 1024)
//   bits 46..47  descriptor version (1)
//   bits 49..51  base offset (0: the buffer is 1024-byte aligned)
//   bit  52      leading-dimension offset mode (0)
//   bits 61..63  layout: 2 = 128-byte swizzle
// Instruction descriptor (32 bits) of kind::f8f6f4:
//   bits 4..5 D format (1 = f32), 7..9 A format (0 = e4m3), 10..12 B format
//   (0 = e4m3), 15 / 16 A / B major (0 = K-major), 17..22 N >> 3,
//   24..28 M >> 4; all other bits 0 (dense, no negation, no saturation).
// Instruction descriptor of kind::mxf8f6f4 (block-scaled, D always f32):
//   bits 4..5 B scale-factor byte, 7..9 / 10..12 A / B format (0 = e4m3),
//   17..22 N >> 3, 23 scale format (1 = UE8M0), 24..28 M >> 4, 29..30 A
//   scale-factor byte.
// Scale factors in tensor memory (scale_vec::1X: one UE8M0 code per row and
// 32-wide K step): a 32-bit TMEM cell holds four codes and the descriptor's
// scale-factor byte picks one. For 128 rows (of A, or a 128-row slice of B)
// the codes sit in 4 consecutive columns: column c, byte b, in every lane
// quadrant at lane 32q + i, holds the code of row i + 32c. That is what
// tcgen05.cp .32x128b.warpx4 writes from a 512-byte shared-memory atom whose
// 16-byte row i holds words (row i, i+32, i+64, i+96); B rows 128..255 use
// the next 4 columns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rq {
namespace umma {

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_byte_addr) {
    uint64_t d = 0;
    d |= uint64_t((smem_byte_addr >> 4) & 0x3fffu);
    d |= uint64_t(1u) << 16;                 // leading byte offset (unused) = 16 B
    d |= uint64_t(1024u >> 4) << 32;         // stride byte offset = 1024 B
    d |= uint64_t(1u) << 46;                 // version
    d |= uint64_t(2u) << 61;                 // 128-byte swizzle
    return d;
}

__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

__host__ __device__ constexpr uint32_t idesc_mx_e4m3_ue8m0(int m, int n, uint32_t sf_byte) {
    return (sf_byte << 4) | (uint32_t(n >> 3) << 17) | (1u << 23) | (uint32_t(m >> 4) << 24) |
           (sf_byte << 29);
}

// Shared-memory descriptor of an unswizzled K-major operand made of 8-row x
// 16-byte core matrices stored one after the other (rows 16 bytes apart):
// stride byte offset 128, leading byte offset unused, layout 0 = no swizzle.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t smem_byte_addr) {
    uint64_t d = 0;
    d |= uint64_t((smem_byte_addr >> 4) & 0x3fffu);
    d |= uint64_t(128u >> 4) << 32;
    d |= uint64_t(1u) << 46;
    return d;
}

// TMEM allocation: one full warp executes these.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T; accumulate when `acc` != 0.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Block-scaled D[tmem] (+)= (A * 2^sfa) * (B * 2^sfb)^T, e4m3 operands, UE8M0
// scale factors read from TMEM columns sfa_tmem / sfb_tmem (byte chosen by
// the instruction descriptor).
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                             uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(acc)
        : "memory");
}

// Copy a 512-byte shared-memory atom (32 rows x 16 bytes) into 4 TMEM columns
// of all four lane quadrants (lane 32q + i, column c = bytes 4c..4c+3 of row
// i). Ordered with this thread's later tcgen05.mma; completion is tracked by
// tcgen05.commit like an MMA.
__device__ __forceinline__ void cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread
// issued so far has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31; the address carries the lane in bits 16..31).
// The load and its tcgen05.wait::ld are one asm statement, so the compiler
// cannot schedule a use of the registers before the wait that makes them
// valid.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 2-D tensor-map TMA load of one box into this CTA's shared memory,
// completing on mbarrier `bar`. x is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster; orders the shared-memory writes
// before it (release) with the reads of any CTA of the cluster after it
// (acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// The address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}

// Hint: bring one box of a 2-D tensor map into L2. It returns no data, so it
// may run before griddepcontrol.wait: the copies that read the box later see
// whatever the previous kernel wrote (L2 is the point of coherence).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// 3-D tensor-map TMA load (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

}  // namespace umma
}  // namespace rq
