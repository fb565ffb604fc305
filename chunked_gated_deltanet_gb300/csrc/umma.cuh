// tcgen05 (5th-generation tensor core) helpers: TMEM allocation, shared-memory
// matrix descriptors for the no-swizzle operand layouts, MMA issue and commit,
// and TMEM loads.
//
// No-swizzle operand layouts. A core matrix is 8 rows x 16 bytes, stored as
// 128 contiguous bytes (row by row).
//   K-major (rows along M/N, the 16 bytes along K): element (r, k) of a bf16
//   operand sits at (r/8)*SBO + (k/8)*LBO + (r%8)*16 + (k%8)*2 bytes.
//   MN-major (rows along K, the 16 bytes along M/N): element (n, k) sits at
//   (n/8)*SBO + (k/8)*LBO + (k%8)*16 + (n%8)*2 bytes.
// In both, the descriptor's leading byte offset (LBO) steps between core
// matrices adjacent along K and the stride byte offset (SBO) between core
// matrices adjacent along M/N (checked on the device for either major-ness).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>
#include "mma.cuh"

namespace gdn {

// byte offset of element (r, k) of a bf16 K-major operand
__host__ __device__ constexpr uint32_t kmajor_bf16_offset(int r, int k, uint32_t lbo, uint32_t sbo) {
    return (uint32_t)(r >> 3) * sbo + (uint32_t)(k >> 3) * lbo + (uint32_t)(r & 7) * 16u + (uint32_t)(k & 7) * 2u;
}
// byte offset of element (n, k) of a bf16 MN-major operand
__host__ __device__ constexpr uint32_t mnmajor_bf16_offset(int n, int k, uint32_t lbo, uint32_t sbo) {
    return (uint32_t)(n >> 3) * sbo + (uint32_t)(k >> 3) * lbo + (uint32_t)(k & 7) * 16u + (uint32_t)(n & 7) * 2u;
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t umma_smem_desc(const void *p, uint32_t lbo, uint32_t sbo) {
    const uint64_t a = smem_addr(p);
    return ((a >> 4) & 0x3FFFull) | (((uint64_t)(lbo >> 4) & 0x3FFFull) << 16) |
           (((uint64_t)(sbo >> 4) & 0x3FFFull) << 32) | (1ull << 46);
}

// Instruction descriptor, fp32 accumulator: kind::f16 with bf16 A and B;
// a_mn / b_mn select the MN-major layout for that operand (else K-major).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, fp32 accumulator: kind::f16 with fp16 A and B (formats 0); a_mn / b_mn as above.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// 2-D tensor copy of one box, global -> this CTA's shared memory, completing on an mbarrier.
// x (innermost, elements) must start on a 16-byte boundary; rows outside the tensor read as zero.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Prefetch of one box of a 2-D tensor into L2 (no shared memory, no completion to wait for); parts outside
// the tensor are skipped. x as for tma_load_2d.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];\n" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Prefetch of [a, a + bytes) into L2 (a and bytes multiples of 16; no completion to wait for).
__device__ __forceinline__ void bulk_prefetch_l2(const void *a, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(a), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// D[tmem] (+)= A * B for one K-step of 16 16-bit elements (bf16 or fp16, as the instruction descriptor says),
// issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier once all previously issued MMAs of this thread have completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_addr(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (lane = thread's lane);
// the values are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
// The same wait, tied to the registers of the load it completes so that no use of them moves above it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// 8 fp16 (one 16-byte core-matrix row) -> fp32
__device__ __forceinline__ void h8_to_f(uint4 u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
// two fp32 -> an fp16 pair (round to nearest even), a in the low half
__device__ __forceinline__ uint32_t f2_to_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}
// 8 fp32 -> one 16-byte row of fp16
__device__ __forceinline__ uint4 f8_to_h8(const float *v) {
    return make_uint4(f2_to_h2(v[0], v[1]), f2_to_h2(v[2], v[3]), f2_to_h2(v[4], v[5]), f2_to_h2(v[6], v[7]));
}

// Packed fp32 pairs (sm_100 and later): each lane rounds as the scalar instruction does, so a pair of
// scalar add / mul / fma chains and its packed form give the same bits.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &a, float &b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r)); }
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld16_nowait(taddr, r);
    tmem_wait_ld(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace gdn
