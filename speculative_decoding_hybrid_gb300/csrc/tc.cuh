// tcgen05 (5th-generation tensor core) helpers for sm_103a: tensor-memory
// allocation, shared-memory matrix descriptors for 128-byte-swizzled K-major
// tiles, single-CTA MMA issue (kind::f16 with bf16 operands, kind::tf32) with
// fp32 accumulation, completion through an mbarrier, and tensor-memory loads.
//
// Tile convention used throughout: a K-major operand tile of R rows stores,
// for every 128-byte slice of K ("atom": 64 bf16 or 32 tf32 elements), R rows
// of 128 bytes; the 16-byte chunks of row r are permuted by (chunk ^ (r & 7))
// -- the 128-byte swizzle -- and 8-row groups are 1024 bytes apart.  Tiles
// start on 1024-byte boundaries.  One MMA consumes 32 bytes of K (16 bf16 or
// 8 tf32 elements), so K steps inside an atom advance the start by 32 bytes.
#pragma once

#include "common.cuh"

namespace tc {

// Byte offset of bf16 element (r, k) inside a swizzled K-major tile of R rows.
__device__ __forceinline__ uint32_t swz_off(int R, int r, int k) {
    const int atom = k >> 6;
    const int kin = k & 63;
    const int chunk = kin >> 3;
    return uint32_t(atom) * uint32_t(R) * 128u + uint32_t(r) * 128u + (uint32_t(chunk ^ (r & 7)) << 4) +
           (uint32_t(kin & 7) << 1);
}

// Byte offset of fp32/tf32 element (r, k) inside a swizzled K-major tile of R
// rows: an atom is 32 elements (128 bytes) of K.
__device__ __forceinline__ uint32_t swz_off_f32(int R, int r, int k) {
    const int atom = k >> 5;
    const int kin = k & 31;
    const int chunk = kin >> 2;
    return uint32_t(atom) * uint32_t(R) * 128u + uint32_t(r) * 128u + (uint32_t(chunk ^ (r & 7)) << 4) +
           (uint32_t(kin & 3) << 2);
}

// Round an fp32 value to tf32 (10 explicit mantissa bits, nearest, ties away),
// so that the tensor core consumes it without a further truncation.
__device__ __forceinline__ float round_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Shared-memory matrix descriptor: start address, leading byte offset 16 B
// (unused for swizzled K-major), stride byte offset 1024 B (8-row groups),
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3fffu);
    d |= uint64_t(1u) << 16;
    d |= uint64_t(1024u >> 4) << 32;
    d |= uint64_t(1u) << 46;
    d |= uint64_t(2u) << 61;
    return d;
}

// Descriptor of the tile `off` bytes after the one `base` describes (off a
// multiple of 16, the start address staying below 256 KB): only the start
// field changes.
__device__ __forceinline__ uint64_t desc_at(uint64_t base, uint32_t off) { return base + (off >> 4); }

// Descriptor of an MN-major 128-byte-swizzled tile (used for B): K rows of
// 64 MN elements (128 B) swizzled like a K-major tile, 8-row K groups 1024 B
// apart, and consecutive 64-element MN blocks `lbo` bytes apart.  One MMA's
// 16 K rows span two K groups, so K steps advance the start by 2048 bytes.
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3fffu);
    d |= uint64_t((lbo >> 4) & 0x3fffu) << 16;
    d |= uint64_t(1024u >> 4) << 32;
    d |= uint64_t(1u) << 46;
    d |= uint64_t(2u) << 61;
    return d;
}

// Instruction-descriptor bit that marks B as MN-major.
constexpr uint32_t kBMnMajor = 1u << 16;

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | (uint32_t(N >> 3) << 17)      // N / 8
           | (uint32_t(M >> 4) << 24);     // M / 16
}

// Instruction descriptor for kind::tf32 with tf32 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4)                       // D format: f32
           | (2u << 7)                     // A format: tf32
           | (2u << 10)                    // B format: tf32
           | (uint32_t(N >> 3) << 17)      // N / 8
           | (uint32_t(M >> 4) << 24);     // M / 16
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction-descriptor bits: A stored MN-major (transposed), and A negated
// (D += -(A B)).
constexpr uint32_t kAMnMajor = 1u << 15;
constexpr uint32_t kNegA = 1u << 13;

// kind::f16 MMA whose A operand lives in tensor memory: row m of A in lane m,
// K elements packed two per 32-bit column (element 2j in the low half), one
// MMA reading K = 16 elements from 8 consecutive columns starting at a_tmem.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier once every MMA issued so far by this thread is done.
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     gdn::smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// Warp-wide: allocate ncols tensor-memory columns; the base address lands in *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(gdn::smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns, without waiting: the registers
// are valid after ld_wait().  Several loads may be in flight together.
__device__ __forceinline__ void ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// After ld_wait(): ties the loaded registers to a point after the wait, so
// that no use of them is scheduled before it.
__device__ __forceinline__ void ld_fence_regs(uint32_t (&r)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp receives
// row (lane base + i), columns col .. col+15.
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 bits, 8 consecutive columns from registers: thread i of the
// warp writes lane (lane base + i), columns col .. col+7; then wait for the
// stores to be done.
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace tc
