// tc.cuh — fifth-generation tensor core (tcgen05) helpers for sm_100-family GPUs (sm_103a):
// tensor-memory (TMEM) allocation, shared-memory matrix descriptors, MMA issue and commit, and
// TMEM loads. Written from the PTX ISA description of the tcgen05 instructions.
#pragma once
#include <stdint.h>

namespace strata {

// ---- TMEM allocation (one warp, all lanes) -------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// ---- ordering of tcgen05 operations around thread synchronisation -------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- shared-memory matrix descriptor, no swizzle --------------------------------------------------
// Operands are K-major "core matrices" of 8 rows x 16 bytes (8 rows of 8 fp16), each 128 contiguous
// bytes. lbo = byte distance between core matrices adjacent along K, sbo = between core matrices
// adjacent along M (or N), i.e. between groups of 8 rows.
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;  // descriptor version of the sm_100 family
    return d;               // base offset 0, layout type 0 (no swizzle)
}

// Instruction descriptor of kind::f16 with fp16 A and B, fp32 accumulation, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4)                            // accumulator format: F32
         | (0u << 7) | (0u << 10)               // A, B format: F16
         | (uint32_t(N >> 3) << 17)             // N / 8
         | (uint32_t(M >> 4) << 24);            // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread; accumulate = 0 overwrites D.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; "
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// the mbarrier receives one arrival when every tcgen05 operation this thread issued so far is done
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(mbar) : "memory");
}

// ---- TMEM -> registers: 32 lanes x 16 consecutive 32-bit columns ---------------------------------
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                   "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                   "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr));
}
// The registers a tcgen05.ld writes are valid only after tcgen05.wait::ld, yet the compiler sees them
// as defined by the load itself and may schedule arithmetic that reads them ahead of a wait that names
// no registers. So the wait takes the loaded registers as read-write operands: every use stays below
// it. Two 16-column loads go out back to back and one wait covers both.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[2][16]) {
    tmem_ld16(taddr, v[0]);
    tmem_ld16(taddr + 16, v[1]);
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0][0]),"+r"(v[0][1]),"+r"(v[0][2]),"+r"(v[0][3]),"+r"(v[0][4]),"+r"(v[0][5]),"+r"(v[0][6]),"+r"(v[0][7]),
                   "+r"(v[0][8]),"+r"(v[0][9]),"+r"(v[0][10]),"+r"(v[0][11]),"+r"(v[0][12]),"+r"(v[0][13]),"+r"(v[0][14]),"+r"(v[0][15]),
                   "+r"(v[1][0]),"+r"(v[1][1]),"+r"(v[1][2]),"+r"(v[1][3]),"+r"(v[1][4]),"+r"(v[1][5]),"+r"(v[1][6]),"+r"(v[1][7]),
                   "+r"(v[1][8]),"+r"(v[1][9]),"+r"(v[1][10]),"+r"(v[1][11]),"+r"(v[1][12]),"+r"(v[1][13]),"+r"(v[1][14]),"+r"(v[1][15])
                 :: "memory");
}

// ---- exact small integers as fp16 pairs ----------------------------------------------------------
// Bytes b0, b1 of `bytes` (selected by `sel`) become the fp16 pair (1024 + b0, 1024 + b1): the
// high byte 0x64 makes 1024 + b for 0 <= b < 1024 exactly.
__device__ __forceinline__ uint32_t bytes_to_h2(uint32_t bytes, uint32_t sel) {
    return __byte_perm(bytes, 0x64646464u, sel);
}
__device__ __forceinline__ uint32_t h2_add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

}  // namespace strata
