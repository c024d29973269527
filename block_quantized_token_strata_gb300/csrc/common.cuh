// common.cuh — device helpers shared by the strata kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace strata {

constexpr int kQK = 32;                  // values per quant block
constexpr int kMaxT = 8;                 // tokens per verify window
constexpr int kMagicBits = 0x4B400000;   // bit pattern of 1.5 * 2^23
constexpr float kMagic = 12582912.0f;    // 1.5 * 2^23

// ---- programmatic dependent launch ----------------------------------------------------------
// wait: block until the grid this launch depends on has completed and its writes are visible
// (a no-op when the launch has no programmatic dependency). launch: allow the next kernel on the
// stream, if launched with programmatic serialization, to start its pre-wait prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- loads ------------------------------------------------------------------------------------
// weights are streamed once: read-only path, no L1 allocation
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ unsigned short ld_stream_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Bulk L2 prefetch of [p, p+bytes) (a hint; issued by one thread). The range is trimmed inward
// to 16-byte boundaries, as the instruction requires.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    uintptr_t b = a + bytes;
    a = (a + 15) & ~uintptr_t(15);
    b &= ~uintptr_t(15);
    while (a < b) {
        uint32_t n = (b - a) > (1u << 20) ? (1u << 20) : uint32_t(b - a);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(a), "r"(n) : "memory");
        a += n;
    }
}

// ---- exact block dots ----------------------------------------------------------------------------
// One 32-value block of weight codes against one token's 32 activation codes, accumulated onto
// c by dp4a. The caller seeds c with kMagicBits - 8*s (Q4: codes q in 0..15 stand for q-8, and
// sum_j (q_j-8)*x_j = sum_j q_j*x_j - 8*s) or kMagicBits (Q8), so that the result is the bit
// pattern of the fp32 number 1.5*2^23 + isum: |isum| <= 32*127*127 < 2^22 keeps it exact.
// Activation layout: xlo = codes 0..15, xhi = codes 16..31 (four per 32-bit word, in order).
// Q4 weight layout: byte j holds code j (low nibble) and code j+16 (high nibble).
__device__ __forceinline__ int dot_q4(const uint4 w, const uint4 xlo, const uint4 xhi, int c) {
    c = __dp4a(int(w.x & 0x0F0F0F0Fu), int(xlo.x), c);
    c = __dp4a(int(w.y & 0x0F0F0F0Fu), int(xlo.y), c);
    c = __dp4a(int(w.z & 0x0F0F0F0Fu), int(xlo.z), c);
    c = __dp4a(int(w.w & 0x0F0F0F0Fu), int(xlo.w), c);
    c = __dp4a(int((w.x >> 4) & 0x0F0F0F0Fu), int(xhi.x), c);
    c = __dp4a(int((w.y >> 4) & 0x0F0F0F0Fu), int(xhi.y), c);
    c = __dp4a(int((w.z >> 4) & 0x0F0F0F0Fu), int(xhi.z), c);
    c = __dp4a(int((w.w >> 4) & 0x0F0F0F0Fu), int(xhi.w), c);
    return c;
}
__device__ __forceinline__ int dot_q8(const uint4 w0, const uint4 w1, const uint4 xlo, const uint4 xhi, int c) {
    c = __dp4a(int(w0.x), int(xlo.x), c);
    c = __dp4a(int(w0.y), int(xlo.y), c);
    c = __dp4a(int(w0.z), int(xlo.z), c);
    c = __dp4a(int(w0.w), int(xlo.w), c);
    c = __dp4a(int(w1.x), int(xhi.x), c);
    c = __dp4a(int(w1.y), int(xhi.y), c);
    c = __dp4a(int(w1.z), int(xhi.z), c);
    c = __dp4a(int(w1.w), int(xhi.w), c);
    return c;
}
// exact int -> float for the magic-seeded dot: one fp32 subtraction on the FMA pipe
__device__ __forceinline__ float magic_to_float(int c) { return __fsub_rn(__int_as_float(c), kMagic); }

}  // namespace strata
