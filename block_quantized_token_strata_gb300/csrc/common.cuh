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

// ---- mbarriers and bulk (TMA) copies -----------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0], %1; }" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }"
                 :: "r"(bar), "r"(bytes) : "memory");
}
// One probe of phase `parity`. If the phase is not complete the thread is suspended in hardware
// (issuing nothing) until it completes or about `hint_ns` pass, whichever comes first.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns = 20000) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase `parity`, bounded: gives up (returns false) after `limit_ns` of wall time (two
// seconds unless a caller asks for less), after an iteration cap as a backstop, or as soon as *abort
// becomes non-zero. The caller then flags the error and leaves without touching the data the
// barrier guards.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitIterCap = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < kWaitIterCap; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// The device error word of the bounded waits (bit 0: a wait ran out; higher bits name the wait).
// The library is built without relocatable device code, so every translation unit that includes
// this header holds its own copy; each unit whose kernels set it exports a host reader (internal.h)
// and strata_device_error combines them.
static __device__ int g_strata_device_error = 0;
// orders this thread's generic-proxy shared-memory accesses (writes, and reads of a slot about to
// be refilled) before later async-proxy (bulk copy, TMA, tensor core) accesses of the same bytes
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// global -> shared bulk copy completing on an mbarrier; dst, src 16-byte aligned, bytes % 16 == 0
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
// bulk L2 prefetch of one 16-byte aligned range (size % 16 == 0), a hint
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
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
// Q5K block (codes 0..31, no offset) against one token's 32 activation codes, onto c. w = the Q4-style
// nibble bytes (byte j: low 4 bits of code j, of code j+16 in the high nibble); hb = the fifth bits,
// code k of four-code group g (g = 0..3: codes 4g..4g+3; g = 4..7: codes 16+4(g-4)..) at bit 8k + g,
// so one shift and one mask put a group's four fifth bits at bit 4 of its four bytes.
__device__ __forceinline__ int dot_q5(const uint4 w, uint32_t hb, const uint4 xlo, const uint4 xhi, int c) {
    c = __dp4a(int((w.x & 0x0F0F0F0Fu) | ((hb << 4) & 0x10101010u)), int(xlo.x), c);
    c = __dp4a(int((w.y & 0x0F0F0F0Fu) | ((hb << 3) & 0x10101010u)), int(xlo.y), c);
    c = __dp4a(int((w.z & 0x0F0F0F0Fu) | ((hb << 2) & 0x10101010u)), int(xlo.z), c);
    c = __dp4a(int((w.w & 0x0F0F0F0Fu) | ((hb << 1) & 0x10101010u)), int(xlo.w), c);
    c = __dp4a(int(((w.x >> 4) & 0x0F0F0F0Fu) | (hb & 0x10101010u)), int(xhi.x), c);
    c = __dp4a(int(((w.y >> 4) & 0x0F0F0F0Fu) | ((hb >> 1) & 0x10101010u)), int(xhi.y), c);
    c = __dp4a(int(((w.z >> 4) & 0x0F0F0F0Fu) | ((hb >> 2) & 0x10101010u)), int(xhi.z), c);
    c = __dp4a(int(((w.w >> 4) & 0x0F0F0F0Fu) | ((hb >> 3) & 0x10101010u)), int(xhi.w), c);
    return c;
}
// Q6 block codes as dp4a operands: words 0..3 hold elements 0..15, words 4..7 elements 16..31, one
// 6-bit code q (0..63) per byte. Layout: lo0/lo1 = code bytes 0..15 (byte j: low 4 bits of element j
// in bits 0-3, of element j+16 in bits 4-7), hi = bytes 16..23 (byte 16+i: the high 2 bits of
// elements i, i+8, i+16, i+24 in bits 0-1, 2-3, 4-5, 6-7).
__device__ __forceinline__ void unpack_q6(const uint2 lo0, const uint2 lo1, const uint2 hi, uint32_t (&q)[8]) {
    const uint32_t L[4] = {lo0.x, lo0.y, lo1.x, lo1.y};
    q[0] = (L[0] & 0x0F0F0F0Fu) | ((hi.x & 0x03030303u) << 4);
    q[1] = (L[1] & 0x0F0F0F0Fu) | ((hi.y & 0x03030303u) << 4);
    q[2] = (L[2] & 0x0F0F0F0Fu) | ((hi.x & 0x0C0C0C0Cu) << 2);
    q[3] = (L[3] & 0x0F0F0F0Fu) | ((hi.y & 0x0C0C0C0Cu) << 2);
    q[4] = ((L[0] >> 4) & 0x0F0F0F0Fu) | (hi.x & 0x30303030u);
    q[5] = ((L[1] >> 4) & 0x0F0F0F0Fu) | (hi.y & 0x30303030u);
    q[6] = ((L[2] >> 4) & 0x0F0F0F0Fu) | ((hi.x & 0xC0C0C0C0u) >> 2);
    q[7] = ((L[3] >> 4) & 0x0F0F0F0Fu) | ((hi.y & 0xC0C0C0C0u) >> 2);
}
// 16 codes (4 words) against 16 activation codes, onto c
__device__ __forceinline__ int dot16(const uint32_t* q, const uint4 x, int c) {
    c = __dp4a(int(q[0]), int(x.x), c);
    c = __dp4a(int(q[1]), int(x.y), c);
    c = __dp4a(int(q[2]), int(x.z), c);
    c = __dp4a(int(q[3]), int(x.w), c);
    return c;
}
// ---- packed fp32 pairs (sm_100+): each half is one IEEE fp32 operation, rounded to nearest --------
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack_f2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f2(f32x2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma_f2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 mul_f2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 add_f2(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// exact int -> float for the magic-seeded dot: one fp32 subtraction on the FMA pipe
__device__ __forceinline__ float magic_to_float(int c) { return __fsub_rn(__int_as_float(c), kMagic); }


// ---- per-thread asynchronous copies global -> shared (cp.async), completion by commit groups -----
// 16 bytes, L2 only; src_bytes < 16 zero-fills the rest (0: nothing is read, the 16 bytes are zero)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// 4 bytes; src_bytes 0 writes zero
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of this thread's groups are still pending
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

}  // namespace strata
